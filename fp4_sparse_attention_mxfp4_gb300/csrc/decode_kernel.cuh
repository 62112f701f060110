// Decode: every cached key of each sequence scored against the sequence's query row(s) on tcgen05
// block-scaled MXFP4 MMA, head-weighted ReLU reduction, and the exact top-k, in one persistent,
// cooperative kernel.
//
// Method ("Score a DSA sparse indexer in FP4", squashed commit message and PR body):
//   logit[q, t] = sum_h w[q, h] * relu(q_h . k_t), keys read in place from the paged two-plane FP4
//   index region; a row's top-k is bounded by its context. With next_n verify rows per sequence
//   (speculative decoding; on the pages the draft folds its batch x next_n verify rows back onto the
//   batch's sequences and rebuilds the schedule for them), row j of a sequence sees keys
//   [0, ctx - next_n + 1 + j) and all rows share one pass over the keys.
//
// GB300 design (the pages' kernels target MI355X MFMA; this is a fresh design):
//   * Stream. CTA c takes the tile range the schedule gives it (at most cap_tiles(next_n) tiles of
//     128 keys). Twelve stage warps each own one stage of a 12-stage ring: a warp issues its tile's
//     eight 1 KB group-chunk bulk copies (cp.async.bulk; a page's chunk g lands at g * 2048 +
//     page * 1024, the canonical no-swizzle K-major operand), loads the two pages' scale words,
//     rebuilds them in the tensor core's scale layout, and issues the tile's two tcgen05.mma
//     kind::mxf4 block_scale MMAs (M = 128 keys, N = next_n * H query heads, K = 64 each) into one
//     of several TMEM accumulators. Three epilogue groups of four warps (one per TMEM lane quarter)
//     read the accumulators with tcgen05.ld, form each key's logits in a fixed order and store their
//     order-preserving 32-bit images in a shared-memory row buffer. Nothing else happens in the
//     stream, so the bulk copies run at the rate of the memory system.
//   * Select. Then every warp of the CTA works on the row buffer. A sequence whose keys all sit in
//     this CTA is selected here (radix passes over the buffer). The units of a longer sequence
//     publish the non-empty bins of their 12-bit key histograms (only bins at or above their own
//     k-th key's bin), wait until every unit of the sequence has published, and each finds the
//     sequence's threshold bin from the published counts. Each then writes only its keys at or
//     above that bin (about k plus one bin's worth over the whole sequence, instead of k per unit)
//     at its offset in the sequence's candidate array, and takes a ticket; the last unit to finish
//     resolves the exact threshold inside the bin and writes the top-k in token order. The logits
//     never reach global memory (unless a debug buffer is passed).
//   * The grid is the SM count, launched cooperatively so that every CTA is resident while units
//     wait on each other's histograms; every wait is bounded and reports a timeout in the status
//     word instead of hanging.
#pragma once
#include <cuda_runtime.h>

#include <cstdint>

#include "block.cuh"
#include "common.cuh"
#include "decode_sched.cuh"
#include "ptx.cuh"

namespace idxfp4 {

// Arguments of one decode call (device pointers owned by the caller).
struct DecodeParams {
  const uint8_t* q_packed;
  const uint8_t* q_scale;
  const float* weights;
  const uint8_t* kv_packed;
  const uint8_t* kv_scale;
  int64_t num_pages;
  const int32_t* block_tables;
  int bt_stride;
  const int32_t* ctx_lens;
  const void* sched;
  size_t sched_bytes;
  int batch;
  int topk;
  void* workspace;
  size_t ws_bytes;
  int32_t* topk_idx;
  float* topk_val;
  float* logits_debug;
  int64_t logits_stride;
  int32_t* status;
};

namespace {

constexpr uint32_t kEpiBarrier = 1;    // the epilogue warps, during the stream
constexpr uint32_t kSelBarrier0 = 2;   // selection group 0 (the stage warps), during the selection
constexpr uint32_t kSelBarrier1 = 3;   // selection group 1 (the epilogue warps), during the selection
constexpr uint32_t kAllBarrier = 4;    // every warp of the CTA
constexpr int kDecodeMaxCtas = 256;    // the decode grid: at most this many CTAs (so a segment holds at most
                                       // this many units)

template <int H, int Q>
struct DecodeCfg {
  static constexpr int N = H * Q;
  static_assert(N % 16 == 0 && N <= 128, "MMA N dimension: next_n * heads, a multiple of 16 up to 128");
  static constexpr int GROUPS = 3;                 // epilogue groups (tiles t with t % GROUPS == g)
  // One query row: 12 tiles in flight and 6 accumulators when N <= 64. Several rows: 9 tiles in
  // flight and 3 accumulators, so that a range of 128 tiles (next_n 2) or 64 (next_n 4) has room for
  // its logits; the stream is then bound by the epilogue's N columns per key, not by the copies.
  static constexpr int ACC = N <= 64 && Q == 1 ? 6 : 3;  // TMEM accumulators
  static constexpr int STAGES = Q == 1 ? 12 : 9;         // tiles in flight; stage warp s streams stage s
  static constexpr int STAGE_WARPS = 12;                 // the stage role (warps past STAGES only select)
  static constexpr int EPI_WARP0 = STAGE_WARPS;
  static constexpr int EPI_WARPS = 4 * GROUPS;
  static constexpr int EPI_THREADS = EPI_WARPS * 32;
  static constexpr int THREADS = (STAGE_WARPS + EPI_WARPS) * 32;
  // Registers: the launch gives 65536 / THREADS each; during the stream the stage warpgroups give
  // some back and the epilogue warpgroups take them (a tile's 64 accumulator columns in flight).
  static constexpr uint32_t LAUNCH_REGS = (65536u / static_cast<uint32_t>(THREADS)) / 8u * 8u;
  static constexpr uint32_t STAGE_REGS = 56u;
  static constexpr uint32_t EPI_REGS =
      (LAUNCH_REGS * (STAGE_WARPS + EPI_WARPS) - STAGE_REGS * STAGE_WARPS) / EPI_WARPS / 8u * 8u;
  static_assert(STAGE_WARPS % 4 == 0 && EPI_WARPS % 4 == 0, "roles are whole warpgroups");
  static_assert(STAGE_WARPS == EPI_WARPS, "the two roles form two equal selection groups");
  static_assert(STAGES <= STAGE_WARPS, "one stage warp per stage");
  static_assert(STAGE_REGS * STAGE_WARPS + EPI_REGS * EPI_WARPS <= LAUNCH_REGS * (STAGE_WARPS + EPI_WARPS),
                "the re-split fits the registers the block is launched with");
  static constexpr int CAP = decode_cap_tiles(Q) * kTileKeys;  // row-buffer keys per query row
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t SFA_COL = ACC * N;
  static constexpr uint32_t SFB_COL = SFA_COL + 4 * STAGES;
  static_assert(ACC % GROUPS == 0, "tiles sharing an accumulator belong to one epilogue group");
  static_assert(SFB_COL + 8 <= TMEM_COLS, "accumulators and scale chunks fit the allocation");
  // shared memory (offsets from a 1024-byte aligned base)
  static constexpr uint32_t OFF_PACKED = 0;                         // [STAGES][4][128][16]
  static constexpr uint32_t OFF_SFA = OFF_PACKED + STAGES * 8192;   // [STAGES][512]
  static constexpr uint32_t OFF_QB = OFF_SFA + STAGES * 512;        // [2][4][N][16]
  static constexpr uint32_t OFF_SFB = OFF_QB + 2 * N * 64;          // [2][512]
  static constexpr uint32_t OFF_W = OFF_SFB + 2 * 512;              // [2][N]
  static constexpr uint32_t OFF_LG = OFF_W + 2 * N * 4;             // [Q][CAP] ordered keys
  // Histograms of the range's first and last units (4096 fine bins and 64 coarse bins of 64): the
  // fine bins counted while streaming, the coarse ones summed from them when the selection starts
  // (one query row; with several rows they are counted after the stream).
  static constexpr bool HIST_IN_STREAM = Q == 1;
  static constexpr int HST_WORDS = kL1Bins + 64;
  static constexpr uint32_t OFF_HST = OFF_LG + Q * CAP * 4;         // [2][HST_WORDS]
  static constexpr uint32_t OFF_SCR = OFF_HST + (HIST_IN_STREAM ? 2 * HST_WORDS * 4 : 0);  // [2][128] scratch
  static constexpr int REL_RING = STAGES / ACC + 2;
  static_assert(STAGES % ACC == 0, "a stage warp keeps to one accumulator");
  // full[STAGES], empty[STAGES], acc_full[ACC], acc_rel[ACC * REL_RING], q_ready[2], q_free[2]
  static constexpr uint32_t NUM_BARS = 2 * STAGES + ACC + ACC * REL_RING + 4;
  static constexpr uint32_t BAR_QREADY = 2 * STAGES + ACC + ACC * REL_RING;
  static constexpr uint32_t BAR_QFREE = BAR_QREADY + 2;
  static constexpr uint32_t OFF_BAR = OFF_SCR + 2 * 128 * 4;
  static constexpr uint32_t OFF_KS = OFF_BAR + NUM_BARS * 8;  // KernelShared
  static constexpr uint32_t SMEM_BYTES = OFF_KS + 512;
  static_assert(SMEM_BYTES <= 227 * 1024, "fits one SM");
  static_assert(OFF_LG % 16 == 0 && OFF_QB % 128 == 0, "operand and row-buffer alignment");
  // The selection phase reuses the stage area (free once the stream has ended): each of the two
  // selection groups gets half of it, in words from the group's base:
  static constexpr int P_WORDS = static_cast<int>(OFF_QB / 4) / 2 / 32 * 32;
  static constexpr int P_HIST = 0;                    // [kL1Bins + 64] histogram, fine and coarse
  static constexpr int P_LIST = P_HIST + kL1Bins + 64;  // [LIST_CAP] keys of the threshold bin
  static constexpr int LIST_CAP = 2048;
  static constexpr int P_EQPRE = P_LIST + LIST_CAP;  // [Q][kDecodeMaxCtas + 4] prefix of the units' bin keys
  // Row-buffer positions (16 bits) of the keys that can still be selected, per row: in the rest of
  // the group's area, or, when the whole CTA selects one unit, in the second group's half.
  static constexpr int P_CIDX = P_EQPRE + Q * (kDecodeMaxCtas + 4);
  static constexpr int CIDX_GROUP = (P_WORDS - P_CIDX) * 2 / Q / 8 * 8;  // positions per row, own area
  // A sequence merge (after the round's exchanges: the bin-key prefixes and positions are dead)
  // stages candidate keys over them and keeps its segment offsets in the area's last words; a merge
  // whose lists exceed CCAP keys reads them from the workspace instead.
  static constexpr int P_CAND = P_EQPRE;
  static constexpr int P_SOFF = P_WORDS - 1040;       // [1024 + 1] segment offsets of a sequence merge
  static constexpr int CCAP = (P_SOFF - P_CAND) / 128 * 128;
  static_assert(P_CIDX < P_WORDS && CCAP >= 2048, "selection areas fit");
  static_assert(P_HIST % 4 == 0 && P_LIST % 4 == 0, "16-byte aligned histograms");
  static constexpr int CIDX_WHOLE = CAP;                                 // positions per row, second half
  static_assert(CAP <= 65536 && (Q > 1 || CAP / 2 <= P_WORDS), "candidate positions fit the second half");
};


// ---- cross-CTA synchronisation in global memory ----------------------------------------------

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ uint32_t atom_add_acq_rel_gpu(uint32_t* p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

__device__ __forceinline__ void red_add_release_gpu(uint32_t* p, uint32_t v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t ldcg_u32(const uint32_t* p) { return __ldcg(p); }
__device__ __forceinline__ uint2 ldcg_u2(const uint2* p) { return __ldcg(p); }

// ---- stream phase -------------------------------------------------------------------------------

struct RangeIter {
  const DecodeUnit* units;
  int first, count;
  __device__ __forceinline__ DecodeUnit at(int i) const { return units[first + i]; }
};

__device__ __forceinline__ int dunit_tiles(const DecodeUnit& u) {
  return u.ke > u.kb ? (u.ke - u.kb + kTileKeys - 1) / kTileKeys : 0;
}

struct Cursor {
  int i, j, nt;
  DecodeUnit u;
};

// Move `steps` tiles forward (skipping units without tiles); false once past the range's last tile.
__device__ __forceinline__ bool cursor_advance(Cursor& c, int steps, const RangeIter& it) {
  while (c.i < it.count && (steps > 0 || c.j >= c.nt)) {
    const int left = c.nt - c.j;
    if (steps < left) {
      c.j += steps;
      steps = 0;
    } else {
      steps -= left;
      ++c.i;
      c.j = 0;
      if (c.i < it.count) {
        c.u = it.at(c.i);
        c.nt = dunit_tiles(c.u);
      }
    }
  }
  return c.i < it.count;
}

// Bounded wait: a timeout raises the CTA's abort flag and the status bit; later waits return at once.
__device__ __forceinline__ bool wait_slow(uint64_t* bar, uint32_t parity, volatile int* abort_flag, int32_t* status) {
  if (*abort_flag) return false;
  if (mbar_wait(bar, parity, kWaitLimitNs)) return true;
  *abort_flag = 1;
  set_status(status, IDX_FP4_DEV_TIMEOUT);
  return false;
}

__device__ __forceinline__ bool bounded_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                             int32_t* status) {
  return mbar_try_wait(bar, parity) || wait_slow(bar, parity, abort_flag, status);
}

// Page id of the tile at cursor c for lane 0 (the tile's first page) and lane 1 (its second, or -1
// when the tile holds one page). A logical page outside the table gives -2 and is not read.
__device__ __forceinline__ int tile_page(const DecodeParams& p, const Cursor& c, int lane) {
  const int lp = c.u.kb / kPage + 2 * c.j + lane;
  const bool needed = lane == 0 || (lane == 1 && c.u.kb + c.j * kTileKeys + kPage < c.u.ke);
  if (!needed) return -1;
  if (lp < 0 || lp >= p.bt_stride) return -2;
  return p.block_tables[static_cast<int64_t>(c.u.seq) * p.bt_stride + lp];
}

// Per-CTA state in shared memory. Every role re-reads it, so that little stays live in registers
// across the warp-role branches (whose register budgets differ).
struct RoundInfo {
  int uf, ul;   // the round's units [uf, ul)
  int tiles;    // tiles this CTA streamed in earlier rounds (ring and accumulator phases)
  int units;    // units this CTA streamed in earlier rounds (query-buffer phases)
};

// The schedule entries of a range's first or last unit, read into shared memory during the stream.
struct RangeMeta {
  DecodeUnit u;
  DecodeSeg sg;
  int ctx;   // its sequence's context
  int nseg;  // its sequence's segments
  int pad[2];
};

// An exchange between the units of a segment row, from its first round to its second.
struct TaskState {
  uint32_t bin;         // threshold bin of the segment row
  uint32_t need;        // keys of that bin among the top-k
  uint32_t gt_before;   // keys above the bin in the segment's earlier units
  uint32_t ok;          // the first round completed
};

struct KernelShared {
  DecodeSchedHeader h;  // the schedule's header
  uint32_t tmem;        // TMEM base address
  int abort;            // a bounded wait gave up: later waits return at once
  RoundInfo round[2];   // round r in slot r & 1 (written before round r's start barrier, read after it;
                        // slot r & 1 is rewritten only after every warp has passed round r + 1's)
  TaskState task[2][kMaxNextN];  // per selection group and row
  uint32_t counter[2][4];        // per selection group
  int pending[2];                // sequence merges deferred to the end of a group's selection
  int pending_seq[2][kMaxNextN];
  RangeMeta meta[2];             // the round's first and last units (written during the stream)
  int ncand[2][kMaxNextN];       // per group and row: candidate positions listed (-1: every key)
};
static_assert(sizeof(KernelShared) <= 512, "fits its slot");

__device__ __forceinline__ DecodeSchedView sched_view(const DecodeParams& p, const DecodeSchedHeader& h) {
  return decode_sched_view(const_cast<void*>(p.sched), h.max_batch, h.ranges_cap, h.units_cap);
}

// Stage warp `ps`: streams the tiles t of this round's range with (st.tiles + t) % STAGES == ps
// through its stage and issues their MMAs.
template <int H, int Q>
__device__ __forceinline__ void stream_stage_warp(const DecodeParams& p, uint8_t* smem, int slot, int ps, int lane) {
  using C = DecodeCfg<H, Q>;
  constexpr int N = C::N, ACC = C::ACC, STAGES = C::STAGES;
  KernelShared* ks = reinterpret_cast<KernelShared*>(smem + C::OFF_KS);
  volatile int* abort_flag = &ks->abort;
  const uint32_t tmem = ks->tmem;
  const RoundInfo st = ks->round[slot];
  const RangeIter it{sched_view(p, ks->h).units, st.uf, st.ul - st.uf};
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* full_bar = bars;
  uint64_t* empty_bar = bars + STAGES;
  uint64_t* acc_full = bars + 2 * STAGES;
  uint64_t* acc_rel = acc_full + ACC;
  uint64_t* q_ready = bars + C::BAR_QREADY;
  uint64_t* q_free = bars + C::BAR_QFREE;
  const uint64_t pol = policy_evict_first();
  uint8_t* stage = smem + C::OFF_PACKED + ps * 8192;
  uint8_t* sfa_s = smem + C::OFF_SFA + ps * 512;
  const uint64_t a_desc = smem_desc(smem_addr(stage), 2048, 128);
  const uint32_t sfa_t = tmem + C::SFA_COL + 4u * static_cast<uint32_t>(ps);
  const uint32_t idesc0 = mxf4_idesc(128, N, 0), idesc2 = mxf4_idesc(128, N, 2);
  // The scale plane's 16x4 row transpose puts rows l%16 + 16*b of a page at byte b of word l%16 of
  // each group's 64 bytes: lane l takes byte l/16 (rows l, l+64 of the tile) and byte 2 + l/16 (rows
  // l+32, l+96); tile row m goes to TMEM lane m%32, column m/32 of the scale chunk.
  const uint32_t sel_lo = static_cast<uint32_t>(lane >> 4), sel_hi = sel_lo + 2u;
  const uint32_t perm_lo = sel_lo | ((sel_lo + 4u) << 4), perm_hi = sel_hi | ((sel_hi + 4u) << 4);
  const int j0 = ((ps - st.tiles) % STAGES + STAGES) % STAGES;  // this warp's first tile of the round
  Cursor c{0, 0, 0, DecodeUnit{}};
  bool have = it.count > 0;
  if (have) {
    c.u = it.at(0);
    c.nt = dunit_tiles(c.u);
    have = cursor_advance(c, j0, it);
  }
  int entry = have ? tile_page(p, c, lane) : -1;
  int f = st.tiles + j0;      // CTA-wide tile number (ring and accumulator phases)
  // Query operands: this warp waits for every unit's operand in order (so that each parity wait
  // names an unambiguous phase) and frees each unit's buffer once its tiles lie behind it.
  int qnext = 0;              // next unit of the round whose operand this warp has waited for
  int qfreed = 0;             // units of the round whose buffer this warp has freed
  int last_f = -1;
  while (have) {
    int pid0 = __shfl_sync(0xFFFFFFFFu, entry, 0);
    int pid1 = __shfl_sync(0xFFFFFFFFu, entry, 1);
    const bool has1 = pid1 != -1;
    if ((pid0 == -2 || pid1 == -2) && lane == 0) set_status(p.status, IDX_FP4_DEV_BAD_CTX);
    if (pid0 < 0 || pid0 >= p.num_pages) {
      if (lane == 0 && pid0 != -2) set_status(p.status, IDX_FP4_DEV_BAD_PAGE);
      pid0 = 0;
    }
    if (has1 && (pid1 < 0 || pid1 >= p.num_pages)) {
      if (lane == 0 && pid1 != -2) set_status(p.status, IDX_FP4_DEV_BAD_PAGE);
      pid1 = 0;
    }
    // the stage's previous tile has been consumed by its MMAs
    if (lane == 0) {
      bounded_wait(&empty_bar[ps], ((f / STAGES) & 1) ^ 1, abort_flag, p.status);
      mbar_arrive_expect_tx(&full_bar[ps], (has1 ? 2u : 1u) * kPageBytes);
    }
    __syncwarp();
    if (lane < 8 && (lane < 4 || has1)) {
      const int pg = lane >> 2, k = lane & 3;
      const int64_t pid = pg == 0 ? pid0 : pid1;
      bulk_load_evict_first(stage + k * 2048 + pg * 1024, p.kv_packed + pid * kPageBytes + k * 1024, 1024,
                            &full_bar[ps], pol);
    }
    uint32_t w0[4], w1[4];
    {
      const uint32_t* s0 = reinterpret_cast<const uint32_t*>(p.kv_scale + static_cast<int64_t>(pid0) * kPageScaleBytes) + (lane & 15);
      const uint32_t* s1 = reinterpret_cast<const uint32_t*>(p.kv_scale + static_cast<int64_t>(has1 ? pid1 : 0) * kPageScaleBytes) + (lane & 15);
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        w0[g] = __ldg(s0 + 16 * g);
        w1[g] = has1 ? __ldg(s1 + 16 * g) : 0x7F7F7F7Fu;
      }
    }
    Cursor nc = c;
    const bool next = cursor_advance(nc, STAGES, it);
    const int next_entry = next ? tile_page(p, nc, lane) : -1;
    {
      const uint32_t c0 = __byte_perm(__byte_perm(w0[0], w0[1], perm_lo), __byte_perm(w0[2], w0[3], perm_lo), 0x5410);
      const uint32_t c1 = __byte_perm(__byte_perm(w0[0], w0[1], perm_hi), __byte_perm(w0[2], w0[3], perm_hi), 0x5410);
      const uint32_t c2 = __byte_perm(__byte_perm(w1[0], w1[1], perm_lo), __byte_perm(w1[2], w1[3], perm_lo), 0x5410);
      const uint32_t c3 = __byte_perm(__byte_perm(w1[0], w1[1], perm_hi), __byte_perm(w1[2], w1[3], perm_hi), 0x5410);
      *reinterpret_cast<uint4*>(sfa_s + lane * 16) = make_uint4(c0, c1, c2, c3);
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      bounded_wait(&full_bar[ps], (f / STAGES) & 1, abort_flag, p.status);
      // in order: wait for unit x's operand, and free it at once when this tile lies past unit x
      // (the operand of unit x + 2 is only prepared once every stage warp has freed unit x)
      while (qnext <= c.i) {
        const int un = st.units + qnext;
        bounded_wait(&q_ready[un & 1], (un >> 1) & 1, abort_flag, p.status);
        ++qnext;
        for (; qfreed < qnext && qfreed < c.i; ++qfreed) mbar_arrive(&q_free[(st.units + qfreed) & 1]);
      }
      const int a = f % ACC, jf = f / ACC;
      if (jf >= 1)  // the accumulator's previous tile has been read out
        bounded_wait(&acc_rel[a * C::REL_RING + (jf - 1) % C::REL_RING],
                     static_cast<uint32_t>((jf - 1) / C::REL_RING) & 1u, abort_flag, p.status);
      tc_fence_after_sync();
      const int par = (st.units + c.i) & 1;
      const uint32_t qb = smem_addr(smem + C::OFF_QB + par * (N * 64));
      const uint32_t sfb = tmem + C::SFB_COL + 4u * static_cast<uint32_t>(par);
      const uint32_t d = tmem + static_cast<uint32_t>(a * N);
      tmem_copy_sf_chunk(sfa_t, smem_addr(sfa_s));
      mma_mxf4(d, a_desc, smem_desc(qb, N * 16, 128), idesc0, sfa_t, sfb, 0u);
      mma_mxf4(d, a_desc + (4096 >> 4), smem_desc(qb + 2 * N * 16, N * 16, 128), idesc2, sfa_t, sfb, 1u);
      tc_commit(&empty_bar[ps]);
      tc_commit(&acc_full[a]);
    }
    __syncwarp();
    last_f = f;
    c = nc;
    have = next;
    entry = next_entry;
    f += STAGES;
  }
  // This warp's last copies and MMAs are done before the stage area is reused; the operands of the
  // round's remaining units are waited for (their scale copies into TMEM completed) and freed.
  if (lane == 0) {
    if (last_f >= 0) {
      mbar_wait(&full_bar[ps], (last_f / STAGES) & 1, kWaitLimitNs);
      mbar_wait(&empty_bar[ps], (last_f / STAGES) & 1, kWaitLimitNs);
    }
    for (; qfreed < it.count; ++qfreed) {
      if (qfreed >= qnext) {
        const int un = st.units + qfreed;
        bounded_wait(&q_ready[un & 1], (un >> 1) & 1, abort_flag, p.status);
        qnext = qfreed + 1;
      }
      mbar_arrive(&q_free[(st.units + qfreed) & 1]);
    }
  }
  __syncwarp();
}

// Query heads of unit i (rows seq * Q .. seq * Q + Q - 1) -> canonical K-major [4 chunks][N][16 B]
// operand, query scales -> the tensor core's scale layout (row n at line n%32, word n/32), weights
// -> plain floats; one thread then copies the scales to TMEM and commits q_ready. The buffers of
// parity un & 1 are free: the unit that used them last has been fully read out.
template <int H, int Q>
__device__ __forceinline__ void prep_query(const DecodeParams& p, const DecodeUnit& u, int un, uint8_t* smem,
                                           uint32_t tmem, int etid) {
  using C = DecodeCfg<H, Q>;
  constexpr int N = C::N;
  uint64_t* q_ready = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR) + C::BAR_QREADY;
  uint64_t* q_free = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR) + C::BAR_QFREE;
  const int par = un & 1;
  // every stage warp is past unit un - 2, the buffers' previous user
  if (un >= 2) {
    const int prev = un - 2;
    if (!mbar_try_wait(&q_free[prev & 1], (prev >> 1) & 1)) {
      volatile int* abort_flag = &reinterpret_cast<KernelShared*>(smem + C::OFF_KS)->abort;
      wait_slow(&q_free[prev & 1], (prev >> 1) & 1, abort_flag, p.status);
    }
  }
  uint8_t* qb = smem + C::OFF_QB + par * (N * 64);
  uint8_t* sfb = smem + C::OFF_SFB + par * 512;
  float* wq = reinterpret_cast<float*>(smem + C::OFF_W) + par * N;
  const int64_t row0 = static_cast<int64_t>(u.seq) * Q;
  const uint8_t* qsrc = p.q_packed + row0 * H * 64;
  for (int cc = etid; cc < 4 * N; cc += C::EPI_THREADS) {
    const int g = cc / N, n = cc % N;
    *reinterpret_cast<uint4*>(qb + g * N * 16 + n * 16) = __ldg(reinterpret_cast<const uint4*>(qsrc + n * 64 + g * 16));
  }
  for (int n = etid; n < 128; n += C::EPI_THREADS) {
    uint32_t wv = 0x7F7F7F7Fu;
    if (n < N) wv = __ldg(reinterpret_cast<const uint32_t*>(p.q_scale + (row0 * H + n) * 4));
    *reinterpret_cast<uint32_t*>(sfb + (n & 31) * 16 + (n >> 5) * 4) = wv;
  }
  for (int x = etid; x < N; x += C::EPI_THREADS) wq[x] = __ldg(p.weights + row0 * H + x);
  fence_proxy_async_smem();
  named_barrier_sync(kEpiBarrier, C::EPI_THREADS);
  if (etid == 0) {
    tc_fence_after_sync();
    tmem_copy_sf_chunk(tmem + C::SFB_COL + 4u * static_cast<uint32_t>(par), smem_addr(sfb));
    tc_commit(&q_ready[par]);
  }
}

// Head-weighted ReLU sum of one query row for this thread's key (TMEM lane): heads h of row r sit in
// accumulator columns r * H + h. Fixed summation order (deterministic).
template <int H>
__device__ __forceinline__ float row_logit(uint32_t col, const float* wr) {
  float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f, s4 = 0.f, s5 = 0.f, s6 = 0.f, s7 = 0.f;
  if constexpr (H == 16) {
    float v[16];
    tmem_load_x16(col, v);
#pragma unroll
    for (int h = 0; h < 16; h += 8) {
      const float4 wa = *reinterpret_cast<const float4*>(wr + h);
      const float4 wb = *reinterpret_cast<const float4*>(wr + h + 4);
      s0 = fmaf(wa.x, fmaxf(v[h], 0.f), s0);
      s1 = fmaf(wa.y, fmaxf(v[h + 1], 0.f), s1);
      s2 = fmaf(wa.z, fmaxf(v[h + 2], 0.f), s2);
      s3 = fmaf(wa.w, fmaxf(v[h + 3], 0.f), s3);
      s4 = fmaf(wb.x, fmaxf(v[h + 4], 0.f), s4);
      s5 = fmaf(wb.y, fmaxf(v[h + 5], 0.f), s5);
      s6 = fmaf(wb.z, fmaxf(v[h + 6], 0.f), s6);
      s7 = fmaf(wb.w, fmaxf(v[h + 7], 0.f), s7);
    }
  } else if constexpr (H % 64 == 0) {
    // packed pairs: heads (h, h+1) share one fma.rn.f32x2
    unsigned long long p01 = 0ull, p23 = 0ull, p45 = 0ull, p67 = 0ull;
#pragma unroll
    for (int cc = 0; cc < H; cc += 64) {
      float v[64];
      tmem_load_2x32(col + cc, col + cc + 32, v);
#pragma unroll
      for (int h = 0; h < 64; h += 8) {
        const float4 wa = *reinterpret_cast<const float4*>(wr + cc + h);
        const float4 wb = *reinterpret_cast<const float4*>(wr + cc + h + 4);
        fma2(p01, wa.x, wa.y, fmaxf(v[h], 0.f), fmaxf(v[h + 1], 0.f));
        fma2(p23, wa.z, wa.w, fmaxf(v[h + 2], 0.f), fmaxf(v[h + 3], 0.f));
        fma2(p45, wb.x, wb.y, fmaxf(v[h + 4], 0.f), fmaxf(v[h + 5], 0.f));
        fma2(p67, wb.z, wb.w, fmaxf(v[h + 6], 0.f), fmaxf(v[h + 7], 0.f));
      }
    }
    const float2 a01 = unpack2(p01), a23 = unpack2(p23), a45 = unpack2(p45), a67 = unpack2(p67);
    s0 = a01.x; s1 = a01.y; s2 = a23.x; s3 = a23.y;
    s4 = a45.x; s5 = a45.y; s6 = a67.x; s7 = a67.y;
  } else {
#pragma unroll
    for (int cc = 0; cc < H; cc += 32) {
      float v[32];
      tmem_load_x32(col + cc, v);
#pragma unroll
      for (int h = 0; h < 32; h += 8) {
        const float4 wa = *reinterpret_cast<const float4*>(wr + cc + h);
        const float4 wb = *reinterpret_cast<const float4*>(wr + cc + h + 4);
        s0 = fmaf(wa.x, fmaxf(v[h], 0.f), s0);
        s1 = fmaf(wa.y, fmaxf(v[h + 1], 0.f), s1);
        s2 = fmaf(wa.z, fmaxf(v[h + 2], 0.f), s2);
        s3 = fmaf(wa.w, fmaxf(v[h + 3], 0.f), s3);
        s4 = fmaf(wb.x, fmaxf(v[h + 4], 0.f), s4);
        s5 = fmaf(wb.y, fmaxf(v[h + 5], 0.f), s5);
        s6 = fmaf(wb.z, fmaxf(v[h + 6], 0.f), s6);
        s7 = fmaf(wb.w, fmaxf(v[h + 7], 0.f), s7);
      }
    }
  }
  return ((s0 + s1) + (s2 + s3)) + ((s4 + s5) + (s6 + s7));
}

// Epilogue warp (group grp, TMEM lane quarter qtr): logits of the tiles t with (st.tiles + t) %
// GROUPS == grp into the row buffer; the query operands of the round's units, two units ahead.
template <int H, int Q>
__device__ __forceinline__ void stream_epilogue_warp(const DecodeParams& p, uint8_t* smem, int slot, int e, int lane) {
  using C = DecodeCfg<H, Q>;
  constexpr int N = C::N, ACC = C::ACC;
  KernelShared* ks = reinterpret_cast<KernelShared*>(smem + C::OFF_KS);
  volatile int* abort_flag = &ks->abort;
  const uint32_t tmem = ks->tmem;
  const DecodeSchedView v = sched_view(p, ks->h);
  const int32_t* seq_ctx = v.seq_ctx;
  const RoundInfo st = ks->round[slot];
  const RangeIter it{v.units, st.uf, st.ul - st.uf};
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* acc_full = bars + 2 * C::STAGES;
  uint64_t* acc_rel = acc_full + ACC;
  const int grp = e >> 2;
  const int qtr = (C::EPI_WARP0 + e) & 3;  // TMEM lane quarter = warp id % 4
  const int etid = e * 32 + lane;
  const int krow = qtr * 32 + lane;
  const uint32_t lane_base = static_cast<uint32_t>(qtr * 32) << 16;
  uint32_t* lg = reinterpret_cast<uint32_t*>(smem + C::OFF_LG);
  uint32_t* hst = reinterpret_cast<uint32_t*>(smem + C::OFF_HST);
  if constexpr (C::HIST_IN_STREAM)
    for (int x = etid; x < 2 * C::HST_WORDS; x += C::EPI_THREADS) hst[x] = 0u;  // ordered by prep's barrier
  if (it.count > 0) prep_query<H, Q>(p, it.at(0), st.units, smem, tmem, etid);
  if (it.count > 1) prep_query<H, Q>(p, it.at(1), st.units + 1, smem, tmem, etid);
  // the last group's first thread, idle until that group's first tile, reads the entries the
  // selection starts from
  if (e == C::EPI_WARPS - 4 && lane == 0 && it.count > 0)
    for (int m = 0; m < 2; ++m) {
      const DecodeUnit u = it.at(m == 0 ? 0 : it.count - 1);
      ks->meta[m] = RangeMeta{u, v.segs[u.seg], seq_ctx[u.seq], v.seq_nseg[u.seq], {0, 0}};
    }
  int t0 = st.tiles;  // CTA-wide number of the unit's first tile
  for (int i = 0; i < it.count; ++i) {
    const DecodeUnit u = it.at(i);
    const float* wsm = reinterpret_cast<const float*>(smem + C::OFF_W) + ((st.units + i) & 1) * N;
    const int ctx = seq_ctx[u.seq];
    const int ntiles = dunit_tiles(u);
    // the range's first and last units may share their sequence with other CTAs: count their keys
    uint32_t* uh = nullptr;
    if constexpr (C::HIST_IN_STREAM) uh = i == 0 ? hst : (i == it.count - 1 ? hst + C::HST_WORDS : nullptr);
    for (int j = ((grp - t0) % C::GROUPS + C::GROUPS) % C::GROUPS; j < ntiles; j += C::GROUPS) {
      const int tt = t0 + j;
      const int a = tt % ACC;
      bounded_wait(&acc_full[a], static_cast<uint32_t>(tt / ACC) & 1u, abort_flag, p.status);
      tc_fence_after_sync();
      float logit[Q];
#pragma unroll
      for (int r = 0; r < Q; ++r) logit[r] = row_logit<H>(tmem + lane_base + a * N + r * H, wsm + r * H);
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_rel[a * C::REL_RING + (tt / ACC) % C::REL_RING]);
      const int key = u.kb + j * kTileKeys + krow;
      const int at = u.buf + j * kTileKeys + krow;  // < CAP: a range holds at most CAP keys
#pragma unroll
      for (int r = 0; r < Q; ++r) {
        const bool valid = key < ctx - Q + 1 + r;
        const uint32_t ok = ordered_key(logit[r]);
        if (at < C::CAP) lg[r * C::CAP + at] = valid ? ok : 0u;
        if (C::HIST_IN_STREAM && valid && uh != nullptr) smem_red_add(&uh[ok >> kL1Shift], 1u);
        if (valid && p.logits_debug != nullptr && key < p.logits_stride)
          p.logits_debug[(static_cast<int64_t>(u.seq) * Q + r) * p.logits_stride + key] = logit[r];
      }
    }
    t0 += ntiles;
    if (i + 2 < it.count) {
      named_barrier_sync(kEpiBarrier, C::EPI_THREADS);  // every group is done with unit i's operand
      prep_query<H, Q>(p, it.at(i + 2), st.units + i + 2, smem, tmem, etid);
    }
  }
}

// ---- selection phase ----------------------------------------------------------------------------

__device__ __forceinline__ int clampi(int x, int lo, int hi) { return x < lo ? lo : (x > hi ? hi : x); }

// Keep every candidate (all) or those above T plus the first `need` equal to T, in token order:
// out(position, key, token) for each kept candidate, positions dense from 0.
template <class KeyAt, class TokAt, class Out>
__device__ __forceinline__ void blk_emit(const Blk& B, KeyAt key, TokAt tok, int n, bool all, uint32_t T,
                                         uint32_t need, Out out) {
  const int2 run = blk_run(B, n);
  uint32_t gt = 0, eq = 0;
  if (all) {
    gt = static_cast<uint32_t>(run.y - run.x);
  } else {
#pragma unroll 1
    for (int x = run.x; x < run.y; ++x) {
      const uint32_t k = key(x);
      gt += k > T ? 1u : 0u;
      eq += k == T ? 1u : 0u;
    }
  }
  const uint2 pre = blk_scan2(B, gt, eq, nullptr, nullptr);
  uint32_t pos = pre.x + min(pre.y, need), eqr = pre.y;
  if (gt + eq != 0u)
#pragma unroll 1
    for (int x = run.x; x < run.y; ++x) {
      const uint32_t k = key(x);
      const bool eqk = !all && k == T;
      const bool keep = all || k > T || (eqk && eqr < need);
      if (keep) out(pos++, k, tok(x));
      eqr += eqk ? 1u : 0u;
    }
}

// Exact top-kk of n candidates in token order (first-level bin unknown: counted here).
template <class KeyAt, class TokAt, class Out>
__device__ __forceinline__ void blk_select(const Blk& B, KeyAt key, TokAt tok, int n, int kk, uint32_t* hist,
                                           uint32_t* list, int list_cap, Out out, const uint32_t* pre = nullptr) {
  if (kk <= 0 || n <= 0) return;
  if (kk >= n) {
    blk_emit(B, key, tok, n, true, 0u, 0u, out);
    return;
  }
  // the first-level histogram (4096 fine bins, then 64 coarse): counted in the stream, or here
  const uint32_t* h = pre;
  if (h == nullptr) {
    blk_zero(B, hist, kL1Bins);
    B.sync();
#pragma unroll 1
    for (int x = B.tid; x < n; x += B.nt) smem_red_add(&hist[key(x) >> kL1Shift], 1u);
    B.sync();
    blk_coarse64(B, hist);
    h = hist;
  }
  B.sync();
  if (B.warp() == 0) {
    const uint2 r = warp_find_bin2<64, 64>(h, h + kL1Bins, static_cast<uint32_t>(kk), B.lane());
    if (B.lane() == 0) {
      B.sc[64] = r.x;
      B.sc[65] = r.y;
    }
  }
  B.sync();
  const uint2 r = make_uint2(B.sc[64], B.sc[65]);
  bool consistent = true;
  const uint2 tn = blk_resolve(B, key, n, r.x, static_cast<uint32_t>(kk) - r.y, hist, list, list_cap, &consistent);
  blk_emit(B, key, tok, n, false, tn.x, tn.y, out);
}

// Where a segment row's selection goes: the final output row (then padded to topk with -1 / -inf),
// or the segment's list when its sequence has several segments.
struct RowOut {
  int32_t* idx;
  float* val;      // nullable
  uint2* list;     // non-null: a segment list instead
  uint32_t limit;  // positions past the row's k are never written
  __device__ __forceinline__ void operator()(uint32_t pos, uint32_t key, int tok) const {
    if (pos >= limit) return;
    if (list != nullptr) {
      list[pos] = make_uint2(key, static_cast<uint32_t>(tok));
    } else {
      idx[pos] = tok;
      if (val != nullptr) val[pos] = key_to_float(key);
    }
  }
};

__device__ __forceinline__ void pad_row(const Blk& B, const DecodeParams& p, int64_t row, int from) {
  int32_t* oi = p.topk_idx + row * p.topk;
  float* ov = p.topk_val != nullptr ? p.topk_val + row * p.topk : nullptr;
  for (int x = from + B.tid; x < p.topk; x += B.nt) {
    oi[x] = -1;
    if (ov != nullptr) ov[x] = -__int_as_float(0x7f800000);
  }
}

// Cross-CTA ordering: a CTA's writes, then a block barrier, then one thread's release (an atomic
// add at GPU scope) publish the writes; another CTA's thread acquires the count (a spin on an
// acquire load, or the acquire half of its own atomic), then a block barrier, and that CTA's
// threads read the published data through L2. The shared flags below are written by one thread
// before a barrier and read after it; the next write to a flag comes after further barriers.

// Bounded wait by one thread until *ctr >= target; the answer is shared with the block.
__device__ __forceinline__ bool blk_wait_count(const Blk& B, uint32_t* ctr, uint32_t target, volatile int* abort_flag,
                                               int32_t* status) {
  if (B.tid == 0) {
    bool ok = *abort_flag == 0;
    if (ok && ld_acquire_gpu(ctr) < target) {
      const uint64_t t0 = global_timer_ns();
      while (ld_acquire_gpu(ctr) < target) {
        if (global_timer_ns() - t0 > kWaitLimitNs) {
          ok = false;
          *abort_flag = 1;
          set_status(status, IDX_FP4_DEV_TIMEOUT);
          break;
        }
      }
    }
    B.sc[72] = ok ? 1u : 0u;
  }
  B.sync();
  return B.sc[72] != 0u;
}

// Publish this CTA's writes for a segment row (count it on *ctr).
__device__ __forceinline__ void blk_publish(const Blk& B, uint32_t* ctr) {
  B.sync();
  if (B.tid == 0) red_add_release_gpu(ctr, 1u);
}

// Ticket after this CTA's writes for a segment row: true for the CTA that arrives last (which has
// then acquired every other arrival's writes).
__device__ __forceinline__ bool blk_ticket(const Blk& B, uint32_t* ctr, uint32_t count) {
  B.sync();
  if (B.tid == 0) B.sc[73] = atom_add_acq_rel_gpu(ctr, 1u) + 1u == count ? 1u : 0u;
  B.sync();
  return B.sc[73] != 0u;
}

struct SegCtx {
  DecodeSeg sg;
  int seg_id, q, row_end, kk;
  int64_t out_row;
};

// Exact top-k of a sequence row over its segments' lists (a sequence spanning several rounds).
// P is the selection group's area.
template <int H, int Q>
__device__ void merge_sequence(const DecodeParams& p, const DecodeSchedView& v, const DecodeWs& ws, int seq, int q,
                               uint32_t* P, const Blk& B) {
  using C = DecodeCfg<H, Q>;
  uint32_t* off = P + C::P_SOFF;
  const int nseg = v.seq_nseg[seq], s0 = v.seq_seg0[seq];
  const int ctx = v.seq_ctx[seq];
  const int row_end = clampi(ctx - Q + 1 + q, 0, ctx);
  const int ns = min(nseg, 1024);
  if (B.tid == 0) {
    uint32_t o = 0;
    for (int k = 0; k < ns; ++k) {
      off[k] = o;
      const DecodeSeg sg = v.segs[s0 + k];
      o += static_cast<uint32_t>(min(p.topk, clampi(row_end - sg.kb, 0, sg.ke - sg.kb)));
    }
    off[ns] = o;
  }
  B.sync();
  const int M = static_cast<int>(off[ns]);
  auto at = [&](int x) {
    int lo = 0, hi = ns - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (static_cast<int>(off[mid]) <= x) lo = mid; else hi = mid - 1;
    }
    return ws.seglists + (static_cast<int64_t>(s0 + lo) * Q + q) * p.topk + (x - static_cast<int>(off[lo]));
  };
  // the keys are staged when they fit (two segments' full lists at least); tokens are read from
  // the lists for the kept keys only
  uint32_t* ckey = P + C::P_CAND;
  const bool staged = M <= C::CCAP;
  if (staged) {
    for (int x = B.tid; x < M; x += B.nt) ckey[x] = ldcg_u2(at(x)).x;
    B.sync();
  }
  auto key = [&](int x) { return staged ? ckey[x] : ldcg_u2(at(x)).x; };
  auto tok = [&](int x) { return static_cast<int>(ldcg_u2(at(x)).y); };
  const int64_t row = static_cast<int64_t>(seq) * Q + q;
  const int kk = min(p.topk, row_end);
  RowOut out{p.topk_idx + row * p.topk, p.topk_val != nullptr ? p.topk_val + row * p.topk : nullptr, nullptr,
             static_cast<uint32_t>(kk)};
  blk_select(B, key, tok, M, kk, P + C::P_HIST, P + C::P_LIST, C::LIST_CAP, out);
  pad_row(B, p, row, kk);
  if (B.tid == 0) ws.seqsync[(static_cast<int64_t>(seq) * Q + q) * 4] = 0u;
  B.sync();
}

// Where a segment row's selection goes: its final output row, or its segment's list when the
// sequence has several segments (then merged by the last segment to finish).
__device__ __forceinline__ RowOut seg_out(const DecodeParams& p, const DecodeWs& ws, const SegCtx& s, int nseg,
                                          int Q) {
  return RowOut{p.topk_idx + s.out_row * p.topk, p.topk_val != nullptr ? p.topk_val + s.out_row * p.topk : nullptr,
                nseg > 1 ? ws.seglists + (static_cast<int64_t>(s.seg_id) * Q + s.q) * p.topk : nullptr,
                static_cast<uint32_t>(max(s.kk, 0))};
}

// Selection of one round's units of this CTA by selection group g (the row buffer holds their
// logits; P is the group's half of the stage area). Group 0 takes the range's first unit, group 1
// its last unit, and the two share the units between them (each a whole sequence). Segments of one
// unit are selected here. The units of a longer segment row run a two-round exchange through the
// workspace, without a merging CTA:
//   A  each unit publishes the non-empty bins of its 12-bit histogram from its own k-th key's bin
//      up (the segment's k-th key lies at or above every unit's, so these bins count it exactly);
//   B1 once every unit has published, each finds the segment's threshold bin and the keys above it
//      from the records, and publishes its keys inside that bin (low 20 bits);
//   B2 once every unit has published those, each resolves the exact threshold key T and how many
//      keys equal to T are kept, works out from the counts how many selected keys the segment's
//      earlier units hold, and writes its own selected keys at that offset, in token order.
// A unit's waits only follow other units' publications, and the two groups run their first and
// last units' exchanges side by side, so no CTA's publication waits behind another exchange.
template <int H, int Q>
__device__ void select_round(const DecodeParams& p, uint8_t* smem, int slot, int g, const Blk& B, bool row_split) {
  using C = DecodeCfg<H, Q>;
  KernelShared* ks = reinterpret_cast<KernelShared*>(smem + C::OFF_KS);
  volatile int* abort_flag = &ks->abort;
  const DecodeSchedView v = sched_view(p, ks->h);
  const DecodeWs ws = decode_ws_view(p.workspace, decode_caps_of(ks->h), ks->h.max_batch, Q);
  const int uf = ks->round[slot].uf, ul = ks->round[slot].ul;
  uint32_t* P = reinterpret_cast<uint32_t*>(smem) + g * C::P_WORDS;
  uint32_t* hist = P + C::P_HIST;
  uint32_t* cnt = ks->counter[g];
  const uint32_t* lg = reinterpret_cast<const uint32_t*>(smem + C::OFF_LG);
  const int topk = p.topk;
  // candidate positions: the second half when the whole CTA selects the range's one unit, else the
  // group's own spare words
  const bool whole = B.nt == C::THREADS;
  const int ccap = whole ? C::CIDX_WHOLE : C::CIDX_GROUP;
  uint16_t* cidx = reinterpret_cast<uint16_t*>(whole ? reinterpret_cast<uint32_t*>(smem) + C::P_WORDS : P + C::P_CIDX);
  const int lane = B.lane(), warp = B.warp();
  // this group's range-end unit, and its rows: all rows, or (row_split: both groups on the range's
  // one unit) every other row from the group's index
  const int ex = g == 0 || row_split ? uf : (ul - 1 > uf ? ul - 1 : -1);
  const int q0 = row_split ? g : 0, qstep = row_split ? 2 : 1;
  auto seg_ctx_of = [&](const DecodeUnit& u, const DecodeSeg& sg, int ctx, int q) {
    SegCtx s;
    s.sg = sg;
    s.seg_id = u.seg;
    s.q = q;
    s.row_end = ctx - Q + 1 + q;
    s.kk = min(topk, clampi(s.row_end - s.sg.kb, 0, s.sg.ke - s.sg.kb));
    s.out_row = static_cast<int64_t>(u.seq) * Q + q;
    return s;
  };
  auto seg_ctx = [&](const DecodeUnit& u, int q) { return seg_ctx_of(u, v.segs[u.seg], v.seq_ctx[u.seq], q); };
  // the range-end unit's schedule entries, read into shared memory during the stream
  DecodeUnit ue{};
  DecodeSeg se{};
  int ctx_e = 0, nseg_e = 0;
  if (ex >= 0) {
    const RangeMeta& m = ks->meta[ex == uf ? 0 : 1];
    ue = m.u;
    se = m.sg;
    ctx_e = m.ctx;
    nseg_e = m.nseg;
  }
  auto seg_keys = [&](const SegCtx& s) { return clampi(s.row_end - s.sg.kb, 0, s.sg.ke - s.sg.kb); };
  auto sync_word = [&](const SegCtx& s, int k) { return &ws.sync[(static_cast<int64_t>(s.seg_id) * Q + s.q) * 4 + k]; };
  // Unit j of a segment: its first tile and tile count follow from the segment's first tile and the
  // range length (unit 0 starts the segment; unit j > 0 starts range seg.tile0 / per + j, or, with
  // ranges aligned to the sequences, j ranges after the segment's first tile), so the other units'
  // areas are found without reading the unit table.
  const int per = ks->h.per;
  const bool aligned = ks->h.aligned != 0;
  auto unit_tile0 = [&](const DecodeSeg& sg, int j) {
    return j == 0 ? sg.tile0 : (aligned ? sg.tile0 + j * per : (sg.tile0 / per + j) * per);
  };
  auto unit_tiles = [&](const DecodeSeg& sg, int j) {
    const int seg_end = sg.tile0 + (sg.ke - sg.kb + kTileKeys - 1) / kTileKeys;
    const int t1 = j + 1 < sg.nunits ? unit_tile0(sg, j + 1) : seg_end;
    return max(0, min(t1, seg_end) - unit_tile0(sg, j));
  };
  // a unit's published bins: a count, then the records
  auto rec_of = [&](const DecodeSeg& sg, int j, int q) {
    return ws.records + q * ws.rec_stride + static_cast<int64_t>(unit_tile0(sg, j)) * kTileKeys + sg.first_unit + j;
  };
  // a unit's list of threshold-bin keys, in its own part of the candidate area
  auto list_of = [&](const DecodeSeg& sg, int j, int q) {
    return reinterpret_cast<uint32_t*>(ws.cands + q * ws.cand_stride + static_cast<int64_t>(unit_tile0(sg, j)) * kTileKeys);
  };
  auto exchanged = [&](const SegCtx& s) { return s.sg.nunits > 1 && s.kk < seg_keys(s); };
  if (B.tid == 0) ks->pending[g] = 0;
  // the stream counted this group's range-end unit (area g) into the fine bins only
  if constexpr (C::HIST_IN_STREAM) blk_coarse64(B, reinterpret_cast<uint32_t*>(smem + C::OFF_HST) + g * C::HST_WORDS);
  // A completed segment row: pad its final row, or count it for its sequence; the last segment of a
  // longer sequence merges the lists at the end of this group's selection (a merge reuses the areas
  // the group's exchanges hold). Only a range-end unit can belong to a sequence spanning rounds, so a
  // group defers at most one merge per row.
  auto segment_done = [&](const SegCtx& s) {
    const int seq = s.sg.seq, nseg = v.seq_nseg[seq];
    if (nseg <= 1) {
      pad_row(B, p, s.out_row, s.kk);
      return;
    }
    if (blk_ticket(B, &ws.seqsync[(static_cast<int64_t>(seq) * Q + s.q) * 4], static_cast<uint32_t>(nseg)) &&
        B.tid == 0) {
      if (ks->pending[g] < kMaxNextN) ks->pending_seq[g][ks->pending[g]++] = seq * kMaxNextN + s.q;
      else set_status(p.status, IDX_FP4_DEV_CAPACITY);
    }
  };
  // The last unit to finish a longer segment row resets the row's counters and completes it.
  auto finish_exchange = [&](const SegCtx& s) {
    if (blk_ticket(B, sync_word(s, 2), static_cast<uint32_t>(s.sg.nunits))) {
      if (B.tid == 0) {
        *sync_word(s, 0) = 0u;
        *sync_word(s, 1) = 0u;
        *sync_word(s, 2) = 0u;
      }
      if (v.seq_nseg[s.sg.seq] > 1) segment_done(s);
    }
  };
  // Selection of a unit that is a whole segment row (nothing to wait for).
  auto select_local = [&](int i, int q) {
    const DecodeUnit u = v.units[i];
    const SegCtx s = seg_ctx(u, q);
    const int un = clampi(s.row_end - u.kb, 0, u.ke - u.kb);
    const uint32_t* keys = lg + q * C::CAP + u.buf;
    auto key = [&](int x) { return keys[x]; };
    auto tok = [&](int x) { return u.kb + x; };
    // a range-end unit's histogram was counted in the stream (one row)
    const uint32_t* pre = nullptr;
    if constexpr (C::HIST_IN_STREAM)
      if (i == uf || i == ul - 1)
        pre = reinterpret_cast<const uint32_t*>(smem + C::OFF_HST) + (i == uf ? 0 : C::HST_WORDS);
    blk_select(B, key, tok, un, s.kk, hist, P + C::P_LIST, C::LIST_CAP, seg_out(p, ws, s, v.seq_nseg[u.seq], Q),
               pre);
    segment_done(s);
    B.sync();
  };

  // ---- A: the range-end unit's rows: whole rows, rows whose every key is selected, published bins
  if (ex >= 0) {
    const DecodeUnit& u = ue;
    const int nseg = nseg_e;
    for (int q = q0; q < Q; q += qstep) {
      const SegCtx s = seg_ctx_of(u, se, ctx_e, q);
      const int un = clampi(s.row_end - u.kb, 0, u.ke - u.kb);
      const uint32_t* keys = lg + q * C::CAP + u.buf;
      if (s.sg.nunits == 1) {
        // a whole segment row: selected with the group's other whole rows below
      } else if (!exchanged(s)) {
        // every key of the segment row is selected: each unit writes its keys at their place
        const RowOut out = seg_out(p, ws, s, nseg, Q);
        const uint32_t base = static_cast<uint32_t>(u.kb - s.sg.kb);
        for (int x = B.tid; x < un; x += B.nt) out(base + static_cast<uint32_t>(x), keys[x], u.kb + x);
        if (u.uidx == 0 && nseg <= 1) pad_row(B, p, s.out_row, s.kk);
        finish_exchange(s);
        B.sync();
      } else {
        const uint32_t* uh;  // fine bins, then 64 coarse bins
        if constexpr (C::HIST_IN_STREAM) {
          uh = reinterpret_cast<const uint32_t*>(smem + C::OFF_HST) + (ex == uf ? 0 : C::HST_WORDS);
        } else {
          blk_zero(B, hist, kL1Bins);
          B.sync();
          for (int x = B.tid; x < un; x += B.nt) smem_red_add(&hist[keys[x] >> kL1Shift], 1u);
          B.sync();
          blk_coarse64(B, hist);
          uh = hist;
        }
        B.sync();
        // the unit's own k-th key's bin (all bins when it holds fewer keys)
        if (warp == 0) {
          const uint32_t bu = un >= s.kk ? warp_find_bin2<64, 64>(uh, uh + kL1Bins, static_cast<uint32_t>(s.kk), lane).x : 0u;
          if (lane == 0) cnt[1] = bu;
        }
        B.sync();
        const uint32_t bu = cnt[1];
        uint32_t* rec = rec_of(s.sg, u.uidx, q);
        const int2 br = blk_run4(B, kL1Bins - static_cast<int>(bu));
        uint32_t nz = 0;
        for (int b = br.x; b < br.y; ++b) nz += uh[bu + b] != 0u ? 1u : 0u;
        uint32_t nrec = 0;
        uint32_t at = 1u + blk_scan2(B, nz, 0u, &nrec, nullptr).x;
        if (nz != 0u)
          for (int b = br.x; b < br.y; ++b) {
            const uint32_t c = uh[bu + b];
            if (c != 0u) rec[at++] = ((bu + static_cast<uint32_t>(b)) << 17) | c;
          }
        if (B.tid == 0) rec[0] = nrec;
        blk_publish(B, sync_word(s, 0));
        {
          // While the other units publish: list the positions of this unit's keys at or above its
          // own k-th key's bin, in token order. The segment's threshold is at or above that bin,
          // so the later passes need only these (all keys when the list would not fit).
          uint16_t* ci = cidx + q * ccap;
          const int2 kr = blk_run4(B, un);
          uint32_t c = 0;
#pragma unroll 4
          for (int x = kr.x; x < kr.y; x += 4) {
            const uint4 vv = *reinterpret_cast<const uint4*>(keys + x);
#pragma unroll
            for (int e = 0; e < 4; ++e) c += (x + e < kr.y && (vec_lane(vv, e) >> kL1Shift) >= bu) ? 1u : 0u;
          }
          uint32_t listed = 0;
          uint32_t at = blk_scan2(B, c, 0u, &listed, nullptr).x;
          const bool fits = listed <= static_cast<uint32_t>(ccap);
          if (fits && c != 0u)
            for (int x = kr.x; x < kr.y; x += 4) {
              const uint4 vv = *reinterpret_cast<const uint4*>(keys + x);
#pragma unroll
              for (int e = 0; e < 4; ++e)
                if (x + e < kr.y && (vec_lane(vv, e) >> kL1Shift) >= bu) ci[at++] = static_cast<uint16_t>(x + e);
            }
          if (B.tid == 0) ks->ncand[g][q] = fits ? static_cast<int>(listed) : -1;
        }
      }
    }
  }
  // whole segment rows: the range-end unit's when its segment is whole, and the units inside the
  // range (whole sequences), shared between the groups by parity (one loop, one copy of the code)
  const bool ex_whole = ex >= 0 && se.nunits == 1;
  const int mfirst = uf + 1 + g;
  const int nmid = mfirst < ul - 1 ? (ul - 1 - mfirst + 1) / 2 : 0;
  for (int k = 0; k < nmid + (ex_whole ? 1 : 0); ++k) {
    const int i = ex_whole ? (k == 0 ? ex : mfirst + 2 * (k - 1)) : mfirst + 2 * k;
    for (int q = q0; q < Q; q += qstep) select_local(i, q);
  }
  if (ex < 0) {
    B.sync();
    return;
  }

  // ---- B1: the threshold bin from every unit's bins; this unit's keys inside it --------------
  const DecodeUnit& u = ue;
  const int nseg = nseg_e;
  for (int q = q0; q < Q; q += qstep) {
    const SegCtx s = seg_ctx_of(u, se, ctx_e, q);
    TaskState& ts = ks->task[g][q];
    if (B.tid == 0) ts.ok = 0u;
    if (s.sg.nunits == 1 || !exchanged(s)) continue;
    const int nu = min(s.sg.nunits, kDecodeMaxCtas);
    if (!blk_wait_count(B, sync_word(s, 0), static_cast<uint32_t>(s.sg.nunits), abort_flag, p.status)) continue;
    // Every unit's records: warp w reads units w, w + warps, ... (the count, then the records, 32
    // words per coalesced load) into the histogram, and keeps its first unit's first words for the
    // second pass. A count is at most the unit's keys and the number of bins: anything else could
    // only come from a workspace that was not zero-filled, and is clamped so that every read stays
    // inside the unit's own area.
    const int nw = B.nw();
    blk_zero(B, hist, kL1Bins + 64);
    B.sync();
    auto rec_count = [&](int j, uint32_t w0) {
      const uint32_t cap = static_cast<uint32_t>(min(kL1Bins, unit_tiles(s.sg, j) * kTileKeys));
      return min(__shfl_sync(0xFFFFFFFFu, w0, 0), cap);
    };
    uint32_t first_w = 0, first_n = 0;
#pragma unroll 1
    for (int j = warp; j < nu; j += nw) {
      const uint32_t* rb = rec_of(s.sg, j, q);
      const uint32_t w0 = ldcg_u32(rb + lane);
      const uint32_t n = rec_count(j, w0);
      if (j == warp) {
        first_w = w0;
        first_n = n;
      }
#pragma unroll 1
      for (uint32_t i = lane; i <= n; i += 32) {
        const uint32_t r = i < 32 ? w0 : ldcg_u32(rb + i);
        if (i >= 1) {
          const uint32_t b = (r >> 17) & (kL1Bins - 1), c = r & 0x1FFFFu;
          smem_red_add(&hist[b], c);
          smem_red_add(&hist[kL1Bins + (b >> 6)], c);
        }
      }
    }
    B.sync();
    if (warp == 0) {
      const uint2 tb = warp_find_bin2<64, 64>(hist, hist + kL1Bins, static_cast<uint32_t>(s.kk), lane);
      if (lane == 0) {
        ts.bin = tb.x;
        ts.need = static_cast<uint32_t>(s.kk) - tb.y;
      }
    }
    uint32_t* eqpre = P + C::P_EQPRE + q * (kDecodeMaxCtas + 4);
    if (B.tid == 0) cnt[2] = 0u;
    B.sync();
    // per unit: its keys inside the bin, and the keys above the bin in the units before this one
    const uint32_t bstar = ts.bin;
    const int me = u.uidx;
#pragma unroll 1
    for (int j = warp; j < nu; j += nw) {
      const uint32_t* rb = rec_of(s.sg, j, q);
      const uint32_t w0 = j == warp ? first_w : ldcg_u32(rb + lane);
      const uint32_t n = j == warp ? first_n : rec_count(j, w0);
      uint32_t eq = 0, gt = 0;
#pragma unroll 1
      for (uint32_t i = lane; i <= n; i += 32) {
        const uint32_t r = i < 32 ? w0 : ldcg_u32(rb + i);
        if (i >= 1) {
          const uint32_t b = (r >> 17) & (kL1Bins - 1), c = r & 0x1FFFFu;
          eq += b == bstar ? c : 0u;
          gt += b > bstar ? c : 0u;
        }
      }
      eq = __reduce_add_sync(0xFFFFFFFFu, eq);
      gt = __reduce_add_sync(0xFFFFFFFFu, gt);
      if (lane == 0) {
        eqpre[j + 1] = eq;
        if (j < me && gt != 0u) atomicAdd(&cnt[2], gt);
      }
    }
    B.sync();
    // prefix of the units' bin keys over the units, by one warp
    if (warp == 0) {
      uint32_t run = 0;
#pragma unroll 1
      for (int base = 0; base < nu; base += 32) {
        const int j = base + lane;
        uint32_t incl = j < nu ? eqpre[j + 1] : 0u;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const uint32_t t = __shfl_up_sync(0xFFFFFFFFu, incl, off);
          if (lane >= off) incl += t;
        }
        if (j < nu) eqpre[j + 1] = run + incl;
        run += __shfl_sync(0xFFFFFFFFu, incl, 31);
      }
      if (lane == 0) {
        eqpre[0] = 0u;
        ts.gt_before = cnt[2];
        ts.ok = 1u;
      }
    }
    B.sync();
    // this unit's keys inside the threshold bin, low 20 bits, in token order
    const int un = clampi(s.row_end - u.kb, 0, u.ke - u.kb);
    const uint32_t* keys = lg + q * C::CAP + u.buf;
    uint32_t* dst = list_of(s.sg, u.uidx, q);
    const uint32_t my_eq = eqpre[me + 1] - eqpre[me];
    // over the listed candidate positions, or every key when the list did not fit
    const int nc = ks->ncand[g][q];
    const uint16_t* ci = cidx + q * ccap;
    auto pos = [&](int f) { return nc >= 0 ? static_cast<int>(ci[f]) : f; };
    uint32_t listed = 0;
    {
      const int2 kr = blk_run(B, nc >= 0 ? nc : un);
      uint32_t c = 0;
#pragma unroll 4
      for (int f = kr.x; f < kr.y; ++f) c += (keys[pos(f)] >> kL1Shift) == bstar ? 1u : 0u;
      uint32_t at = blk_scan2(B, c, 0u, &listed, nullptr).x;
      if (c != 0u)
#pragma unroll 1
        for (int f = kr.x; f < kr.y; ++f) {
          const uint32_t k = keys[pos(f)];
          if ((k >> kL1Shift) == bstar) {
            if (at < my_eq) dst[at] = k & 0xFFFFFu;
            ++at;
          }
        }
    }
    if (B.tid == 0 && listed != my_eq) set_status(p.status, IDX_FP4_DEV_SYNC);
    blk_publish(B, sync_word(s, 1));
  }
  B.sync();  // every row's task state is settled

  // ---- B2: the exact threshold from every unit's bin keys; this unit's selected keys ---------
  for (int q = q0; q < Q; q += qstep) {
    const SegCtx s = seg_ctx_of(u, se, ctx_e, q);
    const TaskState& ts = ks->task[g][q];
    if (ts.ok == 0u) continue;
    const int nu = min(s.sg.nunits, kDecodeMaxCtas);
    if (!blk_wait_count(B, sync_word(s, 1), static_cast<uint32_t>(s.sg.nunits), abort_flag, p.status)) continue;
    // Every unit is past its wait on the second count once all have counted themselves here; the
    // last one then clears the row's counters. With one segment nothing else depends on this ticket,
    // so one thread takes it now and its answer is read at the end (with several segments the
    // ticket also orders the segment lists before the sequence merge, and is taken after them).
    bool last_done = false;
    if (nseg <= 1 && B.tid == 0)
      last_done = atom_add_acq_rel_gpu(sync_word(s, 2), 1u) + 1u == static_cast<uint32_t>(s.sg.nunits);
    const uint32_t* eqpre = P + C::P_EQPRE + q * (kDecodeMaxCtas + 4);
    const int me = u.uidx;
    const int L = static_cast<int>(eqpre[nu]);
    auto src = [&](int x) {
      int lo = 0, hi = nu - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (static_cast<int>(eqpre[mid]) <= x) lo = mid; else hi = mid - 1;
      }
      return list_of(s.sg, lo, q) + (x - static_cast<int>(eqpre[lo]));
    };
    uint32_t* list = P + C::P_LIST;
    const bool staged = L <= C::LIST_CAP;
    blk_zero(B, hist, kL1Bins + 64);  // the levels' histograms (ordered by the barrier below)
    if (!staged) B.sync();
    if (staged) {
      // warp w copies the lists of units w, w + warps, ... (coalesced, loads issued ahead)
      for (int j = warp; j < nu; j += B.nw()) {
        const int a = static_cast<int>(eqpre[j]), n = static_cast<int>(eqpre[j + 1]) - a;
        const uint32_t* from = list_of(s.sg, j, q);
        for (int x0 = 0; x0 < n; x0 += 128) {
          uint32_t r[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int x = x0 + e * 32 + lane;
            r[e] = x < n ? ldcg_u32(from + x) : 0u;
          }
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int x = x0 + e * 32 + lane;
            if (x < n) list[a + x] = r[e];
          }
        }
      }
      B.sync();
    }
    auto low = [&](int x) { return staged ? list[x] : (ldcg_u32(src(x)) & 0xFFFFFu); };
    // Two radix levels (10 + 10 bits) inside the bin. The second level's pass also counts, for the
    // offset of this unit's output, the earlier units' keys above the first level's digit, and
    // histograms the low digits of the earlier units' and this unit's keys at that digit; the four
    // histograms sit in the record histogram's words (zeroed before the lists were staged).
    uint32_t* lv0 = hist;             // [1024 + 32] first digit, fine and coarse
    uint32_t* lv1 = hist + 1056;      // [1024 + 32] second digit of the keys at the first
    uint32_t* h1e = hist + 2112;      // [1024] second digit, earlier units, at the first
    uint32_t* h1m = hist + 3136;      // [1024] second digit, this unit, at the first
    uint32_t* r2 = B.sc + 80;         // the levels' results, shared with the block
    const int e0 = static_cast<int>(eqpre[me]), e1 = static_cast<int>(eqpre[me + 1]);
#pragma unroll 4
    for (int x = B.tid; x < L; x += B.nt) {
      const uint32_t d = low(x) >> 10;
      smem_red_add(&lv0[d], 1u);
      smem_red_add(&lv0[1024 + (d >> 5)], 1u);
    }
    if (B.tid == 0) r2[4] = 0u;
    B.sync();
    if (warp == 0) {
      const uint2 r = warp_find_bin2<32, 32>(lv0, lv0 + 1024, ts.need, lane);
      if (lane == 0) {
        r2[0] = r.x;
        r2[1] = r.y;
      }
    }
    B.sync();
    const uint32_t t0 = r2[0];
    uint32_t need = ts.need - r2[1];
    uint32_t a_gt0 = 0;  // earlier units' keys above the first digit
#pragma unroll 4
    for (int x = B.tid; x < L; x += B.nt) {
      const uint32_t l = low(x);
      const uint32_t d0 = l >> 10, d1 = l & 1023u;
      if (d0 == t0) {
        smem_red_add(&lv1[d1], 1u);
        smem_red_add(&lv1[1024 + (d1 >> 5)], 1u);
        if (x < e0) smem_red_add(&h1e[d1], 1u);
        else if (x < e1) smem_red_add(&h1m[d1], 1u);
      }
      a_gt0 += x < e0 && d0 > t0 ? 1u : 0u;
    }
    a_gt0 = __reduce_add_sync(0xFFFFFFFFu, a_gt0);
    if (lane == 0 && a_gt0 != 0u) atomicAdd(&r2[4], a_gt0);
    B.sync();
    if (warp == 0) {
      const uint2 r = warp_find_bin2<32, 32>(lv1, lv1 + 1024, need, lane);
      uint32_t above = 0;  // earlier units' keys at the first digit, above the second
#pragma unroll 8
      for (int k = 0; k < 32; ++k) {
        const uint32_t b = static_cast<uint32_t>(lane * 32 + k);
        above += b > r.x ? h1e[b] : 0u;
      }
      above = __reduce_add_sync(0xFFFFFFFFu, above);
      if (lane == 0) {
        r2[0] = (t0 << 10) | r.x;  // low 20 bits of T
        r2[1] = r.y;               // keys of the first digit above T
        r2[2] = r2[4] + above;     // earlier units' keys above T (inside the bin)
        r2[3] = h1e[r.x];          // earlier units' keys equal to T
        r2[5] = h1m[r.x];          // this unit's keys equal to T
      }
    }
    B.sync();
    const uint32_t tlow = r2[0];
    need -= r2[1];
    if (B.tid == 0) {
      cnt[0] = r2[2];
      cnt[1] = r2[3];
      cnt[3] = r2[5];
    }
    B.sync();
    const uint32_t T = (ts.bin << kL1Shift) | tlow;
    const uint32_t eq_before = cnt[1];
    const uint32_t take = need > eq_before ? min(need - eq_before, cnt[3]) : 0u;
    const uint32_t off = ts.gt_before + cnt[0] + min(eq_before, need);
    // this unit's selected keys in token order, at `off`
    const int un = clampi(s.row_end - u.kb, 0, u.ke - u.kb);
    const uint32_t* keys = lg + q * C::CAP + u.buf;
    const RowOut out = seg_out(p, ws, s, nseg, Q);
    {
      // over the listed candidate positions, or every key when the list did not fit
      const int nc = ks->ncand[g][q];
      const uint16_t* ci = cidx + q * ccap;
      auto pos_of = [&](int f) { return nc >= 0 ? static_cast<int>(ci[f]) : f; };
      const int2 run = blk_run(B, nc >= 0 ? nc : un);
      uint32_t gt = 0, eq = 0;
#pragma unroll 4
      for (int f = run.x; f < run.y; ++f) {
        const uint32_t k = keys[pos_of(f)];
        gt += k > T ? 1u : 0u;
        eq += k == T ? 1u : 0u;
      }
      const uint2 pre = blk_scan2(B, gt, eq, nullptr, nullptr);
      uint32_t pos = off + pre.x + min(pre.y, take), eqr = pre.y;
      if (gt + eq != 0u)
#pragma unroll 1
        for (int f = run.x; f < run.y; ++f) {
          const int x = pos_of(f);
          const uint32_t k = keys[x];
          const bool eqk = k == T;
          if (k > T || (eqk && eqr < take)) out(pos++, k, u.kb + x);
          eqr += eqk ? 1u : 0u;
        }
    }
    if (nseg > 1) {
      finish_exchange(s);
    } else if (last_done) {
      *sync_word(s, 0) = 0u;
      *sync_word(s, 1) = 0u;
      *sync_word(s, 2) = 0u;
    }
  }
  B.sync();
  const int pending = ks->pending[g];
  for (int k = 0; k < pending; ++k) {
    const int code = ks->pending_seq[g][k];
    merge_sequence<H, Q>(p, v, ws, code / kMaxNextN, code % kMaxNextN, P, B);
  }
  B.sync();
}

template <int H, int Q>
__global__ void __launch_bounds__(DecodeCfg<H, Q>::THREADS, 1) decode_kernel(const __grid_constant__ DecodeParams p) {
  using C = DecodeCfg<H, Q>;
  extern __shared__ __align__(1024) uint8_t smem[];
  KernelShared* ks = reinterpret_cast<KernelShared*>(smem + C::OFF_KS);
  if (threadIdx.x == 0) {
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
    for (int s = 0; s < 2 * C::STAGES + C::ACC; ++s) mbar_init(&bars[s], 1);  // full, empty, acc_full
    for (int x = 0; x < C::ACC * C::REL_RING; ++x) mbar_init(&bars[2 * C::STAGES + C::ACC + x], 4);
    mbar_init(&bars[C::BAR_QREADY], 1);
    mbar_init(&bars[C::BAR_QREADY + 1], 1);
    mbar_init(&bars[C::BAR_QFREE], C::STAGES);
    mbar_init(&bars[C::BAR_QFREE + 1], C::STAGES);
    ks->abort = 0;
    mbar_fence_init();
  }
  pdl_wait();
  pdl_trigger();

  // The schedule must belong to this call and the workspace must hold its layout (checks uniform
  // across the grid; nothing is allocated yet).
  {
    const DecodeSchedHeader h = *static_cast<const DecodeSchedHeader*>(p.sched);
    const DecodeCaps caps = decode_caps_of(h);
    const bool ok = (smem_addr(smem) & 1023u) == 0u && h.magic == kDecodeMagic &&
                    h.ctas == static_cast<int>(gridDim.x) && h.batch == p.batch && h.next_n == Q &&
                    h.max_batch >= h.batch && decode_sched_bytes_for(h.max_batch, caps) <= p.sched_bytes;
    if (!ok) {
      if (threadIdx.x == 0 && blockIdx.x == 0) set_status(p.status, IDX_FP4_DEV_BAD_SCHEDULE);
      return;
    }
    const bool ws_ok = decode_ws_bytes_for(caps, h.max_batch, Q, p.topk) <= p.ws_bytes;
    const DecodeSchedView v = sched_view(p, h);
    // Rows with no keys (or nothing to run) come out empty; the schedule must match the contexts.
    for (int b = blockIdx.x; b < p.batch; b += gridDim.x) {
      if (threadIdx.x == 0 && p.ctx_lens[b] >= 0 && p.ctx_lens[b] != v.seq_ctx[b])
        set_status(p.status, IDX_FP4_DEV_BAD_SCHEDULE);
      if (v.seq_nseg[b] == 0 || !ws_ok || h.ok == 0)
        for (int x = threadIdx.x; x < Q * p.topk; x += C::THREADS) {
          const int64_t at = static_cast<int64_t>(b) * Q * p.topk + x;
          p.topk_idx[at] = -1;
          if (p.topk_val != nullptr) p.topk_val[at] = -__int_as_float(0x7f800000);
        }
    }
    if (!ws_ok) {
      if (threadIdx.x == 0 && blockIdx.x == 0) set_status(p.status, IDX_FP4_DEV_CAPACITY);
      return;
    }
    if (h.ok == 0 || h.rounds == 0) return;
    if (threadIdx.x == 0) ks->h = h;
  }
  const int warp = static_cast<int>(threadIdx.x >> 5), lane = static_cast<int>(threadIdx.x & 31);
  if (warp == C::EPI_WARP0) tmem_alloc(&ks->tmem, C::TMEM_COLS);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  // Rounds: the epilogue warps publish each round's range; the stage warps stream its tiles and the
  // epilogue warps read them out; then every warp, in two selection groups, selects the round's
  // units. Register budgets are re-split for the stream and evened out for the selection.
  const int rounds = ks->h.rounds;
  const bool stage_role = warp < C::STAGE_WARPS;
  int tiles = 0, units = 0;  // streamed in earlier rounds (kept by every epilogue thread alike)
  for (int r = 0; r < rounds; ++r) {
    const int slot = r & 1;
    if (stage_role) {
      warpgroup_regs_dec<C::STAGE_REGS>();
      named_barrier_sync(kAllBarrier, C::THREADS);
      if (warp < C::STAGES && ks->round[slot].uf < ks->round[slot].ul) stream_stage_warp<H, Q>(p, smem, slot, warp, lane);
      warpgroup_regs_inc<C::LAUNCH_REGS>();
    } else {
      warpgroup_regs_inc<C::EPI_REGS>();
      const int etid = static_cast<int>(threadIdx.x) - C::EPI_WARP0 * 32;
      const DecodeSchedView v = sched_view(p, ks->h);
      const int ri = r * ks->h.ctas + static_cast<int>(blockIdx.x);
      const int uf = v.range_first[ri], ul = v.range_first[ri + 1];
      if (etid == 0) ks->round[slot] = RoundInfo{uf, ul, tiles, units};
      named_barrier_sync(kAllBarrier, C::THREADS);
      if (uf < ul) {
        stream_epilogue_warp<H, Q>(p, smem, slot, warp - C::EPI_WARP0, lane);
        for (int i = uf; i < ul; ++i) tiles += dunit_tiles(v.units[i]);
        units += ul - uf;
      }
      warpgroup_regs_dec<C::LAUNCH_REGS>();
    }
    // every tile is read out: the stage area is free and the row buffer complete
    named_barrier_sync(kAllBarrier, C::THREADS);
    if (ks->round[slot].uf < ks->round[slot].ul) {
      // A range inside one sequence (one unit) is selected by every warp of the CTA, as group 0;
      // otherwise the stage warps (group 0) and the epilogue warps (group 1) select side by side.
      // One call site, so the selection's code is laid out once.
      // With several rows, a one-unit range is split by rows between the two groups instead.
      const bool one_unit = ks->round[slot].ul - ks->round[slot].uf == 1;
      const bool whole = one_unit && Q == 1;
      const bool row_split = one_unit && Q > 1;
      const int g = whole || stage_role ? 0 : 1;
      const int gtid = static_cast<int>(threadIdx.x) - (g == 0 ? 0 : C::EPI_WARP0 * 32);
      const Blk B{whole ? static_cast<int>(threadIdx.x) : gtid, whole ? C::THREADS : C::THREADS / 2,
                  g == 0 ? kSelBarrier0 : kSelBarrier1, reinterpret_cast<uint32_t*>(smem + C::OFF_SCR) + g * 128};
      select_round<H, Q>(p, smem, slot, g, B, row_split);
    }
    fence_proxy_async_smem();  // the selection's writes to the stage area precede the next bulk copies
    named_barrier_sync(kAllBarrier, C::THREADS);
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == C::EPI_WARP0) {
    tc_fence_after_sync();
    tmem_dealloc(ks->tmem, C::TMEM_COLS);
  }
}

}  // namespace

template <int H, int Q>
static cudaError_t launch_decode_t(const DecodeParams& p, int grid, cudaStream_t stream) {
  using C = DecodeCfg<H, Q>;
  cudaError_t e = set_smem_once<decode_kernel<H, Q>>(C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  return launch_pdl(decode_kernel<H, Q>, dim3(grid), dim3(C::THREADS), C::SMEM_BYTES, stream, 1, true, p);
}


}  // namespace idxfp4
