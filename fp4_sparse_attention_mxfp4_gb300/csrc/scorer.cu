// Scorer: MXFP4 keys x MXFP4 query heads on tcgen05 block-scaled MMA, fused head-weighted
// ReLU reduction, fused exact top-k. Shared by decode (one query row per unit) and prefill
// (up to two rows of one request per unit).
//
// Method ("Score a DSA sparse indexer in FP4", squashed commit message and PR body):
//   logit[q, t] = sum_h w[q, h] * relu(q_h . k_t), keys read in place from the paged two-plane
//   FP4 index region; the decode top-k is bounded by the row's context and the prefill top-k by
//   the row's [0, row_end) range.
//
// GB300 design (the pages' kernels target MI355X MFMA; this is a fresh design):
//   * A 128-key tile (two pages) is the MMA M dimension, query rows x heads the N dimension:
//     D[128 x N] = K[128 x 128] . Q^T, as two K=64 tcgen05.mma kind::mxf4 block-scaled MMAs
//     accumulating fp32 in TMEM. TMEM lane = key, so the head sum is thread-local.
//   * Eight producer warps each own one stage of an 8-stage ring and fill it with 1-D bulk TMA
//     copies (cp.async.bulk), the ten copies of a tile spread over ten lanes: a page's four 1 KB
//     group chunks land interleaved with the tile's other page, which makes the stage a canonical
//     no-swizzle K-major operand (LBO 2048 B between 32-dim chunks, SBO 128 B between 8-key
//     groups). Bulk copies issued by one warp are processed one after another, so the stream
//     rate grows with the number of issuing warps; eight reach the HBM copy rate.
//   * One MMA warp rebuilds each stage's scale bytes from the cache's 16x4-transposed order into
//     the tensor core's scale-factor layout (key m at lane m%32, column m/32), copies them to
//     TMEM with tcgen05.cp and issues the MMAs; tcgen05.commit frees the stage and hands the
//     accumulator to the epilogue.
//   * Four epilogue warps (one per TMEM lane quarter) read the accumulator with tcgen05.ld, form
//     each key's logit in a fixed order, store its order-preserving key in a shared-memory row
//     buffer and count it in a per-warp histogram. At the end of a unit an exact radix select
//     finds the k-th key and a stable pass writes the selected keys in token order. The logit
//     row never reaches global memory (unless a debug buffer is passed).
//   * Persistent grid, one CTA per SM; every on-chip wait is bounded and reports a timeout in the
//     status word instead of hanging.
#include <cuda_runtime.h>

#include <cstdint>

#include "common.cuh"
#include "ptx.cuh"
#include "topk.cuh"

namespace idxfp4 {
namespace {

constexpr uint32_t kEpiBarrier = 1;

template <int H, int Q>
struct ScorerCfg {
  static constexpr int N = H * Q;
  static constexpr int ACC = N <= 64 ? 6 : 2;  // TMEM accumulators (even: a tile's group is fixed by it)
  static constexpr int STAGES = 12;            // tiles in flight; one stage warp per stage
  static constexpr int EPI_WARP0 = STAGES;
  static constexpr int EPI_WARPS = 8;          // two groups of four (one warp per lane quarter)
  static constexpr int EPI_THREADS = EPI_WARPS * 32;
  static constexpr int THREADS = (STAGES + EPI_WARPS) * 32;
  static constexpr int UCAP = unit_key_cap(Q);   // keys per unit and row (row buffer size)
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t SFA_COL = ACC * N;             // STAGES chunks of 4 columns
  static constexpr uint32_t SFB_COL = SFA_COL + 4 * STAGES;  // 2 chunks of 4 columns (unit parity)
  static_assert(ACC % 2 == 0, "tiles sharing an accumulator belong to one epilogue group");
  static_assert(SFB_COL + 8 <= TMEM_COLS, "accumulators and scale chunks fit the allocation");
  static_assert(UCAP % kTileKeys == 0, "whole tiles per unit");
  // shared memory map (offsets from a 1024-byte aligned base)
  static constexpr uint32_t OFF_PACKED = 0;                              // [STAGES][4][128][16]
  static constexpr uint32_t OFF_SFA = OFF_PACKED + STAGES * 8192;        // [STAGES][512] tensor-core layout
  static constexpr uint32_t OFF_QB = OFF_SFA + STAGES * 512;             // [2][4][N][16]
  static constexpr uint32_t OFF_SFB = OFF_QB + 2 * N * 64;               // [2][512]
  static constexpr uint32_t OFF_W = OFF_SFB + 2 * 512;                   // [2][N] head weights
  static constexpr uint32_t OFF_LG = OFF_W + 2 * N * 4;                  // [Q][UCAP] ordered keys
  static constexpr uint32_t OFF_HW = OFF_LG + Q * UCAP * 4;              // [Q][4 quarters][1024] packed counts
  static constexpr uint32_t OFF_HIST = OFF_HW + Q * 4 * kHistWords * 4;  // [2048]
  static constexpr uint32_t OFF_SCR = OFF_HIST + 2048 * 4;               // [64]
  // Release barriers per accumulator, used in turn. A stage warp's tiles all use one accumulator,
  // STAGES / ACC of its tiles apart; with this many barriers the one it waits on has always seen
  // the completion before the awaited one.
  static constexpr int REL_RING = STAGES / ACC + 2;
  static_assert(STAGES % ACC == 0, "a stage warp keeps to one accumulator");
  static constexpr uint32_t NUM_BARS = 2 * STAGES + ACC + ACC * REL_RING + 2;
  static constexpr uint32_t OFF_BAR = OFF_SCR + 64 * 4;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NUM_BARS * 8;
  static constexpr uint32_t SMEM_BYTES = OFF_MISC + 64;
  static_assert(SMEM_BYTES <= 227 * 1024, "fits one SM");
  static_assert(OFF_LG % 16 == 0 && OFF_SFA % 16 == 0 && OFF_QB % 128 == 0, "operand and row-buffer alignment");
};

struct ScorerParams {
  const uint8_t* q_packed;
  const uint8_t* q_scale;
  const float* weights;
  const uint8_t* kv_packed;
  const uint8_t* kv_scale;
  int64_t num_pages;
  const int32_t* block_tables;
  int bt_stride;
  // unit list: decode (sched != nullptr) uses the schedule's per-CTA table; prefill strides
  // over the workspace's unit list by the grid
  const void* sched;
  size_t sched_bytes;
  const PrefillSchedHeader* prefill;
  int expect_batch;
  const int32_t* row_ends;       // prefill per-row key ends (nullptr: the unit's ke)
  int topk;
  int32_t* topk_idx;
  float* topk_val;
  uint2* cand;                   // candidate slots (see cand_slot_entries)
  int64_t cand_slots;            // slots the caller's buffer holds
  float* logits_debug;
  int64_t logits_stride;
  int32_t* status;
  int stream_once;               // 1: keys are read once (decode) -> L2 evict-first
};

struct UnitIter {
  const Unit* units;
  int first, count, stride;
  bool ok;
  __device__ __forceinline__ Unit at(int i) const { return units[first + i * stride]; }
};

// This CTA's units; `ok` is false when the schedule does not belong to this call.
__device__ __forceinline__ UnitIter unit_range(const ScorerParams& p) {
  UnitIter it{};
  const int c = blockIdx.x;
  if (p.sched != nullptr) {
    const DecodeSchedHeader* h = static_cast<const DecodeSchedHeader*>(p.sched);
    it.ok = h->magic == kDecodeMagic && h->ctas == static_cast<int>(gridDim.x) && h->batch == p.expect_batch &&
            h->max_batch >= h->batch && decode_sched_bytes_for(h->max_batch, h->units_cap) <= p.sched_bytes;
    if (!it.ok) return it;
    const DecodeSchedView v = decode_sched_view(const_cast<void*>(p.sched), h->max_batch);
    it.units = v.units;
    it.first = v.cta_first[c];
    it.count = v.cta_count[c];
    it.stride = 1;
  } else {
    it.ok = p.prefill->magic == kPrefillMagic;
    if (!it.ok) return it;
    const int n = p.prefill->num_units;
    it.units = reinterpret_cast<const Unit*>(reinterpret_cast<const char*>(p.prefill) +
                                             prefill_units_offset(p.prefill->num_rows));
    it.first = c;
    it.count = c < n ? (n - c + static_cast<int>(gridDim.x) - 1) / static_cast<int>(gridDim.x) : 0;
    it.stride = gridDim.x;
  }
  return it;
}

__device__ __forceinline__ int unit_tiles(const Unit& u) {
  return u.ke > u.kb ? (u.ke - u.kb + kTileKeys - 1) / kTileKeys : 0;
}

// Position in this CTA's tile sequence: unit i (of the CTA's list), tile j of that unit.
struct Cursor {
  int i, j, nt;
  Unit u;
};

// Move `steps` tiles forward (skipping units without tiles); false once past the last tile.
__device__ __forceinline__ bool cursor_advance(Cursor& c, int steps, const UnitIter& it) {
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
        c.nt = unit_tiles(c.u);
      }
    }
  }
  return c.i < it.count;
}

// Slow path of a wait: bounded spin; a timeout raises the CTA's abort flag and the status bit,
// after which every later wait of the CTA returns at once.
__device__ __noinline__ bool wait_slow(uint64_t* bar, uint32_t parity, volatile int* abort_flag, int32_t* status) {
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

// Page id of the tile at cursor c: lane 0 reads the tile's first page, lane 1 its second (or -1
// if the tile has one page). A logical page past the table width reads nothing and gives -2.
__device__ __forceinline__ int load_tile_page(const ScorerParams& p, const Cursor& c, int lane) {
  const int lp = c.u.kb / kPage + 2 * c.j + lane;
  const bool needed = lane == 0 || (lane == 1 && c.u.kb + c.j * kTileKeys + kPage < c.u.ke);
  if (!needed) return -1;
  if (lp >= p.bt_stride) return -2;
  return p.block_tables[static_cast<int64_t>(c.u.table) * p.bt_stride + lp];
}

template <int H, int Q>
__global__ void __launch_bounds__(ScorerCfg<H, Q>::THREADS, 1) scorer_kernel(const __grid_constant__ ScorerParams p) {
  using C = ScorerCfg<H, Q>;
  constexpr int N = C::N, ACC = C::ACC, STAGES = C::STAGES;
  // The dynamic shared memory is used through this base directly: pointers derived from it keep
  // the shared state space, so accesses compile to shared-memory instructions.
  extern __shared__ __align__(1024) uint8_t smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // Schedule checks (uniform across the grid; nothing is allocated yet).
  const UnitIter it = unit_range(p);
  if (!it.ok || (smem_addr(smem) & 1023u) != 0u) {
    if (tid == 0 && blockIdx.x == 0) set_status(p.status, IDX_FP4_DEV_BAD_SCHEDULE);
    return;
  }

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* full_bar = bars;                  // stage data landed (TMA transaction count)
  uint64_t* empty_bar = bars + STAGES;        // stage consumed by its MMAs (tcgen05.commit)
  uint64_t* acc_full = bars + 2 * STAGES;     // accumulator written (tcgen05.commit)
  // Release of an accumulator after its j-th tile: acc_rel[a * REL_RING + j % REL_RING]. Tiles of
  // one accumulator are issued by different stage warps, so an issuer skips phases of the
  // accumulator's sequence; spread over REL_RING barriers, the one it waits on is never two
  // phases behind, which keeps parity waits exact.
  uint64_t* acc_rel = acc_full + ACC;
  uint64_t* q_ready = acc_rel + ACC * C::REL_RING;  // unit query operand in place (tcgen05.commit)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);

  if (tid == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int a = 0; a < ACC; ++a) mbar_init(&acc_full[a], 1);
    for (int x = 0; x < ACC * C::REL_RING; ++x) mbar_init(&acc_rel[x], 4);
    mbar_init(&q_ready[0], 1);
    mbar_init(&q_ready[1], 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  {
    uint32_t* hw = reinterpret_cast<uint32_t*>(smem + C::OFF_HW);
    for (int x = tid; x < Q * 4 * kHistWords; x += C::THREADS) hw[x] = 0u;
  }
  if (warp == 0) tmem_alloc(tmem_slot, C::TMEM_COLS);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  if (warp < STAGES) {
    // ---------------- stage warps: warp w streams tiles w, w+12, ... through stage w and issues
    // their MMAs. Issue work is spread over twelve warps because a bulk copy or a tcgen05
    // instruction occupies its issuing warp or thread for a long time; one stage per warp also
    // keeps every wait on a barrier this warp alone advances.
    const int ps = warp;
    const uint64_t pol = policy_evict_first();
    uint8_t* stage = smem + C::OFF_PACKED + ps * 8192;
    uint8_t* sfa_s = smem + C::OFF_SFA + ps * 512;
    const uint64_t a_desc = smem_desc(smem_addr(stage), 2048, 128);
    const uint32_t sfa_t = tmem + C::SFA_COL + 4u * static_cast<uint32_t>(ps);
    const uint32_t idesc0 = mxf4_idesc(128, N, 0), idesc2 = mxf4_idesc(128, N, 2);
    // Scale plane words of this lane: the 16x4 row transpose puts rows l%16 + 16*b at byte b of
    // word l%16, so lane l takes byte l/16 (rows l, l+64 of the tile) and byte 2 + l/16 (rows
    // l+32, l+96) of each group's word; a tile row m goes to TMEM lane m%32, column m/32.
    const uint32_t sel_lo = static_cast<uint32_t>(lane >> 4), sel_hi = sel_lo + 2u;
    const uint32_t perm_lo = sel_lo | ((sel_lo + 4u) << 4), perm_hi = sel_hi | ((sel_hi + 4u) << 4);
    Cursor c{0, 0, 0, Unit{}};
    bool have = it.count > 0;
    if (have) {
      c.u = it.at(0);
      c.nt = unit_tiles(c.u);
      have = cursor_advance(c, ps, it);
    }
    int entry = have ? load_tile_page(p, c, lane) : -1;
    int f = ps;
    int qnext = 0;  // next unit whose query operand this warp has waited for
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
      // the previous tile's MMAs (and its scale copy) are done with the stage
      if (lane == 0) {
        bounded_wait(&empty_bar[ps], ((f / STAGES) & 1) ^ 1, abort_flag, p.status);
        mbar_arrive_expect_tx(&full_bar[ps], (has1 ? 2u : 1u) * kPageBytes);
      }
      __syncwarp();
      // lanes 0..3: group chunks of page 0; lanes 4..7: page 1. A page's chunk g lands at
      // g * 2048 + page * 1024, which makes the stage a canonical no-swizzle K-major operand.
      if (lane < 8 && (lane < 4 || has1)) {
        const int pg = lane >> 2, k = lane & 3;
        const int64_t pid = pg == 0 ? pid0 : pid1;
        uint8_t* dst = stage + k * 2048 + pg * 1024;
        const uint8_t* src = p.kv_packed + pid * kPageBytes + k * 1024;
        if (p.stream_once)
          bulk_load_evict_first(dst, src, 1024, &full_bar[ps], pol);
        else
          bulk_load(dst, src, 1024, &full_bar[ps]);
      }
      // scale bytes: plain loads, in flight together with the bulk copies
      uint32_t w0[4], w1[4];
      {
        const uint32_t* s0 = reinterpret_cast<const uint32_t*>(p.kv_scale + static_cast<int64_t>(pid0) * kPageScaleBytes) + (lane & 15);
        const uint32_t* s1 = reinterpret_cast<const uint32_t*>(p.kv_scale + static_cast<int64_t>(pid1 < 0 ? 0 : pid1) * kPageScaleBytes) + (lane & 15);
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          w0[g] = __ldg(s0 + 16 * g);
          w1[g] = has1 ? __ldg(s1 + 16 * g) : 0x7F7F7F7Fu;
        }
      }
      // the next tile of this stage: its page ids load while this one streams
      Cursor nc = c;
      const bool next = cursor_advance(nc, STAGES, it);
      const int next_entry = next ? load_tile_page(p, nc, lane) : -1;
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
        while (qnext <= c.i) {
          bounded_wait(&q_ready[qnext & 1], (qnext >> 1) & 1, abort_flag, p.status);
          ++qnext;
        }
        const int a = f % ACC, jf = f / ACC;
        if (jf >= 1)  // the accumulator's previous tile has been read out
          bounded_wait(&acc_rel[a * C::REL_RING + (jf - 1) % C::REL_RING],
                       static_cast<uint32_t>((jf - 1) / C::REL_RING) & 1u, abort_flag, p.status);
        tc_fence_after_sync();
        const int par = c.i & 1;
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
      c = nc;
      have = next;
      entry = next_entry;
      f += STAGES;
    }
    // Teardown waits for this warp's last copies and MMAs (they normally finished long ago).
    if (lane == 0 && f - STAGES >= 0) {
      mbar_wait(&full_bar[ps], ((f - STAGES) / STAGES) & 1, kWaitLimitNs);
      mbar_wait(&empty_bar[ps], ((f - STAGES) / STAGES) & 1, kWaitLimitNs);
    }
    __syncwarp();
  } else {
    // ---------------- epilogue: head-weighted ReLU sum, row buffer, exact top-k ----------------
    // Two groups of four warps (one per TMEM lane quarter) take alternate tiles; the epilogue also
    // lays out each unit's query operand and weights, two units ahead.
    const int e = warp - C::EPI_WARP0;
    const int grp = e >> 2;                 // tile parity handled by this warp's group
    const int qtr = warp & 3;               // TMEM lane quarter of this warp
    const int etid = e * 32 + lane;         // rank in the 256-thread epilogue group
    const int krow = qtr * 32 + lane;       // key row within the tile
    const uint32_t lane_base = static_cast<uint32_t>(qtr * 32) << 16;
    uint32_t* lg_base = reinterpret_cast<uint32_t*>(smem + C::OFF_LG);
    uint32_t* hw_base = reinterpret_cast<uint32_t*>(smem + C::OFF_HW);
    uint32_t* hist = reinterpret_cast<uint32_t*>(smem + C::OFF_HIST);
    uint32_t* scr = reinterpret_cast<uint32_t*>(smem + C::OFF_SCR);
    // Query heads of unit i -> canonical K-major [4 chunks][N][16 B] operand (rows past the unit's
    // live rows zeroed), query scales -> the tensor core's scale layout (row n at line n%32, word
    // n/32), weights -> plain floats; then one thread copies the scales to TMEM and commits.
    // The buffers of parity i&1 are free: the unit that used them last has been fully consumed.
    auto prep = [&](int i) {
      const Unit u = it.at(i);
      const int par = i & 1;
      const int live = u.nq * H;
      uint8_t* qb = smem + C::OFF_QB + par * (N * 64);
      uint8_t* sfb = smem + C::OFF_SFB + par * 512;
      float* wq = reinterpret_cast<float*>(smem + C::OFF_W) + par * N;
      const uint8_t* qsrc = p.q_packed + static_cast<int64_t>(u.row) * H * 64;
      for (int cc = etid; cc < 4 * N; cc += C::EPI_THREADS) {
        const int g = cc / N, n = cc % N;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (n < live) v = __ldg(reinterpret_cast<const uint4*>(qsrc + n * 64 + g * 16));
        *reinterpret_cast<uint4*>(qb + g * N * 16 + n * 16) = v;
      }
      for (int n = etid; n < 128; n += C::EPI_THREADS) {
        uint32_t wv = 0x7F7F7F7Fu;
        if (n < live) wv = __ldg(reinterpret_cast<const uint32_t*>(p.q_scale + (static_cast<int64_t>(u.row) * H + n) * 4));
        *reinterpret_cast<uint32_t*>(sfb + (n & 31) * 16 + (n >> 5) * 4) = wv;
      }
      for (int x = etid; x < N; x += C::EPI_THREADS)
        wq[x] = x < live ? __ldg(p.weights + static_cast<int64_t>(u.row) * H + x) : 0.f;
      fence_proxy_async_smem();
      named_barrier_sync(kEpiBarrier, C::EPI_THREADS);
      if (etid == 0) {
        tc_fence_after_sync();
        tmem_copy_sf_chunk(tmem + C::SFB_COL + 4u * static_cast<uint32_t>(par), smem_addr(sfb));
        tc_commit(&q_ready[par]);
      }
    };
    if (it.count > 0) prep(0);
    if (it.count > 1) prep(1);
    int t0 = 0;
    for (int i = 0; i < it.count; ++i) {
      const Unit u = it.at(i);
      const int upar = i & 1;
      const float* wsm = reinterpret_cast<const float*>(smem + C::OFF_W) + upar * N;
      int end[Q];
#pragma unroll
      for (int r = 0; r < Q; ++r) {
        int ee = 0;
        if (r < u.nq) ee = p.row_ends != nullptr ? min(max(p.row_ends[u.row + r], 0), u.ke) : u.ke;
        end[r] = ee;
      }
      const int ntiles = unit_tiles(u);
      for (int j = (grp - t0) & 1; j < ntiles; j += 2) {
        const int tt = t0 + j;
        const int a = tt % ACC;
        bounded_wait(&acc_full[a], static_cast<uint32_t>(tt / ACC) & 1u, abort_flag, p.status);
        tc_fence_after_sync();
        float logit[Q];
#pragma unroll
        for (int r = 0; r < Q; ++r) {
          float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f, s4 = 0.f, s5 = 0.f, s6 = 0.f, s7 = 0.f;
          const uint32_t col = tmem + lane_base + a * N + r * H;
          if constexpr (H == 16) {
            float v[16];
            tmem_load_x16(col, v);
#pragma unroll
            for (int h = 0; h < 16; h += 8) {
              const float4 wa = *reinterpret_cast<const float4*>(wsm + r * H + h);
              const float4 wb = *reinterpret_cast<const float4*>(wsm + r * H + h + 4);
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
#pragma unroll
            for (int cc = 0; cc < H; cc += 64) {
              float v[64];
              tmem_load_2x32(col + cc, col + cc + 32, v);
#pragma unroll
              for (int h = 0; h < 64; h += 8) {
                const float4 wa = *reinterpret_cast<const float4*>(wsm + r * H + cc + h);
                const float4 wb = *reinterpret_cast<const float4*>(wsm + r * H + cc + h + 4);
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
          } else {
#pragma unroll
            for (int cc = 0; cc < H; cc += 32) {
              float v[32];
              tmem_load_x32(col + cc, v);
#pragma unroll
              for (int h = 0; h < 32; h += 8) {
                const float4 wa = *reinterpret_cast<const float4*>(wsm + r * H + cc + h);
                const float4 wb = *reinterpret_cast<const float4*>(wsm + r * H + cc + h + 4);
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
          logit[r] = ((s0 + s1) + (s2 + s3)) + ((s4 + s5) + (s6 + s7));
        }
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_rel[a * C::REL_RING + (tt / ACC) % C::REL_RING]);
        const int rel = j * kTileKeys + krow;  // < UCAP: a unit holds at most UCAP keys
        const int key = u.kb + rel;
#pragma unroll
        for (int r = 0; r < Q; ++r) {
          const bool valid = key < end[r];
          const uint32_t uk = valid ? ordered_key(logit[r]) : 0u;
          lg_base[r * C::UCAP + rel] = uk;
          if (valid) hist16_add(hw_base + (r * 4 + qtr) * kHistWords, uk);
          if (valid && p.logits_debug != nullptr && key < p.logits_stride)
            p.logits_debug[static_cast<int64_t>(u.row + r) * p.logits_stride + key] = logit[r];
        }
      }
      t0 += ntiles;
      named_barrier_sync(kEpiBarrier, C::EPI_THREADS);
      // select each row: exactly min(k, valid keys) keys, in token order
      for (int r = 0; r < u.nq && r < Q; ++r) {
        const uint32_t* keys = lg_base + r * C::UCAP;
        const int nvalid = max(0, end[r] - u.kb);
        const int kk = min(p.topk, nvalid);
        auto load4 = [keys](int x) { return *reinterpret_cast<const uint4*>(keys + x); };
        uint32_t* hw_r = hw_base + r * 4 * kHistWords;
        const int kb = u.kb;
        if (u.slot < 0) {
          const int64_t rowoff = static_cast<int64_t>(u.row + r) * p.topk;
          int32_t* oi = p.topk_idx + rowoff;
          float* ov = p.topk_val != nullptr ? p.topk_val + rowoff : nullptr;
          select_topk<C::EPI_THREADS, 4>(load4, nvalid, kk, hw_r, hist, scr, etid, kEpiBarrier,
                                         [=](int pos, int x, uint32_t kv) {
                                           oi[pos] = kb + x;
                                           if (ov != nullptr) ov[pos] = key_to_float(kv);
                                         });
          for (int x = kk + etid; x < p.topk; x += C::EPI_THREADS) {
            oi[x] = -1;
            if (ov != nullptr) ov[x] = -__int_as_float(0x7f800000);
          }
        } else if (u.slot + r < p.cand_slots) {
          uint2* slot = p.cand + static_cast<int64_t>(u.slot + r) * static_cast<int64_t>(cand_slot_entries(p.topk));
          uint2* oc = slot + 2;
          select_topk<C::EPI_THREADS, 4>(load4, nvalid, kk, hw_r, hist, scr, etid, kEpiBarrier,
                                         [=](int pos, int x, uint32_t kv) {
                                           oc[pos] = make_uint2(kv, static_cast<uint32_t>(kb + x));
                                         });
          // odd counts get one pad entry so every list is a whole number of 16-byte pairs; key 0 is
          // below every logit and never selected
          if (etid == 0) {
            if (kk & 1) oc[kk] = make_uint2(0u, 0xFFFFFFFFu);
            slot[0] = make_uint2(static_cast<uint32_t>(kk), 0u);
          }
        } else if (etid == 0) {
          set_status(p.status, IDX_FP4_DEV_CAPACITY);
        }
      }
      // the next unit counts into cleared histograms
      for (int x = etid; x < Q * 4 * kHistWords; x += C::EPI_THREADS) hw_base[x] = 0u;
      named_barrier_sync(kEpiBarrier, C::EPI_THREADS);
      if (i + 2 < it.count) prep(i + 2);
    }
    // Teardown waits for the last scale copies into TMEM (they normally finished long ago).
    if (etid == 0)
      for (int k = it.count - 2 < 0 ? 0 : it.count - 2; k < it.count; ++k)
        mbar_wait(&q_ready[k & 1], (k >> 1) & 1, kWaitLimitNs);
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------------------------
// Merge of split rows (decode sequences spread over several units, prefill rows cut into key
// chunks): the row's candidate lists (each exactly its unit's top-min(k, keys), in token order)
// are copied into shared memory in key order and the exact selection runs over them. Also
// writes the all-padding output of decode sequences with no keys.
constexpr int kMergeThreads = 512;
constexpr int kMergeCap = 20480;    // candidate entries held at once
constexpr int kMergeKeep = kMaxTopk;
constexpr int kMergeHists = 4;      // level-1 histograms (warp w counts into w % 4)
constexpr size_t kMergeSmem = static_cast<size_t>(kMergeCap) * 8 + static_cast<size_t>(kMergeKeep) * 8 +
                              kMergeHists * kHistWords * 4 + 2048 * 4 + 64 * 4 + 64 * 4 + 2 * kMergeThreads * 4;

struct MergeParams {
  const void* sched;                 // decode: the schedule, else nullptr
  size_t sched_bytes;
  const int32_t* ctx_lens;
  int batch;
  const PrefillSchedHeader* prefill; // prefill: the workspace header, else nullptr
  int topk;
  const uint2* cand;
  int64_t cand_slots;
  int32_t* topk_idx;
  float* topk_val;
  int32_t* status;
};

__global__ void __launch_bounds__(kMergeThreads) merge_kernel(const __grid_constant__ MergeParams mp) {
  extern __shared__ __align__(1024) uint8_t msm[];
  uint2* buf = reinterpret_cast<uint2*>(msm);
  uint2* keep = buf + kMergeCap;
  uint32_t* hw = reinterpret_cast<uint32_t*>(keep + kMergeKeep);
  uint32_t* hist = hw + kMergeHists * kHistWords;
  uint32_t* scr = hist + 2048;
  uint32_t* wsum = scr + 64;  // [0, 32): warp sums of the list scan, [32]: entries of the round
  uint32_t* loff = wsum + 64;  // per list of the round: first entry in the buffer
  uint32_t* lcnt = loff + kMergeThreads;  // per list of the round: entries (even)
  const int row = blockIdx.x, tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int topk = mp.topk;
  int first, nu, stride, kk;
  if (mp.sched != nullptr) {
    const DecodeSchedHeader* h = static_cast<const DecodeSchedHeader*>(mp.sched);
    if (h->magic != kDecodeMagic || h->batch != mp.batch || h->max_batch < mp.batch ||
        decode_sched_bytes_for(h->max_batch, h->units_cap) > mp.sched_bytes)
      return;  // flagged by the scorer
    const DecodeSchedView v = decode_sched_view(const_cast<void*>(mp.sched), h->max_batch);
    const int ctx = v.seq_ctx[row];
    nu = v.seq_units[row];
    first = v.seq_first[row];
    stride = 1;
    kk = min(topk, ctx);
    if (tid == 0 && mp.ctx_lens[row] >= 0 && mp.ctx_lens[row] != ctx) set_status(mp.status, IDX_FP4_DEV_BAD_SCHEDULE);
    if (nu == 0) {
      for (int e = tid; e < topk; e += kMergeThreads) {
        mp.topk_idx[static_cast<int64_t>(row) * topk + e] = -1;
        if (mp.topk_val != nullptr) mp.topk_val[static_cast<int64_t>(row) * topk + e] = -__int_as_float(0x7f800000);
      }
      return;
    }
  } else {
    if (mp.prefill->magic != kPrefillMagic) return;
    const int4 rm = reinterpret_cast<const int4*>(mp.prefill + 1)[row];
    first = rm.x;
    nu = rm.y;
    stride = mp.prefill->rows_per_unit;
    kk = min(topk, rm.z);
  }
  if (nu <= 1) return;  // written by the scorer
  const int64_t orow = static_cast<int64_t>(row) * topk;
  const int64_t slot_entries = static_cast<int64_t>(cand_slot_entries(topk));
  auto list_count = [&](int i) {
    const int64_t s = first + static_cast<int64_t>(i) * stride;
    return s < mp.cand_slots ? min(static_cast<int>(mp.cand[s * slot_entries].x), topk) : 0;
  };
  int kept = 0, next = 0;
  while (next < nu) {
    // The next kMergeThreads lists' sizes load in parallel and a block scan gives each list its
    // offset after the kept prefix; the lists that fit form a prefix of them. A round thus costs
    // one dependent global read instead of one per list.
    const int lx = next + tid;
    const int ce = lx < nu ? (list_count(lx) + 1) & ~1 : 0;
    int incl = ce;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int v = __shfl_up_sync(0xFFFFFFFFu, incl, off);
      if (lane >= off) incl += v;
    }
    if (lane == 31) wsum[w] = incl;
    __syncthreads();
    for (int w2 = 0; w2 < w; ++w2) incl += static_cast<int>(wsum[w2]);
    const bool fits = lx < nu && kept + incl <= kMergeCap;
    const int nfit = __syncthreads_count(fits);
    if (nfit == 0) {  // cannot happen while kMergeCap >= 2 * (kMaxTopk + 1); never spin on it
      if (tid == 0) set_status(mp.status, IDX_FP4_DEV_CAPACITY);
      break;
    }
    if (tid == nfit - 1) wsum[32] = static_cast<uint32_t>(incl);
    if (fits) {
      loff[tid] = static_cast<uint32_t>(kept + incl - ce);
      lcnt[tid] = static_cast<uint32_t>(ce);
    }
    __syncthreads();
    const int last = next + nfit;
    const int total = kept + static_cast<int>(wsum[32]);
    // Every thread copies 16-byte pairs of every list: plain vector loads keep hundreds of
    // requests in flight, where bulk copies issued by one warp would move one after another.
    for (int li = 0; li < nfit; ++li) {
      const uint4* src = reinterpret_cast<const uint4*>(mp.cand + (first + static_cast<int64_t>(next + li) * stride) *
                                                                      slot_entries + 2);
      uint4* dst = reinterpret_cast<uint4*>(buf + loff[li]);
      const int pairs = static_cast<int>(lcnt[li]) >> 1;
      for (int x = tid; x < pairs; x += kMergeThreads) dst[x] = src[x];
    }
    __syncthreads();
    next = last;
    const int n = total;
    const bool final = next >= nu;
    const int kr = final ? kk : min(topk, n);
    // level-1 histograms, one per warp
    for (int wd = tid; wd < kMergeHists * kHistWords; wd += kMergeThreads) hw[wd] = 0u;
    __syncthreads();
    // n is even and the buffer holds whole 16-byte pairs: read two entries per load
    for (int x = 2 * tid; x < n; x += 2 * kMergeThreads) {
      const uint4 v = *reinterpret_cast<const uint4*>(buf + x);
      hist16_add(hw + (w % kMergeHists) * kHistWords, v.x);
      hist16_add(hw + (w % kMergeHists) * kHistWords, v.z);
    }
    __syncthreads();
    auto load4 = [buf](int x) {
      const uint4 a = *reinterpret_cast<const uint4*>(buf + x);
      const uint4 b = *reinterpret_cast<const uint4*>(buf + x + 2);
      return make_uint4(a.x, a.z, b.x, b.z);
    };
    if (final) {
      int32_t* oi = mp.topk_idx + orow;
      float* ov = mp.topk_val != nullptr ? mp.topk_val + orow : nullptr;
      select_topk<kMergeThreads, kMergeHists>(load4, n, kr, hw, hist, scr, tid, 1, [=](int pos, int x, uint32_t kv) {
        oi[pos] = static_cast<int32_t>(buf[x].y);
        if (ov != nullptr) ov[pos] = key_to_float(kv);
      });
      for (int e = kk + tid; e < topk; e += kMergeThreads) {
        oi[e] = -1;
        if (ov != nullptr) ov[e] = -__int_as_float(0x7f800000);
      }
    } else {
      select_topk<kMergeThreads, kMergeHists>(load4, n, kr, hw, hist, scr, tid, 1,
                                              [=](int pos, int x, uint32_t) { keep[pos] = buf[x]; });
      kept = kr;
      for (int x = tid; x < kept; x += kMergeThreads) buf[x] = keep[x];
      if (kept & 1) {
        if (tid == 0) buf[kept] = make_uint2(0u, 0xFFFFFFFFu);
        kept += 1;
      }
      __syncthreads();
    }
  }
}

cudaError_t launch_merge(const MergeParams& mp, int rows, cudaStream_t stream) {
  static bool configured[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !configured[dev]) {
    e = cudaFuncSetAttribute(merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kMergeSmem));
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) configured[dev] = true;
  }
  merge_kernel<<<rows, kMergeThreads, kMergeSmem, stream>>>(mp);
  return cudaGetLastError();
}

// The shared-memory opt-in is set once per device (so that a launch inside stream capture is
// only a launch).
template <class Kernel>
cudaError_t ensure_smem(Kernel k, size_t bytes, bool (&configured)[64]) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !configured[dev]) {
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) configured[dev] = true;
  }
  return cudaSuccess;
}

template <int H, int Q>
cudaError_t launch_scorer_t(const ScorerParams& p, int grid, cudaStream_t stream) {
  using C = ScorerCfg<H, Q>;
  static bool configured[64] = {};
  cudaError_t e = ensure_smem(scorer_kernel<H, Q>, C::SMEM_BYTES, configured);
  if (e != cudaSuccess) return e;
  scorer_kernel<H, Q><<<grid, C::THREADS, C::SMEM_BYTES, stream>>>(p);
  return cudaGetLastError();
}

template <int Q>
cudaError_t launch_scorer_h(int H, const ScorerParams& p, int grid, cudaStream_t stream) {
  switch (H) {
    case 16: return launch_scorer_t<16, Q>(p, grid, stream);
    case 32: return launch_scorer_t<32, Q>(p, grid, stream);
    case 64: return launch_scorer_t<64, Q>(p, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_decode(const uint8_t* q_packed, const uint8_t* q_scale, const float* weights,
                          const uint8_t* kv_packed, const uint8_t* kv_scale, int64_t num_pages,
                          const int32_t* block_tables, int bt_stride, const int32_t* ctx_lens, int batch, int H,
                          int topk, const void* sched, size_t sched_bytes, void* workspace, int64_t cand_slots,
                          int32_t* topk_idx, float* topk_val, float* logits_debug, int64_t logits_stride,
                          int32_t* status, int grid, cudaStream_t stream) {
  ScorerParams p{};
  p.q_packed = q_packed;
  p.q_scale = q_scale;
  p.weights = weights;
  p.kv_packed = kv_packed;
  p.kv_scale = kv_scale;
  p.num_pages = num_pages;
  p.block_tables = block_tables;
  p.bt_stride = bt_stride;
  p.sched = sched;
  p.sched_bytes = sched_bytes;
  p.prefill = nullptr;
  p.expect_batch = batch;
  p.row_ends = nullptr;
  p.topk = topk;
  p.topk_idx = topk_idx;
  p.topk_val = topk_val;
  p.cand = static_cast<uint2*>(workspace);
  p.cand_slots = cand_slots;
  p.logits_debug = logits_debug;
  p.logits_stride = logits_stride;
  p.status = status;
  p.stream_once = 1;
  cudaError_t e = H == 128 ? launch_scorer_t<128, 1>(p, grid, stream) : launch_scorer_h<1>(H, p, grid, stream);
  if (e != cudaSuccess) return e;
  MergeParams mp{};
  mp.sched = sched;
  mp.sched_bytes = sched_bytes;
  mp.ctx_lens = ctx_lens;
  mp.batch = batch;
  mp.prefill = nullptr;
  mp.topk = topk;
  mp.cand = p.cand;
  mp.cand_slots = cand_slots;
  mp.topk_idx = topk_idx;
  mp.topk_val = topk_val;
  mp.status = status;
  return launch_merge(mp, batch, stream);
}

cudaError_t launch_prefill(const uint8_t* q_packed, const uint8_t* q_scale, const float* weights,
                           const uint8_t* kv_packed, const uint8_t* kv_scale, int64_t num_pages,
                           const int32_t* block_tables, int bt_stride, const int32_t* row_ends, int num_rows, int H,
                           int topk, void* workspace, int64_t units_cap, int64_t slots_cap, int32_t* topk_idx,
                           float* topk_val, float* logits_debug, int64_t logits_stride, int32_t* status, int grid,
                           cudaStream_t stream) {
  PrefillSchedHeader* hdr = static_cast<PrefillSchedHeader*>(workspace);
  ScorerParams p{};
  p.q_packed = q_packed;
  p.q_scale = q_scale;
  p.weights = weights;
  p.kv_packed = kv_packed;
  p.kv_scale = kv_scale;
  p.num_pages = num_pages;
  p.block_tables = block_tables;
  p.bt_stride = bt_stride;
  p.sched = nullptr;
  p.prefill = hdr;
  p.row_ends = row_ends;
  p.topk = topk;
  p.topk_idx = topk_idx;
  p.topk_val = topk_val;
  p.cand = reinterpret_cast<uint2*>(static_cast<char*>(workspace) + prefill_slots_offset(num_rows, units_cap));
  p.cand_slots = slots_cap;
  p.logits_debug = logits_debug;
  p.logits_stride = logits_stride;
  p.status = status;
  p.stream_once = 0;
  cudaError_t e = H == 128 ? launch_scorer_t<128, 1>(p, grid, stream) : launch_scorer_h<2>(H, p, grid, stream);
  if (e != cudaSuccess || slots_cap == 0) return e;
  MergeParams mp{};
  mp.sched = nullptr;
  mp.prefill = hdr;
  mp.topk = topk;
  mp.cand = p.cand;
  mp.cand_slots = slots_cap;
  mp.topk_idx = topk_idx;
  mp.topk_val = topk_val;
  mp.status = status;
  return launch_merge(mp, num_rows, stream);
}

}  // namespace idxfp4
