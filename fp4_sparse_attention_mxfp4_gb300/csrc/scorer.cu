// Prefill scorer: MXFP4 keys x MXFP4 query heads on tcgen05 block-scaled MMA, fused head-weighted
// ReLU reduction, fused exact top-k, for up to two query rows of one request per unit.
//
// Method ("Score a DSA sparse indexer in FP4", squashed commit message and PR body):
//   logit[q, t] = sum_h w[q, h] * relu(q_h . k_t), keys read in place from the paged two-plane
//   FP4 index region; the prefill top-k is bounded by the row's [0, row_end) range.
//
// GB300 design (the pages' kernels target MI355X MFMA; this is a fresh design):
//   * A 128-key tile (two pages) is the MMA M dimension, query rows x heads the N dimension:
//     D[128 x N] = K[128 x 128] . Q^T, as two K=64 tcgen05.mma kind::mxf4 block-scaled MMAs
//     accumulating fp32 in TMEM. TMEM lane = key, so the head sum is thread-local.
//   * Stage warps each own one stage of the ring (twelve; eight when the epilogue is two groups wide,
//     which leaves room for the second row's selection areas) and fill it with 1-D bulk copies
//     (cp.async.bulk): a page's four 1 KB group chunks land interleaved with the tile's other page,
//     which makes the stage a canonical no-swizzle K-major operand (LBO 2048 B between 32-dim
//     chunks, SBO 128 B between 8-key groups). The same warp rebuilds the tile's scale bytes from
//     the cache's 16x4-transposed order into the tensor core's scale-factor layout, copies them to
//     TMEM with tcgen05.cp and issues the MMAs; tcgen05.commit frees the stage and hands the
//     accumulator to the epilogue.
//   * Epilogue groups of four warps (one per TMEM lane quarter) read the accumulator with
//     tcgen05.ld, form each key's logit in a fixed order, store its order-preserving key in a
//     shared-memory row buffer and count it in a packed histogram. At the end of a unit an exact
//     radix select finds the k-th key and a stable pass writes the selected keys in token order.
//     The logit row never reaches global memory (unless a debug buffer is passed).
//   * Rows longer than one unit's share are scored in key chunks whose candidate lists are merged
//     by a cluster kernel. Persistent grid, one CTA per SM; every on-chip wait is bounded and
//     reports a timeout in the status word instead of hanging.
#include <cooperative_groups.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "common.cuh"
#include "ptx.cuh"
#include "topk.cuh"

namespace idxfp4 {
namespace {

constexpr uint32_t kEpiBarrier = 1;  // all epilogue warps
constexpr uint32_t kSelBarrier = 2;  // the warps that run the unit-end selection (+1: the second row group)

template <int H, int Q>
struct ScorerCfg {
  static constexpr int N = H * Q;
  // Epilogue groups of four warps (one per TMEM lane quarter) take tiles in turn; tiles that
  // share an accumulator belong to one group (ACC a multiple of GROUPS). Three groups keep up
  // with the stream at up to 64 columns per tile; wider tiles use two, with paired TMEM loads.
  static constexpr int GROUPS = N <= 64 ? 3 : 2;
  static constexpr int ACC = N <= 64 ? 6 : 2;  // TMEM accumulators
  static constexpr int STAGES = GROUPS == 3 ? 12 : 8;  // tiles in flight; one stage warp per stage
  static constexpr int EPI_WARP0 = STAGES;
  static constexpr int EPI_WARPS = 4 * GROUPS;
  static constexpr int EPI_THREADS = EPI_WARPS * 32;
  static constexpr int SEL_THREADS = 256;      // the unit-end selection runs on the first two groups
  // Two rows on two epilogue groups (N = 128): each group selects one of the unit's rows, side by
  // side, with its own histogram, scratch and barrier.
  static constexpr int ROW_GROUPS = Q == 2 && EPI_WARPS == 8 ? 2 : 1;
  static constexpr int SEL_NT = SEL_THREADS / ROW_GROUPS;  // threads selecting one row
  static constexpr int THREADS = (STAGES + EPI_WARPS) * 32;
  // Registers per thread: the launch gets 65536 / THREADS (rounded down to 8); the stage
  // warpgroups give registers back and the epilogue warpgroups take them, enough to hold a
  // tile's 64 accumulator columns in flight at once. The split sums to the launch's share.
  static constexpr uint32_t LAUNCH_REGS = (65536u / static_cast<uint32_t>(THREADS)) / 8u * 8u;
  static constexpr bool RESPLIT = GROUPS == 3;  // two-group tiles already fit at the launch share
  static constexpr uint32_t STAGE_REGS = RESPLIT ? 56u : LAUNCH_REGS;
  static constexpr uint32_t EPI_REGS =
      (LAUNCH_REGS * (STAGES + EPI_WARPS) - STAGE_REGS * STAGES) / EPI_WARPS / 8u * 8u;
  static_assert(STAGES % 4 == 0 && EPI_WARPS % 4 == 0, "roles are whole warpgroups");
  static_assert(STAGE_REGS * STAGES + EPI_REGS * EPI_WARPS <= LAUNCH_REGS * (STAGES + EPI_WARPS),
                "the re-split fits the registers the block is launched with");
  static constexpr int UCAP = unit_key_cap(Q);   // keys per unit and row (row buffer size)
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t SFA_COL = ACC * N;             // STAGES chunks of 4 columns
  static constexpr uint32_t SFB_COL = SFA_COL + 4 * STAGES;  // 2 chunks of 4 columns (unit parity)
  static_assert(ACC % GROUPS == 0, "tiles sharing an accumulator belong to one epilogue group");
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
  static constexpr uint32_t OFF_HIST = OFF_HW + Q * 4 * kHistWords * 4;  // [ROW_GROUPS][2048]
  static constexpr uint32_t OFF_SCR = OFF_HIST + ROW_GROUPS * 2048 * 4;  // [ROW_GROUPS][64]
  // Release barriers per accumulator, used in turn. A stage warp's tiles all use one accumulator,
  // STAGES / ACC of its tiles apart; with this many barriers the one it waits on has always seen
  // the completion before the awaited one.
  static constexpr int REL_RING = STAGES / ACC + 2;
  static_assert(STAGES % ACC == 0, "a stage warp keeps to one accumulator");
  static constexpr uint32_t NUM_BARS = 2 * STAGES + ACC + ACC * REL_RING + 2;
  static constexpr uint32_t OFF_BAR = OFF_SCR + ROW_GROUPS * 64 * 4;
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
  const PrefillSchedHeader* prefill;  // the call's unit list, strided over by the grid
  const int32_t* row_ends;       // per-row key ends
  int topk;
  int32_t* topk_idx;
  float* topk_val;
  uint2* cand;                   // candidate slots (see cand_slot_entries)
  int64_t cand_slots;            // slots the caller's buffer holds
  float* logits_debug;
  int64_t logits_stride;
  int32_t* status;
};

struct UnitIter {
  const Unit* units;
  int first, count, stride;
  bool ok;
  __device__ __forceinline__ Unit at(int i) const { return units[first + i * stride]; }
};

// This CTA's units (every gridDim-th of the call's list); `ok` is false when the workspace holds
// no unit list of this call.
__device__ __forceinline__ UnitIter unit_range(const ScorerParams& p) {
  UnitIter it{};
  const int c = blockIdx.x;
  it.ok = p.prefill->magic == kPrefillMagic;
  if (!it.ok) return it;
  const int n = p.prefill->num_units;
  it.units = reinterpret_cast<const Unit*>(reinterpret_cast<const char*>(p.prefill) +
                                           prefill_units_offset(p.prefill->num_rows));
  it.first = c;
  it.count = c < n ? (n - c + static_cast<int>(gridDim.x) - 1) / static_cast<int>(gridDim.x) : 0;
  it.stride = gridDim.x;
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

// Page id of the tile at cursor c: lane 0 reads the tile's first page, lane 1 its second (or -1
// if the tile has one page). A logical page past the table width reads nothing and gives -2.
__device__ __forceinline__ int load_tile_page(const ScorerParams& p, const Cursor& c, int lane) {
  const int lp = c.u.kb / kPage + 2 * c.j + lane;
  const bool needed = lane == 0 || (lane == 1 && c.u.kb + c.j * kTileKeys + kPage < c.u.ke);
  if (!needed) return -1;
  if (lp < 0 || lp >= p.bt_stride) return -2;
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
  pdl_wait();
  pdl_trigger();

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
    if constexpr (C::RESPLIT) warpgroup_regs_dec<C::STAGE_REGS>();
    // ---------------- stage warps: warp w streams tiles w, w+STAGES, ... through stage w and issues
    // their MMAs. Issue work is spread over many warps because a bulk copy or a tcgen05
    // instruction occupies its issuing warp or thread for a long time; one stage per warp also
    // keeps every wait on a barrier this warp alone advances.
    const int ps = warp;
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
    if constexpr (C::RESPLIT) warpgroup_regs_inc<C::EPI_REGS>();
    // ---------------- epilogue: head-weighted ReLU sum, row buffer, exact top-k ----------------
    // GROUPS groups of four warps (one per TMEM lane quarter; three groups for tiles up to 64
    // columns, two for 128) take tiles in turn; the epilogue also lays out each unit's query
    // operand and weights, two units ahead.
    const int e = warp - C::EPI_WARP0;
    const int grp = e >> 2;                 // tiles t with t % GROUPS == grp are this group's
    const int qtr = warp & 3;               // TMEM lane quarter of this warp
    const int etid = e * 32 + lane;         // rank among the epilogue threads (the first SEL_THREADS select)
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
        if (r < u.nq) ee = min(max(p.row_ends[u.row + r], 0), u.ke);
        end[r] = ee;
      }
      const int ntiles = unit_tiles(u);
      for (int j = ((grp - t0) % C::GROUPS + C::GROUPS) % C::GROUPS; j < ntiles; j += C::GROUPS) {
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
            // accumulator j holds heads j, j+8, ... in order; pairs of them share a packed fma
            unsigned long long p01 = 0ull, p23 = 0ull, p45 = 0ull, p67 = 0ull;
#pragma unroll
            for (int cc = 0; cc < H; cc += 64) {
              float v[64];
              tmem_load_2x32(col + cc, col + cc + 32, v);
#pragma unroll
              for (int h = 0; h < 64; h += 8) {
                const float4 wa = *reinterpret_cast<const float4*>(wsm + r * H + cc + h);
                const float4 wb = *reinterpret_cast<const float4*>(wsm + r * H + cc + h + 4);
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
      // select each row: exactly min(k, valid keys) keys, in token order (first SEL_THREADS; with
      // two row groups each takes every other row)
      const int rg = C::ROW_GROUPS == 1 ? 0 : etid / C::SEL_NT, stid = etid - rg * C::SEL_NT;
      const uint32_t sbar = kSelBarrier + static_cast<uint32_t>(rg);
      uint32_t* hist_g = hist + rg * 2048;
      uint32_t* scr_g = scr + rg * 64;
      for (int r = rg; etid < C::SEL_THREADS && r < u.nq && r < Q; r += C::ROW_GROUPS) {
        const uint32_t* keys = lg_base + r * C::UCAP;
        const int nvalid = max(0, end[r] - u.kb);
        const int kk = min(p.topk, nvalid);
        uint32_t* hw_r = hw_base + r * 4 * kHistWords;
        const int kb = u.kb;
        const bool to_slot = u.slot >= 0;
        if (to_slot && u.slot + r >= p.cand_slots) {
          if (stid == 0) set_status(p.status, IDX_FP4_DEV_CAPACITY);
          continue;
        }
        // The selection is emitted into this row's level-1 histogram area (free by then: 2048
        // (key, index) pairs fit its 16 KB) and then copied out with coalesced stores.
        uint2* sel = reinterpret_cast<uint2*>(hw_r);
        uint2* spare = reinterpret_cast<uint2*>(hist_g) + lane;  // where keys not kept are written
        select_topk<C::SEL_NT, 4>(keys, nvalid, kk, hw_r, hist_g, scr_g, stid, sbar,
                                       [=](bool keep, int pos, int x, uint32_t kv) {
                                         *(keep ? sel + pos : spare) = make_uint2(kv, static_cast<uint32_t>(x));
                                       });
        if (!to_slot) {
          const int64_t rowoff = static_cast<int64_t>(u.row + r) * p.topk;
          int32_t* oi = p.topk_idx + rowoff;
          float* ov = p.topk_val != nullptr ? p.topk_val + rowoff : nullptr;
          for (int x = stid; x < p.topk; x += C::SEL_NT) {
            const uint2 e = x < kk ? sel[x] : make_uint2(0u, 0u);
            oi[x] = x < kk ? kb + static_cast<int>(e.y) : -1;
            if (ov != nullptr) ov[x] = x < kk ? key_to_float(e.x) : -__int_as_float(0x7f800000);
          }
        } else {
          uint2* slot = p.cand + static_cast<int64_t>(u.slot + r) * static_cast<int64_t>(cand_slot_entries(p.topk));
          uint2* oc = slot + 2;
          uint32_t kmin = 0xFFFFFFFFu, kmax = 0u;
          for (int x = stid; x < kk; x += C::SEL_NT) {
            const uint2 e = sel[x];
            oc[x] = make_uint2(e.x, static_cast<uint32_t>(kb) + e.y);
            kmin = min(kmin, e.x);
            kmax = max(kmax, e.x);
          }
          // The header also carries the list's smallest and largest key: the merge bounds the
          // row's threshold from below by the smallest key of a full list, and bins only the
          // keys above that bound.
          kmin = __reduce_min_sync(0xFFFFFFFFu, kmin);
          kmax = __reduce_max_sync(0xFFFFFFFFu, kmax);
          if (lane == 0) {
            scr_g[32 + 2 * (stid >> 5)] = kmin;
            scr_g[33 + 2 * (stid >> 5)] = kmax;
          }
          named_barrier_sync(sbar, C::SEL_NT);
          // odd counts get one pad entry so every list is a whole number of 16-byte pairs; key 0 is
          // below every logit and never selected
          if (stid == 0) {
#pragma unroll
            for (int w2 = 0; w2 < C::SEL_NT / 32; ++w2) {
              kmin = min(kmin, scr_g[32 + 2 * w2]);
              kmax = max(kmax, scr_g[33 + 2 * w2]);
            }
            if (kk & 1) oc[kk] = make_uint2(0u, 0xFFFFFFFFu);
            *reinterpret_cast<uint4*>(slot) = make_uint4(static_cast<uint32_t>(kk), kmin, kmax, 0u);
          }
        }
        named_barrier_sync(sbar, C::SEL_NT);  // the area is reused by the next row
      }
      named_barrier_sync(kEpiBarrier, C::EPI_THREADS);  // selection done before the areas are cleared
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
// Merge of split prefill rows (rows cut into key chunks). A row's candidate lists (each exactly its unit's top-min(k, keys), in token order)
// are merged by one cluster of kMergeG CTAs: CTA r takes the r-th share of the lists'
// concatenation and streams it from L2 in every pass. Each CTA counts its share into local
// radix histograms; the cluster sums them through distributed shared memory, so every CTA
// arrives at the same threshold; each then writes its selected keys at an offset given by the
// counts of the CTAs before it, which keeps the output in token order. Keys are first shifted
// past the bits that all the row's candidates share, so that the first radix level spreads
// them over its bins (the candidates are the top of the row and would otherwise fill a few
// bins).
constexpr int kMergeG = 8;               // CTAs per row (one cluster)
constexpr int kMergeThreads = 256;
constexpr int kMergeNW = kMergeThreads / 32;
constexpr int kMergeMaxLists = 2048;     // lists of one row (rows with more set CAPACITY)
constexpr int kMergeCbuf = 4096;         // keys of the threshold bin a CTA lists
constexpr int kMergeUnion = 4096;        // keys of the threshold bin gathered from the cluster
constexpr int kMergeStage = 6144;        // candidates of a CTA's share staged in shared memory
// shared memory (32-bit words): staged share [2 * kMergeStage] | local histogram [2048] | summed
// histogram [2048] | bin list [kMergeCbuf] | gathered bin [kMergeUnion] | list starts
// [kMergeMaxLists + 1] | scratch [64] | values pulled from the cluster [64] | published values
// [8]. About 104 KB: two CTAs fit an SM, so every row's cluster is resident at once.
constexpr size_t kMergeSmem =
    (2 * kMergeStage + 2048 + 2048 + kMergeCbuf + kMergeUnion + kMergeMaxLists + 1 + 64 + 64 + 8) * 4;

struct MergeParams {
  const PrefillSchedHeader* prefill; // the workspace header
  int topk;
  const uint2* cand;
  int64_t cand_slots;
  int32_t* topk_idx;
  float* topk_val;
  int32_t* status;
};

// Keys below `lo` (a lower bound on the row's threshold) map to 0, never counted or selected;
// keys from lo up, which share their p leading bits, are shifted past them, order-preserving
// (p = 32: all equal). Real keys are nonzero, and so are the images of those kept.
__device__ __forceinline__ uint32_t merge_xform(uint32_t k, uint32_t p, uint32_t lo) {
  return k < lo ? 0u : (p >= 32u ? 1u : ((k << p) | (p != 0u ? 1u : 0u)));
}

__global__ void __launch_bounds__(kMergeThreads) merge_kernel(const __grid_constant__ MergeParams mp) {
  namespace cg = cooperative_groups;
  cg::cluster_group cluster = cg::this_cluster();
  extern __shared__ __align__(16) uint32_t msm[];
  uint2* stage = reinterpret_cast<uint2*>(msm);
  uint32_t* hl = msm + 2 * kMergeStage;     // this CTA's histogram (read by the cluster)
  uint32_t* hs = hl + 2048;                 // cluster sums
  uint32_t* cbuf = hs + 2048;               // this CTA's keys of the threshold bin (read by the cluster)
  uint32_t* ubuf = cbuf + kMergeCbuf;       // the cluster's keys of the threshold bin
  uint32_t* lstart = ubuf + kMergeUnion;
  uint32_t* sc = lstart + kMergeMaxLists + 1;
  uint32_t* rv = sc + 64;                   // values pulled from every CTA of the cluster
  uint32_t* pub = rv + 64;  // [2] keys > T, [3] keys == T, [4] listed keys,
                            // [5] list complete, [6] slice total
  const int rank = static_cast<int>(cluster.block_rank());
  const int row = static_cast<int>(blockIdx.x) / kMergeG;
  pdl_wait();
  pdl_trigger();
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int topk = mp.topk;
  uint32_t* gtw = sc + 16;  // per warp: the largest smallest key of a full list
  uint32_t* eqw = sc + 32;  // per warp: the smallest key of any list
  // Row setup: every CTA of the cluster reads the same row, so every early return below is
  // taken by the whole cluster.
  if (mp.prefill->magic != kPrefillMagic) return;
  const int4 rm = reinterpret_cast<const int4*>(mp.prefill + 1)[row];
  const int first = rm.x, nu = rm.y, stride = mp.prefill->rows_per_unit;
  const int kk = min(topk, rm.z);
  if (nu <= 1) return;  // written by the scorer
  if (nu > kMergeMaxLists) {
    if (rank == 0 && tid == 0) set_status(mp.status, IDX_FP4_DEV_CAPACITY);
    return;
  }
  const int64_t slot_entries = static_cast<int64_t>(cand_slot_entries(topk));
  auto list_base = [&](int li) { return mp.cand + (first + static_cast<int64_t>(li) * stride) * slot_entries + 2; };
  // After a cluster barrier: rv[r * nv + j] = CTA r's pub[j0 + j], read by kMergeG * nv threads at once.
  auto pull = [&](int j0, int nv) {
    if (tid < kMergeG * nv) rv[tid] = cluster.map_shared_rank(pub, tid / nv)[j0 + tid % nv];
    __syncthreads();
  };

  // 1. List starts: block scan of the lists' sizes, and the range of keys that matter, from the
  // lists' headers (every CTA reads all of them). A full list (k keys) is the top-k of its unit,
  // so the row's k-th largest key is at least that list's smallest: `lo` is the largest such
  // bound (with no full list, the smallest key of all). Only keys from lo to the largest key
  // `hi` are binned, shifted past the leading bits lo and hi share.
  uint32_t pbits, lo;
  {
    constexpr int kPerMax = kMergeMaxLists / kMergeThreads;
    const int per = (nu + kMergeThreads - 1) / kMergeThreads;
    const int l0 = min(nu, tid * per);
    uint32_t cnt[kPerMax];
    uint32_t s = 0, lo_full = 0u, lo_all = 0xFFFFFFFFu, hi = 0u;
#pragma unroll
    for (int j = 0; j < kPerMax; ++j) {
      const int li = l0 + j;
      const int64_t sl = first + static_cast<int64_t>(li) * stride;
      cnt[j] = 0u;
      if (j < per && li < nu && sl < mp.cand_slots) {
        const uint4 h = *reinterpret_cast<const uint4*>(mp.cand + sl * slot_entries);
        cnt[j] = static_cast<uint32_t>(min(static_cast<int>(h.x), topk));
        if (cnt[j] != 0u) {
          lo_all = min(lo_all, h.y);
          hi = max(hi, h.z);
          if (h.x >= static_cast<uint32_t>(topk)) lo_full = max(lo_full, h.y);
        }
      }
      s += cnt[j];
    }
    uint32_t incl = s;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, off);
      if (lane >= off) incl += v;
    }
    lo_full = __reduce_max_sync(0xFFFFFFFFu, lo_full);
    lo_all = __reduce_min_sync(0xFFFFFFFFu, lo_all);
    hi = __reduce_max_sync(0xFFFFFFFFu, hi);
    if (lane == 31) sc[w] = incl;
    if (lane == 0) {
      gtw[w] = lo_full;
      eqw[w] = lo_all;
      sc[48 + w] = hi;
    }
    for (int b = tid; b < 2048; b += kMergeThreads) hl[b] = 0u;
    __syncthreads();
    uint32_t run = incl - s;
    for (int w2 = 0; w2 < w; ++w2) run += sc[w2];
    if (tid == 0) lstart[0] = 0u;
#pragma unroll
    for (int j = 0; j < kPerMax; ++j) {
      run += cnt[j];
      if (j < per && l0 + j < nu) lstart[l0 + j + 1] = run;
    }
    lo_full = 0u;
    lo_all = 0xFFFFFFFFu;
    hi = 0u;
#pragma unroll
    for (int w2 = 0; w2 < kMergeNW; ++w2) {
      lo_full = max(lo_full, gtw[w2]);
      lo_all = min(lo_all, eqw[w2]);
      hi = max(hi, sc[48 + w2]);
    }
    lo = lo_full != 0u ? lo_full : lo_all;
    pbits = (lo ^ hi) == 0u ? 32u : static_cast<uint32_t>(__clz(lo ^ hi));
    __syncthreads();
  }
  const int total = static_cast<int>(lstart[nu]);
  const int share = (total + kMergeG - 1) / kMergeG;
  const int p0 = min(total, rank * share), p1 = min(total, p0 + share);
  // the list holding entry p (0 <= p < total): the last list starting at or before p, so
  // lstart[li] <= p < lstart[li + 1]
  auto list_of = [&](int p) {
    int a = 0, b = nu;
    while (b - a > 1) {
      const int mid = (a + b) >> 1;
      if (static_cast<int>(lstart[mid]) <= p) a = mid; else b = mid;
    }
    return a;
  };
  auto entry = [&](int p) {
    const int li = list_of(p);
    return list_base(li)[p - static_cast<int>(lstart[li])];
  };
  // The share is staged in shared memory with independent loads, twelve in flight per thread
  // (a thread's entries are kMergeThreads apart, so it walks its list index forward instead of
  // searching for each); a share too large for the stage (rows of more than kMergeG *
  // kMergeStage candidates) is read from global memory in every pass instead.
  const bool staged = p1 - p0 <= kMergeStage;
  if (staged && p0 + tid < p1) {
    int li = list_of(p0 + tid);
    for (int b = p0; b < p1; b += 12 * kMergeThreads) {
      uint2 v[12];
#pragma unroll
      for (int j = 0; j < 12; ++j) {
        const int p = b + j * kMergeThreads + tid;
        if (p < p1) {
          while (static_cast<int>(lstart[li + 1]) <= p) ++li;
          v[j] = list_base(li)[p - static_cast<int>(lstart[li])];
        }
      }
#pragma unroll
      for (int j = 0; j < 12; ++j) {
        const int p = b + j * kMergeThreads + tid;
        if (p < p1) {
          stage[p - p0] = v[j];
          const uint32_t t = merge_xform(v[j].x, pbits, lo);  // 2. level 1, below
          if (t != 0u) smem_red_add(&hl[t >> 21], 1u);
        }
      }
    }
  }
  auto get = [&](int p) { return staged ? stage[p - p0] : entry(p); };
  // Entries p .. p+3 (p - p0 a multiple of 4); entries at or past `end` come back as zero keys.
  auto get4 = [&](int p, int end, uint2 (&e)[4]) {
    if (staged) {
      const uint4* q = reinterpret_cast<const uint4*>(stage + (p - p0));
      const uint4 a = q[0], b = q[1];
      e[0] = make_uint2(a.x, a.y);
      e[1] = make_uint2(a.z, a.w);
      e[2] = make_uint2(b.x, b.y);
      e[3] = make_uint2(b.z, b.w);
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (p + j >= end) e[j] = make_uint2(0u, 0u);
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j) e[j] = p + j < end ? entry(p + j) : make_uint2(0u, 0u);
    }
  };
  // Each thread's run of the CTA's share, in token order (a multiple of 4 entries long except
  // at the end). The passes below count over runs and turn the counts into list and output
  // offsets with block scans.
  const int2 trun = thread_run<kMergeThreads>(p1 - p0, tid);
  const int ra = p0 + trun.x, rb = p0 + trun.y;
  // exclusive prefix (x, y) and totals (z, w) over the CTA of two per-thread counts
  auto scan2 = [&](uint32_t a, uint32_t b) {
    uint32_t ia = a, ib = b;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const uint32_t va = __shfl_up_sync(0xFFFFFFFFu, ia, off);
      const uint32_t vb = __shfl_up_sync(0xFFFFFFFFu, ib, off);
      if (lane >= off) {
        ia += va;
        ib += vb;
      }
    }
    if (lane == 31) {
      sc[2 * w] = ia;
      sc[2 * w + 1] = ib;
    }
    __syncthreads();
    uint32_t pa = 0, pb = 0, ta = 0, tb = 0;
#pragma unroll
    for (int w2 = 0; w2 < kMergeNW; ++w2) {
      const uint32_t xa = sc[2 * w2], xb = sc[2 * w2 + 1];
      pa += w2 < w ? xa : 0u;
      pb += w2 < w ? xb : 0u;
      ta += xa;
      tb += xb;
    }
    __syncthreads();
    return make_uint4(pa + ia - a, pb + ib - b, ta, tb);
  };

  // 2. Level 1: top 11 bits of the shifted keys (counted while staging, when staged).
  if (!staged)
    for (int p = p0 + tid; p < p1; p += kMergeThreads) {
      const uint32_t t = merge_xform(get(p).x, pbits, lo);
      if (t != 0u) smem_red_add(&hl[t >> 21], 1u);
    }
  cluster.sync();
  // The level-1 bin of the threshold without moving whole histograms: CTA r sums bins
  // [256 r, 256 r + 256) over the cluster (one remote word per thread and CTA) and publishes the
  // slice's total; every CTA then finds the slice holding the kk-th largest key from the eight
  // totals and reads only that slice's sums.
  constexpr int kSlice = 2048 / kMergeG;
  static_assert(kSlice == kMergeThreads, "one bin of the slice per thread");
  {
    uint32_t v[kMergeG];
#pragma unroll
    for (int r = 0; r < kMergeG; ++r) v[r] = cluster.map_shared_rank(hl, r)[rank * kSlice + tid];
    uint32_t sum = 0;
#pragma unroll
    for (int r = 0; r < kMergeG; ++r) sum += v[r];
    hs[rank * kSlice + tid] = sum;
    const uint32_t ws = __reduce_add_sync(0xFFFFFFFFu, sum);
    if (lane == 0) sc[w] = ws;
    __syncthreads();
    if (tid == 0) {
      uint32_t t = 0;
      for (int w2 = 0; w2 < kMergeNW; ++w2) t += sc[w2];
      pub[6] = t;
    }
  }
  cluster.sync();
  pull(6, 1);
  // Fallback sum for the levels below, when the threshold bin is too large to gather.
  auto cluster_sum = [&](int nb) {
    for (int b0 = tid; b0 < nb; b0 += kMergeThreads) {
      uint32_t v[kMergeG];
#pragma unroll
      for (int r = 0; r < kMergeG; ++r) v[r] = cluster.map_shared_rank(hl, r)[b0];
      uint32_t sum = 0;
#pragma unroll
      for (int r = 0; r < kMergeG; ++r) sum += v[r];
      hs[b0] = sum;
    }
    __syncthreads();
  };
  uint32_t thr = 0u, need = 0u;  // keep shifted key > thr, and the first `need` equal to it
  if (kk < total) {
    // slice holding the kk-th largest, scanning slices from the top
    uint32_t above_slice = 0;
    int sl = kMergeG - 1;
    for (; sl > 0; --sl) {
      if (above_slice + rv[sl] >= static_cast<uint32_t>(kk)) break;
      above_slice += rv[sl];
    }
    // the slice's sums land in the gather buffer, which is unused until the gather below
    ubuf[tid] = cluster.map_shared_rank(hs, sl)[sl * kSlice + tid];
    __syncthreads();
    const uint2 r1 = find_bin<kMergeThreads>(ubuf, kSlice, static_cast<uint32_t>(kk) - above_slice, sc, tid, 1);
    const uint32_t bin = static_cast<uint32_t>(sl * kSlice) + r1.x;
    need = static_cast<uint32_t>(kk) - above_slice - r1.y;
    const uint32_t in_bin = ubuf[r1.x];  // the cluster's keys in the threshold bin
    const bool listed = hl[bin] <= static_cast<uint32_t>(kMergeCbuf);
    // The CTA's keys in the threshold bin (low 21 bits), listed in token order: a count over each
    // run, a block scan, and a second walk of the run that writes them.
    uint32_t inb = 0;
    for (int p = ra; p < rb; p += 4) {
      uint2 e[4];
      get4(p, rb, e);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t t = merge_xform(e[j].x, pbits, lo);
        inb += (p + j < rb && t != 0u && (t >> 21) == bin) ? 1u : 0u;
      }
    }
    const uint4 ls = scan2(inb, 0u);
    const int m = static_cast<int>(ls.z);
    if (listed && inb != 0u) {
      uint32_t slot = ls.x;
      for (int p = ra; p < rb; p += 4) {
        uint2 e[4];
        get4(p, rb, e);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint32_t t = merge_xform(e[j].x, pbits, lo);
          if (p + j < rb && t != 0u && (t >> 21) == bin) cbuf[slot++] = t & 0x1FFFFFu;
        }
      }
    }
    if (tid == 0) {
      pub[4] = static_cast<uint32_t>(m);
      pub[5] = listed ? 1u : 0u;
    }
    cluster.sync();  // every CTA's list is complete, and no CTA reads level-1 sums any more
    pull(4, 2);
    bool gather = in_bin <= static_cast<uint32_t>(kMergeUnion);
    uint32_t base_of[kMergeG + 1];
    base_of[0] = 0u;
#pragma unroll
    for (int r = 0; r < kMergeG; ++r) {
      base_of[r + 1] = base_of[r] + rv[2 * r];
      gather = gather && rv[2 * r + 1] != 0u;
    }
    uint32_t low = 0u;
    if (gather) {
      // The bin's keys of the whole cluster, gathered here with independent remote loads:
      // levels 2 and 3 run inside this CTA.
      for (int u = tid; u < static_cast<int>(in_bin); u += kMergeThreads) {
        int r = 0;
#pragma unroll
        for (int q = 1; q < kMergeG; ++q) r += static_cast<uint32_t>(u) >= base_of[q] ? 1 : 0;
        ubuf[u] = cluster.map_shared_rank(cbuf, r)[u - static_cast<int>(base_of[r])] & 0x1FFFFFu;
      }
      __syncthreads();
      if (in_bin <= static_cast<uint32_t>(kMergeThreads)) {
        // Rank selection: thread u holds gathered key u; the threshold's low bits are the key
        // with fewer than `need` keys above it and at least `need` at or above it (equal keys
        // all write the same values).
        if (tid < static_cast<int>(in_bin)) {
          const uint32_t c = ubuf[tid];
          uint32_t gt = 0, ge = 0;
          for (int x = 0; x < static_cast<int>(in_bin); ++x) {
            const uint32_t d = ubuf[x];
            gt += d > c ? 1u : 0u;
            ge += d >= c ? 1u : 0u;
          }
          if (gt < need && need <= ge) {
            sc[60] = c;
            sc[61] = gt;
          }
        }
        __syncthreads();
        low = sc[60];
        need -= sc[61];
      } else {
        // Three radix levels of 8, 8 and 5 bits, over 256 bins (one per thread).
        uint32_t pre = 0u;
#pragma unroll 1
        for (int level = 0; level < 3; ++level) {
          const int sh = level == 0 ? 13 : (level == 1 ? 5 : 0);  // this level's digit
          const int psh = level == 0 ? 21 : sh + (level == 1 ? 8 : 5);  // the digits found so far
          hl[tid] = 0u;
          __syncthreads();
          for (int x = tid; x < static_cast<int>(in_bin); x += kMergeThreads) {
            const uint32_t c = ubuf[x];
            if ((c >> psh) == pre) smem_red_add(&hl[(c >> sh) & (level == 2 ? 31u : 255u)], 1u);
          }
          __syncthreads();
          const uint2 r = find_bin<kMergeThreads>(hl, kMergeThreads, need, sc, tid, 1);
          need -= r.y;
          pre = (pre << (level == 2 ? 5 : 8)) | r.x;
        }
        low = pre;
      }
    } else {
      // Levels 2 and 3 through cluster sums (from the list, or from the share when it did not fit).
#pragma unroll 1
      for (int level = 0; level < 2; ++level) {
        const int nb = level == 0 ? 2048 : 1024;
        if (level == 1) cluster.sync();  // every CTA has finished reading the level-2 histograms
        for (int b0 = tid; b0 < 2048; b0 += kMergeThreads) hl[b0] = 0u;
        __syncthreads();
        auto count = [&](uint32_t c) {
          if (level == 0) smem_red_add(&hl[c >> 10], 1u);
          else if ((c >> 10) == (low >> 10)) smem_red_add(&hl[c & 1023u], 1u);
        };
        if (listed) {
          for (int x = tid; x < m; x += kMergeThreads) count(cbuf[x] & 0x1FFFFFu);
        } else {
          for (int p = p0 + tid; p < p1; p += kMergeThreads) {
            const uint32_t t = merge_xform(get(p).x, pbits, lo);
            if (t != 0u && (t >> 21) == bin) count(t & 0x1FFFFFu);
          }
        }
        __syncthreads();
        cluster.sync();
        cluster_sum(nb);
        const uint2 r = find_bin<kMergeThreads>(hs, nb, need, sc, tid, 1);
        need -= r.y;
        low |= level == 0 ? (r.x << 10) : r.x;
      }
    }
    thr = (bin << 21) | low;
  }
  // Every candidate is kept when kk >= total: thr = 0 and need = 0 keep every key (all are at
  // least lo then, and map to nonzero images).
  // 3. Offsets: per thread, the keys above thr and equal to it; a block scan gives the thread's
  // place in the CTA, the published totals the CTA's place in the cluster.
  uint32_t g = 0, e = 0;
  for (int p = ra; p < rb; p += 4) {
    uint2 en[4];
    get4(p, rb, en);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t t = merge_xform(en[j].x, pbits, lo);  // thr >= 1 when selecting: keys below lo never kept
      g += (p + j < rb && t > thr) ? 1u : 0u;
      e += (p + j < rb && t == thr) ? 1u : 0u;
    }
  }
  const uint4 cs = scan2(g, e);
  if (tid == 0) {
    pub[2] = cs.z;
    pub[3] = cs.w;
  }
  cluster.sync();
  pull(2, 2);
  // That was the last read of another CTA's shared memory: arrive now, and wait for the others
  // only before leaving (no CTA exits while another may still read its published counts).
  asm volatile("barrier.cluster.arrive.relaxed.aligned;\n" ::: "memory");
  uint32_t gb = cs.x, eb = cs.y;  // keys above thr / equal to it before this thread's run
  for (int r = 0; r < rank; ++r) {
    gb += rv[2 * r];
    eb += rv[2 * r + 1];
  }
  // 4. Output in token order: a kept key goes to (keys above thr before it) + min(keys equal to
  // thr before it, need); the first `need` keys equal to thr are kept.
  int32_t* oi = mp.topk_idx + static_cast<int64_t>(row) * topk;
  float* ov = mp.topk_val != nullptr ? mp.topk_val + static_cast<int64_t>(row) * topk : nullptr;
  if (g + min(e, need > eb ? need - eb : 0u) != 0u) {
    for (int p = ra; p < rb; p += 4) {
      uint2 en[4];
      get4(p, rb, en);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t t = merge_xform(en[j].x, pbits, lo);
        const bool gt = p + j < rb && t > thr, eq = p + j < rb && t == thr;
        if (gt || (eq && eb < need)) {
          const uint32_t pos = gb + min(eb, need);
          oi[pos] = static_cast<int32_t>(en[j].y);
          if (ov != nullptr) ov[pos] = key_to_float(en[j].x);
        }
        gb += gt ? 1u : 0u;
        eb += eq ? 1u : 0u;
      }
    }
  }
  if (rank == 0)
    for (int e = kk + tid; e < topk; e += kMergeThreads) {
      oi[e] = -1;
      if (ov != nullptr) ov[e] = -__int_as_float(0x7f800000);
    }
  asm volatile("barrier.cluster.wait.aligned;\n" ::: "memory");
}

cudaError_t launch_merge(const MergeParams& mp, int rows, cudaStream_t stream) {
  cudaError_t e = set_smem_once<merge_kernel>(kMergeSmem);
  if (e != cudaSuccess) return e;
  return launch_pdl(merge_kernel, dim3(static_cast<unsigned>(rows) * kMergeG), dim3(kMergeThreads), kMergeSmem, stream,
                    kMergeG, false, mp);
}

template <int H, int Q>
cudaError_t launch_scorer_t(const ScorerParams& p, int grid, cudaStream_t stream) {
  using C = ScorerCfg<H, Q>;
  cudaError_t e = set_smem_once<scorer_kernel<H, Q>>(C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  return launch_pdl(scorer_kernel<H, Q>, dim3(grid), dim3(C::THREADS), C::SMEM_BYTES, stream, 1, false, p);
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
  cudaError_t e = H == 128 ? launch_scorer_t<128, 1>(p, grid, stream) : launch_scorer_h<2>(H, p, grid, stream);
  if (e != cudaSuccess || slots_cap == 0) return e;
  MergeParams mp{};
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
