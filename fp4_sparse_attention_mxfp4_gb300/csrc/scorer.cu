// Scorer: MXFP4 keys x MXFP4 query heads on tcgen05 block-scaled MMA, fused head-weighted
// ReLU reduction, fused exact top-k. Shared by decode (one query row per unit) and prefill
// (two rows of one request per unit).
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
//   * Warp 0 streams pages with 1-D bulk TMA copies (cp.async.bulk): each page's four 1 KB
//     group chunks land interleaved with the tile's other page, which makes the stage a
//     canonical no-swizzle K-major operand (LBO 2048 B between 32-dim chunks, SBO 128 B
//     between 8-key groups) without any register pass.
//   * Warp 1 rebuilds the stage's scale bytes from the cache's 16x4-transposed order into the
//     tensor core's scale-factor layout (key m at lane m%32, column m/32), copies them to TMEM
//     with tcgen05.cp, and issues the MMAs; tcgen05.commit frees the stage and hands the
//     accumulator to the epilogue.
//   * Warps 2-5 (one per TMEM lane quarter) read the accumulator with tcgen05.ld, form the
//     logit, and push it through a per-row threshold filter into a shared-memory candidate
//     buffer; the buffer is cut back to k with an exact radix select when it fills. The full
//     logit row never reaches global memory (unless a debug buffer is passed).
//   * Persistent grid, one CTA per SM; every on-chip wait is bounded and reports a timeout in
//     the status word instead of hanging.
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
  static constexpr int ACC = N <= 64 ? 4 : 2;  // TMEM accumulator stages
  static constexpr int STAGES = 8;             // key tiles in flight per CTA
  static constexpr int THREADS = 192;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t SFA_COL = 256;            // ACC chunks of 4 columns
  static constexpr uint32_t SFB_COL = 256 + 4 * 4;    // 2 chunks of 4 columns (unit parity)
  static_assert(ACC * N <= 256, "accumulators fit below the scale columns");
  // shared memory map (offsets from a 1024-byte aligned base)
  static constexpr uint32_t OFF_PACKED = 0;                              // [STAGES][4][128][16]
  static constexpr uint32_t OFF_SCALE = OFF_PACKED + STAGES * 8192;      // [STAGES][2 pages][256]
  static constexpr uint32_t OFF_SFA = OFF_SCALE + STAGES * 512;          // [STAGES][512] tensor-core layout
  static constexpr uint32_t RAW_Q = Q * H * 64, RAW_QS = Q * H * 4, RAW_W = Q * H * 4;
  static constexpr uint32_t UNIT_BYTES = RAW_Q + RAW_QS + RAW_W;
  static constexpr uint32_t OFF_UNIT = OFF_SFA + STAGES * 512;           // [2][UNIT_BYTES]
  static constexpr uint32_t OFF_QB = (OFF_UNIT + 2 * UNIT_BYTES + 1023) / 1024 * 1024;  // [2][4][N][16]
  static constexpr uint32_t OFF_SFB = OFF_QB + 2 * N * 64;               // [2][512]
  static constexpr uint32_t OFF_CB = OFF_SFB + 2 * 512;                  // [Q][kCandCap] uint2
  static constexpr uint32_t OFF_HIST = OFF_CB + Q * kCandCap * 8;        // [2048] u32
  static constexpr uint32_t SCR_WORDS = 256;
  static constexpr uint32_t OFF_SCR = OFF_HIST + 2048 * 4;
  static constexpr uint32_t NUM_BARS = 2 * STAGES + 2 * ACC + 6;
  static constexpr uint32_t OFF_BAR = OFF_SCR + SCR_WORDS * 4;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NUM_BARS * 8;
  static constexpr uint32_t SMEM_BYTES = OFF_MISC + 64 + 1024;
  static_assert(SMEM_BYTES <= 227 * 1024, "fits one SM");
  static_assert(UNIT_BYTES % 16 == 0, "bulk copies need 16-byte sizes");
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
  uint2* cand;
  int32_t* cand_count;
  float* logits_debug;
  int64_t logits_stride;
  int32_t* status;
  int stream_once;               // 1: keys are read once (decode) -> L2 evict-first
};

struct UnitIter {
  const Unit* units;
  int first, count, stride;
  bool ok;
};

// This CTA's units; `ok` is false when the schedule does not belong to this call.
__device__ __forceinline__ UnitIter unit_range(const ScorerParams& p) {
  UnitIter it{};
  const int c = blockIdx.x;
  if (p.sched != nullptr) {
    const DecodeSchedHeader* h = static_cast<const DecodeSchedHeader*>(p.sched);
    it.ok = h->magic == kDecodeMagic && h->ctas == static_cast<int>(gridDim.x) && h->batch == p.expect_batch &&
            h->max_batch >= h->batch && decode_sched_bytes(h->max_batch) <= p.sched_bytes;
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
    it.units = reinterpret_cast<const Unit*>(p.prefill + 1);
    it.first = c;
    it.count = c < n ? (n - c + static_cast<int>(gridDim.x) - 1) / static_cast<int>(gridDim.x) : 0;
    it.stride = gridDim.x;
  }
  return it;
}

__device__ __forceinline__ int unit_tiles(const Unit& u) {
  return u.ke > u.kb ? (u.ke - u.kb + kTileKeys - 1) / kTileKeys : 0;
}

__device__ __forceinline__ bool bounded_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                             int32_t* status) {
  if (*abort_flag) return false;
  if (mbar_wait(bar, parity, kWaitLimitNs)) return true;
  *abort_flag = 1;
  set_status(status, IDX_FP4_DEV_TIMEOUT);
  return false;
}

template <int H, int Q>
__global__ void __launch_bounds__(192, 1) scorer_kernel(const __grid_constant__ ScorerParams p) {
  using C = ScorerCfg<H, Q>;
  constexpr int N = C::N, ACC = C::ACC, STAGES = C::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // Schedule checks (uniform across the grid; nothing is allocated yet).
  const UnitIter it = unit_range(p);
  if (!it.ok) {
    if (tid == 0 && blockIdx.x == 0) set_status(p.status, IDX_FP4_DEV_BAD_SCHEDULE);
    return;
  }

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* full_bar = bars;
  uint64_t* empty_bar = bars + STAGES;
  uint64_t* acc_full = bars + 2 * STAGES;
  uint64_t* acc_empty = acc_full + ACC;
  uint64_t* unit_full = acc_empty + ACC;
  uint64_t* unit_empty = unit_full + 2;
  uint64_t* q_free = unit_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);

  if (tid == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int a = 0; a < ACC; ++a) {
      mbar_init(&acc_full[a], 1);
      mbar_init(&acc_empty[a], 128);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&unit_full[i], 1);
      mbar_init(&unit_empty[i], 1 + 128);
      mbar_init(&q_free[i], 1);
    }
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, C::TMEM_COLS);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ---------------- producer: bulk copies of key pages and unit inputs ----------------
    const uint64_t pol = policy_evict_first();
    int f = 0;
    for (int i = 0; i < it.count; ++i) {
      const Unit u = it.units[it.first + i * it.stride];
      const int par = i & 1;
      uint8_t* stage_unit = smem + C::OFF_UNIT + par * C::UNIT_BYTES;
      if (lane == 0) {
        if (i >= 2) bounded_wait(&unit_empty[par], ((i >> 1) - 1) & 1, abort_flag, p.status);
        const uint32_t rq = u.nq * H * 64, rqs = u.nq * H * 4;
        mbar_arrive_expect_tx(&unit_full[par], rq + 2 * rqs);
        bulk_load(stage_unit, p.q_packed + static_cast<int64_t>(u.row) * H * 64, rq, &unit_full[par]);
        bulk_load(stage_unit + C::RAW_Q, p.q_scale + static_cast<int64_t>(u.row) * H * 4, rqs, &unit_full[par]);
        bulk_load(stage_unit + C::RAW_Q + C::RAW_QS, p.weights + static_cast<int64_t>(u.row) * H, rqs,
                  &unit_full[par]);
      }
      const int ntiles = unit_tiles(u);
      const int32_t* table = p.block_tables + static_cast<int64_t>(u.table) * p.bt_stride;
      const int lp_first = u.kb / kPage;
      const int lp_end = (u.ke + kPage - 1) / kPage;  // one past the last logical page read
      int wb = -64, entry = 0;
      for (int j = 0; j < ntiles; ++j) {
        const int lp0 = lp_first + 2 * j;
        const bool has1 = u.kb + j * kTileKeys + kPage < u.ke;
        if (lp0 - wb >= 32) {
          wb = lp0;
          const int lp = wb + lane;
          entry = (lp < lp_end && lp < p.bt_stride) ? table[lp] : 0;
        }
        int pid0 = __shfl_sync(0xFFFFFFFFu, entry, lp0 - wb);
        int pid1 = __shfl_sync(0xFFFFFFFFu, entry, (lp0 + 1 - wb) & 31);
        if (lane == 0) {
          if (lp0 >= p.bt_stride || (has1 && lp0 + 1 >= p.bt_stride)) {
            set_status(p.status, IDX_FP4_DEV_BAD_CTX);
            pid0 = lp0 >= p.bt_stride ? 0 : pid0;
            pid1 = 0;
          }
          if (pid0 < 0 || pid0 >= p.num_pages) {
            set_status(p.status, IDX_FP4_DEV_BAD_PAGE);
            pid0 = 0;
          }
          if (has1 && (pid1 < 0 || pid1 >= p.num_pages)) {
            set_status(p.status, IDX_FP4_DEV_BAD_PAGE);
            pid1 = 0;
          }
          const int s = f % STAGES;
          bounded_wait(&empty_bar[s], ((f / STAGES) & 1) ^ 1, abort_flag, p.status);
          uint8_t* dst = smem + C::OFF_PACKED + s * 8192;
          uint8_t* dsc = smem + C::OFF_SCALE + s * 512;
          mbar_arrive_expect_tx(&full_bar[s], (has1 ? 2u : 1u) * (kPageBytes + kPageScaleBytes));
          const uint8_t* src0 = p.kv_packed + static_cast<int64_t>(pid0) * kPageBytes;
          const uint8_t* src1 = p.kv_packed + static_cast<int64_t>(pid1) * kPageBytes;
          if (p.stream_once) {
#pragma unroll
            for (int g = 0; g < 4; ++g) bulk_load_evict_first(dst + g * 2048, src0 + g * 1024, 1024, &full_bar[s], pol);
            bulk_load_evict_first(dsc, p.kv_scale + static_cast<int64_t>(pid0) * kPageScaleBytes, 256, &full_bar[s], pol);
            if (has1) {
#pragma unroll
              for (int g = 0; g < 4; ++g)
                bulk_load_evict_first(dst + g * 2048 + 1024, src1 + g * 1024, 1024, &full_bar[s], pol);
              bulk_load_evict_first(dsc + 256, p.kv_scale + static_cast<int64_t>(pid1) * kPageScaleBytes, 256,
                                    &full_bar[s], pol);
            }
          } else {
#pragma unroll
            for (int g = 0; g < 4; ++g) bulk_load(dst + g * 2048, src0 + g * 1024, 1024, &full_bar[s]);
            bulk_load(dsc, p.kv_scale + static_cast<int64_t>(pid0) * kPageScaleBytes, 256, &full_bar[s]);
            if (has1) {
#pragma unroll
              for (int g = 0; g < 4; ++g) bulk_load(dst + g * 2048 + 1024, src1 + g * 1024, 1024, &full_bar[s]);
              bulk_load(dsc + 256, p.kv_scale + static_cast<int64_t>(pid1) * kPageScaleBytes, 256, &full_bar[s]);
            }
          }
        }
        __syncwarp();
        ++f;
      }
    }
    // After an abort the consumers stop waiting; drain this CTA's copies before teardown.
    if (lane == 0 && *abort_flag) {
      for (int k = f - STAGES < 0 ? 0 : f - STAGES; k < f; ++k)
        mbar_wait(&full_bar[k % STAGES], (k / STAGES) & 1, kWaitLimitNs);
      for (int i = it.count - 2 < 0 ? 0 : it.count - 2; i < it.count; ++i)
        mbar_wait(&unit_full[i & 1], (i >> 1) & 1, kWaitLimitNs);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    int f = 0, t = 0;
    for (int i = 0; i < it.count; ++i) {
      const Unit u = it.units[it.first + i * it.stride];
      const int par = i & 1;
      const uint8_t* raw = smem + C::OFF_UNIT + par * C::UNIT_BYTES;
      uint8_t* qb = smem + C::OFF_QB + par * (N * 64);
      uint8_t* sfb = smem + C::OFF_SFB + par * 512;
      bounded_wait(&unit_full[par], (i >> 1) & 1, abort_flag, p.status);
      if (lane == 0 && i >= 2) bounded_wait(&q_free[par], ((i >> 1) - 1) & 1, abort_flag, p.status);
      __syncwarp();
      // Plain [rows*H][64 B] query -> canonical K-major [4 chunks][N][16 B]; missing rows zeroed.
      const int live = u.nq * H;
      for (int c = lane; c < 4 * N; c += 32) {
        const int g = c / N, n = c % N;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (n < live) v = *reinterpret_cast<const uint4*>(raw + n * 64 + g * 16);
        *reinterpret_cast<uint4*>(qb + g * N * 16 + n * 16) = v;
      }
      // Query scales -> tensor-core scale layout: row n at line n%32, word n/32.
      for (int n = lane; n < 128; n += 32) {
        uint32_t wv = 0x7F7F7F7Fu;
        if (n < live) wv = *reinterpret_cast<const uint32_t*>(raw + C::RAW_Q + n * 4);
        *reinterpret_cast<uint32_t*>(sfb + (n & 31) * 16 + (n >> 5) * 4) = wv;
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&unit_empty[par]);
        tc_fence_after_sync();
        tmem_copy_sf_chunk(tmem + C::SFB_COL + 4 * par, smem_addr(sfb));
      }
      __syncwarp();
      const int ntiles = unit_tiles(u);
      for (int j = 0; j < ntiles; ++j, ++f, ++t) {
        const int s = f % STAGES;
        bounded_wait(&full_bar[s], (f / STAGES) & 1, abort_flag, p.status);
        // Scale bytes of the two pages -> tensor-core layout; key m = 64*page + row lives in
        // the cache at [page][group][(row % 16) * 4 + row / 16].
        const uint8_t* sc = smem + C::OFF_SCALE + s * 512;
        uint32_t w4[4];
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          const int m = lane + 32 * jj;
          const int pg = m >> 6, row = m & 63;
          const uint8_t* b = sc + pg * 256 + scale_slot(row);
          w4[jj] = static_cast<uint32_t>(b[0]) | (static_cast<uint32_t>(b[64]) << 8) |
                   (static_cast<uint32_t>(b[128]) << 16) | (static_cast<uint32_t>(b[192]) << 24);
        }
        uint8_t* sfa = smem + C::OFF_SFA + s * 512;
        *reinterpret_cast<uint4*>(sfa + lane * 16) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          const int a = t % ACC;
          bounded_wait(&acc_empty[a], ((t / ACC) & 1) ^ 1, abort_flag, p.status);
          tc_fence_after_sync();
          tmem_copy_sf_chunk(tmem + C::SFA_COL + 4 * a, smem_addr(sfa));
          const uint32_t a_base = smem_addr(smem + C::OFF_PACKED + s * 8192);
          const uint32_t b_base = smem_addr(qb);
          const uint32_t d = tmem + a * N;
          mma_mxf4(d, smem_desc(a_base, 2048, 128), smem_desc(b_base, N * 16, 128), mxf4_idesc(128, N, 0),
                   tmem + C::SFA_COL + 4 * a, tmem + C::SFB_COL + 4 * par, 0u);
          mma_mxf4(d, smem_desc(a_base + 4096, 2048, 128), smem_desc(b_base + 2 * N * 16, N * 16, 128),
                   mxf4_idesc(128, N, 2), tmem + C::SFA_COL + 4 * a, tmem + C::SFB_COL + 4 * par, 1u);
          tc_commit(&empty_bar[s]);
          tc_commit(&acc_full[a]);
        }
        __syncwarp();
      }
      if (lane == 0) tc_commit(&q_free[par]);
      __syncwarp();
    }
    if (lane == 0 && it.count > 0) {
      const int i = it.count - 1;
      mbar_wait(&q_free[i & 1], (i >> 1) & 1, kWaitLimitNs);
    }
    __syncwarp();
  } else {
    // ---------------- epilogue: head-weighted ReLU sum + streaming top-k ----------------
    const int qtr = warp & 3;               // TMEM lane quarter of this warp
    const int etid = qtr * 32 + lane;       // key row within the tile, and rank in the group
    const uint32_t lane_base = static_cast<uint32_t>(qtr * 32) << 16;
    uint2* cb_base = reinterpret_cast<uint2*>(smem + C::OFF_CB);
    uint32_t* hist = reinterpret_cast<uint32_t*>(smem + C::OFF_HIST);
    uint32_t* scr = reinterpret_cast<uint32_t*>(smem + C::OFF_SCR);
    uint32_t* wc = scr + 64;  // block_append scratch, 2*Q*4 words
    uint2* cb[Q];
#pragma unroll
    for (int r = 0; r < Q; ++r) cb[r] = cb_base + r * kCandCap;
    int t = 0, par = 0;
    for (int i = 0; i < it.count; ++i) {
      const Unit u = it.units[it.first + i * it.stride];
      const int upar = i & 1;
      const float* wsm = reinterpret_cast<const float*>(smem + C::OFF_UNIT + upar * C::UNIT_BYTES + C::RAW_Q +
                                                        C::RAW_QS);
      bounded_wait(&unit_full[upar], (i >> 1) & 1, abort_flag, p.status);
      int end[Q], cnt[Q];
      uint32_t tau[Q];
#pragma unroll
      for (int r = 0; r < Q; ++r) {
        int e = 0;
        if (r < u.nq) e = p.row_ends != nullptr ? min(max(p.row_ends[u.row + r], 0), u.ke) : u.ke;
        end[r] = e;
        cnt[r] = 0;
        tau[r] = 0u;
      }
      const int ntiles = unit_tiles(u);
      for (int j = 0; j < ntiles; ++j, ++t) {
        const int a = t % ACC;
        bounded_wait(&acc_full[a], (t / ACC) & 1, abort_flag, p.status);
        tc_fence_after_sync();
        float logit[Q];
#pragma unroll
        for (int r = 0; r < Q; ++r) {
          float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
          const uint32_t col = tmem + lane_base + a * N + r * H;
          if constexpr (H == 16) {
            float v[16];
            tmem_load_x16(col, v);
#pragma unroll
            for (int h = 0; h < 16; h += 4) {
              const float4 w = *reinterpret_cast<const float4*>(wsm + r * H + h);
              s0 = fmaf(w.x, fmaxf(v[h], 0.f), s0);
              s1 = fmaf(w.y, fmaxf(v[h + 1], 0.f), s1);
              s2 = fmaf(w.z, fmaxf(v[h + 2], 0.f), s2);
              s3 = fmaf(w.w, fmaxf(v[h + 3], 0.f), s3);
            }
          } else {
#pragma unroll
            for (int c = 0; c < H; c += 32) {
              float v[32];
              tmem_load_x32(col + c, v);
#pragma unroll
              for (int h = 0; h < 32; h += 4) {
                const float4 w = *reinterpret_cast<const float4*>(wsm + r * H + c + h);
                s0 = fmaf(w.x, fmaxf(v[h], 0.f), s0);
                s1 = fmaf(w.y, fmaxf(v[h + 1], 0.f), s1);
                s2 = fmaf(w.z, fmaxf(v[h + 2], 0.f), s2);
                s3 = fmaf(w.w, fmaxf(v[h + 3], 0.f), s3);
              }
            }
          }
          logit[r] = (s0 + s1) + (s2 + s3);
        }
        tc_fence_before_sync();
        mbar_arrive(&acc_empty[a]);
        const int key = u.kb + j * kTileKeys + etid;
        bool keep[Q];
        uint2 val[Q];
#pragma unroll
        for (int r = 0; r < Q; ++r) {
          const bool valid = key < end[r];
          const uint32_t uk = valid ? ordered_key(logit[r]) : 0u;
          keep[r] = valid && uk > tau[r];
          val[r] = make_uint2(uk, static_cast<uint32_t>(key));
          if (valid && p.logits_debug != nullptr && key < p.logits_stride)
            p.logits_debug[static_cast<int64_t>(u.row + r) * p.logits_stride + key] = logit[r];
        }
        block_append<Q, 4>(cb, cnt, keep, val, qtr, lane, wc, par, kEpiBarrier);
#pragma unroll
        for (int r = 0; r < Q; ++r) {
          if (cnt[r] > kCandCap - kTileKeys) {
            tau[r] = block_select<128>(cb[r], cnt[r], p.topk, hist, scr, etid, kEpiBarrier);
            cnt[r] = p.topk;
          }
        }
      }
      // unit inputs are no longer needed
      mbar_arrive(&unit_empty[upar]);
      // finalize each row: exactly min(k, valid keys) entries, in token order
#pragma unroll
      for (int r = 0; r < Q; ++r) {
        if (r >= u.nq) continue;
        const int nvalid = max(0, end[r] - u.kb);
        const int kk = min(p.topk, nvalid);
        if (cnt[r] > kk) {
          block_select<128>(cb[r], cnt[r], kk, hist, scr, etid, kEpiBarrier);
          cnt[r] = kk;
        }
        if (u.slot < 0) {
          const int64_t row = u.row + r;
          for (int e = etid; e < p.topk; e += 128) {
            const bool in = e < kk;
            const uint2 c = in ? cb[r][e] : make_uint2(0u, 0u);
            p.topk_idx[row * p.topk + e] = in ? static_cast<int32_t>(c.y) : -1;
            if (p.topk_val != nullptr) p.topk_val[row * p.topk + e] = in ? key_to_float(c.x) : -__int_as_float(0x7f800000);
          }
        } else {
          for (int e = etid; e < kk; e += 128) p.cand[static_cast<int64_t>(u.slot) * p.topk + e] = cb[r][e];
          if (etid == 0) p.cand_count[u.slot] = kk;
        }
        named_barrier_sync(kEpiBarrier, 128);
      }
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// Merge the per-unit candidate lists of each split sequence into its final top-k; also
// writes the all-padding output of sequences with no keys.
constexpr int kMergeThreads = 256;

__global__ void __launch_bounds__(kMergeThreads) merge_kernel(const void* sched, size_t sched_bytes,
                                                              const int32_t* ctx_lens, int batch, int topk,
                                                              const uint2* __restrict__ cand,
                                                              const int32_t* __restrict__ cand_count,
                                                              int32_t* topk_idx, float* topk_val, int32_t* status) {
  __shared__ uint2 cb[kCandCap];
  __shared__ uint32_t hist[2048];
  __shared__ uint32_t scr[select_scratch_words<kMergeThreads>() + 2 * 8];
  const DecodeSchedHeader* h = static_cast<const DecodeSchedHeader*>(sched);
  const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  if (h->magic != kDecodeMagic || h->batch != batch || h->max_batch < batch ||
      decode_sched_bytes(h->max_batch) > sched_bytes)
    return;  // flagged by the scorer
  const DecodeSchedView v = decode_sched_view(const_cast<void*>(sched), h->max_batch);
  const int ctx = v.seq_ctx[b];
  const int nu = v.seq_units[b];
  if (tid == 0 && ctx_lens[b] >= 0 && ctx_lens[b] != ctx) set_status(status, IDX_FP4_DEV_BAD_SCHEDULE);
  if (nu == 1) return;  // written by the scorer
  const int kk = min(topk, ctx);
  int cnt[1] = {0};
  uint32_t tau = 0u;
  int par = 0;
  uint32_t* wc = scr + select_scratch_words<kMergeThreads>();
  uint2* cbr[1] = {cb};
  for (int ui = 0; ui < nu; ++ui) {
    const int slot = v.seq_first[b] + ui;
    const int n = min(cand_count[slot], topk);
    for (int base = 0; base < n; base += kMergeThreads) {
      const int e = base + tid;
      const uint2 c = e < n ? cand[static_cast<int64_t>(slot) * topk + e] : make_uint2(0u, 0u);
      bool keep[1] = {e < n && c.x > tau};
      uint2 val[1] = {c};
      block_append<1, kMergeThreads / 32>(cbr, cnt, keep, val, w, lane, wc, par, 1);
      if (cnt[0] > kCandCap - kMergeThreads) {
        tau = block_select<kMergeThreads>(cb, cnt[0], topk, hist, scr, tid, 1);
        cnt[0] = topk;
      }
    }
  }
  if (cnt[0] > kk) {
    block_select<kMergeThreads>(cb, cnt[0], kk, hist, scr, tid, 1);
    cnt[0] = kk;
  }
  const int outn = min(cnt[0], kk);
  for (int e = tid; e < topk; e += kMergeThreads) {
    const bool in = e < outn;
    const uint2 c = in ? cb[e] : make_uint2(0u, 0u);
    topk_idx[static_cast<int64_t>(b) * topk + e] = in ? static_cast<int32_t>(c.y) : -1;
    if (topk_val != nullptr)
      topk_val[static_cast<int64_t>(b) * topk + e] = in ? key_to_float(c.x) : -__int_as_float(0x7f800000);
  }
}

template <int H, int Q>
cudaError_t launch_scorer_t(const ScorerParams& p, int grid, cudaStream_t stream) {
  using C = ScorerCfg<H, Q>;
  cudaError_t e = cudaFuncSetAttribute(scorer_kernel<H, Q>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(C::SMEM_BYTES));
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
                          int topk, const void* sched, size_t sched_bytes, void* workspace, int slots,
                          int32_t* topk_idx,
                          float* topk_val, float* logits_debug, int64_t logits_stride, int32_t* status, int grid,
                          cudaStream_t stream) {
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
  p.cand_count = static_cast<int32_t*>(workspace);
  p.cand = reinterpret_cast<uint2*>(static_cast<char*>(workspace) + round_up(sizeof(int32_t) * slots, 16));
  p.logits_debug = logits_debug;
  p.logits_stride = logits_stride;
  p.status = status;
  p.stream_once = 1;
  cudaError_t e = H == 128 ? launch_scorer_t<128, 1>(p, grid, stream) : launch_scorer_h<1>(H, p, grid, stream);
  if (e != cudaSuccess) return e;
  merge_kernel<<<batch, kMergeThreads, 0, stream>>>(sched, sched_bytes, ctx_lens, batch, topk, p.cand, p.cand_count,
                                                    topk_idx, topk_val, status);
  return cudaGetLastError();
}

cudaError_t launch_prefill(const uint8_t* q_packed, const uint8_t* q_scale, const float* weights,
                           const uint8_t* kv_packed, const uint8_t* kv_scale, int64_t num_pages,
                           const int32_t* block_tables, int bt_stride, const int32_t* row_ends, int H, int topk,
                           void* workspace, int32_t* topk_idx, float* topk_val, float* logits_debug,
                           int64_t logits_stride, int32_t* status, int grid, cudaStream_t stream) {
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
  p.logits_debug = logits_debug;
  p.logits_stride = logits_stride;
  p.status = status;
  p.stream_once = 0;
  if (H == 128) return launch_scorer_t<128, 1>(p, grid, stream);
  return launch_scorer_h<2>(H, p, grid, stream);
}

}  // namespace idxfp4
