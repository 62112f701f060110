// Decode schedule builder ("Score a DSA sparse indexer in FP4", squashed commit message and section
// "Decode grid floor": the decode scorer runs on a persistent grid whose CTA schedule is built once
// per step, before the layers, at a CUDA-graph-stable address; a schedule that under-covers rows is an
// error, never a silent truncation).
//
// The pages size their grid as a fixed floor of CTAs and measure the cost of CTAs past the work. Here
// the grid is the SM count and the work is cut to it on the device, from the context lengths the
// step's graph reads: all sequences' 128-key tiles are laid end to end and cut into rounds x ctas
// ranges of `per` tiles. No count on the host depends on device data, so a captured graph replays
// across changing context lengths. One CTA builds the tables with block scans.
//
// A key-range schedule ("Score a DSA sparse indexer in FP4", section "Decode context parallelism":
// each rank scores its own shard of a sequence's keys and its local top-k is merged with the
// others') gives each sequence the keys [key_begin, ctx): the first key is a multiple of the
// 128-key tile, units and segments carry absolute key positions, and the row end stays ctx.
#include <cuda_runtime.h>

#include <cstdint>

#include "common.cuh"
#include "decode_sched.cuh"

namespace idxfp4 {
namespace {

constexpr int kThreads = 1024;
constexpr int kPer = kMaxBatch / kThreads;  // sequences per thread in the scans

// Exclusive scan over the block (one value per thread); the total goes to *total (shared).
__device__ int scan_excl(int v, int* warp_sums, int* total) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int t = __shfl_up_sync(0xFFFFFFFFu, incl, off);
    if (lane >= off) incl += t;
  }
  if (lane == 31) warp_sums[w] = incl;
  __syncthreads();
  if (w == 0) {
    const int s = warp_sums[lane];
    int si = s;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int t = __shfl_up_sync(0xFFFFFFFFu, si, off);
      if (lane >= off) si += t;
    }
    warp_sums[lane] = si - s;
    if (lane == 31) *total = si;
  }
  __syncthreads();
  const int r = warp_sums[w] + incl - v;
  __syncthreads();
  return r;
}

__device__ __forceinline__ void build_decode_schedule_body(const int32_t* __restrict__ ctx_lens,
                                                           const int32_t* __restrict__ key_begin, int batch,
                                                           int next_n, int max_batch, int64_t max_ctx, int ctas,
                                                           DecodeCaps caps, void* sched, int32_t* status) {
  extern __shared__ int s_dyn[];
  int* s_start = s_dyn;                   // [kMaxBatch + 1] first tile of each sequence
  int* s_ne = s_start + kMaxBatch + 1;    // [kMaxBatch + 1] non-empty sequences before each
  int* s_seg0 = s_ne + kMaxBatch + 1;     // [kMaxBatch + 1] segments before each
  int* s_kb0 = s_seg0 + kMaxBatch + 1;    // [kMaxBatch + 1] first key of each sequence's range
  int* s_astart = s_kb0 + kMaxBatch + 1;  // [kMaxBatch + 1] first tile of each sequence, tiles end to end
  __shared__ int warp_sums[32];
  __shared__ int s_total, s_nonempty, s_segs, s_chunk;
  const int tid = threadIdx.x;
  DecodeSchedView v = decode_sched_view(sched, max_batch, caps.ranges_cap, caps.units_cap);

  // 1. tiles per sequence and their prefix sums
  int tiles[kPer], ne[kPer];
  int my_tiles = 0, my_ne = 0;
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const int b = tid * kPer + j;
    int c = 0, k0 = 0;
    if (b < batch) {
      const int64_t raw = ctx_lens[b];
      if (raw < 0 || raw > max_ctx) set_status(status, IDX_FP4_DEV_BAD_CTX);
      else c = static_cast<int>(raw);
      if (key_begin != nullptr) {
        const int64_t kb = key_begin[b];
        if (kb < 0 || kb > c || kb % kTileKeys != 0) {
          set_status(status, IDX_FP4_DEV_BAD_CTX);
          k0 = c;  // no keys
        } else {
          k0 = static_cast<int>(kb);
        }
      }
      s_kb0[b] = k0;
    }
    tiles[j] = (c - k0 + kTileKeys - 1) / kTileKeys;
    ne[j] = tiles[j] > 0 ? 1 : 0;
    my_tiles += tiles[j];
    my_ne += ne[j];
  }
  int off = scan_excl(my_tiles, warp_sums, &s_total);
  int off_ne = scan_excl(my_ne, warp_sums, &s_nonempty);
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const int b = tid * kPer + j;
    s_start[b] = off;
    s_ne[b] = off_ne;
    off += tiles[j];
    off_ne += ne[j];
  }
  if (tid == 0) {
    s_start[kMaxBatch] = s_total;
    s_ne[kMaxBatch] = s_nonempty;
  }
  __syncthreads();
  const int total = s_total;
  for (int b = tid; b <= kMaxBatch; b += kThreads) s_astart[b] = s_start[b];

  // 2. rounds and range length
  const int cap = decode_cap_tiles(next_n);
  const int64_t slab = static_cast<int64_t>(ctas) * cap;
  const int rounds = total > 0 ? static_cast<int>((total + slab - 1) / slab) : 1;
  int per = static_cast<int>((static_cast<int64_t>(total) + static_cast<int64_t>(ctas) * rounds - 1) /
                             (static_cast<int64_t>(ctas) * rounds));
  if (rounds == 1 && per < kMinTilesPerRange) per = kMinTilesPerRange;
  if (per > cap) per = cap;
  if (per < 1) per = 1;

  // 2b. With several query rows, ranges aligned to the sequences when that keeps the rounds: every
  // sequence then starts a range, so no CTA holds the ends of two sequences (whose units each
  // selection group would settle row after row). The ranges are cut from the sequences' tiles
  // padded to whole ranges ("virtual" tiles, s_start); units keep their tile numbers (s_astart).
  // Each warp tries one range length from `per` up and the smallest that fits the ranges wins.
  int aligned = 0;
  if (next_n > 1 && total > 0) {
    const int w = tid >> 5, lane = tid & 31;
    const int step = max(1, (cap - per + 31) / 32);
    const int cand = per + w * step;
    int need = 0;
    if (cand <= cap)
      for (int b = lane; b < batch; b += 32) need += (s_astart[b + 1] - s_astart[b] + cand - 1) / cand;
    need = __reduce_add_sync(0xFFFFFFFFu, need);
    if (lane == 0) warp_sums[w] = cand <= cap && need <= rounds * ctas ? cand : 0x7FFFFFFF;
    __syncthreads();
    if (w == 0) {
      const int best = __reduce_min_sync(0xFFFFFFFFu, warp_sums[lane]);
      if (lane == 0) s_chunk = best;
    }
    __syncthreads();
    if (s_chunk != 0x7FFFFFFF) {
      per = s_chunk;
      aligned = 1;
    }
    __syncthreads();
  }
  int total_v = total;  // tiles of the layout the ranges are cut from
  if (aligned) {
    int vt[kPer], my_v = 0;
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      vt[j] = (tiles[j] + per - 1) / per * per;
      my_v += vt[j];
    }
    int offv = scan_excl(my_v, warp_sums, &s_total);
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      s_start[tid * kPer + j] = offv;
      offv += vt[j];
    }
    if (tid == 0) s_start[kMaxBatch] = s_total;
    __syncthreads();
    total_v = s_total;
  }
  const int ranges = rounds * ctas;
  const int64_t round_tiles = static_cast<int64_t>(ctas) * per;
  bool ok = ranges <= caps.ranges_cap && total <= caps.tiles_cap;

  // the sequence holding tile x: the last b with start[b] <= x (never an empty one)
  auto seq_of = [&](int x) {
    int lo = 0, hi = batch - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_start[mid] <= x) lo = mid; else hi = mid - 1;
    }
    return lo;
  };
  // the end of sequence b's tiles in the layout (before any padding)
  auto seq_end = [&](int b) {
    const int n = b + 1 <= kMaxBatch ? b + 1 : kMaxBatch;
    return s_start[b] + (s_astart[n] - s_astart[b]);
  };

  // 3. segments per sequence: one per round the sequence's tiles touch
  int nseg[kPer], my_segs = 0;
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const int b = tid * kPer + j;
    nseg[j] = 0;
    if (b < batch && tiles[j] > 0) {
      const int64_t r0 = s_start[b] / round_tiles, r1 = (s_start[b] + tiles[j] - 1) / round_tiles;
      nseg[j] = static_cast<int>(r1 - r0 + 1);
    }
    my_segs += nseg[j];
  }
  int off_seg = scan_excl(my_segs, warp_sums, &s_segs);
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const int b = tid * kPer + j;
    s_seg0[b] = off_seg;
    off_seg += nseg[j];
  }
  __syncthreads();
  ok = ok && s_segs <= caps.segs_cap;

  // Everything above read only the caller's inputs; the tables below overwrite the schedule that
  // the kernel before this one may still be reading.
  pdl_wait();
  // the validated context of sequence b
  auto ctx_of = [&](int b) {
    const int64_t raw = ctx_lens[b];
    return raw < 0 || raw > max_ctx ? 0 : static_cast<int>(raw);
  };

  // 4. units per range, and each range's first unit
  int running = 0;
  for (int base = 0; base < ranges; base += kThreads) {
    const int i = base + tid;
    int cnt = 0;
    if (i < ranges) {
      const int64_t lo = static_cast<int64_t>(i) * per;
      if (lo < total_v) {
        const int hi = static_cast<int>(lo + per < total_v ? lo + per : total_v);
        cnt = s_ne[seq_of(hi - 1) + 1] - s_ne[seq_of(static_cast<int>(lo))];
      }
    }
    const int ex = scan_excl(cnt, warp_sums, &s_chunk);
    if (ok && i < ranges) v.range_first[i] = running + ex;
    running += s_chunk;
  }
  const int num_units = running;
  ok = ok && num_units <= caps.units_cap;
  if (ok && tid == 0) v.range_first[ranges] = num_units;

  // 5. units, in range order (= tile order)
  if (ok) {
    for (int i = tid; i < ranges; i += kThreads) {
      const int64_t lo64 = static_cast<int64_t>(i) * per;
      if (lo64 >= total_v) continue;
      const int lo = static_cast<int>(lo64);
      const int hi = lo + per < total_v ? lo + per : total_v;
      const int b0 = seq_of(lo), b1 = seq_of(hi - 1);
      const int r = i / ctas;
      int idx = v.range_first[i];
      for (int b = b0; b <= b1; ++b) {
        const int sb = s_start[b], eb = seq_end(b);
        if (eb == sb) continue;
        const int ulo = lo > sb ? lo : sb, uhi = hi < eb ? hi : eb;
        const int r0 = static_cast<int>(sb / round_tiles);
        const int64_t seg_lo = static_cast<int64_t>(r) * round_tiles > sb ? static_cast<int64_t>(r) * round_tiles : sb;
        DecodeUnit u;
        u.seq = b;
        u.kb = s_kb0[b] + (ulo - sb) * kTileKeys;
        u.ke = min(s_kb0[b] + (uhi - sb) * kTileKeys, ctx_of(b));
        u.buf = (ulo - lo) * kTileKeys;
        u.seg = s_seg0[b] + (r - r0);
        u.uidx = i - static_cast<int>(seg_lo / per);
        u.tile0 = s_astart[b] + (ulo - sb);
        u.pad = 0;
        v.units[idx++] = u;
      }
    }
  }
  __syncthreads();

  // 6. segments, per sequence in round order; sequences with no keys get none
  for (int b = tid; b < batch; b += kThreads) {
    const int sb = s_start[b], eb = seq_end(b);
    const int n = ok ? s_seg0[b + 1 <= kMaxBatch ? b + 1 : kMaxBatch] - s_seg0[b] : 0;
    v.seq_ctx[b] = ctx_of(b);
    v.seq_seg0[b] = s_seg0[b];
    v.seq_nseg[b] = eb > sb ? n : 0;
    if (!ok || eb == sb) continue;
    const int r0 = static_cast<int>(sb / round_tiles);
    for (int k = 0; k < n; ++k) {
      const int r = r0 + k;
      const int64_t rlo = static_cast<int64_t>(r) * round_tiles, rhi = rlo + round_tiles;
      const int slo = static_cast<int>(rlo > sb ? rlo : sb), shi = static_cast<int>(rhi < eb ? rhi : eb);
      const int i0 = slo / per, i1 = (shi - 1) / per;
      DecodeSeg s;
      s.seq = b;
      s.first_unit = v.range_first[i0] + (s_ne[b] - s_ne[seq_of(i0 * per)]);
      s.nunits = i1 - i0 + 1;
      s.kb = s_kb0[b] + (slo - sb) * kTileKeys;
      s.ke = min(s_kb0[b] + (shi - sb) * kTileKeys, ctx_of(b));
      s.rank = k;
      s.tile0 = s_astart[b] + (slo - sb);
      s.pad = 0;
      v.segs[s_seg0[b] + k] = s;
    }
  }
  if (!ok && tid == 0) set_status(status, IDX_FP4_DEV_CAPACITY);
  if (tid == 0) {
    DecodeSchedHeader h{};
    h.magic = kDecodeMagic;
    h.ctas = ctas;
    h.batch = batch;
    h.max_batch = max_batch;
    h.next_n = next_n;
    h.rounds = ok ? rounds : 0;
    h.per = per;
    h.num_units = ok ? num_units : 0;
    h.num_segs = ok ? s_segs : 0;
    h.units_cap = static_cast<int32_t>(caps.units_cap);
    h.segs_cap = static_cast<int32_t>(caps.segs_cap);
    h.ranges_cap = static_cast<int32_t>(caps.ranges_cap);
    h.total_tiles = total;
    h.tiles_cap = static_cast<int32_t>(caps.tiles_cap);
    h.ok = ok ? 1 : 0;
    h.aligned = aligned;
    *v.hdr = h;
  }
}

// The builder reads only its caller's inputs (never what a kernel of this library writes), so it
// starts at once, beside the kernel before it (the writer, when a step runs writer, schedule and
// decode), and waits for that kernel only before its first write to the schedule: its completion
// still implies its predecessor's, which the decode kernel launched after it relies on.
__global__ void __launch_bounds__(kThreads) build_decode_schedule_kernel(const int32_t* __restrict__ ctx_lens,
                                                                        const int32_t* __restrict__ key_begin,
                                                                        int batch, int next_n, int max_batch,
                                                                        int64_t max_ctx, int ctas, DecodeCaps caps,
                                                                        void* sched, int32_t* status) {
  pdl_trigger();
  build_decode_schedule_body(ctx_lens, key_begin, batch, next_n, max_batch, max_ctx, ctas, caps, sched, status);
  pdl_wait();
}

}  // namespace

cudaError_t launch_build_decode_schedule(const int32_t* ctx_lens, const int32_t* key_begin, int batch, int next_n,
                                         int max_batch, int64_t max_ctx, int ctas, const DecodeCaps& caps,
                                         void* sched, int32_t* status, cudaStream_t stream) {
  constexpr size_t smem = sizeof(int) * (5 * (kMaxBatch + 1));
  cudaError_t e = set_smem_once<build_decode_schedule_kernel>(smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(build_decode_schedule_kernel, dim3(1), dim3(kThreads), smem, stream, 1, false, ctx_lens,
                    key_begin, batch, next_n, max_batch, max_ctx, ctas, caps, sched, status);
}

}  // namespace idxfp4
