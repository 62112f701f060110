// Decode work schedule and workspace layout, shared by the schedule builder, the decode kernel and
// the host-side sizing functions.
//
// The schedule ("Score a DSA sparse indexer in FP4", squashed commit message and section "Decode
// grid floor": a persistent-grid CTA schedule built once per step at a CUDA-graph-stable address)
// lays all sequences' 128-key tiles end to end and cuts them into `rounds x ctas` equal ranges of
// `per` tiles; range (r, c) is CTA c's work in round r. A range holds at most cap_tiles(next_n)
// tiles, so its logits fit the CTA's shared-memory row buffer. The piece of a sequence inside one
// range is a unit; the units of one sequence inside one round form a segment. A segment of one unit
// is selected inside its CTA; the units of a longer segment agree on the segment's threshold through
// an exchange in the workspace. A sequence spanning several rounds merges its segments' lists.
// With several query rows the ranges may instead be cut from the tiles with every sequence padded
// to whole ranges (header flag `aligned`), so that each sequence starts a range; a unit's tile0
// stays its position in the unpadded layout, which sizes the workspace.
#pragma once
#include <cstdint>

#include "common.cuh"

namespace idxfp4 {

constexpr uint32_t kDecodeMagic = 0x44534333u;  // "DSC3"
constexpr int kMaxNextN = 4;                     // query rows per sequence (speculative verify rows)
constexpr int kMinTilesPerRange = 32;  // a CTA's share is at least 4096 keys: a short sequence stays in
                                       // one CTA, since streaming 32 tiles there costs less than an exchange
                                       // between CTAs

// Tiles of one CTA range: its logits (4 bytes per key and row) fill the row buffer.
__host__ __device__ constexpr int decode_cap_tiles(int next_n) {
  return next_n <= 2 ? 128 : 64;
}

struct DecodeUnit {  // 32 bytes
  int32_t seq;
  int32_t kb, ke;    // keys [kb, ke) of the sequence
  int32_t buf;       // first row-buffer slot of the unit inside its CTA's range
  int32_t seg;       // segment id
  int32_t uidx;      // index of the unit inside its segment
  int32_t tile0;     // global index of the unit's first tile
  int32_t pad;
};

struct DecodeSeg {   // 32 bytes
  int32_t seq;
  int32_t first_unit;
  int32_t nunits;
  int32_t kb, ke;    // key span of the segment
  int32_t rank;      // index among the sequence's segments (rounds)
  int32_t tile0;     // global index of the segment's first tile
  int32_t pad;
};
static_assert(sizeof(DecodeUnit) == 32 && sizeof(DecodeSeg) == 32, "32-byte records");

struct DecodeSchedHeader {  // 64 bytes
  uint32_t magic;
  int32_t ctas;        // persistent grid the schedule was built for
  int32_t batch;
  int32_t max_batch;
  int32_t next_n;
  int32_t rounds;
  int32_t per;         // tiles per range
  int32_t num_units;
  int32_t num_segs;
  int32_t units_cap;
  int32_t segs_cap;
  int32_t ranges_cap;
  int32_t total_tiles;
  int32_t tiles_cap;   // max_batch * tiles(max_ctx): fixes the workspace's per-row strides
  int32_t ok;          // 0: the schedule could not be built (every row comes out empty)
  int32_t aligned;     // 1: every sequence starts a range (ranges cut from tiles padded per sequence)
};
static_assert(sizeof(DecodeSchedHeader) == 64, "64-byte header");

// Capacities of a schedule for (max_batch, max_ctx), for any next_n and any grid of up to kMaxCtas
// CTAs: rounds * ctas ranges of `per` tiles cover at most tiles / cap_tiles + ctas ranges, each range
// holds at most one unit more than its sequence boundaries, and a segment has at least one unit. The
// sizes depend on the arguments only (nothing is queried from a device); the header carries them and
// the workspace layout follows them.
struct DecodeCaps {
  int64_t tiles_cap, ranges_cap, units_cap, segs_cap;
};

__host__ __device__ inline DecodeCaps decode_caps(int max_batch, int64_t max_ctx) {
  DecodeCaps c;
  c.tiles_cap = static_cast<int64_t>(max_batch) * ((max_ctx + kTileKeys - 1) / kTileKeys);
  const int64_t cap = decode_cap_tiles(kMaxNextN);
  c.ranges_cap = (c.tiles_cap + cap - 1) / cap + kMaxCtas;
  c.units_cap = c.ranges_cap + max_batch;
  c.segs_cap = c.units_cap;
  return c;
}

// A sequence can span several rounds only when the tiles exceed one range.
__host__ __device__ inline bool decode_multi_round(const DecodeCaps& c) {
  return c.tiles_cap > decode_cap_tiles(kMaxNextN);
}

struct DecodeSchedView {
  DecodeSchedHeader* hdr;
  int32_t* range_first;  // [ranges_cap + 1]
  int32_t* seq_ctx;      // [max_batch]
  int32_t* seq_seg0;     // [max_batch] first segment of the sequence
  int32_t* seq_nseg;     // [max_batch] segments of the sequence (0: no keys)
  DecodeUnit* units;     // [units_cap]
  DecodeSeg* segs;       // [segs_cap]
};

__host__ __device__ inline size_t decode_units_offset(int max_batch, int64_t ranges_cap) {
  return round_up(sizeof(DecodeSchedHeader) + sizeof(int32_t) * (static_cast<size_t>(ranges_cap) + 1) +
                      3 * sizeof(int32_t) * static_cast<size_t>(max_batch),
                  32);
}

__host__ __device__ inline size_t decode_sched_bytes_for(int max_batch, const DecodeCaps& c) {
  return decode_units_offset(max_batch, c.ranges_cap) + sizeof(DecodeUnit) * static_cast<size_t>(c.units_cap) +
         sizeof(DecodeSeg) * static_cast<size_t>(c.segs_cap);
}

__host__ __device__ inline DecodeCaps decode_caps_of(const DecodeSchedHeader& h) {
  DecodeCaps c;
  c.tiles_cap = h.tiles_cap;
  c.ranges_cap = h.ranges_cap;
  c.units_cap = h.units_cap;
  c.segs_cap = h.segs_cap;
  return c;
}

__host__ __device__ inline DecodeSchedView decode_sched_view(void* base, int max_batch, int64_t ranges_cap,
                                                             int64_t units_cap) {
  DecodeSchedView v;
  char* p = static_cast<char*>(base);
  v.hdr = reinterpret_cast<DecodeSchedHeader*>(p);
  p += sizeof(DecodeSchedHeader);
  v.range_first = reinterpret_cast<int32_t*>(p);
  p += sizeof(int32_t) * (ranges_cap + 1);
  v.seq_ctx = reinterpret_cast<int32_t*>(p);
  p += sizeof(int32_t) * max_batch;
  v.seq_seg0 = reinterpret_cast<int32_t*>(p);
  p += sizeof(int32_t) * max_batch;
  v.seq_nseg = reinterpret_cast<int32_t*>(p);
  v.units = reinterpret_cast<DecodeUnit*>(static_cast<char*>(base) + decode_units_offset(max_batch, ranges_cap));
  v.segs = reinterpret_cast<DecodeSeg*>(v.units + units_cap);
  return v;
}

// ---- decode workspace -----------------------------------------------------------------------
// The workspace must be zero-filled before its first use; every call leaves its synchronisation
// words at zero again (a call that reports IDX_FP4_DEV_TIMEOUT may not).
//   sync      [segs_cap][next_n] x 4 words: arrivals of the segment's units (histograms published),
//             arrivals after emitting candidates, 0, 0
//   seqsync   [max_batch][next_n] x 4 words: segments of the sequence finished, 0, 0, 0
//   records   [next_n][tiles_cap * 128 + units_cap] words: unit u's histogram records at
//             tile0 * 128 + u (a count, then (bin << 17 | keys) per non-empty bin at or above the
//             unit's own threshold bin)
//   cands     [next_n][tiles_cap * 128] (ordered key, token index) pairs: segment s's candidates at
//             s.tile0 * 128, its units' lists one after another in token order
//   seglists  [segs_cap][next_n][topk] pairs: a segment's exact top-k, when the sequence has several
//             segments (absent when no sequence can span two rounds)
struct DecodeWs {
  uint32_t* sync;
  uint32_t* seqsync;
  uint32_t* records;
  uint2* cands;
  uint2* seglists;
  int64_t rec_stride;   // words per row
  int64_t cand_stride;  // pairs per row
};

__host__ __device__ inline size_t decode_ws_sync_bytes(const DecodeCaps& c, int max_batch, int next_n) {
  return 16 * static_cast<size_t>(next_n) * (static_cast<size_t>(c.segs_cap) + static_cast<size_t>(max_batch));
}

__host__ __device__ inline size_t decode_ws_bytes_for(const DecodeCaps& c, int max_batch, int next_n, int topk) {
  const size_t sync = round_up(decode_ws_sync_bytes(c, max_batch, next_n), 256);
  const size_t rec = round_up(4 * static_cast<size_t>(next_n) * (static_cast<size_t>(c.tiles_cap) * kTileKeys +
                                                                   static_cast<size_t>(c.units_cap)),
                              256);
  const size_t cand = 8 * static_cast<size_t>(next_n) * static_cast<size_t>(c.tiles_cap) * kTileKeys;
  const size_t segl = decode_multi_round(c) ? 8 * static_cast<size_t>(c.segs_cap) * next_n * topk : 0;
  return sync + rec + cand + segl;
}

__host__ __device__ inline DecodeWs decode_ws_view(void* base, const DecodeCaps& c, int max_batch, int next_n) {
  DecodeWs w;
  char* p = static_cast<char*>(base);
  w.sync = reinterpret_cast<uint32_t*>(p);
  w.seqsync = w.sync + 4 * static_cast<size_t>(next_n) * c.segs_cap;
  p += round_up(decode_ws_sync_bytes(c, max_batch, next_n), 256);
  w.records = reinterpret_cast<uint32_t*>(p);
  w.rec_stride = c.tiles_cap * kTileKeys + c.units_cap;
  p += round_up(4 * static_cast<size_t>(next_n) * static_cast<size_t>(w.rec_stride), 256);
  w.cands = reinterpret_cast<uint2*>(p);
  w.cand_stride = c.tiles_cap * kTileKeys;
  p += 8 * static_cast<size_t>(next_n) * static_cast<size_t>(w.cand_stride);
  w.seglists = reinterpret_cast<uint2*>(p);
  return w;
}

}  // namespace idxfp4
