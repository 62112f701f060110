// Test oracle for the MXFP4 DSA lightning indexer.
//
// THIS IS TEST INFRASTRUCTURE. Only the test suite, the package's smoke check and
// the benchmark's CPU-baseline leg may load it. The product path (the CUDA
// library) never calls, links or includes anything in this directory, and this
// file includes no header of the CUDA library.
//
// Plain C++17, every floating-point step in fp64, plain loops, no blocking or
// fusion beyond what the definitions state. The sources it restates:
//
//   [P2] "Score a DSA sparse indexer in FP4" (ROCm/ATOM pull 2216): the squashed
//        commit message (keys kept as packed E2M1 plus e8m0 scales in a paged index
//        region, read in place by decode and prefill; page size 64), the review's
//        second finding (the test oracle's read of the two planes, with the scale
//        plane's in-page row index permuted as (pos % 16) * 4 + pos // 16), the
//        sub-commit "Use the index scale plane's own row order when staging FP4
//        prefill under DCP" (packed plane flat, scale plane a 16x4 transpose), and
//        the sub-commit "Schedule, refuse and document the FP4 indexer paths the
//        review found" (the fused writer skips rows whose slot is negative; the
//        prefill top-k takes per-row [row_start, row_end) bounds).
//   [P1] "PCP correctness fixes" (ROCm/ATOM pull 2125), Technical Details section 3
//        "FP4 indexer padding rows": padding rows sit at position 0 and read no key.
//   The indexer score  logit[q, t] = sum_h w[q, h] * relu(q_h . k_t)  is the DSA
//   lightning-indexer formula the pages score; the MXFP4 block rule (one e8m0 scale
//   per 32 dims, scale = the smallest power of two that brings the block's largest
//   magnitude within the E2M1 range, elements rounded to nearest with ties to the
//   even code) is the workload's stated quantiser.
//
// Readings taken where the pages are silent:
//   R1  Nibble order: element 2i in bits 0..3, element 2i+1 in bits 4..7 of byte i.
//   R2  The sign bit of a code is set iff the input is negative, so a small negative
//       value that rounds to zero encodes as -0 (code 8).
//   R3  An all-zero block takes scale byte 0 (2^-127) and all-zero codes.
//   R4  Packed plane [page][group 0..3][row 0..63][16 bytes]; scale plane
//       [page][group][(row % 16) * 4 + row / 16]. The singleton axis of the page's
//       oracle read is dropped.
//   R5  A prefill row at 0-based position p scores keys [0, p + 1); a padding row
//       has row_end = 0 and scores nothing.
//   R6  Top-k is the set of the min(k, n) best keys by (logit descending, index
//       ascending); the output is padded with index -1 and value -inf.
//   (R7-R11 are the quantiser rule stated above, queries quantised alike, the 68-byte key,
//   the prefill padding variants and the next_n visible-key rule; they need no function here.)
//   R12 Key-sharded decode ([P2], section "Decode context parallelism": each rank scores its
//       shard of the keys, keeps its local top-k, and the gathered candidates are merged): a
//       shard is a contiguous key range [key_begin, key_end) of the sequence; its top-k uses
//       the absolute token index; the merge keeps the min(k, n) best of the union of the
//       shards' lists by the R6 order.

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <thread>
#include <vector>

namespace {

constexpr int kHeadDim = 128;
constexpr int kBlock = 32;                       // dims per e8m0 scale
constexpr int kGroups = kHeadDim / kBlock;       // 4 scale groups per key
constexpr int kPage = 64;                        // keys per page
constexpr int kPackedPerGroup = kBlock / 2;      // 16 bytes of nibbles per group
constexpr int kPageBytes = kGroups * kPage * kPackedPerGroup;  // 4096
constexpr int kPageScaleBytes = kGroups * kPage;               // 256

// E2M1 magnitudes by the low three bits of a code (OCP MX element format E2M1).
const double kE2M1[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

double bf16_to_double(uint16_t h) {
  uint32_t bits = static_cast<uint32_t>(h) << 16;
  float f;
  std::memcpy(&f, &bits, sizeof f);
  return static_cast<double>(f);
}

// Smallest integer e with amax <= 6 * 2^e, clamped to the e8m0 range [-127, 127].
int block_exponent(double amax) {
  if (amax == 0.0) return -127;
  int e = static_cast<int>(std::ceil(std::log2(amax / 6.0)));
  while (std::ldexp(6.0, e) < amax) ++e;        // make the bound hold exactly
  while (std::ldexp(6.0, e - 1) >= amax) --e;   // and make e the smallest such
  if (e < -127) e = -127;
  if (e > 127) e = 127;
  return e;
}

// Round a magnitude (already divided by the block scale) to the E2M1 grid: nearest
// value, ties to the code whose mantissa bit is 0. Returns the 3-bit magnitude code.
int e2m1_round(double y) {
  if (!(y > 0.0)) return 0;
  if (y >= 6.0) return 7;  // saturate (never reached when the scale is chosen above)
  int best = 0;
  double best_d = std::numeric_limits<double>::infinity();
  for (int c = 0; c < 8; ++c) {
    double d = std::fabs(y - kE2M1[c]);
    if (d < best_d || (d == best_d && (c & 1) == 0)) {
      best = c;
      best_d = d;
    }
  }
  return best;
}

double e2m1_value(int code) {
  double v = kE2M1[code & 7];
  return (code & 8) ? -v : v;
}

double e8m0_value(uint8_t s) {
  if (s == 0xFF) return std::numeric_limits<double>::quiet_NaN();
  return std::ldexp(1.0, static_cast<int>(s) - 127);
}

// Encode one 128-dim bf16 vector: 64 packed bytes (R1) and 4 scale bytes.
void encode_vector(const uint16_t* x, uint8_t* packed, uint8_t* scales) {
  for (int g = 0; g < kGroups; ++g) {
    double amax = 0.0;
    for (int i = 0; i < kBlock; ++i) amax = std::max(amax, std::fabs(bf16_to_double(x[g * kBlock + i])));
    const int e = block_exponent(amax);
    scales[g] = static_cast<uint8_t>(e + 127);
    for (int i = 0; i < kBlock; i += 2) {
      uint8_t byte = 0;
      for (int j = 0; j < 2; ++j) {
        const double v = bf16_to_double(x[g * kBlock + i + j]);
        const int mag = e2m1_round(std::fabs(std::ldexp(v, -e)));
        const int code = (v < 0.0 ? 8 : 0) | mag;  // R2
        byte |= static_cast<uint8_t>(code << (4 * j));
      }
      packed[g * kPackedPerGroup + i / 2] = byte;
    }
  }
}

int scale_slot(int row) { return (row % 16) * 4 + row / 16; }  // R4

// Dequantise key (page, row) of the paged cache into 128 doubles.
void read_key(const uint8_t* kv_packed, const uint8_t* kv_scale, int64_t page, int row, double* out) {
  for (int g = 0; g < kGroups; ++g) {
    const uint8_t* src = kv_packed + page * kPageBytes + (static_cast<int64_t>(g) * kPage + row) * kPackedPerGroup;
    const double s = e8m0_value(kv_scale[page * kPageScaleBytes + g * kPage + scale_slot(row)]);
    for (int i = 0; i < kPackedPerGroup; ++i) {
      out[g * kBlock + 2 * i] = e2m1_value(src[i] & 0xF) * s;
      out[g * kBlock + 2 * i + 1] = e2m1_value(src[i] >> 4) * s;
    }
  }
}

// Dequantise a plainly laid out query head: 64 packed bytes + 4 scales.
void read_plain(const uint8_t* packed, const uint8_t* scales, double* out) {
  for (int g = 0; g < kGroups; ++g) {
    const double s = e8m0_value(scales[g]);
    for (int i = 0; i < kPackedPerGroup; ++i) {
      out[g * kBlock + 2 * i] = e2m1_value(packed[g * kPackedPerGroup + i] & 0xF) * s;
      out[g * kBlock + 2 * i + 1] = e2m1_value(packed[g * kPackedPerGroup + i] >> 4) * s;
    }
  }
}

// One query row against one key: sum_h w[h] * max(q_h . k, 0) in fp64.
double score(const std::vector<double>& q /*H*128*/, const float* w, int H, const double* k) {
  double logit = 0.0;
  for (int h = 0; h < H; ++h) {
    double s = 0.0;
    for (int d = 0; d < kHeadDim; ++d) s += q[static_cast<size_t>(h) * kHeadDim + d] * k[d];
    logit += static_cast<double>(w[h]) * std::max(s, 0.0);
  }
  return logit;
}

std::vector<double> read_query(const uint8_t* q_packed, const uint8_t* q_scale, int64_t r, int H) {
  std::vector<double> q(static_cast<size_t>(H) * kHeadDim);
  for (int h = 0; h < H; ++h)
    read_plain(q_packed + (r * H + h) * 64, q_scale + (r * H + h) * 4, q.data() + static_cast<size_t>(h) * kHeadDim);
  return q;
}

// Logits of one query row over keys [t0, t1) of one page table.
void row_logits(const uint8_t* q_packed, const uint8_t* q_scale, const float* w, int64_t r, int H,
                const uint8_t* kv_packed, const uint8_t* kv_scale, const int32_t* table, int64_t t0, int64_t t1,
                double* out) {
  const std::vector<double> q = read_query(q_packed, q_scale, r, H);
  double k[kHeadDim];
  for (int64_t t = t0; t < t1; ++t) {
    read_key(kv_packed, kv_scale, table[t / kPage], static_cast<int>(t % kPage), k);
    out[t - t0] = score(q, w + r * H, H, k);
  }
}

// R6: the min(k, n) best by (value desc, index asc), padded with -1 / -inf.
void select_topk(const double* logits, int64_t n, int k, int32_t* idx, double* val) {
  std::vector<int64_t> order(static_cast<size_t>(n));
  for (int64_t i = 0; i < n; ++i) order[static_cast<size_t>(i)] = i;
  std::sort(order.begin(), order.end(), [&](int64_t a, int64_t b) {
    if (logits[a] != logits[b]) return logits[a] > logits[b];
    return a < b;
  });
  const int64_t m = std::min<int64_t>(k, n);
  for (int64_t i = 0; i < k; ++i) {
    if (i < m) {
      idx[i] = static_cast<int32_t>(order[static_cast<size_t>(i)]);
      val[i] = logits[order[static_cast<size_t>(i)]];
    } else {
      idx[i] = -1;
      val[i] = -std::numeric_limits<double>::infinity();
    }
  }
}

template <class F>
void parallel_for(int64_t n, int threads, F&& f) {
  if (threads <= 1 || n <= 1) {
    for (int64_t i = 0; i < n; ++i) f(i);
    return;
  }
  std::vector<std::thread> pool;
  for (int t = 0; t < threads; ++t)
    pool.emplace_back([&, t] {
      for (int64_t i = t; i < n; i += threads) f(i);
    });
  for (auto& th : pool) th.join();
}

}  // namespace

extern "C" {

int orc_version() { return 1; }

int orc_scale_slot(int row) { return scale_slot(row); }

int orc_block_exponent(double amax) { return block_exponent(amax); }

int orc_e2m1_round(double y) { return e2m1_round(y); }

double orc_e2m1_value(int code) { return e2m1_value(code); }

// Quantise n_vec bf16 vectors of 128 dims into plain [n_vec][64] + [n_vec][4].
void orc_quantize_plain(const uint16_t* x, int64_t n_vec, uint8_t* packed, uint8_t* scales) {
  for (int64_t v = 0; v < n_vec; ++v) encode_vector(x + v * kHeadDim, packed + v * 64, scales + v * 4);
}

// Dequantise n_vec plain vectors into fp64 [n_vec][128].
void orc_dequantize_plain(const uint8_t* packed, const uint8_t* scales, int64_t n_vec, double* out) {
  for (int64_t v = 0; v < n_vec; ++v) read_plain(packed + v * 64, scales + v * 4, out + v * kHeadDim);
}

// Cache writer: token i goes to slot slot_mapping[i] (page = slot / 64, row = slot % 64);
// negative slots are skipped. Returns the number of tokens written, or -1 if a slot
// lies past the pool (nothing is written for such a token).
int64_t orc_quant_and_cache(const uint16_t* k, int64_t num_tokens, const int32_t* slot_mapping, uint8_t* kv_packed,
                            uint8_t* kv_scale, int64_t num_pages) {
  int64_t written = 0;
  bool bad = false;
  for (int64_t i = 0; i < num_tokens; ++i) {
    const int64_t slot = slot_mapping[i];
    if (slot < 0) continue;
    if (slot >= num_pages * kPage) {
      bad = true;
      continue;
    }
    const int64_t page = slot / kPage;
    const int row = static_cast<int>(slot % kPage);
    uint8_t packed[64], scales[4];
    encode_vector(k + i * kHeadDim, packed, scales);
    for (int g = 0; g < kGroups; ++g) {
      std::memcpy(kv_packed + page * kPageBytes + (static_cast<int64_t>(g) * kPage + row) * kPackedPerGroup,
                  packed + g * kPackedPerGroup, kPackedPerGroup);
      kv_scale[page * kPageScaleBytes + g * kPage + scale_slot(row)] = scales[g];
    }
    ++written;
  }
  return bad ? -1 : written;
}

// Read key (page, row) back from the cache as fp64 [128].
void orc_read_key(const uint8_t* kv_packed, const uint8_t* kv_scale, int64_t page, int row, double* out) {
  read_key(kv_packed, kv_scale, page, row, out);
}

// Decode logits: row b scores keys [0, ctx_lens[b]) through block_tables[b]; out is
// [batch][out_stride] fp64, entries past ctx_lens[b] untouched.
void orc_decode_logits(const uint8_t* q_packed, const uint8_t* q_scale, const float* w, const uint8_t* kv_packed,
                       const uint8_t* kv_scale, const int32_t* block_tables, int64_t bt_stride, const int32_t* ctx_lens,
                       int batch, int H, double* out, int64_t out_stride, int threads) {
  parallel_for(batch, threads, [&](int64_t b) {
    row_logits(q_packed, q_scale, w, b, H, kv_packed, kv_scale, block_tables + b * bt_stride, 0, ctx_lens[b],
               out + b * out_stride);
  });
}

// Logits of one query row r over keys [t0, t1) of a page table (for sampled checks).
void orc_row_logits(const uint8_t* q_packed, const uint8_t* q_scale, const float* w, int64_t r, int H,
                    const uint8_t* kv_packed, const uint8_t* kv_scale, const int32_t* table, int64_t t0, int64_t t1,
                    double* out) {
  row_logits(q_packed, q_scale, w, r, H, kv_packed, kv_scale, table, t0, t1, out);
}

// Prefill logits: row r belongs to request g with cu_seqlens[g] <= r < cu_seqlens[g+1]
// and scores keys [0, row_ends[r]) through block_tables[g].
void orc_prefill_logits(const uint8_t* q_packed, const uint8_t* q_scale, const float* w, const uint8_t* kv_packed,
                        const uint8_t* kv_scale, const int32_t* block_tables, int64_t bt_stride,
                        const int32_t* cu_seqlens, const int32_t* row_ends, int num_requests, int num_rows, int H,
                        double* out, int64_t out_stride, int threads) {
  parallel_for(num_rows, threads, [&](int64_t r) {
    int g = 0;
    while (g < num_requests && !(cu_seqlens[g] <= r && r < cu_seqlens[g + 1])) ++g;
    if (g == num_requests) return;
    row_logits(q_packed, q_scale, w, r, H, kv_packed, kv_scale, block_tables + g * bt_stride, 0, row_ends[r],
               out + r * out_stride);
  });
}

void orc_select_topk(const double* logits, int64_t n, int k, int32_t* idx, double* val) {
  select_topk(logits, n, k, idx, val);
}

// R12: the top-k of each sequence over its key range only (absolute indices). Scratch is the
// caller's [batch][scratch_stride], scratch_stride >= the longest range.
void orc_range_topk(const uint8_t* q_packed, const uint8_t* q_scale, const float* w, const uint8_t* kv_packed,
                    const uint8_t* kv_scale, const int32_t* block_tables, int64_t bt_stride, const int32_t* key_begin,
                    const int32_t* key_end, int batch, int H, int k, double* scratch, int64_t scratch_stride,
                    int32_t* topk_idx, double* topk_val, int threads) {
  parallel_for(batch, threads, [&](int64_t b) {
    const int64_t t0 = key_begin[b], t1 = key_end[b];
    const int64_t n = t1 > t0 ? t1 - t0 : 0;
    row_logits(q_packed, q_scale, w, b, H, kv_packed, kv_scale, block_tables + b * bt_stride, t0, t0 + n,
               scratch + b * scratch_stride);
    select_topk(scratch + b * scratch_stride, n, k, topk_idx + b * k, topk_val + b * k);
    for (int i = 0; i < k; ++i)
      if (topk_idx[b * k + i] >= 0) topk_idx[b * k + i] += static_cast<int32_t>(t0);
  });
}

// R12: the merge of candidate lists [lists][rows][k_in] (index < 0 = empty) into each row's
// min(k, n) best of the union by (value descending, index ascending), in that order.
void orc_merge_candidates(const double* vals, const int32_t* idx, int lists, int rows, int k_in, int k,
                          int32_t* out_idx, double* out_val) {
  for (int r = 0; r < rows; ++r) {
    std::vector<std::pair<double, int32_t>> all;
    for (int l = 0; l < lists; ++l)
      for (int i = 0; i < k_in; ++i) {
        const int64_t at = (static_cast<int64_t>(l) * rows + r) * k_in + i;
        if (idx[at] >= 0) all.emplace_back(vals[at], idx[at]);
      }
    std::sort(all.begin(), all.end(), [](const std::pair<double, int32_t>& a, const std::pair<double, int32_t>& b) {
      if (a.first != b.first) return a.first > b.first;
      return a.second < b.second;
    });
    const int64_t m = std::min<int64_t>(k, static_cast<int64_t>(all.size()));
    for (int i = 0; i < k; ++i) {
      out_idx[static_cast<int64_t>(r) * k + i] = i < m ? all[static_cast<size_t>(i)].second : -1;
      out_val[static_cast<int64_t>(r) * k + i] =
          i < m ? all[static_cast<size_t>(i)].first : -std::numeric_limits<double>::infinity();
    }
  }
}

// Full decode path: logits then top-k per row. Scratch is the caller's [batch][scratch_stride].
void orc_decode_topk(const uint8_t* q_packed, const uint8_t* q_scale, const float* w, const uint8_t* kv_packed,
                     const uint8_t* kv_scale, const int32_t* block_tables, int64_t bt_stride, const int32_t* ctx_lens,
                     int batch, int H, int k, double* scratch, int64_t scratch_stride, int32_t* topk_idx,
                     double* topk_val, int threads) {
  orc_decode_logits(q_packed, q_scale, w, kv_packed, kv_scale, block_tables, bt_stride, ctx_lens, batch, H, scratch,
                    scratch_stride, threads);
  parallel_for(batch, threads, [&](int64_t b) {
    select_topk(scratch + b * scratch_stride, ctx_lens[b], k, topk_idx + b * k, topk_val + b * k);
  });
}

// Full prefill path: logits then top-k per row.
void orc_prefill_topk(const uint8_t* q_packed, const uint8_t* q_scale, const float* w, const uint8_t* kv_packed,
                      const uint8_t* kv_scale, const int32_t* block_tables, int64_t bt_stride,
                      const int32_t* cu_seqlens, const int32_t* row_ends, int num_requests, int num_rows, int H, int k,
                      double* scratch, int64_t scratch_stride, int32_t* topk_idx, double* topk_val, int threads) {
  orc_prefill_logits(q_packed, q_scale, w, kv_packed, kv_scale, block_tables, bt_stride, cu_seqlens, row_ends,
                     num_requests, num_rows, H, scratch, scratch_stride, threads);
  parallel_for(num_rows, threads, [&](int64_t r) {
    select_topk(scratch + r * scratch_stride, row_ends[r], k, topk_idx + r * k, topk_val + r * k);
  });
}

}  // extern "C"
