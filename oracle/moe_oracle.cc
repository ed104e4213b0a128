// MoE dispatch + combine: the plain CPU oracle.
//
// TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
// load this file; only the tests, the smoke check and the benchmark's CPU
// baseline leg do.  It shares no code, header or constant with the CUDA
// library: it is written from the definition of the method, single-threaded,
// with no blocking, fusion or reordering, so that it can be checked by eye.
//
// Sources (titles of the pages, with the section used):
//  * "Efficient and portable mixture-of-experts communication" (pplx-kernels):
//    - Introduction: the router keeps the top-K experts per token and the
//      layer output is the router-weighted sum of the experts' outputs.
//    - Portable kernels: per-rank buffers of fixed capacity, reused by every
//      layer, with addresses that follow from offsets alone.
//    - Dispatch: the receiver hands an expert-grouped tensor to the grouped
//      GEMM and keeps, per row, where the token came from (source rank,
//      expert, token index) so that combine can send it back.
//    - Combine: the receiving side computes the weighted sum of all expert
//      contributions of a token, reading the routing table for which buffer to
//      read and which weight to apply.
//  * "Enabling trillion-parameter models on AWS EFA":
//    - Send and receive buffers: with N ranks of T tokens routed to R of E
//      experts, one rank receives at most N*T*max(R, E/N) tokens; the bound is
//      only reached when writes are placed contiguously, which needs the full
//      routing information (per-expert counts exchanged first, then offsets).
//    - Dispatch and combine: tokens per expert are counted, a cumulative sum
//      of the counts gives the offsets of contiguous per-peer buffers, then
//      tokens are packed at those offsets; combine accumulates only on the
//      receiving side.
//
// Readings where the pages are silent:
//  * expert e lives on logical rank floor(e / (E/N)) (contiguous blocks);
//  * inside one expert, rows are ordered by global token index t, which is the
//    same as (source rank, token within rank) because rank s owns tokens
//    [s*T/N, (s+1)*T/N);
//  * out-of-range or repeated expert indices within one token are errors;
//  * router weights are float32; the combine accumulates in float32 with one
//    fused multiply-add per expert in top-k order starting from +0.0, and
//    rounds once to bf16 (round to nearest, ties to even); the weighted sum is
//    not renormalised by the sum of weights.
//  * A second combine evaluates the same sum in double precision and rounds it
//    once to bf16: the plain mathematical definition, for error bounds.
//  * fp8 dispatch payload ("Efficient and portable mixture-of-experts
//    communication", Dispatch: tokens travel with block scaling factors;
//    "Enabling trillion-parameter models on AWS EFA", evaluation: block-scale
//    fp8 dispatch, bf16 combine).  The pages give neither the block nor the
//    scale rule; read as blocks of 128 consecutive elements of a row, E4M3,
//    scale = amax/448 so the largest element maps to the largest finite code,
//    and q = round-to-nearest-even(x * inv), saturating, with inv = 1/scale
//    rounded once per block (the usual form: one multiply per element).
//  * Two-level combine with partial sums on the sending side ("Enabling
//    trillion-parameter models on AWS EFA", evaluation, prefill: DeepEP sums a
//    token's expert outputs on the sender to move less data, which can cost
//    precision; the pages' own kernels sum only at the receiver).  Read as:
//    on each rank r holding some of token t's experts, partial = bf16 of the
//    same float32 fused-multiply-add chain restricted to those experts (top-k
//    order, from +0.0); the token's rank then adds the float32 values of its
//    partials in ascending r from +0.0 and rounds once to bf16.  Partial d of
//    token t (d-th smallest rank) lives in row t*min(K,N) + d.
//  * Two-stage dispatch through per-peer send buffers ("Enabling
//    trillion-parameter models on AWS EFA", dispatch and combine timing: the
//    sender copies tokens into contiguous per-peer send buffers at offsets
//    from the cumulative sum of its per-expert counts; the receiver shuffles
//    them from its receive buffer into the grouped-GEMM input).  Read as:
//    source rank s's (token, slot) pairs, stably sorted by expert (which
//    groups them by destination rank), fill send rows [s*T/N*K, (s+1)*T/N*K);
//    the receiving side then copies each send row to its grouped row.  The
//    result equals the direct placement; only the path (one more copy of every
//    row) differs.
//  * Dense padded all-to-all ("Efficient and portable mixture-of-experts
//    communication", Sharding and parallelism: torch's all_to_all needs
//    padding, or a GPU-CPU synchronisation, because ranks send different
//    numbers of tokens to each peer; Benchmarks: the dense all-to-all
//    primitives are bandwidth-bound and move an order of magnitude more data
//    than the sparse kernels).  Read as: every (source rank s, destination
//    rank r) chunk is a block of `cap` rows, cap fixed ahead of the layer (no
//    count exchange), at least the most rows one source can send to one rank,
//    T/N * min(K, E/N); source s fills block s*N+r with its (token, slot)
//    pairs whose expert lives on r, in (expert, token) order, and leaves the
//    rest of the block as padding; the exchange moves every block whole,
//    padding included (block s*N+r of the send buffer becomes block r*N+s of
//    the receive buffer); the receiver then moves the rows into the grouped
//    layout, expert by expert and source rank by source rank.  Combine
//    returns the expert outputs the same way in reverse and then takes the
//    same float32 chain as the receiver-only combine.
//
// All bf16 values are raw 16-bit patterns.

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

namespace {

enum {
  ORACLE_OK = 0,
  ORACLE_EINVAL = 1,  // bad sizes / pointers
  ORACLE_EROUTE = 3,  // an expert index out of range or repeated in a token
  ORACLE_EBOUND = 5,  // a rank would receive more rows than the printed bound
};

float bf16_to_float(uint16_t b) {
  uint32_t u = static_cast<uint32_t>(b) << 16;
  float f;
  std::memcpy(&f, &u, sizeof f);
  return f;
}

// IEEE round-to-nearest-even of a finite float to bf16: keep the upper 16
// bits, rounding on the lower 16 (add 0x7fff plus the lowest kept bit, then
// truncate).  NaN keeps a quiet-NaN payload.
uint16_t float_to_bf16_rne(float f) {
  uint32_t u;
  std::memcpy(&u, &f, sizeof u);
  if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu) != 0)
    return static_cast<uint16_t>((u >> 16) | 0x0040u);
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7fffu + lsb;
  return static_cast<uint16_t>(u >> 16);
}

// Round a finite double to the nearest bf16 (ties to even) in one step:
// bf16 keeps 8 significant bits; below the smallest normal (2^-126) the
// quantum is fixed at 2^-133.
uint16_t double_to_bf16_rne(double v) {
  if (v == 0.0) return std::signbit(v) ? 0x8000u : 0x0000u;
  int e;
  std::frexp(v, &e);  // |v| = m * 2^e, m in [0.5, 1)
  int q = e - 8;      // quantum exponent for 8 significant bits
  if (q < -133) q = -133;
  double scaled = std::ldexp(v, -q);
  double r = std::nearbyint(scaled);  // default rounding mode: ties to even
  double back = std::ldexp(r, q);
  float f = static_cast<float>(back);  // exact: back has <= 8 significant bits
  if (std::isinf(f) || std::fabs(back) > 3.3895313892515355e38) {
    return std::signbit(v) ? 0xff80u : 0x7f80u;
  }
  uint32_t u;
  std::memcpy(&u, &f, sizeof u);
  return static_cast<uint16_t>(u >> 16);
}

// fp8 E4M3 ("FN" variant: 1 sign, 4 exponent bits with bias 7, 3 mantissa
// bits, no infinities, S.1111.111 is NaN, largest finite 448).  Round to
// nearest, ties to even, saturating to +-448 (finite inputs only).
uint8_t float_to_e4m3_rne_sat(float f) {
  uint32_t u;
  std::memcpy(&u, &f, sizeof u);
  const uint8_t sign = static_cast<uint8_t>((u >> 24) & 0x80u);
  if ((u & 0x7f800000u) == 0x7f800000u) return static_cast<uint8_t>(sign | 0x7f);  // NaN/Inf: NaN
  const double a = std::fabs(static_cast<double>(f));
  if (a >= 448.0) return static_cast<uint8_t>(sign | 0x7e);
  if (a < std::ldexp(1.0, -6)) {
    // Subnormal range: multiples of 2^-9 (a code of 8 is the smallest normal).
    const double m = std::nearbyint(a * 512.0);  // exact scaling; ties to even
    return static_cast<uint8_t>(sign | static_cast<uint8_t>(m));  // m <= 8: 0b0000.mmm or 0b0001.000
  }
  int e;
  std::frexp(a, &e);  // a = f * 2^e, f in [0.5, 1): unbiased exponent e-1
  int ex = e - 1;
  double m = std::nearbyint(std::ldexp(a, 3 - ex));  // in [8, 16]
  if (m >= 16.0) {
    m = 8.0;
    ++ex;
  }
  if (ex > 8) return static_cast<uint8_t>(sign | 0x7e);
  const uint8_t code = static_cast<uint8_t>(((ex + 7) << 3) | (static_cast<int>(m) - 8));
  return static_cast<uint8_t>(sign | (code > 0x7e ? 0x7e : code));
}

double e4m3_to_double(uint8_t b) {
  const int sign = (b & 0x80) ? -1 : 1;
  const int ex = (b >> 3) & 0xf, man = b & 0x7;
  if (ex == 0xf && man == 0x7) return std::nan("");
  if (ex == 0) return sign * std::ldexp(static_cast<double>(man), -9);
  return sign * std::ldexp(static_cast<double>(8 + man), ex - 10);
}

constexpr int kFp8Block = 128;  // elements per scaling block
constexpr float kE4m3Max = 448.0f;

int check_sizes(int32_t T, int32_t H, int32_t K, int32_t E, int32_t N) {
  if (T < 0 || H < 1 || K < 1 || E < 1 || N < 1) return ORACLE_EINVAL;
  if (T % N != 0 || E % N != 0 || K > E) return ORACLE_EINVAL;
  return ORACLE_OK;
}

// Every expert index is in [0, E) and no token names an expert twice
// (top-k yields K distinct experts).
int check_routes(int32_t T, int32_t K, int32_t E, const int32_t* idx) {
  for (int64_t t = 0; t < T; ++t) {
    for (int32_t k = 0; k < K; ++k) {
      int32_t e = idx[t * K + k];
      if (e < 0 || e >= E) return ORACLE_EROUTE;
      for (int32_t j = 0; j < k; ++j)
        if (idx[t * K + j] == e) return ORACLE_EROUTE;
    }
  }
  return ORACLE_OK;
}

struct Triple {
  int32_t e;
  int32_t t;
  int32_t k;
};

}  // namespace

extern "C" {

// Dispatch of one layer.
//   x          bf16 [T, H]   token rows (rank s owns rows [s*T/N, (s+1)*T/N))
//   topk_idx   int32 [T, K]  experts chosen for each token
//   expert_x   bf16 [expert_x_rows, H], expert_x_rows >= T*K; rows [0, T*K)
//              are written in the expert-grouped order, the rest untouched
//   expert_counts   int32 [E]     rows per expert
//   expert_offsets  int32 [E+1]   first row of each expert; last = T*K
//   src_offsets     int32 [E*N]   first row of (expert e, source rank s) at e*N+s
//   rank_offsets    int32 [N+1]   first row of the experts of rank r; last = T*K
//   slot_row        int32 [T*K]   row that (t, k) was written to
//   row_src         int32 [T*K]   for each row, t*K + k of its (token, slot)
// Returns 0, ORACLE_EINVAL, ORACLE_EROUTE or ORACLE_EBOUND; on error nothing
// is written.
int oracle_dispatch(int32_t T, int32_t H, int32_t K, int32_t E, int32_t N,
                    const uint16_t* x, const int32_t* topk_idx,
                    uint16_t* expert_x, int64_t expert_x_rows,
                    int32_t* expert_counts, int32_t* expert_offsets,
                    int32_t* src_offsets, int32_t* rank_offsets,
                    int32_t* slot_row, int32_t* row_src) {
  int rc = check_sizes(T, H, K, E, N);
  if (rc) return rc;
  const int64_t rows = static_cast<int64_t>(T) * K;
  if (expert_x_rows < rows) return ORACLE_EINVAL;
  if (T > 0 && (!x || !topk_idx || !expert_x)) return ORACLE_EINVAL;
  rc = check_routes(T, K, E, topk_idx);
  if (rc) return rc;

  const int32_t Tr = T / N;  // tokens per logical rank
  const int32_t L = E / N;   // experts per logical rank

  // Counts per expert, and per (source rank, expert).
  std::vector<int64_t> cnt(E, 0);
  std::vector<int64_t> src_cnt(static_cast<size_t>(N) * E, 0);
  for (int64_t t = 0; t < T; ++t) {
    int64_t s = t / Tr;
    for (int32_t k = 0; k < K; ++k) {
      int32_t e = topk_idx[t * K + k];
      cnt[e] += 1;
      src_cnt[s * E + e] += 1;
    }
  }

  // Exclusive prefix sum of the counts: first row of each expert.
  std::vector<int64_t> off(E + 1, 0);
  for (int32_t e = 0; e < E; ++e) off[e + 1] = off[e] + cnt[e];

  // Receive bound per rank: N * (T/N) * max(K, E/N) rows.
  const int64_t bound = static_cast<int64_t>(N) * Tr * std::max(K, L);
  for (int32_t r = 0; r < N; ++r) {
    int64_t recv = off[(r + 1) * L] - off[r * L];
    if (recv > bound) return ORACLE_EBOUND;
  }

  // Stable placement: list every (expert, token, slot) in token-major order,
  // then stable-sort by expert.  Row i of the sorted list is row i of the
  // grouped buffer.
  std::vector<Triple> trip;
  trip.reserve(static_cast<size_t>(rows));
  for (int32_t t = 0; t < T; ++t)
    for (int32_t k = 0; k < K; ++k) trip.push_back({topk_idx[static_cast<int64_t>(t) * K + k], t, k});
  std::stable_sort(trip.begin(), trip.end(),
                   [](const Triple& a, const Triple& b) { return a.e < b.e; });

  for (int64_t i = 0; i < rows; ++i) {
    const Triple& p = trip[i];
    int64_t pair = static_cast<int64_t>(p.t) * K + p.k;
    slot_row[pair] = static_cast<int32_t>(i);
    row_src[i] = static_cast<int32_t>(pair);
    std::memcpy(expert_x + i * H, x + static_cast<int64_t>(p.t) * H, sizeof(uint16_t) * H);
  }

  for (int32_t e = 0; e < E; ++e) expert_counts[e] = static_cast<int32_t>(cnt[e]);
  for (int32_t e = 0; e <= E; ++e) expert_offsets[e] = static_cast<int32_t>(off[e]);
  for (int32_t e = 0; e < E; ++e) {
    int64_t run = off[e];
    for (int32_t s = 0; s < N; ++s) {
      src_offsets[static_cast<int64_t>(e) * N + s] = static_cast<int32_t>(run);
      run += src_cnt[static_cast<int64_t>(s) * E + e];
    }
  }
  for (int32_t r = 0; r <= N; ++r) rank_offsets[r] = static_cast<int32_t>(off[r * L]);
  return ORACLE_OK;
}

// Combine of one layer, float32 in top-k order:
//   out[t, h] = bf16_rne( fma(w[t,K-1], y[slot_row[t,K-1], h], ... fma(w[t,0], y[slot_row[t,0], h], +0.0f)) )
//   y         bf16 [y_rows, H]  expert outputs in the grouped row layout
//   topk_w    float32 [T, K]
//   slot_row  int32 [T*K]       from dispatch
//   out       bf16 [T, H]
int oracle_combine(int32_t T, int32_t H, int32_t K, const uint16_t* y, int64_t y_rows,
                   const float* topk_w, const int32_t* slot_row, uint16_t* out) {
  if (T < 0 || H < 1 || K < 1) return ORACLE_EINVAL;
  for (int64_t p = 0; p < static_cast<int64_t>(T) * K; ++p)
    if (slot_row[p] < 0 || slot_row[p] >= y_rows) return ORACLE_EINVAL;
  for (int64_t t = 0; t < T; ++t) {
    for (int64_t h = 0; h < H; ++h) {
      float acc = 0.0f;
      for (int32_t k = 0; k < K; ++k) {
        int64_t row = slot_row[t * K + k];
        acc = std::fmaf(topk_w[t * K + k], bf16_to_float(y[row * H + h]), acc);
      }
      out[t * H + h] = float_to_bf16_rne(acc);
    }
  }
  return ORACLE_OK;
}

// The same weighted sum evaluated in double precision (each product of a
// float32 weight and a bf16 value is exact in double), rounded once to bf16.
// Also returns, per output element, sum_k |w * y| in abs_sum (may be NULL),
// which scales the float32 accumulation error bound.
int oracle_combine_f64(int32_t T, int32_t H, int32_t K, const uint16_t* y, int64_t y_rows,
                       const float* topk_w, const int32_t* slot_row, uint16_t* out,
                       double* exact, double* abs_sum) {
  if (T < 0 || H < 1 || K < 1) return ORACLE_EINVAL;
  for (int64_t p = 0; p < static_cast<int64_t>(T) * K; ++p)
    if (slot_row[p] < 0 || slot_row[p] >= y_rows) return ORACLE_EINVAL;
  for (int64_t t = 0; t < T; ++t) {
    for (int64_t h = 0; h < H; ++h) {
      double acc = 0.0, mag = 0.0;
      for (int32_t k = 0; k < K; ++k) {
        int64_t row = slot_row[t * K + k];
        double term = static_cast<double>(topk_w[t * K + k]) *
                      static_cast<double>(bf16_to_float(y[row * H + h]));
        acc += term;
        mag += std::fabs(term);
      }
      out[t * H + h] = double_to_bf16_rne(acc);
      if (exact) exact[t * H + h] = acc;
      if (abs_sum) abs_sum[t * H + h] = mag;
    }
  }
  return ORACLE_OK;
}

// Two-stage dispatch (per-peer send buffers, then the receiver's shuffle):
//   send_buf   bf16 [T*K, H]: rows [s*T/N*K, (s+1)*T/N*K) hold source rank s's
//              pairs in (expert, token, slot) order, each the token's x row
//   send_dest  int32 [T*K]: the grouped row (slot_row) of each send row
//   expert_x   bf16 [T*K, H]: expert_x[send_dest[j]] = send_buf[j]
//   slot_row   int32 [T*K]: as oracle_dispatch (the grouped placement)
int oracle_dispatch_staged(int32_t T, int32_t H, int32_t K, int32_t E, int32_t N, const uint16_t* x,
                           const int32_t* topk_idx, uint16_t* send_buf, int32_t* send_dest, uint16_t* expert_x,
                           int32_t* slot_row) {
  int rc = check_sizes(T, H, K, E, N);
  if (rc) return rc;
  if (T > 0 && (!x || !topk_idx || !send_buf || !send_dest || !expert_x || !slot_row)) return ORACLE_EINVAL;
  const int64_t rows = static_cast<int64_t>(T) * K;
  // The grouped placement (slot_row) from the direct dispatch.
  std::vector<uint16_t> direct(static_cast<size_t>(rows) * H);
  std::vector<int32_t> counts(E), offsets(E + 1), src_off(static_cast<size_t>(E) * N), rank_off(N + 1),
      row_src(static_cast<size_t>(rows));
  rc = oracle_dispatch(T, H, K, E, N, x, topk_idx, direct.data(), rows, counts.data(), offsets.data(),
                       src_off.data(), rank_off.data(), slot_row, row_src.data());
  if (rc) return rc;
  // Stage 1: each source rank fills its own send rows.
  const int32_t Tr = T / N;
  for (int32_t s = 0; s < N; ++s) {
    std::vector<Triple> trip;
    for (int32_t t = s * Tr; t < (s + 1) * Tr; ++t)
      for (int32_t k = 0; k < K; ++k) trip.push_back({topk_idx[static_cast<int64_t>(t) * K + k], t, k});
    std::stable_sort(trip.begin(), trip.end(), [](const Triple& a, const Triple& b) { return a.e < b.e; });
    const int64_t base = static_cast<int64_t>(s) * Tr * K;
    for (size_t j = 0; j < trip.size(); ++j) {
      const Triple& p = trip[j];
      std::memcpy(send_buf + (base + static_cast<int64_t>(j)) * H, x + static_cast<int64_t>(p.t) * H,
                  sizeof(uint16_t) * H);
      send_dest[base + static_cast<int64_t>(j)] = slot_row[static_cast<int64_t>(p.t) * K + p.k];
    }
  }
  // Stage 2: the receivers move every send row to its grouped row.
  for (int64_t j = 0; j < rows; ++j)
    std::memcpy(expert_x + static_cast<int64_t>(send_dest[j]) * H, send_buf + j * H, sizeof(uint16_t) * H);
  return ORACLE_OK;
}

// Two-level combine (partial sums on the sending side, then on the receiver):
//   topk_idx  int32 [T, K] (the rank of slot k is topk_idx[t,k] / (E/N))
//   partial   bf16 [T * min(K,N), H]: row t*min(K,N)+d holds the partial of the
//             d-th smallest rank among token t's experts; rows past the
//             token's number of ranks are left untouched
//   out       bf16 [T, H]
int oracle_combine_two_level(int32_t T, int32_t H, int32_t K, int32_t E, int32_t N, const uint16_t* y,
                             int64_t y_rows, const int32_t* topk_idx, const float* topk_w,
                             const int32_t* slot_row, uint16_t* partial, uint16_t* out) {
  if (T < 0 || H < 1 || K < 1 || N < 1 || E < N || E % N != 0) return ORACLE_EINVAL;
  for (int64_t p = 0; p < static_cast<int64_t>(T) * K; ++p) {
    if (slot_row[p] < 0 || slot_row[p] >= y_rows) return ORACLE_EINVAL;
    if (topk_idx[p] < 0 || topk_idx[p] >= E) return ORACLE_EROUTE;
  }
  const int32_t L = E / N;
  const int32_t slots = std::min(K, N);
  for (int64_t t = 0; t < T; ++t) {
    // the ranks holding this token's experts, ascending, without repeats
    std::vector<int32_t> ranks;
    for (int32_t k = 0; k < K; ++k) ranks.push_back(topk_idx[t * K + k] / L);
    std::sort(ranks.begin(), ranks.end());
    ranks.erase(std::unique(ranks.begin(), ranks.end()), ranks.end());
    // level 1: one partial per rank
    for (size_t d = 0; d < ranks.size(); ++d) {
      uint16_t* prow = partial + (t * slots + static_cast<int64_t>(d)) * H;
      for (int64_t h = 0; h < H; ++h) {
        float acc = 0.0f;
        for (int32_t k = 0; k < K; ++k) {
          if (topk_idx[t * K + k] / L != ranks[d]) continue;
          int64_t row = slot_row[t * K + k];
          acc = std::fmaf(topk_w[t * K + k], bf16_to_float(y[row * H + h]), acc);
        }
        prow[h] = float_to_bf16_rne(acc);
      }
    }
    // level 2: the receiver adds the partials in rank order
    for (int64_t h = 0; h < H; ++h) {
      float acc = 0.0f;
      for (size_t d = 0; d < ranks.size(); ++d)
        acc = acc + bf16_to_float(partial[(t * slots + static_cast<int64_t>(d)) * H + h]);
      out[t * H + h] = float_to_bf16_rne(acc);
    }
  }
  return ORACLE_OK;
}

// Block-scaled fp8 quantisation of token rows (the dispatch payload with
// "block scaling factors"): for each row and each block of 128 consecutive
// elements, scale = amax / 448 (1 for an all-zero block) and inv = 1 / scale,
// both float32 divisions, and q = e4m3_rne_sat(x * inv) (float32 product).
//   x       bf16 [T, H], H % 128 == 0
//   q       e4m3 [T, H]
//   scales  float32 [T, H/128]
int oracle_quantize_fp8(int32_t T, int32_t H, const uint16_t* x, uint8_t* q, float* scales) {
  if (T < 0 || H < kFp8Block || H % kFp8Block != 0) return ORACLE_EINVAL;
  const int32_t nb = H / kFp8Block;
  for (int64_t t = 0; t < T; ++t) {
    for (int32_t b = 0; b < nb; ++b) {
      const uint16_t* blk = x + t * H + static_cast<int64_t>(b) * kFp8Block;
      float amax = 0.0f;
      for (int i = 0; i < kFp8Block; ++i) amax = std::max(amax, std::fabs(bf16_to_float(blk[i])));
      const float scale = amax > 0.0f ? amax / kE4m3Max : 1.0f;
      const float inv = 1.0f / scale;
      scales[t * nb + b] = scale;
      for (int i = 0; i < kFp8Block; ++i)
        q[t * H + static_cast<int64_t>(b) * kFp8Block + i] = float_to_e4m3_rne_sat(bf16_to_float(blk[i]) * inv);
    }
  }
  return ORACLE_OK;
}

// Element-wise helpers exposed for the pins.
uint16_t oracle_float_to_bf16(float f) { return float_to_bf16_rne(f); }
uint16_t oracle_double_to_bf16(double v) { return double_to_bf16_rne(v); }
float oracle_fmaf(float a, float b, float c) { return std::fmaf(a, b, c); }
uint8_t oracle_float_to_e4m3(float f) { return float_to_e4m3_rne_sat(f); }
double oracle_e4m3_to_double(uint8_t b) { return e4m3_to_double(b); }

// Dense padded all-to-all dispatch (see the header).  cap = rows per
// (source rank, destination rank) block.
//   send_buf  bf16 [N*N*cap, H]: block s*N+r, rows [0, n(s,r)) = the rows
//             source rank s sends to rank r; later rows (padding) untouched
//   recv_buf  bf16 [N*N*cap, H]: block r*N+s = block s*N+r of send_buf, all
//             cap rows
//   expert_x  bf16 [T*K, H]: the grouped layout (as oracle_dispatch)
//   send_pos  int32 [T*K]: the send row of pair t*K+k
// Returns ORACLE_EINVAL when cap < T/N * min(K, E/N), besides the errors of
// oracle_dispatch.
int oracle_dispatch_dense(int32_t T, int32_t H, int32_t K, int32_t E, int32_t N, const uint16_t* x,
                          const int32_t* topk_idx, int64_t cap, uint16_t* send_buf, uint16_t* recv_buf,
                          uint16_t* expert_x, int32_t* send_pos) {
  int rc = check_sizes(T, H, K, E, N);
  if (rc) return rc;
  const int32_t Tr = T / N;
  const int32_t L = E / N;
  if (cap < static_cast<int64_t>(Tr) * std::min(K, L) || cap < 1) return ORACLE_EINVAL;
  if (T > 0 && (!x || !topk_idx || !send_buf || !recv_buf || !expert_x || !send_pos)) return ORACLE_EINVAL;
  rc = check_routes(T, K, E, topk_idx);
  if (rc) return rc;
  // Senders: source s walks the experts of rank r in order, and for each its
  // tokens in order.
  for (int32_t s = 0; s < N; ++s) {
    for (int32_t r = 0; r < N; ++r) {
      const int64_t block = static_cast<int64_t>(s) * N + r;
      int64_t j = 0;
      for (int32_t e = r * L; e < (r + 1) * L; ++e) {
        for (int32_t t = s * Tr; t < (s + 1) * Tr; ++t) {
          for (int32_t k = 0; k < K; ++k) {
            if (topk_idx[static_cast<int64_t>(t) * K + k] != e) continue;
            const int64_t row = block * cap + j;
            std::memcpy(send_buf + row * H, x + static_cast<int64_t>(t) * H, sizeof(uint16_t) * H);
            send_pos[static_cast<int64_t>(t) * K + k] = static_cast<int32_t>(row);
            ++j;
          }
        }
      }
    }
  }
  // The exchange: every block whole, padding included.
  for (int32_t s = 0; s < N; ++s)
    for (int32_t r = 0; r < N; ++r)
      std::memcpy(recv_buf + (static_cast<int64_t>(r) * N + s) * cap * H,
                  send_buf + (static_cast<int64_t>(s) * N + r) * cap * H, sizeof(uint16_t) * cap * H);
  // Receivers: rank r's rows, expert by expert, source rank by source rank.
  int64_t row = 0;
  for (int32_t r = 0; r < N; ++r) {
    std::vector<int64_t> next(N, 0);  // next unread row of block r*N+s
    for (int32_t e = r * L; e < (r + 1) * L; ++e) {
      for (int32_t s = 0; s < N; ++s) {
        // The block's rows of expert e: those of source s's tokens that chose e.
        int64_t n_e = 0;
        for (int32_t t = s * Tr; t < (s + 1) * Tr; ++t)
          for (int32_t k = 0; k < K; ++k) n_e += topk_idx[static_cast<int64_t>(t) * K + k] == e;
        for (int64_t i = 0; i < n_e; ++i, ++row) {
          const int64_t src = (static_cast<int64_t>(r) * N + s) * cap + next[s] + i;
          std::memcpy(expert_x + row * H, recv_buf + src * H, sizeof(uint16_t) * H);
        }
        next[s] += n_e;
      }
    }
  }
  return ORACLE_OK;
}

// Dense padded all-to-all combine: the expert outputs y (grouped layout) go
// back to their source ranks through padded blocks, then the receiver-only
// float32 chain.
//   slot_row   int32 [T*K] grouped row of each pair (from oracle_dispatch)
//   send_pos   int32 [T*K] the dispatch's send row of each pair
//   back_send  bf16 [N*N*cap, H]: block r*N+s, row j = the output for the
//              pair that went to row j of the dispatch's block s*N+r (padding
//              untouched)
//   back_recv  bf16 [N*N*cap, H]: block s*N+r = block r*N+s of back_send
//   out[t, h]  = bf16_rne( fma chain over k of w[t,k] * back_recv[send_pos[t*K+k], h] from +0.0f )
int oracle_combine_dense(int32_t T, int32_t H, int32_t K, int32_t N, const uint16_t* y, int64_t y_rows,
                         const float* topk_w, const int32_t* slot_row, const int32_t* send_pos, int64_t cap,
                         uint16_t* back_send, uint16_t* back_recv, uint16_t* out) {
  if (T < 0 || H < 1 || K < 1 || N < 1 || cap < 1) return ORACLE_EINVAL;
  const int64_t blocks = static_cast<int64_t>(N) * N;
  for (int64_t p = 0; p < static_cast<int64_t>(T) * K; ++p) {
    if (slot_row[p] < 0 || slot_row[p] >= y_rows) return ORACLE_EINVAL;
    if (send_pos[p] < 0 || send_pos[p] >= blocks * cap) return ORACLE_EINVAL;
  }
  // Each expert rank r sends back the outputs of the rows it received from s.
  for (int64_t p = 0; p < static_cast<int64_t>(T) * K; ++p) {
    const int64_t sr = send_pos[p] / cap, j = send_pos[p] % cap;  // block s*N+r, row j
    const int64_t s = sr / N, r = sr % N;
    std::memcpy(back_send + ((r * N + s) * cap + j) * H, y + static_cast<int64_t>(slot_row[p]) * H,
                sizeof(uint16_t) * H);
  }
  for (int64_t s = 0; s < N; ++s)
    for (int64_t r = 0; r < N; ++r)
      std::memcpy(back_recv + (s * N + r) * cap * H, back_send + (r * N + s) * cap * H, sizeof(uint16_t) * cap * H);
  for (int64_t t = 0; t < T; ++t) {
    for (int64_t h = 0; h < H; ++h) {
      float acc = 0.0f;
      for (int32_t k = 0; k < K; ++k) {
        const int64_t row = send_pos[t * K + k];
        acc = std::fmaf(topk_w[t * K + k], bf16_to_float(back_recv[row * H + h]), acc);
      }
      out[t * H + h] = float_to_bf16_rne(acc);
    }
  }
  return ORACLE_OK;
}

}  // extern "C"
