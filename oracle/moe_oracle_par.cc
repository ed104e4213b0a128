// MoE dispatch + combine: the CPU oracle's loops spread over every host core.
//
// TEST INFRASTRUCTURE ONLY, like moe_oracle.cc: the benchmark times it as the
// all-cores CPU baseline next to the single-threaded oracle, and the CPU
// tests check that it writes exactly what the oracle writes.  Nothing on the
// product path calls, links or loads it.
//
// It is the oracle itself (moe_oracle.cc is compiled into the same library)
// plus two functions that run the same steps in the same order with OpenMP
// worksharing over independent iterations:
//  * oracle_dispatch_par: validation, counts, exclusive prefix, receive-bound
//    check and the stable sort by expert run on one thread exactly as in
//    oracle_dispatch; the copy of token rows into the grouped rows (the bulk
//    of the bytes) is a parallel loop over grouped rows, each row written by
//    one thread;
//  * oracle_combine_par: the float32 fused-multiply-add chain of
//    oracle_combine, in the same k order, with a parallel loop over tokens;
//    each output element is computed by one thread, so the result does not
//    depend on the thread count.
// Nothing here changes the arithmetic: every output byte equals the
// single-threaded oracle's.

#include <omp.h>

#include "moe_oracle.cc"

extern "C" {

// Threads a parallel region of this library uses (OpenMP's default team size:
// the cores this process may run on, unless OMP_NUM_THREADS says otherwise).
int oracle_par_threads(void) { return omp_get_max_threads(); }

// Same arguments, results and status codes as oracle_dispatch.
int oracle_dispatch_par(int32_t T, int32_t H, int32_t K, int32_t E, int32_t N,
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

  const int32_t Tr = T / N;
  const int32_t L = E / N;
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
  std::vector<int64_t> off(E + 1, 0);
  for (int32_t e = 0; e < E; ++e) off[e + 1] = off[e] + cnt[e];
  const int64_t bound = static_cast<int64_t>(N) * Tr * std::max(K, L);
  for (int32_t r = 0; r < N; ++r) {
    int64_t recv = off[(r + 1) * L] - off[r * L];
    if (recv > bound) return ORACLE_EBOUND;
  }

  std::vector<Triple> trip;
  trip.reserve(static_cast<size_t>(rows));
  for (int32_t t = 0; t < T; ++t)
    for (int32_t k = 0; k < K; ++k) trip.push_back({topk_idx[static_cast<int64_t>(t) * K + k], t, k});
  std::stable_sort(trip.begin(), trip.end(),
                   [](const Triple& a, const Triple& b) { return a.e < b.e; });

#pragma omp parallel for schedule(static)
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

// Same arguments, results and status codes as oracle_combine.
int oracle_combine_par(int32_t T, int32_t H, int32_t K, const uint16_t* y, int64_t y_rows,
                       const float* topk_w, const int32_t* slot_row, uint16_t* out) {
  if (T < 0 || H < 1 || K < 1) return ORACLE_EINVAL;
  for (int64_t p = 0; p < static_cast<int64_t>(T) * K; ++p)
    if (slot_row[p] < 0 || slot_row[p] >= y_rows) return ORACLE_EINVAL;
#pragma omp parallel for schedule(static)
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

}  // extern "C"
