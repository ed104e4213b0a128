// Self-test of the CPU oracle (test infrastructure only), as a plain C++
// program linked with moe_oracle.cc: the oracle checked against brute force,
// invariants and closed forms, without Python.  Exit status 0 = every check
// passed; each failure prints one line.
//
// What it pins (the method: "Enabling trillion-parameter models on AWS EFA",
// Dispatch and combine, Send and receive buffers; "Efficient and portable
// mixture-of-experts communication", Dispatch, Combine):
//   - every routing of T = 3 tokens to K = 2 of E = 3 experts, for N = 1 and
//     N = 3 logical ranks (216 routings each): counts by brute count, offsets
//     by prefix sum, (expert, source rank) offsets and rank offsets by
//     counting, slot_row a bijection onto the T*K rows with row_src its
//     inverse, rows in (expert, token) order, each grouped row a copy of its
//     token row, and the placement equal to a loop-built one (for each expert
//     in order, each token in order, append the pair if the token chose it);
//   - a repeated or out-of-range expert is rejected;
//   - combine: K = 1 with weight 1 copies, a one-hot weight selects one
//     expert, identity experts with four weights of 1/4 return the input, the
//     chain starts from +0.0 (-0.0 terms give +0.0);
//   - bf16 and E4M3 conversions at hand-worked values (ties to even,
//     saturation, signed zero, the smallest subnormal).
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <vector>

extern "C" {
int oracle_dispatch(int32_t T, int32_t H, int32_t K, int32_t E, int32_t N, const uint16_t* x,
                    const int32_t* topk_idx, uint16_t* expert_x, int64_t expert_x_rows, int32_t* expert_counts,
                    int32_t* expert_offsets, int32_t* src_offsets, int32_t* rank_offsets, int32_t* slot_row,
                    int32_t* row_src);
int oracle_combine(int32_t T, int32_t H, int32_t K, const uint16_t* y, int64_t y_rows, const float* topk_w,
                   const int32_t* slot_row, uint16_t* out);
uint16_t oracle_float_to_bf16(float f);
uint8_t oracle_float_to_e4m3(float f);
double oracle_e4m3_to_double(uint8_t b);
}

namespace {

int failures = 0;
int checks = 0;

void expect(bool ok, const char* what, int a = 0, int b = 0) {
  ++checks;
  if (!ok) {
    ++failures;
    std::printf("FAIL %s (%d, %d)\n", what, a, b);
  }
}

// Every routing of 3 tokens to 2 distinct experts of 3, with N ranks.
void exhaustive_dispatch(int N) {
  const int T = 3, K = 2, E = 3, H = 8;
  const int L = E / N, Tr = T / N;
  std::vector<std::pair<int, int>> choices;
  for (int a = 0; a < E; ++a)
    for (int b = 0; b < E; ++b)
      if (a != b) choices.push_back({a, b});
  const int C = static_cast<int>(choices.size());
  std::vector<uint16_t> x(T * H);
  for (int t = 0; t < T; ++t)
    for (int h = 0; h < H; ++h) x[t * H + h] = static_cast<uint16_t>(0x3F80 + 16 * t + h);
  for (int code = 0; code < C * C * C; ++code) {
    std::vector<int32_t> idx(T * K);
    for (int t = 0, c = code; t < T; ++t, c /= C) {
      idx[t * K] = choices[c % C].first;
      idx[t * K + 1] = choices[c % C].second;
    }
    std::vector<uint16_t> ex(T * K * H, 0);
    std::vector<int32_t> cnt(E), off(E + 1), src(E * N), roff(N + 1), slot(T * K), rsrc(T * K);
    const int rc = oracle_dispatch(T, H, K, E, N, x.data(), idx.data(), ex.data(), T * K, cnt.data(), off.data(),
                                   src.data(), roff.data(), slot.data(), rsrc.data());
    expect(rc == 0, "dispatch status", code, rc);
    if (rc) continue;
    // counts and offsets by brute force
    int run = 0;
    for (int e = 0; e < E; ++e) {
      int n = 0;
      for (int p = 0; p < T * K; ++p) n += idx[p] == e;
      expect(cnt[e] == n, "count", code, e);
      expect(off[e] == run, "offset", code, e);
      int within = 0;
      for (int s = 0; s < N; ++s) {
        expect(src[e * N + s] == run + within, "src offset", code, e * N + s);
        for (int t = s * Tr; t < (s + 1) * Tr; ++t)
          for (int k = 0; k < K; ++k) within += idx[t * K + k] == e;
      }
      run += n;
    }
    expect(off[E] == T * K, "last offset", code, off[E]);
    for (int r = 0; r <= N; ++r) expect(roff[r] == off[r * L], "rank offset", code, r);
    // bijection, inverse, copies
    std::vector<int> seen(T * K, 0);
    for (int p = 0; p < T * K; ++p) {
      const int r = slot[p];
      expect(r >= 0 && r < T * K, "slot in range", code, p);
      if (r < 0 || r >= T * K) continue;
      seen[r] += 1;
      expect(rsrc[r] == p, "row_src inverse", code, p);
      expect(std::memcmp(&ex[r * H], &x[(p / K) * H], H * 2) == 0, "row copy", code, p);
    }
    for (int r = 0; r < T * K; ++r) expect(seen[r] == 1, "bijection", code, r);
    // the loop-built placement: experts in order, tokens in order
    int row = 0;
    for (int e = 0; e < E; ++e)
      for (int t = 0; t < T; ++t)
        for (int k = 0; k < K; ++k)
          if (idx[t * K + k] == e) expect(slot[t * K + k] == row++, "loop placement", code, t * K + k);
  }
}

}  // namespace

namespace {

void routing_errors() {
  const int T = 2, K = 2, E = 4, N = 2, H = 8;
  std::vector<uint16_t> x(T * H, 0x3F80), ex(T * K * H);
  std::vector<int32_t> cnt(E), off(E + 1), src(E * N), roff(N + 1), slot(T * K), rsrc(T * K);
  const int32_t repeated[] = {0, 1, 2, 2};
  const int32_t outside[] = {0, 1, 4, 2};
  const int32_t negative[] = {-1, 1, 3, 2};
  for (const int32_t* idx : {repeated, outside, negative}) {
    const int rc = oracle_dispatch(T, H, K, E, N, x.data(), idx, ex.data(), T * K, cnt.data(), off.data(), src.data(),
                                   roff.data(), slot.data(), rsrc.data());
    expect(rc == 3, "bad routing rejected", rc);
  }
}

uint16_t bf16(float f) { return oracle_float_to_bf16(f); }

void combine_closed_forms() {
  const int H = 4;
  const uint16_t v[H] = {bf16(1.5f), bf16(-0.375f), bf16(3.0e-3f), bf16(-7.0f)};
  // K = 1, w = 1: a copy of the expert row
  {
    const float w[] = {1.0f};
    const int32_t slot[] = {0};
    uint16_t out[H];
    expect(oracle_combine(1, H, 1, v, 1, w, slot, out) == 0, "combine status");
    for (int h = 0; h < H; ++h) expect(out[h] == v[h], "K=1 copy", h);
  }
  // one-hot weight selects one of three expert rows
  {
    std::vector<uint16_t> y(3 * H);
    for (int r = 0; r < 3; ++r)
      for (int h = 0; h < H; ++h) y[r * H + h] = bf16(static_cast<float>(r * 10 + h) - 5.0f);
    const float w[] = {0.0f, 1.0f, 0.0f};
    const int32_t slot[] = {2, 0, 1};
    uint16_t out[H];
    oracle_combine(1, H, 3, y.data(), 3, w, slot, out);
    for (int h = 0; h < H; ++h) expect(out[h] == y[0 * H + h], "one-hot", h);
  }
  // identity experts, four weights of 1/4: every partial sum m*v/4 is exact
  {
    std::vector<uint16_t> y(4 * H);
    for (int r = 0; r < 4; ++r) std::memcpy(&y[r * H], v, sizeof v);
    const float w[] = {0.25f, 0.25f, 0.25f, 0.25f};
    const int32_t slot[] = {3, 1, 0, 2};
    uint16_t out[H];
    oracle_combine(1, H, 4, y.data(), 4, w, slot, out);
    for (int h = 0; h < H; ++h) expect(out[h] == v[h], "identity experts", h);
  }
  // the chain starts from +0.0: -0.0 terms give +0.0
  {
    const uint16_t y[] = {0x8000, 0x8000, 0x8000, 0x8000, 0x8000, 0x8000, 0x8000, 0x8000};
    const float w[] = {0.5f, 0.5f};
    const int32_t slot[] = {0, 1};
    uint16_t out[H];
    oracle_combine(1, H, 2, y, 2, w, slot, out);
    for (int h = 0; h < H; ++h) expect(out[h] == 0x0000, "start value +0.0", h, out[h]);
  }
}

void conversions() {
  expect(bf16(1.0f) == 0x3F80, "bf16 1");
  expect(bf16(-2.5f) == 0xC020, "bf16 -2.5");
  expect(bf16(1.00390625f) == 0x3F80, "bf16 tie to even (down)");      // 1 + 2^-8
  expect(bf16(1.01171875f) == 0x3F82, "bf16 tie to even (up)");        // 1 + 3*2^-8
  expect(bf16(1.00390625f + 0x1p-20f) == 0x3F81, "bf16 above the tie");
  expect(bf16(-0.0f) == 0x8000, "bf16 -0");
  expect(oracle_float_to_e4m3(448.0f) == 0x7E, "e4m3 448");
  expect(oracle_float_to_e4m3(500.0f) == 0x7E, "e4m3 saturates");
  expect(oracle_float_to_e4m3(-448.0f) == 0xFE, "e4m3 -448");
  expect(oracle_float_to_e4m3(0.0f) == 0x00, "e4m3 +0");
  expect(oracle_float_to_e4m3(-0.0f) == 0x80, "e4m3 -0");
  expect(oracle_float_to_e4m3(1.0f) == 0x38, "e4m3 1");
  expect(oracle_float_to_e4m3(1.0625f) == 0x38, "e4m3 tie to even (down)");  // between 1 and 1.125
  expect(oracle_float_to_e4m3(1.1875f) == 0x3A, "e4m3 tie to even (up)");    // between 1.125 and 1.25
  expect(oracle_float_to_e4m3(0x1p-9f) == 0x01, "e4m3 smallest subnormal");
  expect(oracle_e4m3_to_double(0x01) == std::ldexp(1.0, -9), "e4m3 decode subnormal");
  expect(oracle_e4m3_to_double(0x7E) == 448.0, "e4m3 decode max");
  expect(oracle_e4m3_to_double(0x38) == 1.0, "e4m3 decode 1");
}

}  // namespace

int main() {
  exhaustive_dispatch(1);
  exhaustive_dispatch(3);
  routing_errors();
  combine_closed_forms();
  conversions();
  std::printf("oracle self-test: %d checks, %d failed\n", checks, failures);
  return failures == 0 ? 0 : 1;
}
