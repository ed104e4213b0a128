// combine: out[t] = bf16( sum over k of w[t,k] * y[slot_row[t,k]] ).
//
// "Efficient and portable mixture-of-experts communication" (Combine): the
// receiving kernel reads, from the routing table, which buffer holds each of
// a token's expert outputs and which weight goes with it, and writes the
// weighted average into a caller-allocated tensor.  "Enabling
// trillion-parameter models on AWS EFA" (evaluation, prefill): tokens are
// accumulated only on the receiving side, never partially on the sender.
//
// Arithmetic (fixed so the result is reproducible bit for bit): float32
// accumulator starting at +0.0f, one fused multiply-add per expert in top-k
// order k = 0..K-1 (round to nearest), one round-to-nearest-even to bf16.
//
// Layout: one thread per 16-byte column chunk (8 bf16) of one output row.
// Each thread issues all K 16-byte loads of its gathered expert rows before
// the first FMA, so K*16 bytes per thread are in flight.  Gathered rows are
// streamed past L1; the output row is written with coalesced 16-byte stores.

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "moe_kernels.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);  // .x = lo (low half), .y = hi
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ void fma_word(uint32_t word, float w, float& acc_lo, float& acc_hi) {
  acc_lo = __fmaf_rn(w, __uint_as_float(word << 16), acc_lo);
  acc_hi = __fmaf_rn(w, __uint_as_float(word & 0xffff0000u), acc_hi);
}

constexpr int kThreads = 256;

// Flat mapping: thread g handles 16-byte chunk c = g % C of token t = g / C
// (C = H / 8 chunks per row), so a warp reads 512 contiguous bytes of each of
// its K gathered rows.  MIN_BLOCKS sets the register budget: all K loads are
// live at once (4 registers each).
template <int KMAX, int MIN_BLOCKS>
__global__ void __launch_bounds__(kThreads, MIN_BLOCKS) combine_kernel(CombineParams p) {
  ptx::wait_prerequisites();
  const int K = p.K;
  const int64_t C = p.H >> 3;
  const int64_t g = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
  if (g >= static_cast<int64_t>(p.T) * C) return;
  const int64_t t = g / C;
  const int64_t c = g - t * C;
  const int64_t row_bytes = static_cast<int64_t>(p.H) * 2;
  const int32_t* slots = p.slot_row + t * K;

  int bad = 0;
  uint4 v[KMAX];
#pragma unroll
  for (int k = 0; k < KMAX; ++k) {
    if (k < K) {
      const int r = slots[k];
      bad |= r < 0;
      if (r >= 0) v[k] = ptx::ld_stream_v4(p.y + static_cast<int64_t>(r) * row_bytes + c * 16);
    }
  }
  if (bad) return;  // routing error reported by route_count: leave out[t] untouched

  float a[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) a[j] = 0.0f;
  const float* wt = p.w + t * K;
#pragma unroll
  for (int k = 0; k < KMAX; ++k) {
    if (k < K) {
      const float w = __ldg(wt + k);
      fma_word(v[k].x, w, a[0], a[1]);
      fma_word(v[k].y, w, a[2], a[3]);
      fma_word(v[k].z, w, a[4], a[5]);
      fma_word(v[k].w, w, a[6], a[7]);
    }
  }
  uint4 o;
  o.x = pack_bf16x2(a[0], a[1]);
  o.y = pack_bf16x2(a[2], a[3]);
  o.z = pack_bf16x2(a[4], a[5]);
  o.w = pack_bf16x2(a[6], a[7]);
  ptx::st_v4(p.out + t * row_bytes + c * 16, o);
}

template <int KMAX>
cudaError_t launch_k(const CombineParams& p, bool pdl, cudaStream_t stream) {
  constexpr int MIN_BLOCKS = KMAX >= 16 ? 2 : (KMAX >= 8 ? 3 : 4);
  const long long threads = static_cast<long long>(p.T) * (p.H >> 3);
  const long long grid = (threads + kThreads - 1) / kThreads;
  if (grid == 0) return cudaSuccess;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidValue;
  return launch_kernel(combine_kernel<KMAX, MIN_BLOCKS>, dim3(static_cast<unsigned>(grid)), dim3(kThreads), 0,
                       stream, pdl, p);
}

}  // namespace

cudaError_t launch_combine(const CombineParams& p, const CombineLaunch& l, cudaStream_t stream) {
  if (p.K <= 2) return launch_k<2>(p, l.pdl, stream);
  if (p.K <= 4) return launch_k<4>(p, l.pdl, stream);
  if (p.K <= 8) return launch_k<8>(p, l.pdl, stream);
  return launch_k<16>(p, l.pdl, stream);
}

}  // namespace moe
