// Block-scaled E4M3 quantisation of one bf16 token row held in shared
// memory, stored to the row's K destination rows: the fp8 dispatch payload
// of "Efficient and portable mixture-of-experts communication" (Dispatch),
// block-scale fp8 as in "Enabling trillion-parameter models on AWS EFA"
// (evaluation).  Used by the fp8 pack and by route_pack_fp8.
//
//   blocks of 128 consecutive elements, scale = amax / 448 (1 for an all-zero
//   block), inv = 1 / scale (both IEEE float32 divisions, once per block),
//   q = E4M3(x * inv) rounded to nearest even, saturating.
//
// kRowThreads threads share a row: 8 lanes cover one 128-element block (16
// elements each), reduce amax with shuffles, multiply by the block's inverse
// scale, convert two at a time with cvt.rn.satfinite.e4m3x2.f32 and store 16
// fp8 bytes per lane to each of the K destination rows (coalesced); one lane
// per block stores the scale.

#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "ptx.cuh"

namespace moe {
namespace fp8q {

constexpr int kRowThreads = 128;

__device__ __forceinline__ uint4 lds128(const void* p) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(ptx::smem_addr(p)));
  return v;
}

// Two floats to two E4M3 codes: `lo` in the low byte, `hi` in the high byte.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ float lo_f(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float hi_f(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Thread c0 (0..kRowThreads-1) of the row's threads; lane k of every warp
// among them holds destination row k in my_row.  P has K, H (a multiple of
// 128), expert_xq (e4m3 [rows, H]) and expert_scales (float [rows, H/128]).
// Thread c0 takes chunks c0, c0 + kRowThreads, ... of 16 elements.  (Two
// chunks per thread side by side, as independent chains, measured slower on
// GB300: Mixtral-sized fp8 layer through route_pack_fp8 31.8 -> 33.1 us.)
template <int KMAX, class P>
__device__ __forceinline__ void quantize_row(const P& p, const uint8_t* row, int my_row, int c0, int chunks,
                                             int nblk) {
  const int K = p.K, H = p.H;
  // Warp-uniform trip count: every lane reaches the shuffles below; lanes
  // past the end of the row work on zeros and store nothing.
  for (int cb = 0; cb < chunks; cb += kRowThreads) {
    const int c = cb + c0;
    const bool act = c < chunks;
    const uint4 a = act ? lds128(row + c * 32) : make_uint4(0, 0, 0, 0);
    const uint4 b = act ? lds128(row + c * 32 + 16) : make_uint4(0, 0, 0, 0);
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    float amax = 0.0f;
#pragma unroll
    for (int j = 0; j < 8; ++j) amax = fmaxf(fmaxf(amax, fabsf(lo_f(w[j]))), fabsf(hi_f(w[j])));
    // The 8 lanes of one 128-element block are 8 consecutive lanes.
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 4));
    const float scale = amax > 0.0f ? __fdiv_rn(amax, 448.0f) : 1.0f;
    const float inv = __fdiv_rn(1.0f, scale);
    uint4 out;
    uint32_t* o = &out.x;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t lo = e4m3x2(__fmul_rn(lo_f(w[2 * j]), inv), __fmul_rn(hi_f(w[2 * j]), inv));
      const uint32_t hi = e4m3x2(__fmul_rn(lo_f(w[2 * j + 1]), inv), __fmul_rn(hi_f(w[2 * j + 1]), inv));
      o[j] = lo | (hi << 16);
    }
    const int blk = c >> 3;
#pragma unroll
    for (int k = 0; k < KMAX; ++k) {
      if (k < K) {
        const int64_t dst = static_cast<int64_t>(__shfl_sync(0xffffffffu, my_row, k));
        if (act) {
          ptx::st_v4(p.expert_xq + dst * H + static_cast<int64_t>(c) * 16, out);
          if ((c & 7) == 0) p.expert_scales[dst * nblk + blk] = scale;
        }
      }
    }
  }
}

}  // namespace fp8q
}  // namespace moe
