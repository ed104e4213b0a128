// Two-level combine: partial sums on the sending side, then on the receiver.
//
// "Enabling trillion-parameter models on AWS EFA" (evaluation, prefill):
// DeepEP adds up a token's expert outputs on the sending side so that less
// data crosses the network, at some cost in precision; the pages' own kernels
// add only on the receiving side (moe_combine_recv).  This is the sending-side
// form, kept as an alternative so that its traffic and its precision can be
// measured against the receiver-only combine:
//   level 1 (each rank r holding some of token t's experts):
//     partial = bf16( float32 FMA chain over those experts in top-k order,
//                     starting from +0.0 ),
//     stored in row t*S + d of the partial buffer, S = min(K, N), d = the
//     position of r among the token's ranks in ascending order;
//   level 2 (token t's own rank):
//     out[t] = bf16( float32 sum of the token's partials, ascending r, from
//                    +0.0 ).
// On one GPU the partial rows are what would cross the network: level 1
// writes them, level 2 reads them back.
//
// The rank of a dispatched row comes from the layout itself: rank r's rows
// are [rank_offsets[r], rank_offsets[r+1]), so a binary search over the N+1
// offsets (staged in shared memory) places each slot_row entry.
//
// Three kernels: a plan kernel, one thread per token, sorts the token's slots
// by (rank, k) once and marks where each rank's group ends (workspace
// tables); level 1 and level 2 then run one thread per 16-byte column chunk
// (8 bf16) of one token row, flat over (token, chunk), like the vector
// combine, reading the plan.  A token with a routing error (slot_row < 0) is
// skipped: nothing is written for it.

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "moe_kernels.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);  // .x = lo (low half), .y = hi
  return *reinterpret_cast<uint32_t*>(&v);
}

// Largest r in [0, N) with ro[r] <= row (ro[0] = 0 <= row < ro[N]): the rank
// whose row range holds `row`; empty ranks (equal offsets) are never chosen.
__device__ __forceinline__ int rank_of_row(const int32_t* ro, int N, int row) {
  int lo = 0, hi = N;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (ro[mid] <= row) lo = mid;
    else hi = mid;
  }
  return lo;
}

__device__ __forceinline__ void load_rank_offsets(const int32_t* ro, int N, int32_t* s_ro) {
  for (int i = threadIdx.x; i <= N; i += blockDim.x) s_ro[i] = ro[i];
  __syncthreads();
}

// Per token, once: the token's slots sorted by (rank, k), and a bit mask with
// bit i set when sorted slot i is the last of its rank (the partial ends
// there).  plan_mask = 0 marks a token whose routing failed.
template <int KMAX>
__global__ void __launch_bounds__(kThreads) combine_plan_kernel(TwoLevelParams p) {
  extern __shared__ int32_t s_ro[];
  ptx::wait_prerequisites();
  load_rank_offsets(p.rank_offsets, p.N, s_ro);
  const int64_t t = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
  if (t >= p.T) return;
  const int K = p.K;
  int row[KMAX], rk[KMAX];
  int bad = 0;
#pragma unroll
  for (int k = 0; k < KMAX; ++k) {
    row[k] = 0;
    rk[k] = 0x7fffffff;
    if (k < K) {
      row[k] = p.slot_row[t * K + k];
      bad |= row[k] < 0;
      if (kChecked && row[k] >= p.y_rows) {
        atomicCAS(p.error_word, MOE_OK, MOE_ECORRUPT);
        bad = 1;
      }
    }
  }
  if (bad) {
    p.plan_mask[t] = 0;
    return;
  }
#pragma unroll
  for (int k = 0; k < KMAX; ++k)
    if (k < K) rk[k] = rank_of_row(s_ro, p.N, row[k]);
  uint32_t mask = 0;
#pragma unroll
  for (int k = 0; k < KMAX; ++k) {
    if (k < K) {
      int pos = 0;
      bool last = true;
#pragma unroll
      for (int j = 0; j < KMAX; ++j) {
        if (j < K) {
          if (rk[j] < rk[k] || (rk[j] == rk[k] && j < k)) ++pos;
          if (rk[j] == rk[k] && j > k) last = false;
        }
      }
      p.plan_row[t * K + pos] = row[k];
      p.plan_w[t * K + pos] = p.w[t * K + k];
      if (last) mask |= 1u << pos;
    }
  }
  p.plan_mask[t] = static_cast<int32_t>(mask);
}

// Level 1: thread (t, c) runs the FMA chain over the sorted slots and stores
// one bf16 partial at each group end.
template <int KMAX>
__global__ void __launch_bounds__(kThreads) combine_partial_kernel(TwoLevelParams p) {
  ptx::wait_prerequisites();
  const int K = p.K;
  const int64_t C = p.H >> 3;
  const int64_t g = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
  if (g >= static_cast<int64_t>(p.T) * C) return;
  const int64_t t = g / C;
  const int64_t c = g - t * C;
  const int64_t row_bytes = static_cast<int64_t>(p.H) * 2;
  const uint32_t mask = static_cast<uint32_t>(p.plan_mask[t]);
  if (mask == 0) return;  // routing error: nothing is written
  uint4 v[KMAX];
  float wk[KMAX];
#pragma unroll
  for (int i = 0; i < KMAX; ++i) {
    if (i < K) {
      const int r = p.plan_row[t * K + i];
      wk[i] = p.plan_w[t * K + i];
      v[i] = ptx::ld_stream_v4(p.y + static_cast<int64_t>(r) * row_bytes + c * 16);
    }
  }
  const int S = K < p.N ? K : p.N;
  uint8_t* prow = p.partial + (t * S) * row_bytes + c * 16;
  float a[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) a[j] = 0.0f;
  int d = 0;
#pragma unroll
  for (int i = 0; i < KMAX; ++i) {
    if (i < K) {
      const uint32_t wd[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        a[2 * j] = __fmaf_rn(wk[i], __uint_as_float(wd[j] << 16), a[2 * j]);
        a[2 * j + 1] = __fmaf_rn(wk[i], __uint_as_float(wd[j] & 0xffff0000u), a[2 * j + 1]);
      }
      if ((mask >> i) & 1u) {
        uint4 o;
        o.x = pack_bf16x2(a[0], a[1]);
        o.y = pack_bf16x2(a[2], a[3]);
        o.z = pack_bf16x2(a[4], a[5]);
        o.w = pack_bf16x2(a[6], a[7]);
        ptx::st_v4(prow + static_cast<int64_t>(d) * row_bytes, o);
        ++d;
#pragma unroll
        for (int j = 0; j < 8; ++j) a[j] = 0.0f;
      }
    }
  }
}

// Level 2: thread (t, c) adds the token's D partials in rank order.
template <int KMAX>
__global__ void __launch_bounds__(kThreads) combine_reduce_kernel(TwoLevelParams p) {
  ptx::wait_prerequisites();
  const int64_t C = p.H >> 3;
  const int64_t g = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
  if (g >= static_cast<int64_t>(p.T) * C) return;
  const int64_t t = g / C;
  const int64_t c = g - t * C;
  const int64_t row_bytes = static_cast<int64_t>(p.H) * 2;
  const uint32_t mask = static_cast<uint32_t>(p.plan_mask[t]);
  if (mask == 0) return;
  const int D = __popc(mask);
  const int S = p.K < p.N ? p.K : p.N;
  const uint8_t* prow = p.partial + (t * S) * row_bytes + c * 16;
  uint4 v[KMAX];
#pragma unroll
  for (int d = 0; d < KMAX; ++d)
    if (d < D) v[d] = ptx::ld_stream_v4(prow + static_cast<int64_t>(d) * row_bytes);
  float a[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) a[j] = 0.0f;
#pragma unroll
  for (int d = 0; d < KMAX; ++d) {
    if (d < D) {
      const uint32_t wd[4] = {v[d].x, v[d].y, v[d].z, v[d].w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        a[2 * j] = __fadd_rn(a[2 * j], __uint_as_float(wd[j] << 16));
        a[2 * j + 1] = __fadd_rn(a[2 * j + 1], __uint_as_float(wd[j] & 0xffff0000u));
      }
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
cudaError_t launch_two_level_k(const TwoLevelParams& p, bool pdl, cudaStream_t stream) {
  const long long threads = static_cast<long long>(p.T) * (p.H >> 3);
  const long long grid = (threads + kThreads - 1) / kThreads;
  if (grid == 0) return cudaSuccess;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidValue;
  const size_t smem = static_cast<size_t>(p.N + 1) * sizeof(int32_t);
  const unsigned plan_grid = static_cast<unsigned>((p.T + kThreads - 1) / kThreads);
  cudaError_t err = launch_kernel(combine_plan_kernel<KMAX>, dim3(plan_grid), dim3(kThreads), smem, stream, pdl, p);
  if (err != cudaSuccess) return err;
  err = launch_kernel(combine_partial_kernel<KMAX>, dim3(static_cast<unsigned>(grid)), dim3(kThreads), 0, stream,
                      pdl, p);
  if (err != cudaSuccess) return err;
  return launch_kernel(combine_reduce_kernel<KMAX>, dim3(static_cast<unsigned>(grid)), dim3(kThreads), 0, stream,
                       pdl, p);
}

}  // namespace

cudaError_t launch_combine_two_level(const TwoLevelParams& p, bool pdl, cudaStream_t stream) {
  if (p.K <= 2) return launch_two_level_k<2>(p, pdl, stream);
  if (p.K <= 4) return launch_two_level_k<4>(p, pdl, stream);
  if (p.K <= 8) return launch_two_level_k<8>(p, pdl, stream);
  return launch_two_level_k<16>(p, pdl, stream);
}

}  // namespace moe
