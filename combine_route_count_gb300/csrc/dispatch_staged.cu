// staged_layout: send rows of the two-stage dispatch.
//
// "Enabling trillion-parameter models on AWS EFA" (dispatch and combine
// timing): the sender copies its tokens into contiguous per-peer send buffers
// at offsets from the cumulative sum of its per-expert token counts; the
// receiver shuffles them from its receive buffer into the grouped-GEMM input.
// moe_dispatch_send places rows directly at their grouped position (send and
// receive memory coincide on one GPU); moe_dispatch_send_staged keeps the
// pages' two copies so that the cost of the extra one can be measured.
//
// Source rank s owns send rows [s*T_r*K, (s+1)*T_r*K) (T_r = T/N), filled with
// its (token, slot) pairs in (expert, token) order, which groups them by
// destination rank.  From the routing tables:
//   cnt(e, s)  = rows of (expert e, source s) = next src offset - src_offsets[e*N+s]
//   pre(e, s)  = sum over e' < e of cnt(e', s)              (block scan)
//   send row of pair (t, k) with expert e = idx[t,k]:
//     s*T_r*K + pre(e, s) + (slot_row[t,k] - src_offsets[e*N+s])
// because rows of (e, s) sit in token order in both layouts.  One block per
// source rank; send_dest is the inverse (send row -> grouped row).  After a
// routing error every entry is -1 and the packs that read them write nothing.

#include <cuda_runtime.h>

#include "moe_kernels.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kThreads = 1024;  // >= MOE_MAX_EXPERTS: one thread per expert in the scan

__device__ __forceinline__ int warp_inclusive_scan(int v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int u = __shfl_up_sync(0xffffffffu, v, d);
    if (lane >= d) v += u;
  }
  return v;
}

__global__ void __launch_bounds__(kThreads) staged_layout_kernel(StagedLayoutParams p) {
  __shared__ int32_t pre[MOE_MAX_EXPERTS];
  __shared__ int32_t wsum[kThreads / 32];
  ptx::wait_prerequisites();  // slot_row and the offsets come from routing
  const int s = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t n = static_cast<int64_t>(p.T / p.N) * p.K;
  const int64_t base = static_cast<int64_t>(s) * n;

  int bad = 0;
  for (int64_t q = tid; q < n; q += kThreads) bad |= p.slot_row[base + q] < 0;
  if (__syncthreads_or(bad)) {
    for (int64_t q = tid; q < n; q += kThreads) {
      p.send_pos[base + q] = -1;
      p.send_dest[base + q] = -1;
    }
    return;
  }

  int cnt = 0;
  if (tid < p.E) {
    const int64_t i = static_cast<int64_t>(tid) * p.N + s;
    const int next = s + 1 < p.N ? p.src_offsets[i + 1] : p.expert_offsets[tid + 1];
    cnt = next - p.src_offsets[i];
  }
  const int incl = warp_inclusive_scan(cnt);
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int v = wsum[lane];
    wsum[lane] = warp_inclusive_scan(v) - v;
  }
  __syncthreads();
  if (tid < p.E) pre[tid] = incl - cnt + wsum[warp];
  __syncthreads();

  for (int64_t q = tid; q < n; q += kThreads) {
    const int64_t pair = base + q;
    const int e = p.topk_idx[pair];
    const int g = p.slot_row[pair];
    const int64_t j = base + pre[e] + (g - p.src_offsets[static_cast<int64_t>(e) * p.N + s]);
    if (kChecked && (j < base || j >= base + n)) {
      atomicCAS(p.error_word, MOE_OK, MOE_ECORRUPT);
      p.send_pos[pair] = -1;
      continue;
    }
    p.send_pos[pair] = static_cast<int32_t>(j);
    p.send_dest[j] = g;
  }
}

}  // namespace

cudaError_t launch_staged_layout(const StagedLayoutParams& p, bool pdl, cudaStream_t stream) {
  if (p.T == 0) return cudaSuccess;
  return launch_kernel(staged_layout_kernel, dim3(p.N), dim3(kThreads), 0, stream, pdl, p);
}

}  // namespace moe
