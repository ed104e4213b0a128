// Dense padded all-to-all: the pages' comparison system, emulated on one GPU.
//
// "Efficient and portable mixture-of-experts communication" (Sharding and
// parallelism): torch's all_to_all is not suited to MoE dispatch because it
// needs padding (or a GPU-CPU synchronisation) when ranks send different
// numbers of tokens to each peer; (Benchmarks) the dense all-to-all is
// bandwidth-bound and moves an order of magnitude more data than the sparse
// kernels.  Here every (source rank s, destination rank r) chunk is a block
// of `cap` rows fixed before the layer, so no count has to be exchanged:
//
//   dense_layout   per (token, slot): its row in the send buffer,
//                  (s*N + r)*cap + j, and in the receive buffer,
//                  (r*N + s)*cap + j, j = its rank among source s's rows to
//                  rank r in (expert, token) order (from the routing tables);
//   (bulk pack)    x rows into the send blocks (the context's pack kernel);
//   dense_a2a      the exchange: every block whole, padding included, block
//                  s*N+r of one buffer to block r*N+s of the other;
//   row_move       the receive side's copy from the receive blocks to the
//                  grouped rows (and, for combine, the expert outputs into
//                  their blocks);
//   (combine)      the receiver-only combine reads the rows back from the
//                  blocks, so its float32 chain and result are unchanged.
//
// Padding rows are sent as they are (the emulation does not clear them): the
// exchange moves N*N*cap rows whatever the counts.

#include <cuda_runtime.h>

#include "moe_kernels.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads) dense_layout_kernel(DenseLayoutParams p) {
  ptx::wait_prerequisites();  // the routing tables come from the previous kernel
  const int64_t pairs = static_cast<int64_t>(p.T) * p.K;
  const int Tr = p.T / p.N, L = p.E / p.N;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; i < pairs;
       i += static_cast<int64_t>(gridDim.x) * kThreads) {
    const int32_t row = p.slot_row[i];
    if (row < 0) {  // routing error: nothing moves
      p.send_pos[i] = -1;
      p.recv_pos[i] = -1;
      continue;
    }
    const int t = static_cast<int>(i / p.K);
    const int e = p.topk_idx[i];
    const int s = t / Tr, r = e / L;
    // Rows of source s to the experts of rank r before e, then e's rows of
    // tokens before t.
    int64_t j = row - p.src_offsets[static_cast<int64_t>(e) * p.N + s];
    for (int q = r * L; q < e; ++q) {
      const int32_t lo = p.src_offsets[static_cast<int64_t>(q) * p.N + s];
      const int32_t hi = s + 1 < p.N ? p.src_offsets[static_cast<int64_t>(q) * p.N + s + 1] : p.expert_offsets[q + 1];
      j += hi - lo;
    }
    if (kChecked && (j < 0 || j >= p.cap)) {
      atomicCAS(p.error_word, MOE_OK, MOE_ECORRUPT);
      p.send_pos[i] = -1;
      p.recv_pos[i] = -1;
      continue;
    }
    p.send_pos[i] = static_cast<int32_t>((static_cast<int64_t>(s) * p.N + r) * p.cap + j);
    p.recv_pos[i] = static_cast<int32_t>((static_cast<int64_t>(r) * p.N + s) * p.cap + j);
  }
}

// Block s*N+r of `in` to block r*N+s of `out`, 16 bytes per thread and step,
// four steps in flight.  Skipped after a routing error.
__global__ void __launch_bounds__(kThreads) dense_a2a_kernel(DenseA2aParams p) {
  ptx::wait_prerequisites();
  if (p.error_word && *reinterpret_cast<volatile const int32_t*>(p.error_word) == MOE_EROUTE) return;
  const int64_t block_chunks = p.cap * (p.row_bytes >> 4);
  const int64_t total = static_cast<int64_t>(p.N) * p.N * block_chunks;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
  for (int64_t c0 = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; c0 < total; c0 += 4 * stride) {
    uint4 v[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int64_t c = c0 + q * stride;
      if (c < total) v[q] = ptx::ld_stream_v4(p.in + c * 16);
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int64_t c = c0 + q * stride;
      if (c < total) {
        const int64_t b = c / block_chunks;
        const int64_t rest = c - b * block_chunks;
        const int64_t ob = (b % p.N) * p.N + b / p.N;
        ptx::st_v4(p.out + (ob * block_chunks + rest) * 16, v[q]);
      }
    }
  }
}

// dst[dst_row[i]] = src[src_row[i]] for i < n (rows of row_bytes, 16-byte
// chunks, one warp per row); an entry < 0 skips the row.
__global__ void __launch_bounds__(kThreads) row_move_kernel(RowMoveParams p) {
  ptx::wait_prerequisites();
  const int lane = threadIdx.x & 31;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (kThreads >> 5);
  const int64_t chunks = p.row_bytes >> 4;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * (kThreads >> 5) + (threadIdx.x >> 5); i < p.n; i += warps) {
    const int32_t sr = p.src_row[i], dr = p.dst_row[i];
    if (sr < 0 || dr < 0) continue;
    if (kChecked && (sr >= p.src_rows || dr >= p.dst_rows)) {
      if (lane == 0) atomicCAS(p.error_word, MOE_OK, MOE_ECORRUPT);
      continue;
    }
    const uint8_t* src = p.src + static_cast<int64_t>(sr) * p.row_bytes;
    uint8_t* dst = p.dst + static_cast<int64_t>(dr) * p.row_bytes;
    for (int64_t c0 = lane; c0 < chunks; c0 += 4 * 32) {
      uint4 v[4];
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (c0 + q * 32 < chunks) v[q] = ptx::ld_stream_v4(src + (c0 + q * 32) * 16);
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (c0 + q * 32 < chunks) ptx::st_v4(dst + (c0 + q * 32) * 16, v[q]);
    }
  }
}

int grid_for(int64_t work, int64_t per_cta, int sms) {
  int64_t g = (work + per_cta - 1) / per_cta;
  const int64_t cap = static_cast<int64_t>(sms) * 8;
  if (g > cap) g = cap;
  if (g < 1) g = 1;
  return static_cast<int>(g);
}

}  // namespace

cudaError_t launch_dense_layout(const DenseLayoutParams& p, int sms, bool pdl, cudaStream_t stream) {
  const int64_t pairs = static_cast<int64_t>(p.T) * p.K;
  if (pairs == 0) return cudaSuccess;
  return launch_kernel(dense_layout_kernel, dim3(grid_for(pairs, kThreads, sms)), dim3(kThreads), 0, stream, pdl, p);
}

cudaError_t launch_dense_a2a(const DenseA2aParams& p, int sms, bool pdl, cudaStream_t stream) {
  const int64_t total = static_cast<int64_t>(p.N) * p.N * p.cap * (p.row_bytes >> 4);
  if (total == 0) return cudaSuccess;
  return launch_kernel(dense_a2a_kernel, dim3(grid_for(total, 4 * kThreads, sms)), dim3(kThreads), 0, stream, pdl,
                       p);
}

cudaError_t launch_row_move(const RowMoveParams& p, int sms, bool pdl, cudaStream_t stream) {
  if (p.n == 0) return cudaSuccess;
  return launch_kernel(row_move_kernel, dim3(grid_for(p.n, kThreads >> 5, sms)), dim3(kThreads), 0, stream, pdl, p);
}

}  // namespace moe
