// Routing spread over many SMs: route_local + route_finalize.
//
// Same results as route_count (stable placement by expert, then token; the
// counts, exclusive-scan offsets, per-(expert, source rank) and per-rank
// offsets of "Enabling trillion-parameter models on AWS EFA", Dispatch and
// combine / Send and receive buffers), computed by B blocks instead of one.
// One block walks all T*K routing entries in about 40 us at DeepSeek size,
// bound by one SM's issue rate; here each block handles a chunk of tokens:
//
// route_local (block c, tokens [c*CT, (c+1)*CT)), in sub-chunks of 256:
//   per-(expert, warp) bitmasks set with atomicOr -> the stable rank of each
//   (t, k) among the chunk's tokens with the same expert, and the chunk's
//   histogram hist[c][e]; the rank counted up to each rank boundary s*T/N in
//   the chunk; range / repeat check of every index (one flag per block).
// route_finalize (block c), after route_local completes:
//   total[e] = sum over all chunks, prefix[e] = sum over chunks before c,
//   expert_offsets = exclusive scan of total, and for the chunk's tokens
//   slot_row[t,k] = expert_offsets[e] + prefix[e] + local rank.
//   Block 0 also writes counts, offsets, rank offsets and the error word.
//
// No block waits on another inside a kernel: the only ordering is the kernel
// boundary (programmatic dependent launch lets each next grid start early).

#include <cuda_runtime.h>

#include "moe_kernels.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kThreads = kSplitThreads;  // tokens per sub-chunk, one per thread
constexpr int kW = kThreads / 32;        // warps per sub-chunk
constexpr int kS = kW + 1;               // padded mask stride per expert

template <int KMAX, int VEC>
__device__ __forceinline__ void load_row(const int32_t* __restrict__ row, int K, int (&e)[KMAX]) {
#pragma unroll
  for (int k = 0; k < KMAX; k += VEC) {
    if (k < K) {
      if constexpr (VEC == 4) {
        const int4 v = *reinterpret_cast<const int4*>(row + k);
        e[k] = v.x;
        e[k + 1] = v.y;
        e[k + 2] = v.z;
        e[k + 3] = v.w;
      } else if constexpr (VEC == 2) {
        const int2 v = *reinterpret_cast<const int2*>(row + k);
        e[k] = v.x;
        e[k + 1] = v.y;
      } else {
        e[k] = row[k];
      }
    }
  }
}

template <int KMAX, int VEC>
__device__ __forceinline__ void store_row(int32_t* __restrict__ row, int K, const int (&r)[KMAX]) {
#pragma unroll
  for (int k = 0; k < KMAX; k += VEC) {
    if (k < K) {
      if constexpr (VEC == 4) {
        *reinterpret_cast<int4*>(row + k) = make_int4(r[k], r[k + 1], r[k + 2], r[k + 3]);
      } else if constexpr (VEC == 2) {
        *reinterpret_cast<int2*>(row + k) = make_int2(r[k], r[k + 1]);
      } else {
        row[k] = r[k];
      }
    }
  }
}

__device__ __forceinline__ int warp_incl_scan(int v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  return v;
}

template <int KMAX, int VEC>
__global__ void __launch_bounds__(kThreads) route_local_kernel(RouteSplitParams p) {
  extern __shared__ __align__(16) int32_t smem[];
  const int E = p.E, K = p.K, N = p.N, T = p.T;
  uint32_t* mask = reinterpret_cast<uint32_t*>(smem);  // [E * kS]
  int32_t* lbase = smem + E * kS;                      // [E * kS] chunk-local rank of each warp's first token
  int32_t* carry = lbase + E * kS;                     // [E] tokens of earlier sub-chunks per expert
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int c = blockIdx.x;
  const int c0 = c * p.chunk;
  const int c1 = min(T, c0 + p.chunk);
  const int Tr = T / N;

  ptx::launch_dependents();
  // The pack's and the combine's unit queues restart at 0 (this kernel is
  // launched without programmatic serialisation: every earlier kernel has
  // ended).
  if (p.queue && c == 0 && tid == 0) {
    p.queue[0] = 0ull;  // the pack's units
    p.queue[1] = 0ull;  // the combine's units
  }

  for (int i = tid; i < E; i += kThreads) carry[i] = 0;
  bool bad = false;
  for (int s0 = c0; s0 < c1; s0 += kThreads) {
    for (int i = tid; i < E * kS; i += kThreads) mask[i] = 0u;
    __syncthreads();
    const int t = s0 + tid;
    const bool mine = t < c1;
    int e[KMAX];
    if (mine) {
      load_row<KMAX, VEC>(p.topk_idx + static_cast<int64_t>(t) * K, K, e);
#pragma unroll
      for (int k = 0; k < KMAX; ++k) {
        if (k < K) {
          if (static_cast<unsigned>(e[k]) >= static_cast<unsigned>(E)) {
            bad = true;
            e[k] = 0;  // keep the index in range; the whole layer is rejected anyway
          } else {
#pragma unroll
            for (int j = 0; j < k; ++j) bad |= (e[j] == e[k]);
            atomicOr(&mask[e[k] * kS + warp], 1u << lane);
          }
        }
      }
    }
    __syncthreads();
    // Chunk-local base of each warp word, per expert (kW words, in order).
    for (int ex = tid; ex < E; ex += kThreads) {
      int run = carry[ex];
#pragma unroll
      for (int w = 0; w < kW; ++w) {
        lbase[ex * kS + w] = run;
        run += __popc(mask[ex * kS + w]);
      }
      carry[ex] = run;
    }
    __syncthreads();
    if (mine) {
      const uint32_t lower = (1u << lane) - 1u;
      int r[KMAX];
#pragma unroll
      for (int k = 0; k < KMAX; ++k) {
        if (k < K) {
          const int i = e[k] * kS + warp;
          r[k] = lbase[i] + __popc(mask[i] & lower);
        }
      }
      store_row<KMAX, VEC>(p.slot_row + static_cast<int64_t>(t) * K, K, r);  // chunk-local for now
    }
    // Chunk-local count of each expert before every rank boundary b = s*Tr
    // in this sub-chunk (finalize adds the chunk's base).
    if (Tr > 0) {
      const int sub1 = min(c1, s0 + kThreads);
      const int s_lo = (s0 + Tr - 1) / Tr;
      const int s_hi = min(N, (sub1 + Tr - 1) / Tr);
      for (int s = s_lo; s < s_hi; ++s) {
        const int pos = s * Tr - s0;
        const uint32_t below = (1u << (pos & 31)) - 1u;
        for (int ex = tid; ex < E; ex += kThreads) {
          const int i = ex * kS + (pos >> 5);
          p.src_offsets[static_cast<int64_t>(ex) * N + s] = lbase[i] + __popc(mask[i] & below);
        }
      }
    }
    __syncthreads();
  }
  for (int ex = tid; ex < E; ex += kThreads) p.hist[static_cast<int64_t>(c) * E + ex] = carry[ex];
  bad = __syncthreads_or(bad);
  if (tid == 0) p.block_err[c] = bad ? 1 : 0;
}

// Exclusive scan of v over the block (E <= 4 * kThreads values, each thread
// owning four consecutive entries).  Returns the total.
__device__ int block_exclusive_scan4(const int32_t* in, int32_t* out, int E, int32_t* wsum) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int v[4], s = 0;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int i = tid * 4 + q;
    v[q] = i < E ? in[i] : 0;
    s += v[q];
  }
  const int incl = warp_incl_scan(s, lane);
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int x = lane < kW ? wsum[lane] : 0;
    const int xi = warp_incl_scan(x, lane);
    if (lane < kW) wsum[lane] = xi - x;
    if (lane == 31) wsum[kW] = xi;
  }
  __syncthreads();
  int run = incl - s + wsum[warp];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int i = tid * 4 + q;
    if (i < E) out[i] = run;
    run += v[q];
  }
  const int total = wsum[kW];
  __syncthreads();
  return total;
}

template <int KMAX, int VEC>
__global__ void __launch_bounds__(kThreads) route_finalize_kernel(RouteSplitParams p) {
  extern __shared__ __align__(16) int32_t smem[];
  const int E = p.E, K = p.K, N = p.N, T = p.T;
  int32_t* total = smem;         // [E]
  int32_t* off = total + E;      // [E] exclusive scan of total
  int32_t* base = off + E;       // [E] first row of this chunk's tokens per expert
  int32_t* wsum = base + E;      // [kW + 1]
  const int tid = threadIdx.x;
  const int c = blockIdx.x;
  const int B = gridDim.x;
  const int c0 = c * p.chunk;
  const int c1 = min(T, c0 + p.chunk);
  const int L = E / N;
  const int Tr = T / N;

  ptx::launch_dependents();   // the pack kernel may start fetching token rows
  ptx::wait_prerequisites();  // route_local's histograms and local ranks

  bool bad = false;
  for (int i = tid; i < B; i += kThreads) bad |= p.block_err[i] != 0;
  if (__syncthreads_or(bad)) {
    // Malformed routing: nothing is placed; slot_row = -1 makes the pack and
    // combine kernels skip every pair.
    for (int64_t i = static_cast<int64_t>(c0) * K + tid; i < static_cast<int64_t>(c1) * K; i += kThreads)
      p.slot_row[i] = -1;
    if (c == 0) {
      for (int i = tid; i < E; i += kThreads) p.expert_counts[i] = 0;
      for (int i = tid; i <= E; i += kThreads) p.expert_offsets[i] = 0;
      for (int i = tid; i <= N; i += kThreads) p.rank_offsets[i] = 0;
      for (int i = tid; i < E * N; i += kThreads) p.src_offsets[i] = 0;
      if (tid == 0) *p.error_word = MOE_EROUTE;
    }
    return;
  }

  for (int ex = tid; ex < E; ex += kThreads) {
    int tot = 0, pre = 0;
#pragma unroll 8
    for (int b = 0; b < B; ++b) {
      const int h = p.hist[static_cast<int64_t>(b) * E + ex];
      tot += h;
      pre += b < c ? h : 0;
    }
    total[ex] = tot;
    base[ex] = pre;
  }
  __syncthreads();
  block_exclusive_scan4(total, off, E, wsum);
  for (int ex = tid; ex < E; ex += kThreads) base[ex] += off[ex];
  __syncthreads();

  // Final rows of this chunk's tokens.
  for (int t = c0 + tid; t < c1; t += kThreads) {
    int e[KMAX], r[KMAX];
    load_row<KMAX, VEC>(p.topk_idx + static_cast<int64_t>(t) * K, K, e);
    load_row<KMAX, VEC>(p.slot_row + static_cast<int64_t>(t) * K, K, r);
#pragma unroll
    for (int k = 0; k < KMAX; ++k) {
      if (k < K) {
        r[k] += base[e[k]];
        p.row_src[r[k]] = t * K + k;
      }
    }
    store_row<KMAX, VEC>(p.slot_row + static_cast<int64_t>(t) * K, K, r);
  }
  // Rank boundaries that fall in this chunk.
  if (Tr > 0) {
    const int s_lo = (c0 + Tr - 1) / Tr;
    const int s_hi = min(N, (c1 + Tr - 1) / Tr);
    for (int s = s_lo; s < s_hi; ++s)
      for (int ex = tid; ex < E; ex += kThreads) p.src_offsets[static_cast<int64_t>(ex) * N + s] += base[ex];
  } else if (c == 0) {
    for (int i = tid; i < E * N; i += kThreads) p.src_offsets[i] = 0;
  }

  if (c == 0) {
    for (int ex = tid; ex < E; ex += kThreads) {
      p.expert_counts[ex] = total[ex];
      p.expert_offsets[ex] = off[ex];
    }
    if (tid == 0) p.expert_offsets[E] = T * K;
    for (int r = tid; r <= N; r += kThreads) p.rank_offsets[r] = r < N ? off[r * L] : T * K;
    // Receive bound of one rank: N * (T/N) * max(K, E/N) rows.
    const int64_t bound = static_cast<int64_t>(N) * Tr * (K > L ? K : L);
    bool over = false;
    for (int r = tid; r < N; r += kThreads) {
      const int hi = r + 1 < N ? off[(r + 1) * L] : T * K;
      over |= (hi - off[r * L]) > bound;
    }
    over = __syncthreads_or(over);
    if (tid == 0) *p.error_word = over ? MOE_EBOUND : MOE_OK;
  }
}

template <int KMAX, int VEC>
cudaError_t launch_split(const RouteSplitParams& p, int blocks, cudaStream_t stream) {
  auto* k1 = route_local_kernel<KMAX, VEC>;
  auto* k2 = route_finalize_kernel<KMAX, VEC>;
  const size_t s1 = route_local_smem_bytes(p.E);
  const size_t s2 = sizeof(int32_t) * (3 * static_cast<size_t>(p.E) + kW + 1);
  cudaError_t err = set_kernel_limits(reinterpret_cast<const void*>(k1), s1);
  if (err != cudaSuccess) return err;
  err = launch_kernel(k1, dim3(blocks), dim3(kThreads), s1, stream, false, p);
  if (err != cudaSuccess) return err;
  return launch_kernel(k2, dim3(blocks), dim3(kThreads), s2, stream, true, p);
}

}  // namespace

size_t route_local_smem_bytes(int E) {
  return sizeof(int32_t) * (2 * static_cast<size_t>(E) * kS + E);
}

int route_split_chunk(int T) {
  // At most kMaxSplitBlocks chunks; each a multiple of the 256-token sub-chunk.
  int chunk = kThreads;
  while (static_cast<int64_t>(chunk) * kMaxSplitBlocks < T) chunk *= 2;
  return chunk;
}

cudaError_t launch_route_split(const RouteSplitParams& p, int idx_vec, cudaStream_t stream) {
  // Wider index loads need K to be a multiple of the width (the caller also
  // checks the pointer's alignment).
  if (idx_vec != 1 && p.K % idx_vec != 0) idx_vec = 1;
  const int blocks = p.T > 0 ? (p.T + p.chunk - 1) / p.chunk : 1;
  if (p.K <= 8) {
    if (idx_vec == 4) return launch_split<8, 4>(p, blocks, stream);
    if (idx_vec == 2) return launch_split<8, 2>(p, blocks, stream);
    return launch_split<8, 1>(p, blocks, stream);
  }
  if (idx_vec == 4) return launch_split<16, 4>(p, blocks, stream);
  if (idx_vec == 2) return launch_split<16, 2>(p, blocks, stream);
  return launch_split<16, 1>(p, blocks, stream);
}

}  // namespace moe
