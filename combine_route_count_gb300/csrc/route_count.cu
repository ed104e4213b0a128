// route_count: the routing half of dispatch, in one thread block.
//
// "Enabling trillion-parameter models on AWS EFA" (Dispatch and combine):
// dispatch-send aggregates the routing information and counts tokens per
// expert with atomic adds in shared memory inside a single block, then takes
// the cumulative sum of the counts to find where each token goes in
// contiguous buffers.  "Efficient and portable mixture-of-experts
// communication" (Dispatch) keeps, next to the grouped rows, where each row
// came from so that combine can send it back.
//
// The block computes, for T tokens with K distinct experts each:
//   pass 1  cnt[e]            shared-memory atomicAdd histogram, plus the
//                             range / duplicate check of every index
//   scan    expert_offsets    exclusive warp-shuffle scan of cnt (E <= 1024,
//                             one expert per thread), rank_offsets, bound check
//   pass 2  slot_row, row_src stable rank of (t, k) inside expert e:
//                             slot_row[t,k] = expert_offsets[e] + #{t' < t : e in idx[t']}
//           src_offsets       the same count taken at each rank boundary s*T/N
//
// Pass 2 walks the tokens in chunks of 32*W (one token per thread).  Each
// token sets its bit in a per-(expert, warp) 32-bit mask with atomicOr (the
// result does not depend on the order of the atomics), a warp-shuffle scan
// over the W mask popcounts of each expert gives every warp's base, and a
// token's rank is that base plus the popcount of the lower lanes' bits.  No
// slot is grabbed with an atomic counter, so the placement is deterministic
// and stable by token, i.e. by (source rank, token within rank).

#include <cuda_runtime.h>

#include "moe_kernels.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kThreads = kRouteThreads;

// Warps of tokens per chunk: 32 (1024 tokens) unless the per-expert masks
// would not fit in shared memory.
__host__ __device__ inline int chunk_warps(int E) { return E <= 768 ? 32 : 16; }

struct Smem {
  int32_t* cnt;    // [E] histogram, then the running per-expert carry
  int32_t* off;    // [E+1] expert offsets
  int32_t* wsum;   // [32] scan scratch
  uint32_t* mask;  // [E*S] per (expert, warp) token bitmask, S = W + 1 (padding)
  int32_t* base;   // [E*S] rank of the warp's first token inside the expert
};

__device__ inline Smem carve(void* raw, int E) {
  const int S = chunk_warps(E) + 1;
  int32_t* p = static_cast<int32_t*>(raw);
  Smem s;
  s.cnt = p;
  s.off = s.cnt + E;
  s.wsum = s.off + E + 1;
  s.mask = reinterpret_cast<uint32_t*>(s.wsum + 32);
  s.base = reinterpret_cast<int32_t*>(s.mask + E * S);
  return s;
}

template <int KMAX, int VEC>
__device__ __forceinline__ void load_choices(const int32_t* __restrict__ row, int K, int (&e)[KMAX]) {
#pragma unroll
  for (int k = 0; k < KMAX; k += VEC) {
    if (k < K) {
      if constexpr (VEC == 4) {
        int4 v = __ldg(reinterpret_cast<const int4*>(row + k));
        e[k] = v.x;
        e[k + 1] = v.y;
        e[k + 2] = v.z;
        e[k + 3] = v.w;
      } else if constexpr (VEC == 2) {
        int2 v = __ldg(reinterpret_cast<const int2*>(row + k));
        e[k] = v.x;
        e[k + 1] = v.y;
      } else {
        e[k] = __ldg(row + k);
      }
    }
  }
}

template <int KMAX, int VEC>
__device__ __forceinline__ void store_slots(int32_t* __restrict__ row, int K, const int (&r)[KMAX]) {
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

__device__ __forceinline__ int warp_inclusive_scan(int v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  return v;
}

// Range check and repeated-expert check of one token's choices; counts the
// valid ones.  Returns true if the token is malformed.
template <int KMAX>
__device__ __forceinline__ bool count_token(const int (&e)[KMAX], int K, int E, int32_t* cnt) {
  bool bad = false;
#pragma unroll
  for (int k = 0; k < KMAX; ++k) {
    if (k < K) {
      if (static_cast<unsigned>(e[k]) >= static_cast<unsigned>(E)) {
        bad = true;
      } else {
#pragma unroll
        for (int j = 0; j < k; ++j) bad |= (e[j] == e[k]);
        atomicAdd(&cnt[e[k]], 1);
      }
    }
  }
  return bad;
}

// U = tokens each thread loads per round in pass 1 (more loads in flight).
template <int KMAX, int VEC, int U>
__global__ void __launch_bounds__(kThreads, 1) route_count_kernel(RouteCountParams p) {
  extern __shared__ __align__(16) int32_t smem_raw[];
  const int E = p.E, K = p.K, N = p.N, T = p.T;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int W = chunk_warps(E), S = W + 1, CH = 32 * W;
  Smem sm = carve(smem_raw, E);

  // The pack kernel may start loading token rows now: they do not depend on
  // anything this kernel writes.
  ptx::launch_dependents();
  // The pack's and the combine's unit queues restart at 0 for this layer
  // (units are claimed from them only after this grid has completed).
  // Launched without programmatic serialisation, this kernel starts after
  // every earlier kernel has ended.
  if (p.queue && tid == 0) {
    p.queue[0] = 0ull;  // the pack's units
    p.queue[1] = 0ull;  // the combine's units
  }

  for (int i = tid; i < E; i += kThreads) sm.cnt[i] = 0;
  __syncthreads();

  // ---- pass 1: histogram + validation ----
  bool bad = false;
  for (int t0 = tid; t0 < T; t0 += U * kThreads) {
    int e[U][KMAX];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int t = t0 + u * kThreads;
      if (t < T) load_choices<KMAX, VEC>(p.topk_idx + static_cast<int64_t>(t) * K, K, e[u]);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int t = t0 + u * kThreads;
      if (t < T) bad |= count_token<KMAX>(e[u], K, E, sm.cnt);
    }
  }
  if (__syncthreads_or(bad)) {
    // Malformed routing: no row is placed.  slot_row = -1 tells the pack and
    // combine kernels to skip every (token, slot).
    const int64_t pairs = static_cast<int64_t>(T) * K;
    for (int64_t i = tid; i < pairs; i += kThreads) p.slot_row[i] = -1;
    for (int i = tid; i < E; i += kThreads) p.expert_counts[i] = 0;
    for (int i = tid; i <= E; i += kThreads) p.expert_offsets[i] = 0;
    for (int i = tid; i <= N; i += kThreads) p.rank_offsets[i] = 0;
    for (int i = tid; i < E * N; i += kThreads) p.src_offsets[i] = 0;
    if (tid == 0) *p.error_word = MOE_EROUTE;
    return;
  }

  // ---- exclusive scan of the counts (E <= kThreads: one expert per thread) ----
  {
    const int v = tid < E ? sm.cnt[tid] : 0;
    const int incl = warp_inclusive_scan(v, lane);
    if (lane == 31) sm.wsum[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      const int ws = sm.wsum[lane];
      const int wi = warp_inclusive_scan(ws, lane);
      sm.wsum[lane] = wi - ws;
    }
    __syncthreads();
    const int excl = incl - v + sm.wsum[warp];
    if (tid < E) {
      sm.off[tid] = excl;
      sm.cnt[tid] = excl;  // carry for pass 2
      p.expert_counts[tid] = v;
      p.expert_offsets[tid] = excl;
    }
    if (tid == E - 1) {
      sm.off[E] = excl + v;
      p.expert_offsets[E] = excl + v;
    }
    __syncthreads();
  }
  const int L = E / N;
  const int Tr = T / N;
  for (int r = tid; r <= N; r += kThreads) p.rank_offsets[r] = sm.off[r * L];
  // Receive bound of one rank: N * (T/N) * max(K, E/N) rows.
  const int64_t bound = static_cast<int64_t>(N) * Tr * (K > L ? K : L);
  bool over = false;
  for (int r = tid; r < N; r += kThreads) over |= (sm.off[(r + 1) * L] - sm.off[r * L]) > bound;
  over = __syncthreads_or(over);

  if (T == 0) {
    for (int i = tid; i < E * N; i += kThreads) p.src_offsets[i] = 0;
  }

  // ---- pass 2: stable ranks, one chunk of CH tokens at a time ----
  for (int c0 = 0; c0 < T; c0 += CH) {
    for (int i = tid; i < E * S; i += kThreads) sm.mask[i] = 0u;
    __syncthreads();
    const int t = c0 + tid;
    const bool mine = tid < CH && t < T;
    int e[KMAX];
    if (mine) {
      load_choices<KMAX, VEC>(p.topk_idx + static_cast<int64_t>(t) * K, K, e);
#pragma unroll
      for (int k = 0; k < KMAX; ++k)
        if (k < K) atomicOr(&sm.mask[e[k] * S + warp], 1u << lane);
    }
    __syncthreads();
    // Per expert: scan the W warp popcounts (one lane per warp word).
    for (int ex = warp; ex < E; ex += kThreads / 32) {
      const uint32_t m = lane < W ? sm.mask[ex * S + lane] : 0u;
      const int v = __popc(m);
      const int incl = warp_inclusive_scan(v, lane);
      const int carry = sm.cnt[ex];
      if (lane < W) sm.base[ex * S + lane] = carry + incl - v;
      const int total = __shfl_sync(0xffffffffu, incl, 31);
      __syncwarp();
      if (lane == 0) sm.cnt[ex] = carry + total;
    }
    __syncthreads();
    if (mine) {
      const uint32_t lower = (1u << lane) - 1u;
      int r[KMAX];
#pragma unroll
      for (int k = 0; k < KMAX; ++k) {
        if (k < K) {
          const int i = e[k] * S + warp;
          r[k] = sm.base[i] + __popc(sm.mask[i] & lower);
          p.row_src[r[k]] = t * K + k;
        }
      }
      store_slots<KMAX, VEC>(p.slot_row + static_cast<int64_t>(t) * K, K, r);
    }
    // src_offsets at every rank boundary b = s*Tr that falls in [c0, c0+CH).
    {
      const int c1 = min(T, c0 + CH);
      const int s_lo = (c0 + Tr - 1) / Tr;
      const int s_hi = min(N, (c1 + Tr - 1) / Tr);
      const int pairs = (s_hi - s_lo) * E;
      for (int j = tid; j < pairs; j += kThreads) {
        const int s = s_lo + j / E, ex = j % E;
        const int pos = s * Tr - c0;
        const int i = ex * S + (pos >> 5);
        p.src_offsets[ex * N + s] = sm.base[i] + __popc(sm.mask[i] & ((1u << (pos & 31)) - 1u));
      }
    }
    __syncthreads();
  }
  if (tid == 0) *p.error_word = over ? MOE_EBOUND : MOE_OK;
}

template <int KMAX, int VEC>
cudaError_t launch_kmax_vec(const RouteCountParams& p, cudaStream_t stream) {
  constexpr int U = KMAX <= 8 ? 4 : 2;
  auto* kern = route_count_kernel<KMAX, VEC, U>;
  const size_t smem = route_count_smem_bytes(p.E);
  cudaError_t err = set_kernel_limits(reinterpret_cast<const void*>(kern), smem);
  if (err != cudaSuccess) return err;
  return launch_kernel(kern, dim3(1), dim3(kThreads), smem, stream, false, p);
}

}  // namespace

size_t route_count_smem_bytes(int E) {
  const int S = chunk_warps(E) + 1;
  return sizeof(int32_t) * (static_cast<size_t>(E) + (E + 1) + 32 + 2 * static_cast<size_t>(E) * S);
}

cudaError_t launch_route_count(const RouteCountParams& p, int idx_vec, cudaStream_t stream) {
  // Wider index loads need K to be a multiple of the width (the caller also
  // checks the pointer's alignment).
  if (idx_vec != 1 && p.K % idx_vec != 0) idx_vec = 1;
  if (p.K <= 8) {
    if (idx_vec == 4) return launch_kmax_vec<8, 4>(p, stream);
    if (idx_vec == 2) return launch_kmax_vec<8, 2>(p, stream);
    return launch_kmax_vec<8, 1>(p, stream);
  }
  if (idx_vec == 4) return launch_kmax_vec<16, 4>(p, stream);
  if (idx_vec == 2) return launch_kmax_vec<16, 2>(p, stream);
  return launch_kmax_vec<16, 1>(p, stream);
}

}  // namespace moe
