// route_cluster: the routing of dispatch in one thread-block cluster.
//
// Same results as route_count (stable placement by expert, then token; the
// counts, exclusive-scan offsets, per-(expert, source rank) and per-rank
// offsets of "Enabling trillion-parameter models on AWS EFA", Dispatch and
// combine / Send and receive buffers).  The pages count in one block with
// shared-memory atomics; one SM takes ~40 us for the 32K routing entries of a
// DeepSeek-sized layer, bound by its issue rate.  Here C <= 16 CTAs of one
// cluster each take a contiguous chunk of tokens:
//
//   1. per sub-chunk of 32*W tokens (one per thread): per-(expert, warp)
//      bitmasks set with shared-memory atomicOr give each (t, k) its stable
//      rank among the chunk's tokens with the same expert; the chunk's
//      per-expert histogram accumulates in shared memory;
//   2. cluster barrier; every CTA reads all C histograms through distributed
//      shared memory: total[e] and prefix[e] (chunks before its own);
//   3. warp-shuffle exclusive scan of total -> expert offsets;
//      slot_row[t,k] = offset[e] + prefix[e] + local rank, row_src inverse,
//      src_offsets at the rank boundaries in the chunk;
//   4. CTA 0 writes counts, offsets, rank offsets and the error word;
//      cluster barrier (no CTA leaves while others may still read its
//      shared memory).
//
// The cluster barriers are hardware barriers that every CTA reaches on every
// path; no thread spins on memory.

#include <cuda_runtime.h>

#include "moe_kernels.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kThreads = kClusterThreads;  // largest CTA (one token per thread)

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.release;" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire;" ::: "memory"); }
__device__ __forceinline__ void cluster_sync() {
  cluster_arrive();
  cluster_wait();
}
// Address of the same shared-memory variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t dsmem_addr(const void* local, uint32_t rank) {
  uint32_t out;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(out) : "r"(ptx::smem_addr(local)), "r"(rank));
  return out;
}
__device__ __forceinline__ int ld_dsmem(uint32_t addr) {
  int v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}

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

struct Smem {
  uint32_t* mask;  // [E*S]
  int32_t* lbase;  // [E*S]
  int32_t* hist;   // [E] this chunk's per-expert totals (read by the whole cluster)
  int32_t* base;   // [E] first row of this chunk's tokens per expert
  int32_t* off;    // [E] expert offsets
  int32_t* wsum;   // [64] scan scratch (two scans of up to 32 warp sums)
  int32_t* flag;   // [1] routing error in this chunk (read by the whole cluster)
  int32_t* lofs;   // [E] chunk-local first row of each expert (staged row_src only)
  int32_t* sval;   // [chunk*K] staged row_src values, grouped by expert
  int16_t* sexp;   // [chunk*K] expert of each staged value
};

__device__ inline Smem carve(int32_t* raw, int E, int S, int staged_pairs) {
  Smem s;
  s.mask = reinterpret_cast<uint32_t*>(raw);
  s.lbase = raw + E * S;
  s.hist = s.lbase + E * S;
  s.base = s.hist + E;
  s.off = s.base + E;
  s.wsum = s.off + E;
  s.flag = s.wsum + 64;
  s.lofs = s.flag + 4;
  s.sval = s.lofs + E;
  s.sexp = reinterpret_cast<int16_t*>(s.sval + staged_pairs);
  return s;
}

// Two exclusive scans in one pass: a[] in place, and (if `second`) b[] into
// b_out[] (b[] itself is left intact: other CTAs may still read it).
__device__ void cta_exclusive_scan2(int32_t* a, const int32_t* b, int32_t* b_out, int E, int32_t* wsum,
                                    bool second) {
  const int nt = blockDim.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = nt >> 5;
  const int per = (E + nt - 1) / nt;
  const int lo = min(E, tid * per), hi = min(E, lo + per);
  int sa = 0, sb = 0;
  for (int i = lo; i < hi; ++i) {
    sa += a[i];
    if (second) sb += b[i];
  }
  const int ia = warp_incl_scan(sa, lane);
  const int ib = warp_incl_scan(sb, lane);
  if (lane == 31) {
    wsum[warp] = ia;
    wsum[32 + warp] = ib;
  }
  __syncthreads();
  if (warp == 0) {
    const int xa = lane < nw ? wsum[lane] : 0;
    const int xb = lane < nw ? wsum[32 + lane] : 0;
    const int ya = warp_incl_scan(xa, lane);
    const int yb = warp_incl_scan(xb, lane);
    __syncwarp();
    if (lane < nw) {
      wsum[lane] = ya - xa;
      wsum[32 + lane] = yb - xb;
    }
  }
  __syncthreads();
  int ra = ia - sa + wsum[warp];
  int rb = ib - sb + wsum[32 + warp];
  for (int i = lo; i < hi; ++i) {
    const int va = a[i];
    a[i] = ra;
    ra += va;
    if (second) {
      b_out[i] = rb;
      rb += b[i];
    }
  }
  __syncthreads();
}

template <int KMAX, int VEC>
__global__ void __launch_bounds__(kThreads, 1) route_cluster_kernel(RouteClusterParams p) {
  extern __shared__ __align__(16) int32_t smem_raw[];
  const int E = p.E, K = p.K, N = p.N, T = p.T;
  const int W = p.warps, S = W + 1, SUB = 32 * W;  // blockDim.x == SUB: one token per thread
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t rank = cluster_ctarank();
  const int C = gridDim.x;  // the grid is one cluster
  const int c0 = min(T, static_cast<int>(rank) * p.chunk);
  const int c1 = min(T, c0 + p.chunk);
  const int Tr = T / N;
  Smem sm = carve(smem_raw, E, S, p.staged ? p.chunk * K : 0);

  // Inputs may come from the previous kernel in the stream: wait for it,
  // then let the pack kernel start fetching token rows.
  ptx::wait_prerequisites();
  ptx::launch_dependents();
  // The pack's and the combine's unit queues restart at 0 for this layer;
  // units are claimed from them only after this grid has completed.
  if (p.queue && rank == 0 && tid == 0) {
    p.queue[0] = 0ull;  // the pack's units
    p.queue[1] = 0ull;  // the combine's units
  }

  // First sub-chunk's indices are requested before the shared-memory set-up.
  int e[KMAX], r[KMAX];
  if (c0 + tid < c1) load_row<KMAX, VEC>(p.topk_idx + static_cast<int64_t>(c0 + tid) * K, K, e);
  for (int i = tid; i < E; i += SUB) sm.hist[i] = 0;
  if (tid == 0) *sm.flag = 0;
  bool bad = false;
  // The last sub-chunk keeps its ranks in registers and its masks in shared
  // memory across the cluster barrier; earlier ones park their chunk-local
  // ranks in slot_row and their boundary counts in src_offsets.
  int last_s0 = c1;
  for (int s0 = c0; s0 < c1; s0 += SUB) {
    const int t = s0 + tid;
    const bool mine = t < c1;
    if (s0 != c0 && mine) load_row<KMAX, VEC>(p.topk_idx + static_cast<int64_t>(t) * K, K, e);
    for (int i = tid; i < E * S; i += SUB) sm.mask[i] = 0u;
    __syncthreads();
    if (mine) {
#pragma unroll
      for (int k = 0; k < KMAX; ++k) {
        if (k < K) {
          if (static_cast<unsigned>(e[k]) >= static_cast<unsigned>(E)) {
            bad = true;
            e[k] = 0;  // keep the index in range; the layer is rejected anyway
          } else {
#pragma unroll
            for (int j = 0; j < k; ++j) bad |= (e[j] == e[k]);
            atomicOr(&sm.mask[e[k] * S + warp], 1u << lane);
          }
        }
      }
    }
    __syncthreads();
    // Per expert: chunk-local base of each warp word.  Few words: one thread
    // per expert walks them; many: one warp per expert, shuffle scan.
    if (W <= 8) {
      for (int ex = tid; ex < E; ex += SUB) {
        int run = sm.hist[ex];
        for (int w = 0; w < W; ++w) {
          sm.lbase[ex * S + w] = run;
          run += __popc(sm.mask[ex * S + w]);
        }
        sm.hist[ex] = run;
      }
    } else {
      for (int ex = warp; ex < E; ex += W) {
        const int v = lane < W ? __popc(sm.mask[ex * S + lane]) : 0;
        const int incl = warp_incl_scan(v, lane);
        const int carry = sm.hist[ex];
        if (lane < W) sm.lbase[ex * S + lane] = carry + incl - v;
        const int tot = __shfl_sync(0xffffffffu, incl, 31);
        __syncwarp();
        if (lane == 0) sm.hist[ex] = carry + tot;
      }
    }
    __syncthreads();
    if (mine) {
      const uint32_t lower = (1u << lane) - 1u;
#pragma unroll
      for (int k = 0; k < KMAX; ++k) {
        if (k < K) {
          const int i = e[k] * S + warp;
          r[k] = sm.lbase[i] + __popc(sm.mask[i] & lower);
        }
      }
    }
    if (s0 + SUB >= c1) {
      last_s0 = s0;
    } else {
      if (mine) store_row<KMAX, VEC>(p.slot_row + static_cast<int64_t>(t) * K, K, r);
      if (Tr > 0) {
        const int s_lo = (s0 + Tr - 1) / Tr;
        const int s_hi = min(N, (s0 + SUB + Tr - 1) / Tr);
        for (int ex = tid; ex < E; ex += SUB) {
          for (int s = s_lo; s < s_hi; ++s) {
            const int pos = s * Tr - s0;
            const int i = ex * S + (pos >> 5);
            p.src_offsets[static_cast<int64_t>(ex) * N + s] =
                sm.lbase[i] + __popc(sm.mask[i] & ((1u << (pos & 31)) - 1u));
          }
        }
      }
      __syncthreads();  // masks are cleared for the next sub-chunk
    }
  }
  if (__syncthreads_or(bad) && tid == 0) *sm.flag = 1;

  // ---- exchange the chunk histograms through distributed shared memory ----
  cluster_sync();
  bool any_bad = false;
  if (tid < C) any_bad = ld_dsmem(dsmem_addr(sm.flag, tid)) != 0;
  {
    // G threads per expert (G a power of two, G | 32, G * E <= threads)
    // split the C loads.
    const int G = p.dsmem_group;
    const int gshift = __ffs(G) - 1;
    const int sub = tid & (G - 1);
    const int rounds = (E * G + SUB - 1) / SUB;
    for (int rd = 0; rd < rounds; ++rd) {
      const int ex = (rd * SUB + tid) >> gshift;
      int tot = 0, before = 0;
      if (ex < E) {
        int h[kMaxClusterCtas];
#pragma unroll
        for (int q = 0; q < kMaxClusterCtas; ++q)
          h[q] = (q < C && (q & (G - 1)) == sub) ? ld_dsmem(dsmem_addr(sm.hist + ex, q)) : 0;
#pragma unroll
        for (int q = 0; q < kMaxClusterCtas; ++q) {
          tot += h[q];
          before += q < static_cast<int>(rank) ? h[q] : 0;
        }
      }
      for (int o = 1; o < G; o <<= 1) {
        tot += __shfl_xor_sync(0xffffffffu, tot, o);
        before += __shfl_xor_sync(0xffffffffu, before, o);
      }
      if (ex < E && sub == 0) {
        sm.off[ex] = tot;  // totals for now; scanned below
        sm.base[ex] = before;
      }
    }
  }
  any_bad = __syncthreads_or(any_bad);
  // Done reading the other CTAs' shared memory: signal it now, wait for the
  // others only at exit, so the writes below overlap the barrier.
  cluster_arrive();

  if (any_bad) {
    // Malformed routing: nothing is placed; slot_row = -1 makes the pack and
    // combine kernels skip every pair.
    for (int64_t i = static_cast<int64_t>(c0) * K + tid; i < static_cast<int64_t>(c1) * K; i += SUB)
      p.slot_row[i] = -1;
    if (rank == 0) {
      for (int i = tid; i < E; i += SUB) p.expert_counts[i] = 0;
      for (int i = tid; i <= E; i += SUB) p.expert_offsets[i] = 0;
      for (int i = tid; i <= N; i += SUB) p.rank_offsets[i] = 0;
      for (int i = tid; i < E * N; i += SUB) p.src_offsets[i] = 0;
      if (tid == 0) *p.error_word = MOE_EROUTE;
    }
    cluster_wait();
    return;
  }

  if (rank == 0)
    for (int ex = tid; ex < E; ex += SUB) p.expert_counts[ex] = sm.off[ex];
  // In place: expert offsets from the totals and, for staging, the
  // chunk-local offsets from this chunk's histogram, in one pass.
  cta_exclusive_scan2(sm.off, sm.hist, sm.lofs, E, sm.wsum, p.staged != 0);
  for (int ex = tid; ex < E; ex += SUB) sm.base[ex] += sm.off[ex];
  __syncthreads();

  // Final rows: sub-chunks parked in slot_row, then the one in registers.
  for (int s0 = c0; s0 < last_s0; s0 += SUB) {
    const int t = s0 + tid;
    int ee[KMAX], rr[KMAX];
    load_row<KMAX, VEC>(p.topk_idx + static_cast<int64_t>(t) * K, K, ee);
    load_row<KMAX, VEC>(p.slot_row + static_cast<int64_t>(t) * K, K, rr);
#pragma unroll
    for (int k = 0; k < KMAX; ++k) {
      if (k < K) {
        rr[k] += sm.base[ee[k]];
        p.row_src[rr[k]] = t * K + k;
      }
    }
    store_row<KMAX, VEC>(p.slot_row + static_cast<int64_t>(t) * K, K, rr);
  }
  if (p.staged) {
    // One sub-chunk: r[] are chunk-local ranks.  Stage row_src grouped by
    // expert in shared memory, then write each expert's run of rows with
    // consecutive threads (coalesced) instead of one scattered store per pair.
    if (last_s0 < c1 && last_s0 + tid < c1) {
      const int t = last_s0 + tid;
#pragma unroll
      for (int k = 0; k < KMAX; ++k) {
        if (k < K) {
          const int pos = sm.lofs[e[k]] + r[k];
          sm.sval[pos] = t * K + k;
          sm.sexp[pos] = static_cast<int16_t>(e[k]);
          r[k] += sm.base[e[k]];
        }
      }
      store_row<KMAX, VEC>(p.slot_row + static_cast<int64_t>(t) * K, K, r);
    }
    __syncthreads();
    const int pairs = (c1 - c0) * K;
    for (int i = tid; i < pairs; i += SUB) {
      const int ex = sm.sexp[i];
      p.row_src[sm.base[ex] + (i - sm.lofs[ex])] = sm.sval[i];
    }
  } else if (last_s0 < c1 && last_s0 + tid < c1) {
    const int t = last_s0 + tid;
#pragma unroll
    for (int k = 0; k < KMAX; ++k) {
      if (k < K) {
        r[k] += sm.base[e[k]];
        p.row_src[r[k]] = t * K + k;
      }
    }
    store_row<KMAX, VEC>(p.slot_row + static_cast<int64_t>(t) * K, K, r);
  }
  // src_offsets at the rank boundaries of this chunk.
  if (Tr > 0) {
    const int s_lo = (c0 + Tr - 1) / Tr;
    const int s_hi = min(N, (c1 + Tr - 1) / Tr);
    for (int ex = tid; ex < E; ex += SUB) {
      const int bx = sm.base[ex];
      for (int s = s_lo; s < s_hi; ++s) {
        const int b = s * Tr;
        int32_t* dst = p.src_offsets + static_cast<int64_t>(ex) * N + s;
        if (b >= last_s0) {  // masks of the last sub-chunk are still in shared memory
          const int pos = b - last_s0;
          const int i = ex * S + (pos >> 5);
          *dst = bx + sm.lbase[i] + __popc(sm.mask[i] & ((1u << (pos & 31)) - 1u));
        } else {
          *dst += bx;
        }
      }
    }
  } else if (rank == 0) {
    for (int i = tid; i < E * N; i += SUB) p.src_offsets[i] = 0;
  }

  if (rank == 0) {
    const int L = E / N;
    for (int ex = tid; ex < E; ex += SUB) p.expert_offsets[ex] = sm.off[ex];
    if (tid == 0) p.expert_offsets[E] = T * K;
    for (int q = tid; q <= N; q += SUB) p.rank_offsets[q] = q < N ? sm.off[q * L] : T * K;
    // Receive bound of one rank: N * (T/N) * max(K, E/N) rows.
    const int64_t bound = static_cast<int64_t>(N) * Tr * (K > L ? K : L);
    bool over = false;
    for (int q = tid; q < N; q += SUB) {
      const int hi = q + 1 < N ? sm.off[(q + 1) * L] : T * K;
      over |= (hi - sm.off[q * L]) > bound;
    }
    over = __syncthreads_or(over);
    if (tid == 0) *p.error_word = over ? MOE_EBOUND : MOE_OK;
  }
  cluster_wait();  // no CTA leaves while another may still read its shared memory
}

template <int KMAX, int VEC>
cudaError_t launch_kv(const RouteClusterParams& p, int cluster, cudaStream_t stream, bool query_only, int* ok) {
  auto* kern = route_cluster_kernel<KMAX, VEC>;
  const size_t smem = route_cluster_smem_bytes(p.E, p.warps, p.staged ? p.chunk * p.K : 0);
  cudaError_t err = set_kernel_limits(reinterpret_cast<const void*>(kern), smem, cluster > 8);
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cluster);
  cfg.blockDim = dim3(32 * p.warps);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = query_only ? 1 : 2;
  if (query_only) {
    int n = 0;
    err = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
    *ok = (err == cudaSuccess && n > 0) ? 1 : 0;
    if (err != cudaSuccess) cudaGetLastError();  // clear a refused query; the caller falls back
    return cudaSuccess;
  }
  return cudaLaunchKernelEx(&cfg, kern, p);
}

template <int KMAX, int VEC>
cudaError_t dispatch_kv2(const RouteClusterParams& p, int cluster, cudaStream_t s, bool q, int* ok) {
  return launch_kv<KMAX, VEC>(p, cluster, s, q, ok);
}

cudaError_t dispatch_kv(const RouteClusterParams& p, int idx_vec, int cluster, cudaStream_t s, bool q, int* ok) {
  if (p.K <= 8) {
    if (idx_vec == 4) return dispatch_kv2<8, 4>(p, cluster, s, q, ok);
    if (idx_vec == 2) return dispatch_kv2<8, 2>(p, cluster, s, q, ok);
    return dispatch_kv2<8, 1>(p, cluster, s, q, ok);
  }
  if (idx_vec == 4) return dispatch_kv2<16, 4>(p, cluster, s, q, ok);
  if (idx_vec == 2) return dispatch_kv2<16, 2>(p, cluster, s, q, ok);
  return dispatch_kv2<16, 1>(p, cluster, s, q, ok);
}

}  // namespace

size_t route_cluster_smem_bytes(int E, int warps, int staged_pairs) {
  const size_t S = warps + 1;
  return sizeof(int32_t) * (2 * static_cast<size_t>(E) * S + 4 * static_cast<size_t>(E) + 64 + 4) +
         static_cast<size_t>(staged_pairs) * (sizeof(int32_t) + sizeof(int16_t));
}

void route_cluster_shape(int T, int E, int max_cluster, int* cluster, int* chunk, int* warps) {
  // Chunks of at least 256 tokens, at most max_cluster of them.
  int c = (T + 255) / 256;
  if (c < 1) c = 1;
  if (c > max_cluster) c = max_cluster;
  int ch = (T + c - 1) / c;
  ch = (ch + 31) / 32 * 32;
  if (ch < 32) ch = 32;
  // Sub-chunk (= CTA size): up to 32 warps of tokens (16 when E > 768, to
  // fit the masks); the whole chunk when it is smaller.
  const int wmax = E <= 768 ? 32 : 16;
  int w = (ch + 31) / 32;
  if (w > wmax) w = wmax;
  *cluster = c;
  *chunk = ch;
  *warps = w;
}

void route_cluster_plan(RouteClusterParams* p, int cluster, int max_smem) {
  const int threads = 32 * p->warps;
  // Stage row_src when each CTA's chunk is a single sub-chunk and it fits.
  p->staged = 0;
  if (p->chunk <= threads &&
      route_cluster_smem_bytes(p->E, p->warps, p->chunk * p->K) <= static_cast<size_t>(max_smem))
    p->staged = 1;
  int g = 1;
  while (g * 2 <= kMaxClusterCtas && g * 2 <= cluster && g * 2 * p->E <= threads) g *= 2;
  p->dsmem_group = g;
}

bool route_cluster_supported(const RouteClusterParams& p, int idx_vec, int cluster) {
  int ok = 0;
  if (dispatch_kv(p, idx_vec, cluster, nullptr, true, &ok) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return ok != 0;
}

cudaError_t launch_route_cluster(const RouteClusterParams& p, int idx_vec, int cluster, cudaStream_t stream) {
  // Wider index loads need K to be a multiple of the width (the caller also
  // checks the pointer's alignment).
  if (idx_vec != 1 && p.K % idx_vec != 0) idx_vec = 1;
  int ok = 0;
  return dispatch_kv(p, idx_vec, cluster, stream, false, &ok);
}

}  // namespace moe
