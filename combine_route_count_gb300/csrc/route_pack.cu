// route_pack: the routing and the pack of dispatch in one kernel, for small
// layers.
//
// "Enabling trillion-parameter models on AWS EFA" (Dispatch and combine)
// counts the tokens per expert, takes the cumulative sum of the counts and
// then packs every token at its offset.  As two kernels (route_cluster, then
// dispatch_pack) the pack cannot start copying before the routing grid has
// finished and its writes are visible, so every layer pays the routing
// kernel's launch, its dependent steps and the grid boundary in series.  For
// a small layer that is most of the layer: a Mixtral-sized layer (4096
// tokens, 8 experts, top-2) spends ~3 us of 36 there, a 64-token layer half
// of its time.
//
// Here one CTA per SM computes the whole routing itself from topk_idx (which
// is small for these layers) while its first token rows are already in
// flight, then its first P warps copy units, each warp with its own ring of
// shared-memory stages (P "virtual" pack CTAs per SM, as the two-kernel path
// runs P pack CTAs per SM; one routing per SM instead of P):
//
//   0. one bulk copy (TMA) brings all of topk_idx into shared memory; it is
//      issued before the token rows so that it does not queue behind them;
//   1. per 32-token word q and expert e, a bitmask of the tokens of q that
//      chose e, one warp per word: per group of 32 experts, each lane (token)
//      sets one bit per chosen expert and a 32x32 bit transpose across the
//      warp (five shuffle stages) hands lane x the mask of expert x: no
//      atomics, no per-expert loop.  The range and duplicate check of every
//      index rides along;
//   2. per (expert, chunk of 32 words), side by side: an exclusive
//      warp-shuffle scan of the word popcounts, and the chunk's total;
//   3. one exclusive scan of the chunk totals in (expert, chunk) order:
//      the expert offsets and every chunk's first row at once;
//   4. the stable row of (t, k) with e = idx[t, k] is
//        cpre[e][chunk of t] + pre[e][t/32] + popc(mask[e][t/32] & lanes below t%32),
//      the same placement as route_count and route_cluster (by expert, then
//      by token); the CTA writes slot_row and row_src of tokens b, b+G, ...;
//      CTA 0 writes counts, offsets, per-(expert, source rank) and per-rank
//      offsets and the status word;
//   5. warps w < P run the bulk pack's static copy loop as virtual CTA
//      v = b*P + w of G*P (units v, v+GP, ...), taking destination rows from
//      the tables in shared memory; or, when a copy warp has at most two
//      small whole rows (VEC), it loads them into registers right after the
//      dependency wait and stores them once the tables are built.
//
// The redundant routing costs each CTA a T*K*4-byte copy from L2 and
// ~T*K/32 warp instructions; the host picks this kernel only when that is
// small (see route_pack_eligible).  Reading the indices from shared memory
// matters: with per-lane global loads the compiler may issue each word's
// loads just before their use, and a Mixtral-sized layer spent ~15 us of
// serialised round trips (queued behind the token rows) in step 1.  Every
// CTA reaches the same verdict on a malformed routing, so after a routing
// error no CTA copies anything and every slot_row entry becomes -1 (the
// combine then writes nothing).

#include <cuda_runtime.h>

#include "moe_kernels.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kMaxStages = 16;
constexpr int kBarBytes = 512;  // mbarriers: copy warps' stages (<= 63), then the index copy's
constexpr int kIdxBar = kBarBytes / 8 - 1;
constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s

__device__ __forceinline__ unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ bool wait_phase(uint64_t* bar, uint32_t parity) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const unsigned long long start = globaltimer();
  while (!ptx::mbar_try_wait(bar, parity)) {
    if (globaltimer() - start > kWaitLimitNs) return false;
  }
  return true;
}

__device__ __forceinline__ void wait_reads_at_most(int depth) {
  switch (depth) {
    case 0: ptx::bulk_wait_read<0>(); break;
    case 1: ptx::bulk_wait_read<1>(); break;
    case 2: ptx::bulk_wait_read<2>(); break;
    case 3: ptx::bulk_wait_read<3>(); break;
    case 4: ptx::bulk_wait_read<4>(); break;
    case 5: ptx::bulk_wait_read<5>(); break;
    case 6: ptx::bulk_wait_read<6>(); break;
    default: ptx::bulk_wait_read<7>(); break;
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

// 32x32 bit-matrix transpose across a warp: bit j of the result in lane i
// is bit i of the argument in lane j.  Five butterfly stages; stage s swaps,
// between lanes i and i^s, the bits j whose bit s differs from bit s of i.
__device__ __forceinline__ uint32_t warp_transpose32(uint32_t x, int lane) {
  constexpr uint32_t lo[5] = {0x0000ffffu, 0x00ff00ffu, 0x0f0f0f0fu, 0x33333333u, 0x55555555u};
#pragma unroll
  for (int i = 0; i < 5; ++i) {
    const int sh = 16 >> i;
    const uint32_t y = __shfl_xor_sync(0xffffffffu, x, sh);
    x = (lane & sh) ? ((x & ~lo[i]) | ((y & ~lo[i]) >> sh)) : ((x & lo[i]) | ((y & lo[i]) << sh));
  }
  return x;
}

// Words are scanned in chunks of 32 (one warp scan each): the first row of
// word q's tokens of expert e is cpre[e][q/32] (the expert's offset plus its
// rows in earlier chunks) + pre[e][q] (earlier words of its chunk).
struct Tables {
  uint32_t* mask;  // [E*NW] tokens of word q that chose expert e, at e*NW+q
  int32_t* pre;    // [E*NW] #{t in [32*32*(q/32), 32q) : e in idx[t]}
  int32_t* cpre;   // [E*NC] first row of expert e's tokens in chunk c, at e*NC+c
  int32_t* off;    // [E+1] expert offsets
};

__host__ __device__ inline size_t tables_bytes(int T, int E) {
  const size_t NW = (static_cast<size_t>(T) + 31) / 32;
  const size_t NC = (NW + 31) / 32;
  const size_t b =
      sizeof(int32_t) * (2 * static_cast<size_t>(E) * NW + static_cast<size_t>(E) * NC + static_cast<size_t>(E) + 1);
  return (b + 15) / 16 * 16;  // the index copy that follows starts 16-byte aligned
}

__host__ __device__ inline size_t index_bytes(int T, int K) {
  return (static_cast<size_t>(T) * K * sizeof(int32_t) + 15) / 16 * 16;
}

// VEC (small rows, at most kVecUnits units of at most kVecChunks*512 bytes
// per copy warp): the copy warps hold their rows in registers, loaded with
// 16-byte loads while the tables are built, and store them with 16-byte
// stores; no stages, no mbarriers, nothing to wait for before exiting.
constexpr int kVecUnits = 2;
constexpr int kVecChunks = 2;

template <int KMAX, bool VEC>
__global__ void __launch_bounds__(kRoutePackThreads, 1)
    route_pack_kernel(RoutePackParams p, int copy_warps, int stages, int hints, int depth) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int T = p.T, K = p.K, E = p.E, N = p.N;
  const int NW = (T + 31) / 32;
  const int NC = (NW + 31) / 32;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, W = blockDim.x >> 5;
  const bool copier = warp < copy_warps;
  // This warp's stage ring and mbarriers (copy warps only).
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem) + (copier ? warp * stages : 0);
  uint8_t* stage_buf = smem + kBarBytes + (copier ? static_cast<size_t>(warp) * stages * p.piece_bytes : 0);
  Tables tb;
  tb.mask = reinterpret_cast<uint32_t*>(smem + kBarBytes + static_cast<size_t>(copy_warps) * stages * p.piece_bytes);
  tb.pre = reinterpret_cast<int32_t*>(tb.mask + static_cast<size_t>(E) * NW);
  tb.cpre = tb.pre + static_cast<size_t>(E) * NW;
  tb.off = tb.cpre + static_cast<size_t>(E) * NC;
  // topk_idx, copied whole: the choices of token t at sidx[t*K .. t*K+K).
  int32_t* sidx = reinterpret_cast<int32_t*>(reinterpret_cast<uint8_t*>(tb.mask) + tables_bytes(T, E));
  uint64_t* idx_bar = reinterpret_cast<uint64_t*>(smem) + kIdxBar;
  const int pairs = T * K;
  const int bulk_ints = (reinterpret_cast<uintptr_t>(p.topk_idx) & 15) == 0 ? (pairs & ~3) : 0;
  const int64_t units = static_cast<int64_t>(T) * p.pieces;
  const int64_t first = static_cast<int64_t>(blockIdx.x) * copy_warps + warp;  // virtual CTA
  const int64_t step = static_cast<int64_t>(gridDim.x) * copy_warps;
  const int64_t mine = copier && units > first ? (units - first + step - 1) / step : 0;

  if (!VEC && copier && lane == 0) {
    for (int s = 0; s < stages; ++s) ptx::mbar_init(&bars[s], 1);
    ptx::mbar_fence_init();
  }
  if (tid == 32 * (W - 1)) {
    ptx::mbar_init(idx_bar, 1);
    ptx::mbar_fence_init();
  }
  // The indices and the token rows may come from the previous kernel, and the
  // previous combine still reads the routing tables: wait for it.
  ptx::wait_prerequisites();
  // Routing only (no copy warps, one CTA): the pack kernel that follows may
  // start now and fetch its first token rows while the tables are built.
  if (copy_warps == 0) ptx::launch_dependents();
  // 0. the indices: one bulk copy of their 16-byte-aligned prefix, issued by
  // the thread that set up its barrier before any token row is requested (so
  // that it does not queue behind the rows), plain loads for the rest.
  if (tid == 32 * (W - 1)) {
    ptx::mbar_arrive_expect_tx(idx_bar, static_cast<uint32_t>(bulk_ints) * 4u);
    if (bulk_ints > 0) ptx::bulk_g2s(sidx, p.topk_idx, static_cast<uint32_t>(bulk_ints) * 4u, idx_bar);
  }
  if (blockIdx.x == 0 && tid == 0) {
    *p.error_word = MOE_OK;  // routing problems are added below; timeouts with atomicCAS
    if (p.queue) {
      p.queue[0] = 0ull;  // the pack's unit queue (unused here)
      p.queue[1] = 0ull;  // the combine's token queue
    }
  }
  for (int i = bulk_ints + tid; i < pairs; i += blockDim.x) sidx[i] = __ldg(p.topk_idx + i);
  __syncthreads();

  auto piece_bytes = [&](int j) -> uint32_t {
    const int64_t left = p.row_bytes - static_cast<int64_t>(j) * p.piece_bytes;
    return static_cast<uint32_t>(left < p.piece_bytes ? left : p.piece_bytes);
  };
  const uint64_t pol = hints ? ptx::policy_evict_first() : 0;
  auto issue_load = [&](int64_t i) {
    const int64_t u = first + i * step;
    const int64_t t = u / p.pieces;
    const int j = static_cast<int>(u - t * p.pieces);
    const uint32_t bytes = piece_bytes(j);
    const int s = static_cast<int>(i % stages);
    ptx::mbar_arrive_expect_tx(&bars[s], bytes);
    if (hints & kHintPackLoads)
      ptx::bulk_g2s_hint(stage_buf + static_cast<size_t>(s) * p.piece_bytes,
                         p.x + t * p.row_bytes + static_cast<int64_t>(j) * p.piece_bytes, bytes, &bars[s], pol);
    else
      ptx::bulk_g2s(stage_buf + static_cast<size_t>(s) * p.piece_bytes,
                    p.x + t * p.row_bytes + static_cast<int64_t>(j) * p.piece_bytes, bytes, &bars[s]);
  };
  // Each copy warp's first token rows travel while the tables are built;
  // its later rows go to L2.  (VEC: all its rows, into registers.)
  const int64_t prologue = VEC ? 0 : (mine < stages ? mine : stages);
  const int64_t row_chunks = p.row_bytes >> 4;
  uint4 vrow[VEC ? kVecUnits : 1][VEC ? kVecChunks : 1];
  if (VEC && copier) {
#pragma unroll
    for (int u = 0; u < (VEC ? kVecUnits : 1); ++u) {
      if (u < mine) {
        const int64_t t = first + u * step;  // whole rows: unit = token
#pragma unroll
        for (int c = 0; c < (VEC ? kVecChunks : 1); ++c) {
          const int64_t ch = static_cast<int64_t>(c) * 32 + lane;
          if (ch < row_chunks) vrow[u][c] = ptx::ld_stream_v4(p.x + t * p.row_bytes + ch * 16);
        }
      }
    }
  }
  if (!VEC && copier) {
    if (lane == 0)
      for (int64_t i = 0; i < prologue; ++i) issue_load(i);
    for (int64_t i = prologue + lane; i < mine; i += 32) {
      const int64_t u = first + i * step;
      const int64_t t = u / p.pieces;
      const int j = static_cast<int>(u - t * p.pieces);
      ptx::bulk_prefetch_l2(p.x + t * p.row_bytes + static_cast<int64_t>(j) * p.piece_bytes, piece_bytes(j));
    }
  }

  const bool idx_ok = __syncthreads_and(wait_phase(idx_bar, 0));
  if (!idx_ok) {
    // The index copy did not complete in time: report it, wait (bounded)
    // for it and for the row loads issued so far, copy nothing.
    if (tid == 0) atomicCAS(p.error_word, MOE_OK, MOE_ETIMEDOUT);
    if (tid == 32 * (W - 1)) wait_phase(idx_bar, 0);
    if (copier && lane == 0)
      for (int64_t i = 0; i < prologue; ++i) wait_phase(&bars[i % stages], static_cast<uint32_t>((i / stages) & 1));
    return;
  }

  // 1. per-(expert, word) token masks; index checks.
  bool bad = false;
  for (int q = warp; q < NW; q += W) {
    const int t = q * 32 + lane;
    int e[KMAX];
#pragma unroll
    for (int k = 0; k < KMAX; ++k) e[k] = (k < K && t < T) ? sidx[t * K + k] : -1;
    if (t < T) {
#pragma unroll
      for (int k = 0; k < KMAX; ++k) {
        if (k < K) {
          if (static_cast<unsigned>(e[k]) >= static_cast<unsigned>(E)) {
            bad = true;
            e[k] = -1;
          } else {
#pragma unroll
            for (int j = 0; j < k; ++j) bad |= (e[j] == e[k]);
          }
        }
      }
    }
    // Per group of 32 experts: lane t sets bit x for each expert 32g+x it
    // chose; transposing that 32x32 bit matrix across the warp leaves in lane
    // x the word's mask of expert 32g+x.
    for (int g0 = 0; g0 < E; g0 += 32) {
      uint32_t bits = 0u;
#pragma unroll
      for (int k = 0; k < KMAX; ++k)
        if (k < K && e[k] >= g0 && e[k] < g0 + 32) bits |= 1u << (e[k] - g0);
      bits = warp_transpose32(bits, lane);
      if (g0 + lane < E) tb.mask[(g0 + lane) * NW + q] = bits;
    }
  }
  bad = __syncthreads_or(bad);

  // 2. per (expert, chunk of 32 words): exclusive prefix of the word
  // popcounts inside the chunk, and the chunk's total.
  for (int pc = warp; pc < E * NC; pc += W) {
    const int ex = pc / NC;
    const int q = (pc - ex * NC) * 32 + lane;
    const int c = q < NW ? __popc(tb.mask[ex * NW + q]) : 0;
    const int incl = warp_incl_scan(c, lane);
    if (q < NW) tb.pre[ex * NW + q] = incl - c;
    if (lane == 31) tb.cpre[pc] = incl;
  }
  __syncthreads();
  // 3. one exclusive scan over the chunk totals in (expert, chunk) order
  // gives both: cpre[e][c] becomes the first row of expert e's tokens in
  // chunk c, so cpre[e][0] is the expert's offset.  One warp, each lane a
  // run of consecutive totals.
  if (warp == 0) {
    const int L = E * NC;
    const int m = (L + 31) / 32;
    const int lo = min(L, lane * m), hi = min(L, lo + m);
    int sum = 0;
    for (int i = lo; i < hi; ++i) sum += tb.cpre[i];
    const int incl = warp_incl_scan(sum, lane);
    int run = incl - sum;
    for (int i = lo; i < hi; ++i) {
      const int v = tb.cpre[i];
      tb.cpre[i] = run;
      run += v;
    }
    const int total = __shfl_sync(0xffffffffu, incl, 31);
    __syncwarp();
    for (int ex = lane; ex < E; ex += 32) tb.off[ex] = tb.cpre[ex * NC];
    if (lane == 0) tb.off[E] = total;
  }
  __syncthreads();

  // Stable row of token t's choice of expert e (t < T).
  auto row_of = [&](int t, int e) -> int {
    const int q = t >> 5;
    return tb.cpre[e * NC + (q >> 5)] + tb.pre[e * NW + q] + __popc(tb.mask[e * NW + q] & ((1u << (t & 31)) - 1u));
  };

  // 4. this CTA's tokens b, b+G, ...: slot_row and row_src.
  const int G = gridDim.x;
  const int my_tokens = T > static_cast<int>(blockIdx.x) ? (T - static_cast<int>(blockIdx.x) + G - 1) / G : 0;
  for (int i = tid; i < my_tokens * K; i += blockDim.x) {
    const int t = static_cast<int>(blockIdx.x) + (i / K) * G;
    const int k = i - (i / K) * K;
    const int64_t pair = static_cast<int64_t>(t) * K + k;
    if (bad) {
      p.slot_row[pair] = -1;
    } else {
      const int r = row_of(t, sidx[pair]);
      p.slot_row[pair] = r;
      p.row_src[r] = static_cast<int32_t>(pair);
    }
  }
  if (blockIdx.x == 0) {
    if (bad) {
      for (int i = tid; i < E; i += blockDim.x) p.expert_counts[i] = 0;
      for (int i = tid; i <= E; i += blockDim.x) p.expert_offsets[i] = 0;
      for (int i = tid; i <= N; i += blockDim.x) p.rank_offsets[i] = 0;
      for (int i = tid; i < E * N; i += blockDim.x) p.src_offsets[i] = 0;
      if (tid == 0) atomicExch(p.error_word, MOE_EROUTE);
    } else {
      const int Tr = T / N, L = E / N;
      for (int i = tid; i < E; i += blockDim.x) p.expert_counts[i] = tb.off[i + 1] - tb.off[i];
      for (int i = tid; i <= E; i += blockDim.x) p.expert_offsets[i] = tb.off[i];
      for (int r = tid; r <= N; r += blockDim.x) p.rank_offsets[r] = r < N ? tb.off[r * L] : tb.off[E];
      // First row of (expert e, source rank s): the rows of e that tokens
      // before s*T/N took.
      for (int i = tid; i < E * N; i += blockDim.x) {
        const int ex = i / N, s = i - (i / N) * N;
        p.src_offsets[i] = row_of(s * Tr, ex);
      }
      // Receive bound of one rank: N * (T/N) * max(K, E/N) rows.
      const int64_t bound = static_cast<int64_t>(N) * Tr * (K > L ? K : L);
      bool over = false;
      for (int r = tid; r < N; r += blockDim.x) over |= (tb.off[(r + 1) * L] - tb.off[r * L]) > bound;
      over = __syncthreads_or(over);
      if (tid == 0 && over) atomicCAS(p.error_word, MOE_OK, MOE_EBOUND);
    }
  }
  if (!copier) return;

  if (bad) {
    // Nothing is copied; the prologue's loads are waited for (bounded)
    // before shared memory goes away.
    if (lane == 0)
      for (int64_t i = 0; i < prologue; ++i) wait_phase(&bars[i % stages], static_cast<uint32_t>((i / stages) & 1));
    __syncwarp();
    return;
  }

  if (VEC) {
#pragma unroll
    for (int u = 0; u < (VEC ? kVecUnits : 1); ++u) {
      if (u < mine) {
        const int t = static_cast<int>(first + u * step);
        const int my_row = lane < K ? row_of(t, sidx[t * K + lane]) : -1;
        for (int k = 0; k < K; ++k) {
          const int row = __shfl_sync(0xffffffffu, my_row, k);
          if (kChecked && row >= p.dst_rows) {
            if (lane == 0) atomicCAS(p.error_word, MOE_OK, MOE_ECORRUPT);
            continue;
          }
          uint8_t* dst = p.expert_x + static_cast<int64_t>(row) * p.row_bytes;
#pragma unroll
          for (int c = 0; c < (VEC ? kVecChunks : 1); ++c) {
            const int64_t ch = static_cast<int64_t>(c) * 32 + lane;
            if (ch < row_chunks) ptx::st_v4(dst + ch * 16, vrow[u][c]);
          }
        }
      }
    }
    return;
  }

  // 5. the static bulk copy loop of this virtual CTA; destination rows one
  // unit ahead.
  auto dest_row = [&](int64_t unit_index) -> int {
    const int tt = static_cast<int>((first + unit_index * step) / p.pieces);
    return lane < K ? row_of(tt, sidx[tt * K + lane]) : -1;
  };
  int64_t i = 0;
  bool ok = true;
  int next_row = mine > 0 ? dest_row(0) : -1;
  for (; i < mine; ++i) {
    const int64_t u = first + i * step;
    const int64_t t = u / p.pieces;
    const int j = static_cast<int>(u - t * p.pieces);
    const int s = static_cast<int>(i % stages);
    const int row = next_row;
    if (i + 1 < mine) next_row = dest_row(i + 1);
    const bool arrived = wait_phase(&bars[s], static_cast<uint32_t>((i / stages) & 1));
    if (!__all_sync(0xffffffffu, arrived)) {
      ok = false;
      break;
    }
    int row_ok = row;
    if (kChecked && row >= 0 && row >= p.dst_rows) {
      atomicCAS(p.error_word, MOE_OK, MOE_ECORRUPT);
      row_ok = -1;
    }
    if (row_ok >= 0) {
      uint8_t* dst = p.expert_x + static_cast<int64_t>(row) * p.row_bytes + static_cast<int64_t>(j) * p.piece_bytes;
      const uint8_t* src = stage_buf + static_cast<size_t>(s) * p.piece_bytes;
      if (hints & kHintPackStores)
        ptx::bulk_s2g_hint(dst, src, piece_bytes(j), pol);
      else
        ptx::bulk_s2g(dst, src, piece_bytes(j));
    }
    ptx::bulk_commit();
    const int64_t r = i - depth + 1;
    if (r >= 0 && r + stages < mine) {
      wait_reads_at_most(depth - 1);
      __syncwarp();
      if (lane == 0) issue_load(r + stages);
    }
  }
  if (!ok) {
    if (lane == 0) {
      atomicCAS(p.error_word, MOE_OK, MOE_ETIMEDOUT);
      int64_t last = prologue - 1;
      if (i - depth + stages > last) last = i - depth + stages;
      if (last > mine - 1) last = mine - 1;
      for (int64_t q = i; q <= last; ++q) wait_phase(&bars[q % stages], static_cast<uint32_t>((q / stages) & 1));
    }
    __syncwarp();
  }
  ptx::bulk_wait<0>();
}

int clamp_depth(int depth, int stages) {
  if (depth < 1) depth = 1;
  if (depth > 8) depth = 8;
  if (depth > stages - 1) depth = stages - 1;
  return depth < 1 ? 1 : depth;
}

}  // namespace

size_t route_pack_tables_bytes(int T, int E) { return tables_bytes(T, E); }

size_t route_pack_smem_bytes(int T, int K, int E, int copy_warps, int stages, int piece_bytes) {
  return kBarBytes + static_cast<size_t>(copy_warps) * stages * piece_bytes + tables_bytes(T, E) + index_bytes(T, K);
}

bool route_pack_eligible(int T, int K, int E) {
  if (T <= 0) return false;
  const int64_t words = (static_cast<int64_t>(T) + 31) / 32 * E;
  return static_cast<int64_t>(T) * K <= kRoutePackMaxPairs && words <= kRoutePackMaxMaskWords;
}

int route_pack_max_stages(int copy_warps) {
  const int n = kIdxBar / (copy_warps < 1 ? 1 : copy_warps);
  return n < kMaxStages ? n : kMaxStages;
}

cudaError_t prepare_route_pack(int max_smem_bytes) {
  const void* kernels[] = {reinterpret_cast<const void*>(route_pack_kernel<2, false>),
                           reinterpret_cast<const void*>(route_pack_kernel<4, false>),
                           reinterpret_cast<const void*>(route_pack_kernel<8, false>),
                           reinterpret_cast<const void*>(route_pack_kernel<16, false>),
                           reinterpret_cast<const void*>(route_pack_kernel<2, true>),
                           reinterpret_cast<const void*>(route_pack_kernel<4, true>),
                           reinterpret_cast<const void*>(route_pack_kernel<8, true>)};
  for (const void* k : kernels) {
    const cudaError_t err = set_kernel_limits(k, static_cast<size_t>(max_smem_bytes));
    if (err != cudaSuccess) return err;
  }
  return cudaSuccess;
}

bool route_pack_vec_ok(int64_t row_bytes, int64_t units_per_warp) {
  return row_bytes <= kVecChunks * 512 && units_per_warp <= kVecUnits;
}

cudaError_t launch_route_pack(const RoutePackParams& p, const RoutePackLaunch& l, cudaStream_t stream) {
  const bool vec = l.vec && p.K <= 8;  // K > 8 keeps its rows in stages (registers would spill)
  const int maxst = route_pack_max_stages(l.copy_warps);
  const int stages = vec ? 0 : (l.stages < 2 ? 2 : (l.stages > maxst ? maxst : l.stages));
  const size_t smem = route_pack_smem_bytes(p.T, p.K, p.E, l.copy_warps, stages, p.piece_bytes);
  const int depth = vec ? 1 : clamp_depth(l.depth, stages);
  const int threads = l.threads >= 32 * (l.copy_warps > 1 ? l.copy_warps : 1) && l.threads <= kRoutePackThreads
                          ? l.threads / 32 * 32
                          : kRoutePackThreads;
  const dim3 grid(l.grid), block(threads);
#define MOE_RP_LAUNCH(KM)                                                                                      \
  return vec ? launch_kernel(route_pack_kernel<KM, true>, grid, block, smem, stream, l.pdl, p, l.copy_warps, \
                               stages, l.hints, depth)                                                         \
               : launch_kernel(route_pack_kernel<KM, false>, grid, block, smem, stream, l.pdl, p, l.copy_warps, \
                               stages, l.hints, depth)
  if (p.K <= 2) MOE_RP_LAUNCH(2);
  if (p.K <= 4) MOE_RP_LAUNCH(4);
  if (p.K <= 8) MOE_RP_LAUNCH(8);
#undef MOE_RP_LAUNCH
  return launch_kernel(route_pack_kernel<16, false>, grid, block, smem, stream, l.pdl, p, l.copy_warps, stages,
                       l.hints, depth);
}

}  // namespace moe
