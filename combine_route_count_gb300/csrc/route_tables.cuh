// Routing of one layer inside one CTA, from topk_idx staged in shared memory:
// the device steps shared by the kernels that route and pack in one launch
// (route_pack for the bf16 payload, route_pack_fp8 for the fp8 one).
//
// "Enabling trillion-parameter models on AWS EFA" (Dispatch and combine):
// count the tokens per expert, take the cumulative sum of the counts, place
// every token at its expert's offset.  Here the counts are per-(expert,
// 32-token word) bitmasks, and the placement is stable (by expert, then by
// token), as in every other routing kernel of this library:
//
//   1. token_masks: one warp per 32-token word; per group of 32 experts each
//      lane (token) sets one bit per chosen expert and a 32x32 bit transpose
//      across the warp leaves in lane x the word's mask of expert x.  The
//      range and duplicate checks of every index ride along;
//   2. expert_scans: per (expert, chunk of 32 words) an exclusive warp scan
//      of the word popcounts and the chunk's total, then one scan of the
//      chunk totals in (expert, chunk) order: the expert offsets and every
//      chunk's first row;
//   3. row_of(t, e) = cpre[e][chunk of t] + pre[e][t/32]
//                     + popc(mask[e][t/32] & lanes below t%32);
//   4. write_routing: slot_row and row_src of the CTA's tokens b, b+G, ...;
//      CTA 0 also the counts, offsets, per-(expert, source rank) and per-rank
//      offsets and the status word.
//
// Every CTA computes the same tables and reaches the same decision on a
// malformed routing.

#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "moe_kernels.cuh"
#include "ptx.cuh"

namespace moe {
namespace rtab {

constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s

__device__ __forceinline__ unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Bounded mbarrier wait: false after kWaitLimitNs without the phase.
__device__ __forceinline__ bool wait_phase(uint64_t* bar, uint32_t parity) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const unsigned long long start = globaltimer();
  while (!ptx::mbar_try_wait(bar, parity)) {
    if (globaltimer() - start > kWaitLimitNs) return false;
  }
  return true;
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
  int NW, NC;      // words of 32 tokens, chunks of 32 words
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

// The tables at `base`; the staged topk_idx follows them at base + tables_bytes.
__device__ __forceinline__ Tables carve_tables(uint8_t* base, int T, int E) {
  Tables tb;
  tb.NW = (T + 31) / 32;
  tb.NC = (tb.NW + 31) / 32;
  tb.mask = reinterpret_cast<uint32_t*>(base);
  tb.pre = reinterpret_cast<int32_t*>(tb.mask + static_cast<size_t>(E) * tb.NW);
  tb.cpre = tb.pre + static_cast<size_t>(E) * tb.NW;
  tb.off = tb.cpre + static_cast<size_t>(E) * tb.NC;
  return tb;
}

// Step 0, after the CTA's prerequisite wait: thread `issuer` (which set up
// idx_bar) bulk-copies the 16-byte-aligned prefix of topk_idx (bulk_ints
// ints) into sidx; CTA 0 resets the status word and the queues; every
// thread loads part of the unaligned tail.  The caller synchronises the CTA
// before anything reads sidx and waits for idx_bar before the prefix.
template <class P>
__device__ __forceinline__ void start_index_copy(const P& p, int32_t* sidx, uint64_t* idx_bar, int bulk_ints,
                                                 int issuer) {
  const int tid = threadIdx.x;
  if (tid == issuer) {
    ptx::mbar_arrive_expect_tx(idx_bar, static_cast<uint32_t>(bulk_ints) * 4u);
    if (bulk_ints > 0) ptx::bulk_g2s(sidx, p.topk_idx, static_cast<uint32_t>(bulk_ints) * 4u, idx_bar);
  }
  if (blockIdx.x == 0 && tid == 0) {
    *p.error_word = MOE_OK;  // routing problems are added later; timeouts with atomicCAS
    if (p.queue) {
      p.queue[0] = 0ull;  // the pack's unit queue
      p.queue[1] = 0ull;  // the combine's token queue
    }
  }
  const int pairs = p.T * p.K;
  for (int i = bulk_ints + tid; i < pairs; i += blockDim.x) sidx[i] = __ldg(p.topk_idx + i);
}

// Step 1: the per-(expert, word) token masks, one warp per word.  Returns
// whether this thread saw a malformed index (out of range or repeated in its
// token); the caller reduces it over the CTA.
template <int KMAX>
__device__ __forceinline__ bool token_masks(const int32_t* sidx, const Tables& tb, int T, int K, int E) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, W = blockDim.x >> 5;
  bool bad = false;
  for (int q = warp; q < tb.NW; q += W) {
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
      if (g0 + lane < E) tb.mask[(g0 + lane) * tb.NW + q] = bits;
    }
  }
  return bad;
}

// Step 2, all threads of the CTA, after the masks are complete (the caller's
// barrier); ends with the CTA synchronised and the tables ready.
__device__ __forceinline__ void expert_scans(const Tables& tb, int E) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, W = blockDim.x >> 5;
  const int NW = tb.NW, NC = tb.NC;
  if (E * NC <= 32 && NW <= 8) {
    // Few experts and words (up to 256 tokens): one warp, lane pc walks the
    // words of its chunk (word prefixes and the chunk total), then one warp
    // scan over the chunk totals in (expert, chunk) order; one CTA barrier
    // instead of two.  Measured on GB300 (A/B, 20-layer graphs): 64-token
    // layer 4.82 -> 4.61 us, its fp8 form 5.64 -> 5.43 us.  With 32 words per
    // chunk the serial walk is slower than the two scans (Mixtral-sized layer
    // 34.15 -> 36.6 us).
    if (warp == 0) {
      const int L = E * NC;
      int total = 0;
      if (lane < L) {
        const int ex = lane / NC;
        const int q0 = (lane - ex * NC) * 32;
        const int q1 = q0 + 32 < NW ? q0 + 32 : NW;
        for (int q = q0; q < q1; ++q) {
          tb.pre[ex * NW + q] = total;
          total += __popc(tb.mask[ex * NW + q]);
        }
      }
      const int incl = warp_incl_scan(total, lane);
      if (lane < L) tb.cpre[lane] = incl - total;
      const int all = __shfl_sync(0xffffffffu, incl, 31);
      __syncwarp();
      for (int ex = lane; ex < E; ex += 32) tb.off[ex] = tb.cpre[ex * NC];
      if (lane == 0) tb.off[E] = all;
    }
    __syncthreads();
    return;
  }
  // Per (expert, chunk of 32 words): exclusive prefix of the word popcounts
  // inside the chunk, and the chunk's total.
  for (int pc = warp; pc < E * NC; pc += W) {
    const int ex = pc / NC;
    const int q = (pc - ex * NC) * 32 + lane;
    const int c = q < NW ? __popc(tb.mask[ex * NW + q]) : 0;
    const int incl = warp_incl_scan(c, lane);
    if (q < NW) tb.pre[ex * NW + q] = incl - c;
    if (lane == 31) tb.cpre[pc] = incl;
  }
  __syncthreads();
  // One exclusive scan over the chunk totals in (expert, chunk) order gives
  // both: cpre[e][c] becomes the first row of expert e's tokens in chunk c,
  // so cpre[e][0] is the expert's offset.  One warp, each lane a run of
  // consecutive totals.
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
}

// Stable row of token t's choice of expert e (t < T).
__device__ __forceinline__ int row_of(const Tables& tb, int t, int e) {
  const int q = t >> 5;
  return tb.cpre[e * tb.NC + (q >> 5)] + tb.pre[e * tb.NW + q] +
         __popc(tb.mask[e * tb.NW + q] & ((1u << (t & 31)) - 1u));
}

// Step 4, all threads of the CTA: slot_row and row_src of tokens b, b+G, ...
// (every slot_row entry -1 after a routing error); CTA 0 writes the counts,
// offsets and status.  `bad` is the CTA-wide decision.
template <class P>
__device__ __forceinline__ void write_routing(const P& p, const Tables& tb, const int32_t* sidx, bool bad) {
  const int T = p.T, K = p.K, E = p.E, N = p.N;
  const int tid = threadIdx.x;
  const int G = gridDim.x;
  const int my_tokens = T > static_cast<int>(blockIdx.x) ? (T - static_cast<int>(blockIdx.x) + G - 1) / G : 0;
  for (int i = tid; i < my_tokens * K; i += blockDim.x) {
    const int t = static_cast<int>(blockIdx.x) + (i / K) * G;
    const int k = i - (i / K) * K;
    const int64_t pair = static_cast<int64_t>(t) * K + k;
    if (bad) {
      p.slot_row[pair] = -1;
    } else {
      const int r = row_of(tb, t, sidx[pair]);
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
        p.src_offsets[i] = row_of(tb, s * Tr, ex);
      }
      // Receive bound of one rank: N * (T/N) * max(K, E/N) rows.
      const int64_t bound = static_cast<int64_t>(N) * Tr * (K > L ? K : L);
      bool over = false;
      for (int r = tid; r < N; r += blockDim.x) over |= (tb.off[(r + 1) * L] - tb.off[r * L]) > bound;
      over = __syncthreads_or(over);
      if (tid == 0 && over) atomicCAS(p.error_word, MOE_OK, MOE_EBOUND);
    }
  }
}

}  // namespace rtab
}  // namespace moe
