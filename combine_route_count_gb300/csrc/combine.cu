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

// Flat mapping: thread g handles CPT 16-byte chunks c0, c0 + C/CPT, ... of
// token t = g / (C/CPT), c0 = g % (C/CPT) (C = H / 8 chunks per row), so a
// warp reads 512 contiguous bytes of each of its K gathered rows per chunk
// step, and a thread keeps CPT*K loads in flight behind one read of the
// token's slot rows.  MIN_BLOCKS sets the register budget: all CPT*K loads
// are live at once (4 registers each).
template <int KMAX, int MIN_BLOCKS, int CPT>
__global__ void __launch_bounds__(kThreads, MIN_BLOCKS) combine_kernel(CombineParams p) {
  ptx::wait_prerequisites();
  const int K = p.K;
  const int64_t CT = (p.H >> 3) / CPT;  // threads per token
  const int64_t g = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
  if (g >= static_cast<int64_t>(p.T) * CT) return;
  const int64_t t = g / CT;
  const int64_t c0 = g - t * CT;
  const int64_t row_bytes = static_cast<int64_t>(p.H) * 2;
  const int32_t* slots = p.slot_row + t * K;

  int bad = 0;
  uint4 v[CPT][KMAX];
#pragma unroll
  for (int k = 0; k < KMAX; ++k) {
    if (k < K) {
      const int r = slots[k];
      const bool out_of_range = kChecked && r >= p.y_rows;
      if (out_of_range) atomicCAS(p.error_word, MOE_OK, MOE_ECORRUPT);
      bad |= r < 0 || out_of_range;
      if (r >= 0 && !out_of_range) {
#pragma unroll
        for (int i = 0; i < CPT; ++i)
          v[i][k] = ptx::ld_stream_v4(p.y + static_cast<int64_t>(r) * row_bytes + (c0 + i * CT) * 16);
      }
    }
  }
  if (bad) return;  // routing error reported by the routing kernel: leave out[t] untouched

  float wk[KMAX];
  const float* wt = p.w + t * K;
#pragma unroll
  for (int k = 0; k < KMAX; ++k)
    if (k < K) wk[k] = __ldg(wt + k);
#pragma unroll
  for (int i = 0; i < CPT; ++i) {
    float a[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) a[j] = 0.0f;
#pragma unroll
    for (int k = 0; k < KMAX; ++k) {
      if (k < K) {
        fma_word(v[i][k].x, wk[k], a[0], a[1]);
        fma_word(v[i][k].y, wk[k], a[2], a[3]);
        fma_word(v[i][k].z, wk[k], a[4], a[5]);
        fma_word(v[i][k].w, wk[k], a[6], a[7]);
      }
    }
    uint4 o;
    o.x = pack_bf16x2(a[0], a[1]);
    o.y = pack_bf16x2(a[2], a[3]);
    o.z = pack_bf16x2(a[4], a[5]);
    o.w = pack_bf16x2(a[6], a[7]);
    ptx::st_v4(p.out + t * row_bytes + (c0 + i * CT) * 16, o);
  }
}

// ---- bulk variant: a producer warp gathers with the TMA engine ---------------
//
// Work unit = (token t, column piece j of the row).  CTA b takes every piece
// of tokens b, b+G, b+2G, ... (or, as an option, a contiguous range of
// units), so the K rows of one token serve its consecutive pieces and the
// next token's slot_row entries are fetched while the current token is in
// flight.  Stage s holds the K gathered row pieces (K * piece bytes):
//   producer (warp 0): waits until stage s is free, lane 0 posts the expected
//     bytes on full[s], lanes k < K each bulk-load row slot_row[t,k]'s piece;
//   consumers (warps 1..): wait on full[s], each thread reads its 16-byte
//     column chunk of the K pieces from shared memory in k order, runs the
//     FMA chain, stores 16 bytes of out[t], and its warp arrives on empty[s].
// All waits are bounded (2 s); a timeout sets MOE_ETIMEDOUT in the error word.

constexpr int kBulkBarBytes = 256;  // full[8] + empty[8] mbarriers + skip flags
constexpr int kMaxBulkStages = 8;
constexpr int kBulkMaxPiece = 4096;                    // 256 consumer threads
constexpr int kBulkMaxThreads = 32 + kBulkMaxPiece / 16;  // producer warp + consumers
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ bool wait_parity(uint64_t* bar, uint32_t parity) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const unsigned long long start = globaltimer_ns();
  while (!ptx::mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - start > kWaitLimitNs) return false;
  }
  return true;
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(ptx::smem_addr(bar)) : "memory");
}

__device__ __forceinline__ uint4 lds128(const void* p) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(ptx::smem_addr(p)));
  return v;
}

// DROP = true only for the failure-injection hook: a separate instance, since
// even this one warp-uniform compare in the producer's per-unit path was
// measured to slow the normal kernel down (DeepSeek-sized layer 168.8 ->
// 170.9 us).  STRIDED picks the tokens of a CTA: false = one contiguous range
// of units; true = tokens b, b+G, b+2G, ... (G CTAs), all pieces of each, so
// that the CTAs work on a window of consecutive tokens at any moment and the
// rows they gather sit close together inside each expert's region.
template <int KMAX, bool DROP, bool STRIDED>
__global__ void __launch_bounds__(kBulkMaxThreads, 2) combine_bulk_kernel(CombineParams p, BulkCombineShape sh) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty = full + kMaxBulkStages;
  int32_t* skip = reinterpret_cast<int32_t*>(empty + kMaxBulkStages);
  uint8_t* stage_buf = smem + kBulkBarBytes;
  const int S = sh.stages, P = sh.pieces, PB = sh.piece_bytes;
  const int K = p.K;
  const int64_t row_bytes = static_cast<int64_t>(p.H) * 2;
  const int64_t stage_bytes = static_cast<int64_t>(K) * PB;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int consumer_warps = (blockDim.x >> 5) - 1;

  // Units of this CTA: a contiguous range starting at u0; or (STRIDED) all
  // pieces of tokens blockIdx.x + m * G for the R = T / G full rounds, then a
  // contiguous share, starting at remainder unit v0, of the (T - R*G) * P units
  // left over, so that no CTA gets a whole token more than another.
  const int64_t G = gridDim.x;
  const int64_t R = p.T / G;
  int64_t u0 = 0, n = 0, strided_units = 0, v0 = 0;
  if constexpr (STRIDED) {
    strided_units = R * P;
    const int64_t rest = (p.T - R * G) * P;
    const int64_t q = rest / G, rem = rest % G;
    v0 = blockIdx.x * q + (blockIdx.x < rem ? blockIdx.x : rem);
    n = strided_units + q + (blockIdx.x < rem ? 1 : 0);
  } else {
    const int64_t units = static_cast<int64_t>(p.T) * P;
    const int64_t q = units / G, rem = units % G;
    u0 = blockIdx.x * q + (blockIdx.x < rem ? blockIdx.x : rem);
    n = q + (blockIdx.x < rem ? 1 : 0);
  }
  // (token, piece) of the CTA's i-th unit.
  auto unit_at = [&](int64_t i, int64_t& t, int& j) {
    if constexpr (STRIDED) {
      if (i < strided_units) {
        const int64_t m = i / P;
        j = static_cast<int>(i - m * P);
        t = blockIdx.x + m * G;
      } else {
        const int64_t v = v0 + (i - strided_units);
        const int64_t tr = v / P;
        j = static_cast<int>(v - tr * P);
        t = R * G + tr;
      }
    } else {
      const int64_t u = u0 + i;
      t = u / P;
      j = static_cast<int>(u - t * P);
    }
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], consumer_warps);
    }
    ptx::mbar_fence_init();
  }
  __syncthreads();
  ptx::wait_prerequisites();  // y and slot_row come from earlier kernels

  auto piece_len = [&](int j) -> uint32_t {
    const int64_t left = row_bytes - static_cast<int64_t>(j) * PB;
    return static_cast<uint32_t>(left < PB ? left : PB);
  };

  if (warp == 0) {
    // ---------------- producer ----------------
    const int hints = sh.hints;
    const uint64_t pol = hints ? ptx::policy_evict_first() : 0;
    int64_t t_cur = -1;
    int row = -1, next_row = -1;
    if (n > 0 && lane < K) {
      int64_t t0;
      int j0;
      unit_at(0, t0, j0);
      next_row = p.slot_row[t0 * K + lane];
    }
    bool ok = true;
    for (int64_t i = 0; i < n; ++i) {
      const int s = static_cast<int>(i % S);
      int64_t t;
      int j;
      unit_at(i, t, j);
      if (t != t_cur) {
        t_cur = t;
        row = next_row;
        // Prefetch the next token's rows while this one is in flight.
        if constexpr (STRIDED) {
          // This CTA's pieces of token t are consecutive from piece j on.
          const int64_t i_next = i + (P - j);
          if (i_next < n) {
            int64_t tn;
            int jn;
            unit_at(i_next, tn, jn);
            if (lane < K) next_row = p.slot_row[tn * K + lane];
          }
        } else {
          const int64_t tn = t + 1;
          if (lane < K && tn * P < u0 + n) next_row = p.slot_row[tn * K + lane];
        }
      }
      if (i >= S) {
        const bool freed = wait_parity(&empty[s], static_cast<uint32_t>(((i / S) - 1) & 1));
        if (!__all_sync(0xffffffffu, freed)) {
          ok = false;
          break;
        }
      }
      // Failure-injection hook (tests only): nothing is posted for this unit,
      // so its consumers' bounded wait runs out and reports MOE_ETIMEDOUT.
      if (DROP && t * P + j == sh.drop_unit) continue;
      const bool out_of_range = kChecked && lane < K && row >= p.y_rows;
      if (out_of_range) atomicCAS(p.error_word, MOE_OK, MOE_ECORRUPT);
      const bool bad = __any_sync(0xffffffffu, lane < K && (row < 0 || out_of_range));
      const uint32_t bytes = piece_len(j);
      if (lane == 0) {
        skip[s] = bad ? 1 : 0;
        if (bad) {
          mbar_arrive(&full[s]);  // nothing to load: release the consumers, who skip the unit
        } else {
          ptx::mbar_arrive_expect_tx(&full[s], static_cast<uint32_t>(K) * bytes);
        }
      }
      __syncwarp();
      if (!bad && lane < K) {
        uint8_t* dst = stage_buf + s * stage_bytes + static_cast<int64_t>(lane) * PB;
        const uint8_t* src = p.y + static_cast<int64_t>(row) * row_bytes + static_cast<int64_t>(j) * PB;
        if (hints & kHintCombineLoads)
          ptx::bulk_g2s_hint(dst, src, bytes, &full[s], pol);
        else
          ptx::bulk_g2s(dst, src, bytes, &full[s]);
      }
    }
    if (!ok && lane == 0) atomicCAS(p.error_word, MOE_OK, MOE_ETIMEDOUT);
  } else {
    // ---------------- consumers ----------------
    const int c = threadIdx.x - 32;  // 16-byte column chunk within the piece
    int64_t t_cur = -1;
    float wk[KMAX];
    for (int64_t i = 0; i < n; ++i) {
      const int s = static_cast<int>(i % S);
      int64_t t;
      int j;
      unit_at(i, t, j);
      if (t != t_cur) {
        t_cur = t;
#pragma unroll
        for (int k = 0; k < KMAX; ++k)
          if (k < K) wk[k] = __ldg(p.w + t * K + k);
      }
      const bool arrived = wait_parity(&full[s], static_cast<uint32_t>((i / S) & 1));
      if (!__all_sync(0xffffffffu, arrived)) {
        if (lane == 0) atomicCAS(p.error_word, MOE_OK, MOE_ETIMEDOUT);
        break;
      }
      const uint32_t bytes = piece_len(j);
      if (!skip[s] && static_cast<uint32_t>(c) * 16 < bytes) {
        const uint8_t* src = stage_buf + s * stage_bytes + static_cast<int64_t>(c) * 16;
        uint4 v[KMAX];
#pragma unroll
        for (int k = 0; k < KMAX; ++k)
          if (k < K) v[k] = lds128(src + static_cast<int64_t>(k) * PB);
        float a[8];
#pragma unroll
        for (int q2 = 0; q2 < 8; ++q2) a[q2] = 0.0f;
#pragma unroll
        for (int k = 0; k < KMAX; ++k) {
          if (k < K) {
            fma_word(v[k].x, wk[k], a[0], a[1]);
            fma_word(v[k].y, wk[k], a[2], a[3]);
            fma_word(v[k].z, wk[k], a[4], a[5]);
            fma_word(v[k].w, wk[k], a[6], a[7]);
          }
        }
        uint4 o;
        o.x = pack_bf16x2(a[0], a[1]);
        o.y = pack_bf16x2(a[2], a[3]);
        o.z = pack_bf16x2(a[4], a[5]);
        o.w = pack_bf16x2(a[6], a[7]);
        ptx::st_v4(p.out + t * row_bytes + static_cast<int64_t>(j) * PB + static_cast<int64_t>(c) * 16, o);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
  }
}

// Token queue.  The static orders give every CTA the same number of units,
// but inside a layer the CTAs do not progress at the same rate (the write-back
// of the previous kernel's dirty lines and DRAM contention fall unevenly), so
// the last CTAs finish well after the median one.  Here CTA b takes token b,
// then claims tokens G, G+1, ... from a counter that the routing kernel sets
// to 0, and copies all P pieces of each claimed token one after another (as
// in the static orders, whose row locality this keeps).  The producer
// publishes each stage's unit (t*P + j) and its K weights in shared memory
// before the stage's full barrier completes, loads the next unit's rows and
// weights while the current one is issued, and keeps two claims in flight.
// Unit -1 ends a CTA's sequence.
constexpr int kBulkQueueHeaderBytes = 1024;  // full[8], empty[8], skip[8], stage_unit[8], stage_w[8][16]

template <int KMAX>
__global__ void __launch_bounds__(kBulkMaxThreads, 2) combine_bulk_queue_kernel(CombineParams p, BulkCombineShape sh) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty = full + kMaxBulkStages;
  int32_t* skip = reinterpret_cast<int32_t*>(empty + kMaxBulkStages);
  int64_t* stage_unit = reinterpret_cast<int64_t*>(skip + kMaxBulkStages);
  float* stage_w = reinterpret_cast<float*>(stage_unit + kMaxBulkStages);  // [kMaxBulkStages][MOE_MAX_TOP_K]
  uint8_t* stage_buf = smem + kBulkQueueHeaderBytes;
  const int S = sh.stages, P = sh.pieces, PB = sh.piece_bytes;
  const int K = p.K;
  const int64_t row_bytes = static_cast<int64_t>(p.H) * 2;
  const int64_t stage_bytes = static_cast<int64_t>(K) * PB;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int consumer_warps = (blockDim.x >> 5) - 1;
  const int64_t G = gridDim.x;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], consumer_warps);
    }
    ptx::mbar_fence_init();
  }
  __syncthreads();
  ptx::wait_prerequisites();  // y and slot_row come from earlier kernels; routing reset the queue

  auto piece_len = [&](int j) -> uint32_t {
    const int64_t left = row_bytes - static_cast<int64_t>(j) * PB;
    return static_cast<uint32_t>(left < PB ? left : PB);
  };

  if (warp == 0) {
    // ---------------- producer ----------------
    const uint64_t pol = sh.hints ? ptx::policy_evict_first() : 0;
    // Lane 0: this CTA's next unit (called in order); -1 = none.  Token b
    // first, then tokens G, G+1, ... claimed whole: all P pieces of a token
    // go to the CTA that claimed it, one after another.
    bool claiming = static_cast<int64_t>(p.T) > G;
    unsigned long long q0 = 0, q1 = 0;
    if (lane == 0 && claiming) {
      q0 = atomicAdd(p.queue, 1ull);
      q1 = atomicAdd(p.queue, 1ull);
    }
    bool first = true;
    int64_t tok = -1;
    int jj = P;
    auto unit_of = [&](int64_t) -> int64_t {
      if (jj >= P) {
        if (first) {
          first = false;
          tok = blockIdx.x < p.T ? static_cast<int64_t>(blockIdx.x) : -1;
        } else if (!claiming) {
          tok = -1;
        } else {
          const int64_t c = G + static_cast<int64_t>(q0);
          if (c >= p.T) {
            claiming = false;
            tok = -1;
          } else {
            tok = c;
            q0 = q1;
            q1 = atomicAdd(p.queue, 1ull);
          }
        }
        jj = 0;
        if (tok < 0) return -1;
      }
      return tok * P + jj++;
    };
    // Rows and weight of unit u for lane k < K.
    auto fetch = [&](int64_t u, int& row, float& wk) {
      row = -1;
      wk = 0.0f;
      if (u >= 0 && lane < K) {
        const int64_t t = u / P;
        row = p.slot_row[t * K + lane];
        wk = __ldg(p.w + t * K + lane);
      }
    };
    int64_t u_cur = 0;
    if (lane == 0) u_cur = unit_of(0);
    u_cur = __shfl_sync(0xffffffffu, u_cur, 0);
    int row, nrow;
    float wk, nw;
    fetch(u_cur, row, wk);
    bool ok = true;
    for (int64_t i = 0;; ++i) {
      const int s = static_cast<int>(i % S);
      int64_t u_nxt = 0;
      if (lane == 0) u_nxt = u_cur >= 0 ? unit_of(i + 1) : -1;
      u_nxt = __shfl_sync(0xffffffffu, u_nxt, 0);
      fetch(u_nxt, nrow, nw);
      if (i >= S) {
        const bool freed = wait_parity(&empty[s], static_cast<uint32_t>(((i / S) - 1) & 1));
        if (!__all_sync(0xffffffffu, freed)) {
          ok = false;
          break;
        }
      }
      if (u_cur < 0) {
        if (lane == 0) {
          stage_unit[s] = -1;
          mbar_arrive(&full[s]);  // the end of this CTA's sequence
        }
        break;
      }
      const int j = static_cast<int>(u_cur % P);
      const bool out_of_range = kChecked && lane < K && row >= p.y_rows;
      if (out_of_range) atomicCAS(p.error_word, MOE_OK, MOE_ECORRUPT);
      const bool bad = __any_sync(0xffffffffu, lane < K && (row < 0 || out_of_range));
      const uint32_t bytes = piece_len(j);
      if (lane < K) stage_w[s * MOE_MAX_TOP_K + lane] = wk;
      if (lane == 0) {
        stage_unit[s] = u_cur;
        skip[s] = bad ? 1 : 0;
      }
      __syncwarp();
      if (lane == 0) {
        if (bad)
          mbar_arrive(&full[s]);  // nothing to load: release the consumers, who skip the unit
        else
          ptx::mbar_arrive_expect_tx(&full[s], static_cast<uint32_t>(K) * bytes);
      }
      __syncwarp();
      if (!bad && lane < K) {
        uint8_t* dst = stage_buf + s * stage_bytes + static_cast<int64_t>(lane) * PB;
        const uint8_t* src = p.y + static_cast<int64_t>(row) * row_bytes + static_cast<int64_t>(j) * PB;
        if (sh.hints & kHintCombineLoads)
          ptx::bulk_g2s_hint(dst, src, bytes, &full[s], pol);
        else
          ptx::bulk_g2s(dst, src, bytes, &full[s]);
      }
      u_cur = u_nxt;
      row = nrow;
      wk = nw;
    }
    if (!ok && lane == 0) atomicCAS(p.error_word, MOE_OK, MOE_ETIMEDOUT);
  } else {
    // ---------------- consumers ----------------
    const int c = threadIdx.x - 32;  // 16-byte column chunk within the piece
    for (int64_t i = 0;; ++i) {
      const int s = static_cast<int>(i % S);
      const bool arrived = wait_parity(&full[s], static_cast<uint32_t>((i / S) & 1));
      if (!__all_sync(0xffffffffu, arrived)) {
        if (lane == 0) atomicCAS(p.error_word, MOE_OK, MOE_ETIMEDOUT);
        break;
      }
      const int64_t u = stage_unit[s];
      if (u < 0) break;
      const int64_t t = u / P;
      const int j = static_cast<int>(u - t * P);
      const uint32_t bytes = piece_len(j);
      if (!skip[s] && static_cast<uint32_t>(c) * 16 < bytes) {
        const uint8_t* src = stage_buf + s * stage_bytes + static_cast<int64_t>(c) * 16;
        uint4 v[KMAX];
#pragma unroll
        for (int k = 0; k < KMAX; ++k)
          if (k < K) v[k] = lds128(src + static_cast<int64_t>(k) * PB);
        float a[8];
#pragma unroll
        for (int q2 = 0; q2 < 8; ++q2) a[q2] = 0.0f;
#pragma unroll
        for (int k = 0; k < KMAX; ++k) {
          if (k < K) {
            const float w = stage_w[s * MOE_MAX_TOP_K + k];
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
        ptx::st_v4(p.out + t * row_bytes + static_cast<int64_t>(j) * PB + static_cast<int64_t>(c) * 16, o);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
  }
}

template <int KMAX>
cudaError_t launch_bulk_k(const CombineParams& p, const CombineLaunch& l, cudaStream_t stream) {
  const BulkCombineShape& sh = l.shape;
  const size_t smem = combine_bulk_smem_bytes(sh, p.K);
  auto* kern = sh.queue && p.queue ? combine_bulk_queue_kernel<KMAX>
               : sh.strided ? (sh.drop_unit >= 0 ? combine_bulk_kernel<KMAX, true, true>
                                                 : combine_bulk_kernel<KMAX, false, true>)
                            : (sh.drop_unit >= 0 ? combine_bulk_kernel<KMAX, true, false>
                                                 : combine_bulk_kernel<KMAX, false, false>);
  cudaError_t err = set_kernel_limits(reinterpret_cast<const void*>(kern), smem);
  if (err != cudaSuccess) return err;
  const int threads = 32 + (sh.piece_bytes / 16 + 31) / 32 * 32;
  return launch_kernel(kern, dim3(l.grid), dim3(threads), smem, stream, l.pdl, p, sh);
}

template <int KMAX>
cudaError_t launch_k(const CombineParams& p, bool pdl, int sms, cudaStream_t stream) {
  constexpr int MIN_BLOCKS = KMAX >= 16 ? 2 : (KMAX >= 8 ? 3 : 4);
  // K <= 2: four chunks per thread when the row splits evenly (more loads in
  // flight per thread; measured on GB300: Mixtral-sized layer 34.82 -> 34.19
  // us), unless that leaves SMs without a CTA: a small layer keeps one chunk
  // per thread and more CTAs (64-token layer in 20-layer graphs: 4.61 ->
  // 4.21 us, its fp8 form 5.53 -> 5.13 us).
  const long long chunks = static_cast<long long>(p.T) * (p.H >> 3);
  const int cpt = KMAX <= 2 && (p.H >> 3) % 4 == 0 && chunks / 4 >= static_cast<long long>(sms) * kThreads ? 4 : 1;
  const long long threads = static_cast<long long>(p.T) * ((p.H >> 3) / cpt);
  const long long grid = (threads + kThreads - 1) / kThreads;
  if (grid == 0) return cudaSuccess;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidValue;
  if constexpr (KMAX <= 2) {
    if (cpt == 4)
      return launch_kernel(combine_kernel<KMAX, MIN_BLOCKS, 4>, dim3(static_cast<unsigned>(grid)), dim3(kThreads), 0,
                           stream, pdl, p);
  }
  return launch_kernel(combine_kernel<KMAX, MIN_BLOCKS, 1>, dim3(static_cast<unsigned>(grid)), dim3(kThreads), 0,
                       stream, pdl, p);
}

}  // namespace

size_t combine_bulk_smem_bytes(const BulkCombineShape& sh, int K) {
  return (sh.queue ? kBulkQueueHeaderBytes : kBulkBarBytes) + static_cast<size_t>(sh.stages) * K * sh.piece_bytes;
}

BulkCombineShape combine_bulk_shape(int H, int K, int stages, int piece_bytes, int max_smem, int auto_piece_max) {
  BulkCombineShape sh;
  sh.hints = 0;
  sh.drop_unit = -1;
  sh.strided = 0;
  const int64_t row_bytes = static_cast<int64_t>(H) * 2;
  if (piece_bytes <= 0) {
    // Pieces of at most auto_piece_max bytes (one consumer thread per 16
    // bytes), equal up to 16 bytes.
    const int64_t pieces = (row_bytes + auto_piece_max - 1) / auto_piece_max;
    piece_bytes = static_cast<int>((row_bytes / 16 + pieces - 1) / pieces * 16);
  }
  if (piece_bytes > kBulkMaxPiece) piece_bytes = kBulkMaxPiece;
  if (piece_bytes > row_bytes) piece_bytes = static_cast<int>(row_bytes);
  sh.piece_bytes = piece_bytes;
  sh.pieces = static_cast<int>((row_bytes + piece_bytes - 1) / piece_bytes);
  if (stages <= 0) {
    // About 100 KiB of stages per CTA: two CTAs per SM.
    stages = static_cast<int>((100 * 1024) / (static_cast<int64_t>(K) * piece_bytes));
  }
  if (stages < 2) stages = 2;
  if (stages > kMaxBulkStages) stages = kMaxBulkStages;
  while (stages > 2 && combine_bulk_smem_bytes(BulkCombineShape{stages, sh.piece_bytes, sh.pieces, 0, -1, 0}, K) >
                           static_cast<size_t>(max_smem))
    --stages;
  sh.stages = stages;
  return sh;
}

cudaError_t launch_combine(const CombineParams& p, const CombineLaunch& l, cudaStream_t stream) {
  if (l.variant == kCombineBulk) {
    if (p.K <= 2) return launch_bulk_k<2>(p, l, stream);
    if (p.K <= 4) return launch_bulk_k<4>(p, l, stream);
    if (p.K <= 8) return launch_bulk_k<8>(p, l, stream);
    return launch_bulk_k<16>(p, l, stream);
  }
  if (p.K <= 2) return launch_k<2>(p, l.pdl, l.sms, stream);
  if (p.K <= 4) return launch_k<4>(p, l.pdl, l.sms, stream);
  if (p.K <= 8) return launch_k<8>(p, l.pdl, l.sms, stream);
  return launch_k<16>(p, l.pdl, l.sms, stream);
}

}  // namespace moe
