// dispatch_pack_fp8: the dispatch payload as block-scaled fp8.
//
// "Efficient and portable mixture-of-experts communication" (Dispatch): the
// dispatch kernel sends tokens together with their block scaling factors;
// "Enabling trillion-parameter models on AWS EFA" (evaluation): block-scale
// fp8 dispatch, bf16 combine.  Each token row is quantised once and written
// to its K destination rows (block scales of 128 elements, fp8_quant.cuh):
//   expert_xq[slot_row[t,k]] = q[t], expert_scales[slot_row[t,k]] = scales[t].
//
// CTA = 1 producer warp + 4 consumer warps; unit = one token row; each CTA
// takes a contiguous range of tokens.  The producer bulk-loads rows into
// shared-memory stages (the first ones before griddepcontrol.wait: rows do
// not depend on routing); the 128 consumer threads quantise each row
// together.  Waits are bounded (2 s) and report MOE_ETIMEDOUT.

#include <cuda_runtime.h>

#include "moe_kernels.cuh"
#include "fp8_quant.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kConsumers = fp8q::kRowThreads;
constexpr int kMaxFp8Stages = 8;
constexpr int kFp8BarBytes = 256;
// Queue variant: mbarriers, stage_tok[8] and stage_rows[8][16] before the stages.
constexpr int kFp8QueueHeaderBytes = 1024;
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ unsigned long long now_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ bool wait_parity(uint64_t* bar, uint32_t parity) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const unsigned long long start = now_ns();
  while (!ptx::mbar_try_wait(bar, parity)) {
    if (now_ns() - start > kWaitLimitNs) return false;
  }
  return true;
}

__device__ __forceinline__ void arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(ptx::smem_addr(bar)) : "memory");
}

// STRIDED: CTA b takes tokens b, b+G, b+2G, ... (G CTAs), so that the CTAs
// work on a window of consecutive tokens and their destination rows lie close
// together in each expert's region; otherwise one contiguous token range.
template <int KMAX, bool STRIDED>
__global__ void __launch_bounds__(32 + kConsumers, KMAX <= 4 ? 8 : 1) dispatch_pack_fp8_kernel(PackFp8Params p, int stages) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty = full + kMaxFp8Stages;
  uint8_t* stage_buf = smem + kFp8BarBytes;
  const int K = p.K, H = p.H;
  const int64_t row_bytes = static_cast<int64_t>(H) * 2;
  const int nblk = H / 128;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const int64_t q = p.T / gridDim.x, rem = p.T % gridDim.x;
  const int64_t t0 = STRIDED ? static_cast<int64_t>(blockIdx.x) : blockIdx.x * q + (blockIdx.x < rem ? blockIdx.x : rem);
  const int64_t n = q + (blockIdx.x < rem ? 1 : 0);
  // token step between a CTA's consecutive tokens
  const int dt = STRIDED ? static_cast<int>(gridDim.x) : 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], kConsumers / 32);
    }
    ptx::mbar_fence_init();
  }
  __syncthreads();

  if (warp == 0) {
    // ---------------- producer ----------------
    // The CTA's rows past its first `stages` go to L2 now, while routing
    // runs, so that their loads after the routing hit L2; with the evict-last
    // policy, so that the stream of code rows written meanwhile does not push
    // them out first (each row returns to normal priority once quantised).
    // Measured on GB300 (A/B in one call, twice): DeepSeek-sized fp8 layer
    // 137.8 -> 137.1 us with a plain prefetch, 137.6 -> 132.6 us with
    // evict-last; Kimi-sized (token queue, no prefetch) unchanged.
    {
      const uint64_t last = ptx::policy_evict_last();
      for (int64_t i = stages + lane; i < n; i += 32)
        ptx::bulk_prefetch_l2_hint(p.x + (t0 + i * dt) * row_bytes, static_cast<uint32_t>(row_bytes), last);
    }
    if (lane == 0) {
      bool ok = true;
      int64_t t = t0;
      for (int64_t i = 0; i < n; ++i, t += dt) {
        const int s = static_cast<int>(i % stages);
        if (i >= stages && !wait_parity(&empty[s], static_cast<uint32_t>(((i / stages) - 1) & 1))) {
          ok = false;
          break;
        }
        ptx::mbar_arrive_expect_tx(&full[s], static_cast<uint32_t>(row_bytes));
        ptx::bulk_g2s(stage_buf + s * row_bytes, p.x + t * row_bytes, static_cast<uint32_t>(row_bytes), &full[s]);
      }
      if (!ok) atomicCAS(p.error_word, MOE_OK, MOE_ETIMEDOUT);
    }
    return;
  }

  // ---------------- consumers ----------------
  ptx::wait_prerequisites();  // slot_row is written by the routing kernel
  const int c0 = threadIdx.x - 32;  // 0..127: 16-element chunk within each 2048-element span
  const int chunks = H / 16;
  int next_row = -1;
  if (n > 0 && lane < K) next_row = p.slot_row[t0 * K + lane];
  int64_t t = t0;
  for (int64_t i = 0; i < n; ++i, t += dt) {
    const int s = static_cast<int>(i % stages);
    int my_row = next_row;
    if (i + 1 < n && lane < K) next_row = p.slot_row[(t + dt) * K + lane];
    if (kChecked && lane < K && my_row >= 0 && my_row >= p.dst_rows) {
      atomicCAS(p.error_word, MOE_OK, MOE_ECORRUPT);
      my_row = -1;  // treated like a routing error: the token is skipped
    }
    const bool arrived = wait_parity(&full[s], static_cast<uint32_t>((i / stages) & 1));
    if (!__all_sync(0xffffffffu, arrived)) {
      if (lane == 0) atomicCAS(p.error_word, MOE_OK, MOE_ETIMEDOUT);
      break;
    }
    // Routing error: slot_row is -1 everywhere, nothing is written.
    const bool skip = __any_sync(0xffffffffu, lane < K && my_row < 0);
    const uint8_t* row = stage_buf + s * row_bytes;
    if (!skip) {
      fp8q::quantize_row<KMAX>(p, row, my_row, c0, chunks, nblk);
    }
    // A prefetched row's lines back to normal L2 priority once it is read.
    if (i >= stages)
      for (int64_t l = c0; l < row_bytes / 128; l += kConsumers) ptx::l2_priority_normal(p.x + t * row_bytes + l * 128);
    __syncwarp();
    if (lane == 0) arrive(&empty[s]);
  }
}

// Token queue: CTA b quantises tokens b, b+G, ..., b+(stages-1)G (its
// prologue, loaded while routing runs), then claims tokens stages*G, ... in
// increasing order from a counter that the routing kernel resets, so that
// CTAs that progress faster take more tokens.  The producer warp publishes
// each stage's token and its K destination rows in shared memory; full[s]
// counts two arrivals per phase (the load's expect_tx, then "rows written"),
// and token -1 with two plain arrivals ends a CTA's sequence.
template <int KMAX>
__global__ void __launch_bounds__(32 + kConsumers, KMAX <= 4 ? 8 : 1)
    dispatch_pack_fp8_queue_kernel(PackFp8Params p, int stages) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty = full + kMaxFp8Stages;
  int64_t* stage_tok = reinterpret_cast<int64_t*>(empty + kMaxFp8Stages);      // [kMaxFp8Stages]
  int32_t* stage_rows = reinterpret_cast<int32_t*>(stage_tok + kMaxFp8Stages);  // [kMaxFp8Stages][MOE_MAX_TOP_K]
  uint8_t* stage_buf = smem + kFp8QueueHeaderBytes;
  const int K = p.K, H = p.H;
  const int64_t row_bytes = static_cast<int64_t>(H) * 2;
  const int nblk = H / 128;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t G = gridDim.x, T = p.T;
  const int64_t static_end = static_cast<int64_t>(stages) * G;
  const int64_t static_tok = T < static_end ? T : static_end;
  const int64_t nstatic = static_tok > blockIdx.x ? (static_tok - blockIdx.x + G - 1) / G : 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      ptx::mbar_init(&full[s], 2);
      ptx::mbar_init(&empty[s], kConsumers / 32);
    }
    ptx::mbar_fence_init();
  }
  __syncthreads();

  if (warp == 0) {
    // ---------------- producer ----------------
    auto load = [&](int s, int64_t t) {
      ptx::mbar_arrive_expect_tx(&full[s], static_cast<uint32_t>(row_bytes));
      ptx::bulk_g2s(stage_buf + s * row_bytes, p.x + t * row_bytes, static_cast<uint32_t>(row_bytes), &full[s]);
    };
    if (lane == 0) {
      for (int i = 0; i < stages; ++i) {
        const int64_t t = i < nstatic ? blockIdx.x + i * G : -1;
        stage_tok[i] = t;
        if (t >= 0) load(i, t);
      }
    }
    __syncwarp();
    ptx::wait_prerequisites();  // slot_row, and the queue reset, come from routing
    bool claiming = T > static_end;
    unsigned long long claim = 0;
    if (lane == 0 && claiming) claim = atomicAdd(p.queue, 1ull);
    for (int64_t i = 0;; ++i) {
      const int s = static_cast<int>(i % stages);
      int64_t t;
      if (i < stages) {
        t = stage_tok[s];
      } else {
        // The stage is free once the consumers of sequence i - stages are done.
        const bool freed = wait_parity(&empty[s], static_cast<uint32_t>(((i / stages) - 1) & 1));
        if (!__all_sync(0xffffffffu, freed)) {
          if (lane == 0) atomicCAS(p.error_word, MOE_OK, MOE_ETIMEDOUT);
          break;
        }
        t = -1;
        if (lane == 0) {
          if (claiming) {
            const int64_t c = static_end + static_cast<int64_t>(claim);
            if (c < T) {
              t = c;
              claim = atomicAdd(p.queue, 1ull);
            } else {
              claiming = false;
            }
          }
          stage_tok[s] = t;
          if (t >= 0) load(s, t);
        }
        t = __shfl_sync(0xffffffffu, t, 0);
      }
      // The token's destination rows, published with the stage.
      if (lane < K) stage_rows[s * MOE_MAX_TOP_K + lane] = t >= 0 ? p.slot_row[t * K + lane] : -1;
      __syncwarp();
      if (lane == 0) {
        if (t < 0) arrive(&full[s]);  // no load: its arrival too
        arrive(&full[s]);
      }
      if (t < 0) break;
    }
    return;
  }

  // ---------------- consumers ----------------
  const int c0 = threadIdx.x - 32;
  const int chunks = H / 16;
  for (int64_t i = 0;; ++i) {
    const int s = static_cast<int>(i % stages);
    const bool arrived = wait_parity(&full[s], static_cast<uint32_t>((i / stages) & 1));
    if (!__all_sync(0xffffffffu, arrived)) {
      if (lane == 0) atomicCAS(p.error_word, MOE_OK, MOE_ETIMEDOUT);
      break;
    }
    if (stage_tok[s] < 0) break;
    int my_row = lane < K ? stage_rows[s * MOE_MAX_TOP_K + lane] : -1;
    if (kChecked && lane < K && my_row >= 0 && my_row >= p.dst_rows) {
      atomicCAS(p.error_word, MOE_OK, MOE_ECORRUPT);
      my_row = -1;
    }
    // Routing error: slot_row is -1 everywhere, nothing is written.
    if (!__any_sync(0xffffffffu, lane < K && my_row < 0))
      fp8q::quantize_row<KMAX>(p, stage_buf + s * row_bytes, my_row, c0, chunks, nblk);
    __syncwarp();
    if (lane == 0) arrive(&empty[s]);
  }
}

template <int KMAX>
cudaError_t launch_fp8_k(const PackFp8Params& p, int sms, int per_sm, int stages, bool pdl, bool strided,
                         cudaStream_t stream) {
  auto* kern = p.queue ? dispatch_pack_fp8_queue_kernel<KMAX>
               : strided ? dispatch_pack_fp8_kernel<KMAX, true>
                         : dispatch_pack_fp8_kernel<KMAX, false>;
  const size_t smem = pack_fp8_smem_bytes(stages, p.H, p.queue != nullptr);
  cudaError_t err = set_kernel_limits(reinterpret_cast<const void*>(kern), smem);
  if (err != cudaSuccess) return err;
  // A persistent grid larger than what can be resident runs a second wave:
  // never ask for more CTAs per SM than the registers and shared memory allow.
  const int resident = resident_ctas_per_sm(reinterpret_cast<const void*>(kern), 32 + kConsumers, smem);
  if (resident > 0 && per_sm > resident) per_sm = resident;
  if (per_sm < 1) per_sm = 1;
  int64_t grid = static_cast<int64_t>(sms) * per_sm;
  if (grid > p.T) grid = p.T;
  if (grid < 1) grid = 1;
  return launch_kernel(kern, dim3(static_cast<unsigned>(grid)), dim3(32 + kConsumers), smem, stream, pdl, p, stages);
}

}  // namespace

size_t pack_fp8_smem_bytes(int stages, int H, bool queue) {
  return (queue ? kFp8QueueHeaderBytes : kFp8BarBytes) + static_cast<size_t>(stages) * H * 2;
}

int pack_fp8_max_stages() { return kMaxFp8Stages; }

cudaError_t launch_dispatch_pack_fp8(const PackFp8Params& p, int sms, int per_sm, int stages, bool pdl, bool strided,
                                     cudaStream_t stream) {
  if (stages < 2) stages = 2;
  if (stages > kMaxFp8Stages) stages = kMaxFp8Stages;
  if (p.K <= 2) return launch_fp8_k<2>(p, sms, per_sm, stages, pdl, strided, stream);
  if (p.K <= 4) return launch_fp8_k<4>(p, sms, per_sm, stages, pdl, strided, stream);
  if (p.K <= 8) return launch_fp8_k<8>(p, sms, per_sm, stages, pdl, strided, stream);
  return launch_fp8_k<16>(p, sms, per_sm, stages, pdl, strided, stream);
}

}  // namespace moe
