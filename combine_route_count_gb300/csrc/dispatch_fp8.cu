// dispatch_pack_fp8: the dispatch payload as block-scaled fp8.
//
// "Efficient and portable mixture-of-experts communication" (Dispatch): the
// dispatch kernel sends tokens together with their block scaling factors;
// "Enabling trillion-parameter models on AWS EFA" (evaluation): block-scale
// fp8 dispatch, bf16 combine.  Each token row is quantised once and written
// to its K destination rows:
//   blocks of 128 consecutive elements, scale = amax / 448 (1 for an all-zero
//   block), inv = 1 / scale (both IEEE float32 divisions, once per block),
//   q = E4M3(x * inv) rounded to nearest even, saturating;
//   expert_xq[slot_row[t,k]] = q[t], expert_scales[slot_row[t,k]] = scales[t].
//
// CTA = 1 producer warp + 4 consumer warps; unit = one token row; each CTA
// takes a contiguous range of tokens.  The producer bulk-loads rows into
// shared-memory stages (the first ones before griddepcontrol.wait: rows do
// not depend on routing).  Consumers: 8 lanes cover one 128-element block (16
// elements each), reduce amax with shuffles, multiply by the block's inverse
// scale, convert two at a time with cvt.rn.satfinite.e4m3x2.f32 and store 16
// fp8 bytes per lane to
// each of the K destination rows (coalesced); one lane per block stores the
// scale.  Waits are bounded (2 s) and report MOE_ETIMEDOUT.

#include <cuda_runtime.h>

#include "moe_kernels.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kConsumers = 128;
constexpr int kMaxFp8Stages = 8;
constexpr int kFp8BarBytes = 256;
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

__device__ __forceinline__ uint4 lds128(const void* p) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(ptx::smem_addr(p)));
  return v;
}

// Two floats to two E4M3 codes: `lo` in the low byte, `hi` in the high byte.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
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
      // Warp-uniform trip count: every lane reaches the shuffles below; lanes
      // past the end of the row work on zeros and store nothing.
      for (int cb = 0; cb < chunks; cb += kConsumers) {
        const int c = cb + c0;
        const bool act = c < chunks;
        const uint4 a = act ? lds128(row + c * 32) : make_uint4(0, 0, 0, 0);
        const uint4 b = act ? lds128(row + c * 32 + 16) : make_uint4(0, 0, 0, 0);
        const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
        float f[16];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          f[2 * j] = __uint_as_float(w[j] << 16);
          f[2 * j + 1] = __uint_as_float(w[j] & 0xffff0000u);
        }
        float amax = 0.0f;
#pragma unroll
        for (int j = 0; j < 16; ++j) amax = fmaxf(amax, fabsf(f[j]));
        // The 8 lanes of one 128-element block are 8 consecutive lanes.
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 4));
        const float scale = amax > 0.0f ? __fdiv_rn(amax, 448.0f) : 1.0f;
        const float inv = __fdiv_rn(1.0f, scale);
        uint4 out;
        uint32_t* o = &out.x;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint32_t lo = e4m3x2(__fmul_rn(f[4 * j], inv), __fmul_rn(f[4 * j + 1], inv));
          const uint32_t hi = e4m3x2(__fmul_rn(f[4 * j + 2], inv), __fmul_rn(f[4 * j + 3], inv));
          o[j] = lo | (hi << 16);
        }
        const int blk = c >> 3;
#pragma unroll
        for (int k = 0; k < KMAX; ++k) {
          if (k < K) {
            const int64_t dst = static_cast<int64_t>(__shfl_sync(0xffffffffu, my_row, k));
            if (act) {
              ptx::st_v4(p.expert_xq + dst * H + static_cast<int64_t>(c) * 16, out);
              if ((c & 7) == 0) p.expert_scales[dst * nblk + blk] = scale;
            }
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) arrive(&empty[s]);
  }
}

template <int KMAX>
cudaError_t launch_fp8_k(const PackFp8Params& p, int sms, int per_sm, int stages, bool pdl, bool strided,
                         cudaStream_t stream) {
  auto* kern = strided ? dispatch_pack_fp8_kernel<KMAX, true> : dispatch_pack_fp8_kernel<KMAX, false>;
  const size_t smem = pack_fp8_smem_bytes(stages, p.H);
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

size_t pack_fp8_smem_bytes(int stages, int H) {
  return kFp8BarBytes + static_cast<size_t>(stages) * H * 2;
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
