// route_pack_fp8: the routing and the fp8 pack of dispatch in one kernel, for
// small layers.
//
// The fp8 payload ("Efficient and portable mixture-of-experts communication",
// Dispatch: tokens travel with their block scales) behind routing as in
// "Enabling trillion-parameter models on AWS EFA" (Dispatch and combine:
// counts, their cumulative sum, every token at its offset).  With routing in
// a kernel of its own, the fp8 pack cannot quantise a row before the routing
// grid has finished: on a Mixtral-sized layer that routing stays exposed
// (~3 us of a ~33 us layer), unlike the bf16 pack, which ends its routing
// wait with the rows already staged and has only stores left.
//
// Here one CTA per SM computes the whole routing from topk_idx staged in
// shared memory (route_tables.cuh, the same steps and tables as route_pack)
// while its token rows are already in flight.  The CTA's threads form groups
// of 128 (four warps); group g of CTA b is virtual group v = b*groups + g and
// quantises tokens v, v + G*groups, ... in order, each group with its own
// ring of whole-row stages that its first thread fills by bulk copies (TMA):
//
//   before the routing: the group's first `stages` rows into its stages and
//   the rest of its rows into L2;
//   after the routing:  per token, wait for the stage, quantise the row with
//   the 128 threads (fp8_quant.cuh: codes and scales to the K destination
//   rows from the tables in shared memory), a barrier of the group, refill
//   the stage with the group's token `stages` further on.
//
// After a routing error every CTA reaches the same decision: nothing is
// written but slot_row = -1 and the zeroed tables.  Waits are bounded (2 s)
// and report MOE_ETIMEDOUT; a group that gives up waits (bounded) for its
// loads in flight before it exits.

#include <cuda_runtime.h>

#include "fp8_quant.cuh"
#include "moe_kernels.cuh"
#include "ptx.cuh"
#include "route_tables.cuh"

namespace moe {
namespace {

constexpr int kGroupThreads = kRoutePackFp8GroupThreads;
static_assert(kGroupThreads == fp8q::kRowThreads, "a group quantises one row");
constexpr int kMaxGroups = kRoutePackThreads / kGroupThreads;
constexpr int kMaxStages = 16;
constexpr int kBarBytes = 512;  // mbarriers: the groups' stages (<= 63), then the index copy's
constexpr int kIdxBar = kBarBytes / 8 - 1;

// Named barrier of group g (ids 1..kMaxGroups; 0 is the CTA's).
__device__ __forceinline__ void group_sync(int g) {
  asm volatile("bar.sync %0, %1;" ::"r"(g + 1), "r"(kGroupThreads) : "memory");
}
// The same barrier, returning whether `v` holds for every thread of the group.
__device__ __forceinline__ bool group_all(int g, bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(v)), "r"(g + 1), "r"(kGroupThreads)
      : "memory");
  return r != 0;
}

template <int KMAX>
__global__ void __launch_bounds__(kRoutePackThreads, 1) route_pack_fp8_kernel(RoutePackFp8Params p, int stages) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int T = p.T, K = p.K, E = p.E;
  const int tid = threadIdx.x, lane = tid & 31, W = blockDim.x >> 5;
  const int groups = blockDim.x / kGroupThreads;
  const int g = tid / kGroupThreads, c0 = tid - g * kGroupThreads;
  const bool leader = c0 == 0;
  const int64_t row_bytes = static_cast<int64_t>(p.H) * 2;
  // This group's stage ring and mbarriers.
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem) + g * stages;
  uint8_t* stage_buf = smem + kBarBytes + static_cast<size_t>(g) * stages * row_bytes;
  const rtab::Tables tb = rtab::carve_tables(smem + kBarBytes + static_cast<size_t>(groups) * stages * row_bytes, T, E);
  // topk_idx, copied whole: the choices of token t at sidx[t*K .. t*K+K).
  int32_t* sidx = reinterpret_cast<int32_t*>(reinterpret_cast<uint8_t*>(tb.mask) + rtab::tables_bytes(T, E));
  uint64_t* idx_bar = reinterpret_cast<uint64_t*>(smem) + kIdxBar;
  const int pairs = T * K;
  const int bulk_ints = (reinterpret_cast<uintptr_t>(p.topk_idx) & 15) == 0 ? (pairs & ~3) : 0;
  const int64_t first = static_cast<int64_t>(blockIdx.x) * groups + g;  // virtual group
  const int64_t step = static_cast<int64_t>(gridDim.x) * groups;
  const int64_t mine = T > first ? (T - first + step - 1) / step : 0;

  if (leader) {
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
  rtab::start_index_copy(p, sidx, idx_bar, bulk_ints, 32 * (W - 1));
  __syncthreads();

  auto issue_load = [&](int64_t i) {
    const int s = static_cast<int>(i % stages);
    const int64_t t = first + i * step;
    ptx::mbar_arrive_expect_tx(&bars[s], static_cast<uint32_t>(row_bytes));
    ptx::bulk_g2s(stage_buf + static_cast<size_t>(s) * row_bytes, p.x + t * row_bytes,
                  static_cast<uint32_t>(row_bytes), &bars[s]);
  };
  // Bounded waits for the loads of the group's tokens lo..hi (leader only).
  auto drain = [&](int64_t lo, int64_t hi) {
    for (int64_t q = lo; q <= hi; ++q) rtab::wait_phase(&bars[q % stages], static_cast<uint32_t>((q / stages) & 1));
  };
  // The group's first rows travel while the tables are built; its later
  // rows go to L2.
  const int64_t prologue = mine < stages ? mine : stages;
  if (leader)
    for (int64_t i = 0; i < prologue; ++i) issue_load(i);
  if (c0 < 32)
    for (int64_t i = prologue + lane; i < mine; i += 32)
      ptx::bulk_prefetch_l2(p.x + (first + i * step) * row_bytes, static_cast<uint32_t>(row_bytes));

  const bool idx_ok = __syncthreads_and(rtab::wait_phase(idx_bar, 0));
  if (!idx_ok) {
    // The index copy did not complete in time: report it, wait (bounded)
    // for it and for the row loads issued so far, write nothing.
    if (tid == 0) atomicCAS(p.error_word, MOE_OK, MOE_ETIMEDOUT);
    if (tid == 32 * (W - 1)) rtab::wait_phase(idx_bar, 0);
    if (leader) drain(0, prologue - 1);
    return;
  }

  // The routing tables, the CTA's slot_row / row_src entries and (CTA 0) the
  // counts, offsets and status.
  const bool bad = __syncthreads_or(rtab::token_masks<KMAX>(sidx, tb, T, K, E));
  rtab::expert_scans(tb, E);
  rtab::write_routing(p, tb, sidx, bad);
  if (bad) {
    // Nothing is written; the prologue's loads are waited for (bounded)
    // before shared memory goes away.
    if (leader) drain(0, prologue - 1);
    return;
  }

  const int chunks = p.H / 16, nblk = p.H / 128;
  int64_t i = 0;
  bool ok = true;
  for (; i < mine; ++i) {
    const int s = static_cast<int>(i % stages);
    const int t = static_cast<int>(first + i * step);
    int my_row = lane < K ? rtab::row_of(tb, t, sidx[t * K + lane]) : -1;
    if (kChecked && my_row >= p.dst_rows) {
      atomicCAS(p.error_word, MOE_OK, MOE_ECORRUPT);
      my_row = -1;  // the token is skipped
    }
    if (!group_all(g, rtab::wait_phase(&bars[s], static_cast<uint32_t>((i / stages) & 1)))) {
      ok = false;
      break;
    }
    if (!__any_sync(0xffffffffu, lane < K && my_row < 0))
      fp8q::quantize_row<KMAX>(p, stage_buf + static_cast<size_t>(s) * row_bytes, my_row, c0, chunks, nblk);
    group_sync(g);  // every thread of the group is done with stage s
    if (leader && i + stages < mine) issue_load(i + stages);
  }
  if (!ok && leader) {
    atomicCAS(p.error_word, MOE_OK, MOE_ETIMEDOUT);
    // Loads issued: tokens up to i - 1 + stages.
    drain(i, (i - 1 + stages < mine - 1) ? i - 1 + stages : mine - 1);
  }
}

}  // namespace

size_t route_pack_fp8_smem_bytes(int T, int K, int E, int H, int groups, int stages) {
  return kBarBytes + static_cast<size_t>(groups) * stages * H * 2 + rtab::tables_bytes(T, E) + rtab::index_bytes(T, K);
}

int route_pack_fp8_max_stages(int groups) {
  const int n = kIdxBar / (groups < 1 ? 1 : groups);
  return n < kMaxStages ? n : kMaxStages;
}

cudaError_t prepare_route_pack_fp8(int max_smem_bytes) {
  const void* kernels[] = {reinterpret_cast<const void*>(route_pack_fp8_kernel<2>),
                           reinterpret_cast<const void*>(route_pack_fp8_kernel<4>),
                           reinterpret_cast<const void*>(route_pack_fp8_kernel<8>),
                           reinterpret_cast<const void*>(route_pack_fp8_kernel<16>)};
  for (const void* k : kernels) {
    const cudaError_t err = set_kernel_limits(k, static_cast<size_t>(max_smem_bytes));
    if (err != cudaSuccess) return err;
  }
  return cudaSuccess;
}

cudaError_t launch_route_pack_fp8(const RoutePackFp8Params& p, int grid, int groups, int stages, bool pdl,
                                  cudaStream_t stream) {
  if (groups < 1) groups = 1;
  if (groups > kMaxGroups) groups = kMaxGroups;
  const int maxst = route_pack_fp8_max_stages(groups);
  if (stages > maxst) stages = maxst;
  if (stages < 1) stages = 1;
  const size_t smem = route_pack_fp8_smem_bytes(p.T, p.K, p.E, p.H, groups, stages);
  const dim3 g(grid < 1 ? 1 : grid), block(groups * kGroupThreads);
  if (p.K <= 2) return launch_kernel(route_pack_fp8_kernel<2>, g, block, smem, stream, pdl, p, stages);
  if (p.K <= 4) return launch_kernel(route_pack_fp8_kernel<4>, g, block, smem, stream, pdl, p, stages);
  if (p.K <= 8) return launch_kernel(route_pack_fp8_kernel<8>, g, block, smem, stream, pdl, p, stages);
  return launch_kernel(route_pack_fp8_kernel<16>, g, block, smem, stream, pdl, p, stages);
}

}  // namespace moe
