// moe_dispatch_send_noalloc: dispatch (route_count + the bulk dispatch_pack)
// for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc at all: code that runs inside another
// framework's memory pool with no allocator handle, allocation-free runtime
// sections, or environments where the process may not grow its device
// footprint after start-up.  For them the routing tables that dispatch needs
// between its two kernels (slot_row, row_src, per-(expert, rank) offsets,
// per-rank offsets) live in one file-scope device array of fixed size instead
// of a caller-allocated workspace.  Every GPU that loads this library holds
// the array (MOE_NOALLOC_SCRATCH_BYTES) until the process exits.
//
// Set-up: the first call on a device, with that device current, looks up the
// array's device address with cudaGetSymbolAddress (in host code the array's
// name is only a host-side stand-in, never a device address) and raises the
// pack kernel's shared-memory limit.  That first call should therefore come
// before any stream capture on that device.
//
// All calls share the array and it keeps the last call's contents.  Nothing
// in it has to start at zero: route_count writes every entry it later reads.
// Calls whose kernels overlap on the GPU (different streams without ordering,
// or several host threads) race on the array; calls in one stream do not.

#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "moe.h"
#include "moe_kernels.cuh"

#define MOE_API extern "C" __attribute__((visibility("default")))

namespace {

constexpr int64_t kMaxPairs = MOE_NOALLOC_MAX_PAIRS;
constexpr int64_t kMaxExpertRanks = MOE_NOALLOC_MAX_EXPERT_RANKS;
constexpr int64_t kRankSlots = MOE_MAX_EXPERTS + 64;  // >= N + 1 for every valid N
constexpr size_t kScratchInts = 2 * kMaxPairs + kMaxExpertRanks + kRankSlots;
static_assert(kScratchInts * 4 == MOE_NOALLOC_SCRATCH_BYTES, "scratch size must match the header");

// slot_row [kMaxPairs] | row_src [kMaxPairs] | src_offsets [kMaxExpertRanks] | rank_offsets [kRankSlots]
static __device__ __align__(256) int32_t g_noalloc_scratch[kScratchInts];

struct DeviceSetup {
  bool ready;
  int32_t* scratch;  // device address of g_noalloc_scratch on this device
  int num_sms;
  int max_smem_optin;
};

constexpr int kMaxDevices = 64;
std::mutex g_setup_mu;
DeviceSetup g_setup[kMaxDevices];

int setup_device(int dev, DeviceSetup* out) {
  if (dev < 0 || dev >= kMaxDevices) return MOE_EINVAL;
  std::lock_guard<std::mutex> lock(g_setup_mu);
  DeviceSetup& s = g_setup[dev];
  if (!s.ready) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return MOE_ECUDA;
    int sms = 0, optin = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return MOE_ECUDA;
    if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) return MOE_ECUDA;
    if (moe::prepare_pack(optin) != cudaSuccess) return MOE_ECUDA;
    s.scratch = static_cast<int32_t*>(p);
    s.num_sms = sms;
    s.max_smem_optin = optin;
    s.ready = true;
  }
  *out = s;
  return MOE_OK;
}

bool aligned_to(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

MOE_API int moe_dispatch_send_noalloc(const moe_config* cfg, const void* x, const int32_t* topk_idx, void* expert_x,
                                      int64_t expert_x_rows, int32_t* expert_counts, int32_t* expert_offsets,
                                      int32_t* status, void* stream) {
  const int rc = moe_validate_config(cfg);
  if (rc) return rc;
  const int64_t pairs = static_cast<int64_t>(cfg->num_tokens) * cfg->top_k;
  // Sizes beyond the fixed scratch array are refused before anything runs.
  if (pairs > kMaxPairs) return MOE_EINVAL;
  if (static_cast<int64_t>(cfg->num_experts) * cfg->num_ranks > kMaxExpertRanks) return MOE_EINVAL;
  if (expert_x_rows < pairs) return MOE_EINVAL;
  if (!expert_counts || !expert_offsets || !status) return MOE_EINVAL;
  if (!aligned_to(expert_counts, 4) || !aligned_to(expert_offsets, 4) || !aligned_to(status, 4)) return MOE_EINVAL;
  if (cfg->num_tokens > 0) {
    if (!x || !topk_idx || !expert_x) return MOE_EINVAL;
    if (!aligned_to(x, 16) || !aligned_to(expert_x, 16) || !aligned_to(topk_idx, 4)) return MOE_EINVAL;
  }

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ECUDA;
  DeviceSetup ds;
  const int src = setup_device(dev, &ds);
  if (src) return src;
  if (moe::route_count_smem_bytes(cfg->num_experts) > static_cast<size_t>(ds.max_smem_optin)) return MOE_EINVAL;

  int32_t* slot_row = ds.scratch;
  int32_t* row_src = slot_row + kMaxPairs;
  int32_t* src_offsets = row_src + kMaxPairs;
  int32_t* rank_offsets = src_offsets + kMaxExpertRanks;
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  moe::RouteCountParams rp = {};
  rp.topk_idx = topk_idx;
  rp.T = cfg->num_tokens;
  rp.K = cfg->top_k;
  rp.E = cfg->num_experts;
  rp.N = cfg->num_ranks;
  rp.expert_counts = expert_counts;
  rp.expert_offsets = expert_offsets;
  rp.src_offsets = src_offsets;
  rp.rank_offsets = rank_offsets;
  rp.slot_row = slot_row;
  rp.row_src = row_src;
  rp.error_word = status;
  int vec = 1;
  if (cfg->top_k % 4 == 0 && aligned_to(topk_idx, 16)) vec = 4;
  else if (cfg->top_k % 2 == 0 && aligned_to(topk_idx, 8)) vec = 2;
  if (moe::launch_route_count(rp, vec, s) != cudaSuccess) return MOE_ECUDA;
  if (cfg->num_tokens == 0) return MOE_OK;

  moe::PackParams pp = {};
  pp.x = static_cast<const uint8_t*>(x);
  pp.expert_x = static_cast<uint8_t*>(expert_x);
  pp.slot_row = slot_row;
  pp.error_word = status;
  pp.T = cfg->num_tokens;
  pp.K = cfg->top_k;
  pp.dst_rows = expert_x_rows;
  pp.row_bytes = static_cast<int64_t>(cfg->hidden) * 2;
  // A fixed launch shape, simpler than moe_dispatch_send's automatic one (no
  // unit queue, no L2 prefetch or cache hints, one store group in flight):
  // pieces of at most 16 KiB, 4 bulk stages, as many CTAs per SM as shared
  // memory allows.
  const int64_t npieces = (pp.row_bytes + 16384 - 1) / 16384;
  pp.piece_bytes = static_cast<int32_t>((pp.row_bytes / 16 + npieces - 1) / npieces * 16);
  pp.pieces = static_cast<int32_t>((pp.row_bytes + pp.piece_bytes - 1) / pp.piece_bytes);
  moe::PackLaunch pl = {};
  pl.variant = moe::kPackBulk;
  pl.stages = 4;
  while (pl.stages > 2 && moe::pack_bulk_smem_bytes(pl.stages, pp.piece_bytes) > static_cast<size_t>(ds.max_smem_optin))
    --pl.stages;
  const size_t smem = moe::pack_bulk_smem_bytes(pl.stages, pp.piece_bytes);
  if (smem > static_cast<size_t>(ds.max_smem_optin)) return MOE_EINVAL;
  const int per_sm = moe::smem_ctas_per_sm(smem);
  int64_t grid = static_cast<int64_t>(ds.num_sms) * per_sm;
  const int64_t units = static_cast<int64_t>(pp.T) * pp.pieces;
  if (grid > units) grid = units;
  pl.grid = static_cast<int>(grid);
  pl.pdl = true;
  pl.prefetch = 0;
  pl.prefetch_units = 0;
  pl.hints = 0;
  pl.depth = 0;
  if (moe::launch_dispatch_pack(pp, pl, s) != cudaSuccess) return MOE_ECUDA;
  return MOE_OK;
}
