// The C ABI of libmoe.so (declared in include/moe.h): argument checks, the
// workspace layout, the send/recv phase machine and the kernel launches.
//
// The split send/recv pairs follow "Efficient and portable
// mixture-of-experts communication" (Portable kernels: each kernel pair owns
// fixed-capacity buffers that every layer reuses; Dispatch; Combine) and
// "Enabling trillion-parameter models on AWS EFA" (Dispatch and combine).
// On one GPU nothing travels between ranks, so the receive halves are
// ordering points: dispatch_recv hands out the layout, combine_send registers
// the expert outputs, and the gather + weighted sum runs in combine_recv.

#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include <climits>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <new>
#include <tuple>
#include <utility>

#include "moe.h"
#include "moe_kernels.cuh"

namespace {

// NVTX range around the host side of one entry point (what it enqueues shows
// under this name in Nsight tools; ncu --nvtx --nvtx-include selects kernels by
// it).  Costs a few nanoseconds when no tool is attached.
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

}  // namespace

#define MOE_API extern "C" __attribute__((visibility("default")))

namespace moe {

cudaError_t set_kernel_limits(const void* kernel, size_t bytes, bool nonportable_cluster) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  static std::mutex mu;
  static std::map<std::pair<int, const void*>, std::pair<size_t, bool>> done;
  std::lock_guard<std::mutex> lock(mu);
  auto& entry = done[{dev, kernel}];
  if (bytes > entry.first) {
    err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
    if (err != cudaSuccess) return err;
    entry.first = bytes;
  }
  if (nonportable_cluster && !entry.second) {
    err = cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (err != cudaSuccess) return err;
    entry.second = true;
  }
  return cudaSuccess;
}

int resident_ctas_per_sm(const void* kernel, int threads, size_t smem) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  static std::mutex mu;
  static std::map<std::tuple<int, const void*, int, size_t>, int> known;
  std::lock_guard<std::mutex> lock(mu);
  auto it = known.find({dev, kernel, threads, smem});
  if (it != known.end()) return it->second;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, smem) != cudaSuccess) return 0;
  known[{dev, kernel, threads, smem}] = n;
  return n;
}

int smem_ctas_per_sm(size_t smem) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  static std::mutex mu;
  static std::map<int, std::pair<int, int>> known;  // device -> (shared memory per SM, reserve per CTA)
  int per_sm = 0, reserve = 0;
  {
    std::lock_guard<std::mutex> lock(mu);
    auto it = known.find(dev);
    if (it == known.end()) {
      if (cudaDeviceGetAttribute(&per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess ||
          cudaDeviceGetAttribute(&reserve, cudaDevAttrReservedSharedMemoryPerBlock, dev) != cudaSuccess) {
        cudaGetLastError();
        return 1;
      }
      known[dev] = {per_sm, reserve};
    } else {
      per_sm = it->second.first;
      reserve = it->second.second;
    }
  }
  const int n = static_cast<int>(static_cast<size_t>(per_sm) / (smem + static_cast<size_t>(reserve)));
  return n < 1 ? 1 : n;
}

}  // namespace moe

namespace {

enum Phase { kIdle = 0, kDispatched = 1, kReceived = 2, kCombineSent = 3 };

constexpr size_t kAlign = 256;

size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

struct WorkspaceLayout {
  size_t error_word, expert_counts, expert_offsets, src_offsets, rank_offsets, slot_row, row_src, hist, block_err,
      send_pos, send_dest, plan_row, plan_w, plan_mask, queue, total;
};

WorkspaceLayout layout_of(const moe_config& c) {
  WorkspaceLayout l;
  const size_t pairs = static_cast<size_t>(c.num_tokens) * c.top_k;
  size_t o = 0;
  l.error_word = o;
  o += align_up(sizeof(int32_t));
  l.expert_counts = o;
  o += align_up(sizeof(int32_t) * c.num_experts);
  l.expert_offsets = o;
  o += align_up(sizeof(int32_t) * (c.num_experts + 1));
  l.src_offsets = o;
  o += align_up(sizeof(int32_t) * static_cast<size_t>(c.num_experts) * c.num_ranks);
  l.rank_offsets = o;
  o += align_up(sizeof(int32_t) * (c.num_ranks + 1));
  l.slot_row = o;
  o += align_up(sizeof(int32_t) * pairs);
  l.row_src = o;
  o += align_up(sizeof(int32_t) * pairs);
  l.hist = o;  // per-chunk expert histograms of the split routing kernels
  o += align_up(sizeof(int32_t) * static_cast<size_t>(moe::kMaxSplitBlocks) * c.num_experts);
  l.block_err = o;
  o += align_up(sizeof(int32_t) * moe::kMaxSplitBlocks);
  l.send_pos = o;  // two-stage dispatch: send row of each (token, slot) pair
  o += align_up(sizeof(int32_t) * pairs);
  l.send_dest = o;  // two-stage dispatch: grouped row of each send row
  o += align_up(sizeof(int32_t) * pairs);
  l.plan_row = o;  // two-level combine: sorted slots, weights, group ends
  o += align_up(sizeof(int32_t) * pairs);
  l.plan_w = o;
  o += align_up(sizeof(float) * pairs);
  l.plan_mask = o;
  o += align_up(sizeof(int32_t) * static_cast<size_t>(c.num_tokens));
  l.queue = o;  // the pack's and the combine's unit queues (set to 0 by the routing of every dispatch)
  o += align_up(2 * sizeof(unsigned long long));
  l.total = o;
  return l;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

struct moe_ctx {
  moe_config cfg;
  uint8_t* ws;
  size_t ws_bytes;
  int device;
  int num_sms;
  int max_sms;  // MOE_OPT_MAX_SMS: 0 = every SM
  int64_t test_drop_unit;  // MOE_OPT_TEST_DROP_COMBINE_UNIT (-1: off)
  int combine_order;       // MOE_OPT_COMBINE_ORDER
  int fp8_order;           // MOE_OPT_FP8_ORDER
  int kernel_events;       // MOE_OPT_KERNEL_EVENTS
  bool events_created;
  cudaEvent_t ev[4];       // before/after the pack kernel, before/after the combine kernel
  bool pack_timed, combine_timed;
  int max_smem_optin;
  int l2_bytes;
  int phase;
  const void* expert_y;
  int64_t expert_y_rows;
  int32_t* error_word;
  int32_t* expert_counts;
  int32_t* expert_offsets;
  int32_t* src_offsets;
  int32_t* rank_offsets;
  int32_t* slot_row;
  int32_t* row_src;
  int32_t* hist;
  int32_t* block_err;
  int32_t* send_pos;
  int32_t* send_dest;
  int32_t* plan_row;
  float* plan_w;
  int32_t* plan_mask;
  unsigned long long* queue;
  // launch options (MOE_OPT_* in moe.h)
  int pack_variant;
  int pack_stages;
  int pack_piece_bytes;  // 0 = automatic
  int pack_ctas_per_sm;  // 0 = as many as fit
  int pack_prefetch;     // 1 = prefetch the CTA's later token rows into L2 before routing completes
  int cache_hints;       // MOE_OPT_CACHE_HINTS bit flags
  int pack_depth;        // MOE_OPT_PACK_STORE_DEPTH (0 = default)
  int pack_schedule;     // MOE_OPT_PACK_SCHEDULE (-1 = automatic)
  int combine_schedule;  // MOE_OPT_COMBINE_SCHEDULE (-1 = automatic)
  int pdl;
  int route_variant;  // MOE_OPT_ROUTE_VARIANT
  int combine_variant;      // MOE_OPT_COMBINE_VARIANT
  int combine_stages;       // 0 = automatic
  int combine_piece_bytes;  // 0 = automatic
  int combine_ctas_per_sm;  // 0 = as many as fit
  bool route_pack_ok;  // the one-kernel route+pack path can run this configuration
  bool route_pack_fp8_ok;  // ... and its fp8 form (moe_dispatch_send_fp8)
  int64_t dense_cap;   // capacity of the last dispatch if it was moe_dispatch_send_dense, else 0
  int cluster_ctas;   // route_cluster shape for this configuration (0 = cannot be scheduled)
  int cluster_chunk;
  int cluster_warps;
  int cluster_staged;
  int cluster_group;
};

MOE_API int moe_validate_config(const moe_config* c) {
  if (!c) return MOE_EINVAL;
  if (c->num_tokens < 0 || c->num_ranks < 1 || c->num_experts < 1 || c->top_k < 1) return MOE_EINVAL;
  if (c->hidden < 8 || c->hidden % 8 != 0) return MOE_EINVAL;
  if (c->top_k > MOE_MAX_TOP_K || c->top_k > c->num_experts) return MOE_EINVAL;
  if (c->num_experts > MOE_MAX_EXPERTS) return MOE_EINVAL;
  if (c->num_tokens % c->num_ranks != 0 || c->num_experts % c->num_ranks != 0) return MOE_EINVAL;
  if (static_cast<int64_t>(c->num_tokens) * c->top_k > INT32_MAX) return MOE_EINVAL;
  if (static_cast<int64_t>(c->num_experts) * c->num_ranks > INT32_MAX / 4) return MOE_EINVAL;
  return MOE_OK;
}

MOE_API int moe_workspace_bytes(const moe_config* cfg, size_t* bytes) {
  if (!bytes) return MOE_EINVAL;
  const int rc = moe_validate_config(cfg);
  if (rc) return rc;
  *bytes = layout_of(*cfg).total;
  return MOE_OK;
}

MOE_API int moe_recv_bound_rows(const moe_config* cfg, int64_t* rows) {
  if (!rows) return MOE_EINVAL;
  const int rc = moe_validate_config(cfg);
  if (rc) return rc;
  const int64_t Tr = cfg->num_tokens / cfg->num_ranks;
  const int64_t L = cfg->num_experts / cfg->num_ranks;
  *rows = static_cast<int64_t>(cfg->num_ranks) * Tr * (cfg->top_k > L ? cfg->top_k : L);
  return MOE_OK;
}

MOE_API int moe_ctx_create(const moe_config* cfg, void* workspace, size_t workspace_bytes, moe_ctx** out) {
  if (!out) return MOE_EINVAL;
  *out = nullptr;
  int rc = moe_validate_config(cfg);
  if (rc) return rc;
  const WorkspaceLayout l = layout_of(*cfg);
  if (!workspace || workspace_bytes < l.total || !aligned(workspace, kAlign)) return MOE_EINVAL;

  int dev = 0, sms = 0, optin = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ECUDA;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return MOE_ECUDA;
  if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) return MOE_ECUDA;
  int l2 = 0;
  if (cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev) != cudaSuccess) return MOE_ECUDA;
  if (moe::route_count_smem_bytes(cfg->num_experts) > static_cast<size_t>(optin)) return MOE_EINVAL;
  if (moe::route_local_smem_bytes(cfg->num_experts) > static_cast<size_t>(optin)) return MOE_EINVAL;
  if (moe::prepare_pack(optin) != cudaSuccess) return MOE_ECUDA;
  if (moe::prepare_route_pack(optin) != cudaSuccess) return MOE_ECUDA;
  if (moe::prepare_route_pack_fp8(optin) != cudaSuccess) return MOE_ECUDA;

  moe_ctx* c = new (std::nothrow) moe_ctx;
  if (!c) return MOE_EINVAL;
  std::memset(c, 0, sizeof *c);
  c->cfg = *cfg;
  c->ws = static_cast<uint8_t*>(workspace);
  c->ws_bytes = workspace_bytes;
  c->device = dev;
  c->num_sms = sms;
  c->max_smem_optin = optin;
  c->l2_bytes = l2;
  c->phase = kIdle;
  c->error_word = reinterpret_cast<int32_t*>(c->ws + l.error_word);
  c->expert_counts = reinterpret_cast<int32_t*>(c->ws + l.expert_counts);
  c->expert_offsets = reinterpret_cast<int32_t*>(c->ws + l.expert_offsets);
  c->src_offsets = reinterpret_cast<int32_t*>(c->ws + l.src_offsets);
  c->rank_offsets = reinterpret_cast<int32_t*>(c->ws + l.rank_offsets);
  c->slot_row = reinterpret_cast<int32_t*>(c->ws + l.slot_row);
  c->row_src = reinterpret_cast<int32_t*>(c->ws + l.row_src);
  c->hist = reinterpret_cast<int32_t*>(c->ws + l.hist);
  c->block_err = reinterpret_cast<int32_t*>(c->ws + l.block_err);
  c->send_pos = reinterpret_cast<int32_t*>(c->ws + l.send_pos);
  c->send_dest = reinterpret_cast<int32_t*>(c->ws + l.send_dest);
  c->plan_row = reinterpret_cast<int32_t*>(c->ws + l.plan_row);
  c->plan_w = reinterpret_cast<float*>(c->ws + l.plan_w);
  c->plan_mask = reinterpret_cast<int32_t*>(c->ws + l.plan_mask);
  c->queue = reinterpret_cast<unsigned long long*>(c->ws + l.queue);
  c->pack_schedule = -1;
  c->combine_schedule = -1;
  c->pack_variant = moe::kPackBulk;
  c->pack_stages = 0;  // automatic: about 200 KiB of stages per SM
  c->pack_prefetch = 2;
  c->cache_hints = moe::kHintPackLoads | moe::kHintPackStores | moe::kHintCombineLoads;
  c->pack_piece_bytes = 0;
  c->pack_ctas_per_sm = 0;
  c->pdl = 1;
  c->route_variant = 0;
  c->combine_variant = -1;  // automatic
  c->test_drop_unit = -1;
  c->combine_order = -1;  // automatic
  // fp8 pack in the strided token order (measured on GB300: DeepSeek-sized
  // fp8 layer 141.4 -> 139.0 us, Kimi-sized 545 -> 543 us, Mixtral-sized
  // unchanged).
  c->fp8_order = 1;
  // One-kernel route+pack: small routing tables, and two stages of the
  // automatic piece size fit next to them in one CTA.
  {
    const int64_t row_bytes = static_cast<int64_t>(cfg->hidden) * 2;
    const int64_t pieces = (row_bytes + 8191) / 8192;
    const int64_t piece = (row_bytes / 16 + pieces - 1) / pieces * 16;
    c->route_pack_ok = moe::route_pack_eligible(cfg->num_tokens, cfg->top_k, cfg->num_experts) &&
                       moe::route_pack_smem_bytes(cfg->num_tokens, cfg->top_k, cfg->num_experts, 1, 2,
                                                  static_cast<int>(piece)) <=
                           static_cast<size_t>(optin);
    // The fp8 form: two whole bf16 rows of one group next to the tables.
    c->route_pack_fp8_ok = moe::route_pack_eligible(cfg->num_tokens, cfg->top_k, cfg->num_experts) &&
                           cfg->hidden % MOE_FP8_BLOCK == 0 &&
                           moe::route_pack_fp8_smem_bytes(cfg->num_tokens, cfg->top_k, cfg->num_experts,
                                                          cfg->hidden, 1, 2) <= static_cast<size_t>(optin);
  }
  // Largest cluster of route_cluster CTAs this device can schedule for this
  // configuration (16, else 8, 4, 2, 1), or none.
  for (int maxc = moe::kMaxClusterCtas; maxc >= 1; maxc /= 2) {
    int ctas = 0, chunk = 0, warps = 0;
    moe::route_cluster_shape(cfg->num_tokens, cfg->num_experts, maxc, &ctas, &chunk, &warps);
    moe::RouteClusterParams q = {};
    q.T = cfg->num_tokens;
    q.K = cfg->top_k;
    q.E = cfg->num_experts;
    q.N = cfg->num_ranks;
    q.chunk = chunk;
    q.warps = warps;
    moe::route_cluster_plan(&q, ctas, optin);
    if (moe::route_cluster_smem_bytes(q.E, warps, q.staged ? chunk * q.K : 0) > static_cast<size_t>(optin)) continue;
    if (moe::route_cluster_supported(q, 1, ctas)) {
      c->cluster_ctas = ctas;
      c->cluster_chunk = chunk;
      c->cluster_warps = warps;
      c->cluster_staged = q.staged;
      c->cluster_group = q.dsmem_group;
      break;
    }
  }
  *out = c;
  return MOE_OK;
}

MOE_API int moe_ctx_destroy(moe_ctx* ctx) {
  if (ctx && ctx->events_created)
    for (cudaEvent_t e : ctx->ev) cudaEventDestroy(e);
  delete ctx;
  return MOE_OK;
}

namespace {

// Automatic choices, from steady-state sweeps on GB300: with K >= 4 the TMA
// gather combine and 2 pack CTAs per SM are fastest (DeepSeek, Kimi, worst
// case); with K <= 2 each unit carries too little work for the bulk combine's
// per-CTA pipeline and 3 pack CTAs per SM issue faster (Mixtral).
int combine_variant_of(const moe_ctx* c) {
  if (c->combine_variant >= 0) return c->combine_variant;
  return c->cfg.top_k >= 4 ? moe::kCombineBulk : moe::kCombineVector;
}
// Bulk pack CTAs per SM: 2 when a token row has K >= 4 destinations, else 3.
int pack_ctas_auto(int K) { return K >= 4 ? 2 : 3; }

// SMs the persistent grids may spread over (MOE_OPT_MAX_SMS).
int grid_sms(const moe_ctx* c) { return c->max_sms > 0 && c->max_sms < c->num_sms ? c->max_sms : c->num_sms; }

// Whether moe_dispatch_send routes and packs in one kernel (route_pack):
// forced by MOE_OPT_ROUTE_VARIANT 4, or automatic for small layers with the
// default bulk pack and its static split.  Measured on GB300 (A/B, one box,
// against route_cluster + the bulk pack): 64-token layer 9.23 -> 7.17 us in
// a CUDA graph, Mixtral-sized layer 34.96 -> 34.70 us; not eligible from
// T*K > 16384 on (a DeepSeek-sized layer exposes ~0.4 us of routing).
bool dispatch_uses_route_pack(const moe_ctx* c) {
  if (!c->route_pack_ok) return false;
  if (c->route_variant == 4) return true;
  return c->route_variant == 0 && c->pack_variant == moe::kPackBulk && c->pack_schedule != 1;
}

// Whether moe_dispatch_send_fp8 routes and quantises in one kernel
// (route_pack_fp8): forced by MOE_OPT_ROUTE_VARIANT 4, or automatic for the
// same small layers, in the strided token order and without the token queue.
bool dispatch_fp8_uses_route_pack(const moe_ctx* c) {
  if (!c->route_pack_fp8_ok) return false;
  if (c->route_variant == 4) return true;
  return c->route_variant == 0 && c->fp8_order == 1 && c->pack_schedule != 1;
}

}  // namespace

MOE_API int moe_ctx_set_option(moe_ctx* ctx, int option, int64_t value) {
  if (!ctx) return MOE_EINVAL;
  switch (option) {
    case MOE_OPT_PACK_VARIANT:
      if (value != moe::kPackBulk && value != moe::kPackVector) return MOE_EINVAL;
      ctx->pack_variant = static_cast<int>(value);
      return MOE_OK;
    case MOE_OPT_PACK_STAGES:
      if (value != 0 && (value < 2 || value > 16)) return MOE_EINVAL;
      ctx->pack_stages = static_cast<int>(value);
      return MOE_OK;
    case MOE_OPT_PACK_PIECE_BYTES:
      if (value < 0 || value % 16 != 0 || value > 65536) return MOE_EINVAL;
      ctx->pack_piece_bytes = static_cast<int>(value);
      return MOE_OK;
    case MOE_OPT_PACK_CTAS_PER_SM:
      if (value < 0 || value > 32) return MOE_EINVAL;
      ctx->pack_ctas_per_sm = static_cast<int>(value);
      return MOE_OK;
    case MOE_OPT_PDL:
      if (value != 0 && value != 1) return MOE_EINVAL;
      ctx->pdl = static_cast<int>(value);
      return MOE_OK;
    case MOE_OPT_PACK_PREFETCH:
      if (value < 0 || value > 2) return MOE_EINVAL;
      ctx->pack_prefetch = static_cast<int>(value);
      return MOE_OK;
    case MOE_OPT_CACHE_HINTS:
      if (value < 0 || value > 7) return MOE_EINVAL;
      ctx->cache_hints = static_cast<int>(value);
      return MOE_OK;
    case MOE_OPT_PACK_STORE_DEPTH:
      if (value < 0 || value > 8) return MOE_EINVAL;
      ctx->pack_depth = static_cast<int>(value);
      return MOE_OK;
    case MOE_OPT_PACK_SCHEDULE:
      if (value < -1 || value > 1) return MOE_EINVAL;
      ctx->pack_schedule = static_cast<int>(value);
      return MOE_OK;
    case MOE_OPT_COMBINE_SCHEDULE:
      if (value < -1 || value > 1) return MOE_EINVAL;
      ctx->combine_schedule = static_cast<int>(value);
      return MOE_OK;
    case MOE_OPT_COMBINE_VARIANT:
      if (value != -1 && value != moe::kCombineBulk && value != moe::kCombineVector) return MOE_EINVAL;
      ctx->combine_variant = static_cast<int>(value);
      return MOE_OK;
    case MOE_OPT_COMBINE_STAGES:
      if (value != 0 && (value < 2 || value > 8)) return MOE_EINVAL;
      ctx->combine_stages = static_cast<int>(value);
      return MOE_OK;
    case MOE_OPT_COMBINE_PIECE_BYTES:
      if (value < 0 || value % 16 != 0 || value > 16384) return MOE_EINVAL;
      ctx->combine_piece_bytes = static_cast<int>(value);
      return MOE_OK;
    case MOE_OPT_COMBINE_CTAS_PER_SM:
      if (value < 0 || value > 32) return MOE_EINVAL;
      ctx->combine_ctas_per_sm = static_cast<int>(value);
      return MOE_OK;
    case MOE_OPT_MAX_SMS:
      if (value < 0 || value > ctx->num_sms) return MOE_EINVAL;
      ctx->max_sms = static_cast<int>(value);
      return MOE_OK;
    case MOE_OPT_TEST_DROP_COMBINE_UNIT:
      if (value < -1) return MOE_EINVAL;
      ctx->test_drop_unit = value;
      return MOE_OK;
    case MOE_OPT_COMBINE_ORDER:
      if (value < -1 || value > 1) return MOE_EINVAL;
      ctx->combine_order = static_cast<int>(value);
      return MOE_OK;
    case MOE_OPT_FP8_ORDER:
      if (value < 0 || value > 1) return MOE_EINVAL;
      ctx->fp8_order = static_cast<int>(value);
      return MOE_OK;
    case MOE_OPT_KERNEL_EVENTS:
      if (value < 0 || value > 1) return MOE_EINVAL;
      if (value == 1 && !ctx->events_created) {
        for (int i = 0; i < 4; ++i) {
          if (cudaEventCreate(&ctx->ev[i]) != cudaSuccess) {
            for (int j = 0; j < i; ++j) cudaEventDestroy(ctx->ev[j]);
            return MOE_ECUDA;
          }
        }
        ctx->events_created = true;
      }
      ctx->kernel_events = static_cast<int>(value);
      return MOE_OK;
    case MOE_OPT_ROUTE_VARIANT:
      if (value < 0 || value > 5) return MOE_EINVAL;
      if (value == 3 && ctx->cluster_ctas == 0) return MOE_EINVAL;
      if ((value == 4 || value == 5) && !ctx->route_pack_ok) return MOE_EINVAL;
      ctx->route_variant = static_cast<int>(value);
      return MOE_OK;
    default:
      return MOE_EINVAL;
  }
}

MOE_API int moe_ctx_get_option(const moe_ctx* ctx, int option, int64_t* value) {
  if (!ctx || !value) return MOE_EINVAL;
  switch (option) {
    case MOE_OPT_PACK_VARIANT:
      *value = ctx->pack_variant;
      return MOE_OK;
    case MOE_OPT_PACK_STAGES:
      *value = ctx->pack_stages;
      return MOE_OK;
    case MOE_OPT_PACK_PIECE_BYTES:
      *value = ctx->pack_piece_bytes;
      return MOE_OK;
    case MOE_OPT_PACK_CTAS_PER_SM:
      *value = ctx->pack_ctas_per_sm;
      return MOE_OK;
    case MOE_OPT_PDL:
      *value = ctx->pdl;
      return MOE_OK;
    case MOE_OPT_PACK_PREFETCH:
      *value = ctx->pack_prefetch;
      return MOE_OK;
    case MOE_OPT_CACHE_HINTS:
      *value = ctx->cache_hints;
      return MOE_OK;
    case MOE_OPT_PACK_STORE_DEPTH:
      *value = ctx->pack_depth;
      return MOE_OK;
    case MOE_OPT_PACK_SCHEDULE:
      *value = ctx->pack_schedule;
      return MOE_OK;
    case MOE_OPT_COMBINE_SCHEDULE:
      *value = ctx->combine_schedule;
      return MOE_OK;
    case MOE_OPT_ROUTE_VARIANT:
      *value = ctx->route_variant != 0    ? ctx->route_variant
               : dispatch_uses_route_pack(ctx) ? 4
               : ctx->cluster_ctas > 0         ? 3
                                               : 2;
      return MOE_OK;
    case MOE_OPT_ROUTE_CLUSTER_CTAS:
      *value = ctx->cluster_ctas;
      return MOE_OK;
    case MOE_OPT_ROUTE_VARIANT_FP8:
      *value = dispatch_fp8_uses_route_pack(ctx)                                ? 4
               : ctx->route_variant != 0 && ctx->route_variant != 4           ? ctx->route_variant
               : ctx->cluster_ctas > 0                                          ? 3
                                                                                : 2;
      return MOE_OK;
    case MOE_OPT_COMBINE_VARIANT:
      *value = combine_variant_of(ctx);
      return MOE_OK;
    case MOE_OPT_COMBINE_STAGES:
      *value = ctx->combine_stages;
      return MOE_OK;
    case MOE_OPT_COMBINE_PIECE_BYTES:
      *value = ctx->combine_piece_bytes;
      return MOE_OK;
    case MOE_OPT_COMBINE_CTAS_PER_SM:
      *value = ctx->combine_ctas_per_sm;
      return MOE_OK;
    case MOE_OPT_MAX_SMS:
      *value = ctx->max_sms;
      return MOE_OK;
    case MOE_OPT_TEST_DROP_COMBINE_UNIT:
      *value = ctx->test_drop_unit;
      return MOE_OK;
    case MOE_OPT_COMBINE_ORDER:
      *value = ctx->combine_order;
      return MOE_OK;
    case MOE_OPT_FP8_ORDER:
      *value = ctx->fp8_order;
      return MOE_OK;
    case MOE_OPT_KERNEL_EVENTS:
      *value = ctx->kernel_events;
      return MOE_OK;
    default:
      return MOE_EINVAL;
  }
}

namespace {

// Packs that write more than this use whole rows as units (see pack_piece_bytes)
// and one store group in flight.
constexpr int64_t kLargePackBytes = int64_t{1} << 30;

// Bytes per pack unit: the whole row when it is at most 8 KiB, else the row
// split into equal 16-byte-multiple pieces of at most 8 KiB; for packs that
// write more than kLargePackBytes, whole rows of up to 16 KiB (measured on
// GB300, Kimi-sized layer with 14 KiB rows: 645.2 -> 630.0 us with 6 stages;
// DeepSeek-sized, 470 MB of writes, 161.4 -> 161.9 us, so it keeps 7 KiB pieces).
int pack_piece_bytes(const moe_ctx* c, int64_t row_bytes, int64_t dest_bytes) {
  int64_t pb = c->pack_piece_bytes;
  if (pb <= 0) {
    const int64_t max_piece = dest_bytes > kLargePackBytes && row_bytes <= 16384 ? 16384 : 8192;
    const int64_t pieces = (row_bytes + max_piece - 1) / max_piece;
    pb = (row_bytes / 16 + pieces - 1) / pieces * 16;
  }
  if (pb > row_bytes) pb = row_bytes;
  return static_cast<int>(pb);
}

int pack_grid(const moe_ctx* c, const moe::PackParams& p, int variant, int stages) {
  const bool bulk = variant == moe::kPackBulk;
  const int64_t units = static_cast<int64_t>(p.T) * p.pieces;
  int per_sm = c->pack_ctas_per_sm > 0 ? c->pack_ctas_per_sm : (bulk ? pack_ctas_auto(p.K) : 0);
  if (bulk) {
    const size_t smem = moe::pack_bulk_smem_bytes(stages, p.piece_bytes);
    const int fit = moe::smem_ctas_per_sm(smem);
    if (per_sm <= 0 || per_sm > fit) per_sm = fit;
    if (per_sm < 1) per_sm = 1;
  } else if (per_sm <= 0) {
    per_sm = 8;  // 8 x 256 threads
  }
  int64_t grid = static_cast<int64_t>(grid_sms(c)) * per_sm;
  const int64_t useful = bulk ? units : (units + 7) / 8;
  if (grid > useful) grid = useful;
  if (grid < 1) grid = 1;
  return static_cast<int>(grid);
}

}  // namespace

namespace {

// Enqueues the routing kernels of the context's variant (counts, offsets,
// slot_row, row_src, error word).  MOE_OK or MOE_ECUDA.
int enqueue_routing(moe_ctx* ctx, const int32_t* topk_idx, cudaStream_t s) {
  const moe_config& c = ctx->cfg;
  moe::RouteCountParams rp = {};
  rp.topk_idx = topk_idx;
  rp.T = c.num_tokens;
  rp.K = c.top_k;
  rp.E = c.num_experts;
  rp.N = c.num_ranks;
  rp.expert_counts = ctx->expert_counts;
  rp.expert_offsets = ctx->expert_offsets;
  rp.src_offsets = ctx->src_offsets;
  rp.rank_offsets = ctx->rank_offsets;
  rp.slot_row = ctx->slot_row;
  rp.row_src = ctx->row_src;
  rp.error_word = ctx->error_word;
  rp.queue = ctx->queue;
  int vec = 1;
  if (c.top_k % 4 == 0 && aligned(topk_idx, 16)) vec = 4;
  else if (c.top_k % 2 == 0 && aligned(topk_idx, 8)) vec = 2;
  // Variant 4 (one-kernel route+pack) exists only for moe_dispatch_send and
  // moe_dispatch_send_fp8; every other dispatch form routes as in the
  // automatic choice.
  const bool use_cluster =
      (ctx->route_variant == 0 || ctx->route_variant == 3 || ctx->route_variant == 4) && ctx->cluster_ctas > 0;
  if (ctx->route_variant == 1) {
    if (moe::launch_route_count(rp, vec, s) != cudaSuccess) return MOE_ECUDA;
  } else if (ctx->route_variant == 5 && c.num_tokens > 0) {
    // route_pack's routing alone, in one CTA (no copy warps).
    moe::RoutePackParams qp = {};
    qp.topk_idx = topk_idx;
    qp.T = c.num_tokens;
    qp.K = c.top_k;
    qp.E = c.num_experts;
    qp.N = c.num_ranks;
    qp.row_bytes = 16;
    qp.piece_bytes = 16;
    qp.pieces = 1;
    qp.expert_counts = ctx->expert_counts;
    qp.expert_offsets = ctx->expert_offsets;
    qp.src_offsets = ctx->src_offsets;
    qp.rank_offsets = ctx->rank_offsets;
    qp.slot_row = ctx->slot_row;
    qp.row_src = ctx->row_src;
    qp.error_word = ctx->error_word;
    qp.queue = ctx->queue;
    moe::RoutePackLaunch ql = {};
    ql.threads = moe::kRoutePackThreads;
    ql.grid = 1;
    ql.copy_warps = 0;
    ql.stages = 2;
    ql.depth = 1;
    ql.pdl = ctx->pdl != 0;
    if (moe::launch_route_pack(qp, ql, s) != cudaSuccess) return MOE_ECUDA;
  } else if (use_cluster) {
    moe::RouteClusterParams cp = {};
    cp.topk_idx = topk_idx;
    cp.T = c.num_tokens;
    cp.K = c.top_k;
    cp.E = c.num_experts;
    cp.N = c.num_ranks;
    cp.chunk = ctx->cluster_chunk;
    cp.warps = ctx->cluster_warps;
    cp.staged = ctx->cluster_staged;
    cp.dsmem_group = ctx->cluster_group;
    cp.expert_counts = ctx->expert_counts;
    cp.expert_offsets = ctx->expert_offsets;
    cp.src_offsets = ctx->src_offsets;
    cp.rank_offsets = ctx->rank_offsets;
    cp.slot_row = ctx->slot_row;
    cp.row_src = ctx->row_src;
    cp.error_word = ctx->error_word;
    cp.queue = ctx->queue;
    if (moe::launch_route_cluster(cp, vec, ctx->cluster_ctas, s) != cudaSuccess) return MOE_ECUDA;
  } else {
    moe::RouteSplitParams sp = {};
    sp.topk_idx = topk_idx;
    sp.T = c.num_tokens;
    sp.K = c.top_k;
    sp.E = c.num_experts;
    sp.N = c.num_ranks;
    sp.chunk = moe::route_split_chunk(c.num_tokens);
    sp.expert_counts = ctx->expert_counts;
    sp.expert_offsets = ctx->expert_offsets;
    sp.src_offsets = ctx->src_offsets;
    sp.rank_offsets = ctx->rank_offsets;
    sp.slot_row = ctx->slot_row;
    sp.row_src = ctx->row_src;
    sp.error_word = ctx->error_word;
    sp.hist = ctx->hist;
    sp.block_err = ctx->block_err;
    sp.queue = ctx->queue;
    if (moe::launch_route_split(sp, vec, s) != cudaSuccess) return MOE_ECUDA;
  }
  return MOE_OK;
}

}  // namespace

namespace {

// Enqueues the pack kernel of the context's variant: dst[table[t*K+k]] = src[t]
// for T source rows of H bf16 each (a table entry < 0 is skipped).  The
// bulk pack reads its first source rows before waiting on the previous
// kernel, so `pdl` must be false when src is that kernel's output.
// `after_routing` marks the first pack after the routing kernels: it may
// prefetch source rows into L2 while routing runs (the context's prefetch
// mode) and claim units from the queue that routing has just reset (the
// context's schedule); `variant` < 0 takes the context's pack variant.
int enqueue_pack(moe_ctx* ctx, const void* src, void* dst, int64_t dst_rows, const int32_t* table, int32_t T,
                 int32_t K, int64_t row_bytes, bool pdl, bool after_routing, int variant, cudaStream_t s) {
  moe::PackParams pp = {};
  pp.x = static_cast<const uint8_t*>(src);
  pp.expert_x = static_cast<uint8_t*>(dst);
  pp.slot_row = table;
  pp.error_word = ctx->error_word;
  pp.T = T;
  pp.K = K;
  pp.dst_rows = dst_rows;
  pp.row_bytes = row_bytes;
  const int64_t dest_bytes = static_cast<int64_t>(T) * K * pp.row_bytes;
  pp.piece_bytes = pack_piece_bytes(ctx, pp.row_bytes, dest_bytes);
  pp.pieces = static_cast<int32_t>((pp.row_bytes + pp.piece_bytes - 1) / pp.piece_bytes);
  moe::PackLaunch pl = {};
  pl.variant = variant >= 0 ? variant : ctx->pack_variant;
  pl.stages = ctx->pack_stages;
  if (pl.stages <= 0) {
    // About 200 KiB of stages per SM split over the automatic CTAs per SM
    // (two for K >= 4: ~100 KiB each; three otherwise), 2..16 stages.
    pl.stages = static_cast<int>((200 * 1024) / pack_ctas_auto(K) / pp.piece_bytes);
    // Whole-row units of large packs: about 96 KiB of stages (6 of 14 KiB rows).
    if (pp.piece_bytes > 8192) pl.stages = static_cast<int>((96 * 1024) / pp.piece_bytes);
    if (pl.stages > 16) pl.stages = 16;
    if (pl.stages < 2) pl.stages = 2;
  }
  if (pl.variant == moe::kPackBulk) {
    // Shrink the pipeline if the stages do not fit in one CTA's shared memory.
    while (pl.stages > 2 &&
           moe::pack_bulk_smem_bytes(pl.stages, pp.piece_bytes) > static_cast<size_t>(ctx->max_smem_optin))
      --pl.stages;
    if (moe::pack_bulk_smem_bytes(pl.stages, pp.piece_bytes) > static_cast<size_t>(ctx->max_smem_optin))
      return MOE_EINVAL;
  }
  pl.grid = pack_grid(ctx, pp, pl.variant, pl.stages);
  pl.prefetch = after_routing ? ctx->pack_prefetch : 0;
  pl.prefetch_units = -1;
  if (pl.prefetch == 2) {
    // Evict-last prefetch when every row a CTA still needs after its
    // prologue fits, across the grid, in a third of L2.  (Measured on
    // GB300: it pays at DeepSeek size even beyond the device's persisting
    // L2 carve-out, so that carve-out does not bound it.)
    const int64_t budget = static_cast<int64_t>(ctx->l2_bytes) / 3;
    const int64_t units = static_cast<int64_t>(pp.T) * pp.pieces;
    const int64_t per_cta = (units + pl.grid - 1) / pl.grid - pl.stages;  // units past the prologue
    const int64_t fit = budget > 0 ? budget / (static_cast<int64_t>(pl.grid) * pp.piece_bytes) : 0;
    if (per_cta > 0 && fit >= per_cta) {
      pl.prefetch_units = static_cast<int>(per_cta);
    } else {
      // The token rows do not fit: marking part of them evict-last was
      // measured slower (Kimi-sized layers) than prefetching all normally.
      pl.prefetch = 1;
    }
  }
  pl.pdl = pdl;
  pl.hints = ctx->cache_hints;
  // Store groups in flight (measured on GB300 with the destination rows
  // loaded one unit ahead): two for DeepSeek-, worst-case- and Mixtral-sized
  // layers and the two-stage dispatch; one when the pack writes more than
  // 1 GiB (Kimi-sized layers: 3 % faster than with two).
  pl.depth = ctx->pack_depth > 0 ? ctx->pack_depth : (dest_bytes > kLargePackBytes ? 1 : 2);
  // Unit queue (bulk pack, first pack after routing): automatic when a CTA
  // has more than 1.5x its prologue's worth of units.  Measured on GB300:
  // the DeepSeek-, Kimi- and worst-case-sized layers gain from it; with about
  // one prologue of units per CTA (Mixtral-sized layers) the claims of all
  // CTAs at once cost more than the balance gives back.
  if (after_routing && pl.variant == moe::kPackBulk && ctx->pack_schedule != 0) {
    const int64_t units = static_cast<int64_t>(T) * pp.pieces;
    pl.dynamic = ctx->pack_schedule == 1 || 2 * units > 3 * static_cast<int64_t>(pl.stages) * pl.grid;
    if (pl.dynamic) pp.queue = ctx->queue;
  }
  if (moe::launch_dispatch_pack(pp, pl, s) != cudaSuccess) return MOE_ECUDA;
  return MOE_OK;
}

}  // namespace

namespace {

// Enqueues route_pack: routing and the bulk pack of x into expert_x in one
// kernel (moe_dispatch_send of a small layer), one CTA per SM.  Its copy
// warps stand for the two-kernel path's static bulk-pack CTAs: as many per SM
// (MOE_OPT_PACK_CTAS_PER_SM, else 2 for K >= 4 and 3 otherwise), the same
// pieces, stage budget (about 200 KiB per SM), cache hints and store depth;
// the stages shrink until everything fits next to the routing tables.
// MOE_OK, MOE_EINVAL or MOE_ECUDA.
int enqueue_route_pack(moe_ctx* ctx, const void* x, const int32_t* topk_idx, void* expert_x, int64_t expert_x_rows,
                       cudaStream_t s) {
  const moe_config& c = ctx->cfg;
  moe::RoutePackParams rp = {};
  rp.topk_idx = topk_idx;
  rp.x = static_cast<const uint8_t*>(x);
  rp.expert_x = static_cast<uint8_t*>(expert_x);
  rp.T = c.num_tokens;
  rp.K = c.top_k;
  rp.E = c.num_experts;
  rp.N = c.num_ranks;
  rp.row_bytes = static_cast<int64_t>(c.hidden) * 2;
  const int64_t dest_bytes = static_cast<int64_t>(c.num_tokens) * c.top_k * rp.row_bytes;
  rp.piece_bytes = pack_piece_bytes(ctx, rp.row_bytes, dest_bytes);
  rp.pieces = static_cast<int32_t>((rp.row_bytes + rp.piece_bytes - 1) / rp.piece_bytes);
  rp.dst_rows = expert_x_rows;
  rp.expert_counts = ctx->expert_counts;
  rp.expert_offsets = ctx->expert_offsets;
  rp.src_offsets = ctx->src_offsets;
  rp.rank_offsets = ctx->rank_offsets;
  rp.slot_row = ctx->slot_row;
  rp.row_src = ctx->row_src;
  rp.error_word = ctx->error_word;
  rp.queue = ctx->queue;

  moe::RoutePackLaunch rl = {};
  // Small layers (at most 32 words of 32 tokens) route with 8 warps per CTA
  // (measured on GB300, 64-token layer in a graph: 7.3-8.2 -> 7.17 us against
  // 32 warps); larger ones with 32 (one or a few words per warp).
  rl.threads = (c.num_tokens + 31) / 32 <= 32 ? 256 : moe::kRoutePackThreads;
  int warps = ctx->pack_ctas_per_sm > 0 ? ctx->pack_ctas_per_sm : pack_ctas_auto(c.top_k);
  if (warps > rl.threads / 32) warps = rl.threads / 32;
  auto smem_of = [&](int w, int st) { return moe::route_pack_smem_bytes(rp.T, rp.K, rp.E, w, st, rp.piece_bytes); };
  while (warps > 1 && smem_of(warps, 2) > static_cast<size_t>(ctx->max_smem_optin)) --warps;
  int stages = ctx->pack_stages > 0 ? ctx->pack_stages : static_cast<int>((200 * 1024) / warps / rp.piece_bytes);
  const int maxst = moe::route_pack_max_stages(warps);
  if (stages > maxst) stages = maxst;
  if (stages < 2) stages = 2;
  while (stages > 2 && smem_of(warps, stages) > static_cast<size_t>(ctx->max_smem_optin)) --stages;
  if (smem_of(warps, stages) > static_cast<size_t>(ctx->max_smem_optin)) return MOE_EINVAL;
  const int64_t units = static_cast<int64_t>(rp.T) * rp.pieces;
  int64_t grid = (units + warps - 1) / warps;
  if (grid > grid_sms(ctx)) grid = grid_sms(ctx);
  if (grid < 1) grid = 1;
  rl.grid = static_cast<int>(grid);
  rl.copy_warps = warps;
  rl.stages = stages;
  // Small rows, at most two per copy warp (a 64-token layer): through
  // registers, no stages.
  rl.vec = c.top_k <= 8 && rp.pieces == 1 &&
           moe::route_pack_vec_ok(rp.row_bytes, (units + grid * warps - 1) / (grid * warps));
  rl.hints = ctx->cache_hints;
  rl.depth = ctx->pack_depth > 0 ? ctx->pack_depth : 2;
  rl.pdl = ctx->pdl != 0;
  if (moe::launch_route_pack(rp, rl, s) != cudaSuccess) return MOE_ECUDA;
  return MOE_OK;
}

// Enqueues route_pack_fp8: routing and the fp8 pack of x into expert_xq /
// expert_scales in one kernel (moe_dispatch_send_fp8 of a small layer), one
// CTA per SM.  Groups of 128 threads per CTA (MOE_OPT_PACK_CTAS_PER_SM, else
// 2 for layers of at most 32 words of 32 tokens, whose routing is fastest
// with 8 warps as for route_pack, and 7 otherwise), whole-row stages per
// group (MOE_OPT_PACK_STAGES, else as many as fit next to the routing
// tables); groups drop until two stages fit.  Measured on GB300 (A/B, one
// box), Mixtral-sized fp8 layer with 2..8 groups: 42.8, 36.6, 34.2, 33.5,
// 32.9, 31.8 (7 groups of 3 stages; 31.8 with 2 stages too) and 33.1 us (8
// groups of 2 stages), against 33.6 us for route_cluster + the fp8 pack; the
// 64-token layer in a graph: 6.05 us with 1 or 2 groups, 6.6 with 4, against
// 8.6 us.  MOE_OK, MOE_EINVAL or MOE_ECUDA.
int enqueue_route_pack_fp8(moe_ctx* ctx, const void* x, const int32_t* topk_idx, void* expert_xq,
                           float* expert_scales, int64_t expert_rows, cudaStream_t s) {
  const moe_config& c = ctx->cfg;
  moe::RoutePackFp8Params rp = {};
  rp.topk_idx = topk_idx;
  rp.x = static_cast<const uint8_t*>(x);
  rp.expert_xq = static_cast<uint8_t*>(expert_xq);
  rp.expert_scales = expert_scales;
  rp.T = c.num_tokens;
  rp.K = c.top_k;
  rp.E = c.num_experts;
  rp.N = c.num_ranks;
  rp.H = c.hidden;
  rp.dst_rows = expert_rows;
  rp.expert_counts = ctx->expert_counts;
  rp.expert_offsets = ctx->expert_offsets;
  rp.src_offsets = ctx->src_offsets;
  rp.rank_offsets = ctx->rank_offsets;
  rp.slot_row = ctx->slot_row;
  rp.row_src = ctx->row_src;
  rp.error_word = ctx->error_word;
  rp.queue = ctx->queue;

  const int max_groups = moe::kRoutePackThreads / moe::kRoutePackFp8GroupThreads;
  auto smem_of = [&](int g, int st) { return moe::route_pack_fp8_smem_bytes(rp.T, rp.K, rp.E, rp.H, g, st); };
  const size_t optin = static_cast<size_t>(ctx->max_smem_optin);
  auto stages_for = [&](int g) {  // as many as fit, or as asked; 0 if two do not fit
    int st = ctx->pack_stages > 0 ? ctx->pack_stages : 16;
    const int maxst = moe::route_pack_fp8_max_stages(g);
    if (st > maxst) st = maxst;
    while (st > 2 && smem_of(g, st) > optin) --st;
    return smem_of(g, st) <= optin ? st : 0;
  };
  auto grid_for = [&](int g) {
    int64_t grid = (static_cast<int64_t>(rp.T) + g - 1) / g;
    if (grid > grid_sms(ctx)) grid = grid_sms(ctx);
    return grid < 1 ? static_cast<int64_t>(1) : grid;
  };
  int groups = ctx->pack_ctas_per_sm > 0 ? ctx->pack_ctas_per_sm : ((c.num_tokens + 31) / 32 <= 32 ? 2 : 7);
  if (groups > max_groups) groups = max_groups;
  while (groups > 1 && stages_for(groups) == 0) --groups;
  const int stages = stages_for(groups);
  if (groups < 1 || stages < 1 || smem_of(groups, stages) > optin) return MOE_EINVAL;
  const int64_t grid = grid_for(groups);
  if (moe::launch_route_pack_fp8(rp, static_cast<int>(grid), groups, stages, ctx->pdl != 0, s) != cudaSuccess)
    return MOE_ECUDA;
  return MOE_OK;
}

}  // namespace

MOE_API int moe_dispatch_send(moe_ctx* ctx, const void* x, const int32_t* topk_idx, void* expert_x,
                              int64_t expert_x_rows, void* stream) {
  NvtxRange nvtx_range("moe_dispatch_send");
  if (!ctx) return MOE_EINVAL;
  if (ctx->phase != kIdle) return MOE_ESTATE;
  const moe_config& c = ctx->cfg;
  const int64_t pairs = static_cast<int64_t>(c.num_tokens) * c.top_k;
  if (expert_x_rows < pairs) return MOE_EINVAL;
  if (c.num_tokens > 0) {
    if (!x || !topk_idx || !expert_x) return MOE_EINVAL;
    if (!aligned(x, 16) || !aligned(expert_x, 16) || !aligned(topk_idx, 4)) return MOE_EINVAL;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (c.num_tokens > 0 && dispatch_uses_route_pack(ctx)) {
    const bool timed = ctx->kernel_events != 0;
    if (timed && cudaEventRecord(ctx->ev[0], s) != cudaSuccess) return MOE_ECUDA;
    const int frc = enqueue_route_pack(ctx, x, topk_idx, expert_x, expert_x_rows, s);
    if (frc != MOE_OK) return frc;
    if (timed && cudaEventRecord(ctx->ev[1], s) != cudaSuccess) return MOE_ECUDA;
    ctx->pack_timed = timed;
    ctx->dense_cap = 0;
    ctx->phase = kDispatched;
    return MOE_OK;
  }
  const int rrc = enqueue_routing(ctx, topk_idx, s);
  if (rrc != MOE_OK) return rrc;

  if (c.num_tokens > 0) {
    const bool timed = ctx->kernel_events != 0;
    if (timed && cudaEventRecord(ctx->ev[0], s) != cudaSuccess) return MOE_ECUDA;
    const int64_t row_bytes = static_cast<int64_t>(c.hidden) * 2;
    const int prc = enqueue_pack(ctx, x, expert_x, expert_x_rows, ctx->slot_row, c.num_tokens, c.top_k, row_bytes, ctx->pdl != 0,
                                 true, -1, s);
    if (prc != MOE_OK) return prc;
    if (timed && cudaEventRecord(ctx->ev[1], s) != cudaSuccess) return MOE_ECUDA;
    ctx->pack_timed = timed;
  }
  ctx->dense_cap = 0;
  ctx->phase = kDispatched;
  return MOE_OK;
}

MOE_API int moe_dispatch_send_staged(moe_ctx* ctx, const void* x, const int32_t* topk_idx, void* send_buf,
                                     int64_t send_rows, void* expert_x, int64_t expert_x_rows, void* stream) {
  NvtxRange nvtx_range("moe_dispatch_send_staged");
  if (!ctx) return MOE_EINVAL;
  if (ctx->phase != kIdle) return MOE_ESTATE;
  const moe_config& c = ctx->cfg;
  const int64_t pairs = static_cast<int64_t>(c.num_tokens) * c.top_k;
  if (expert_x_rows < pairs || send_rows < pairs) return MOE_EINVAL;
  if (c.num_tokens > 0) {
    if (!x || !topk_idx || !send_buf || !expert_x) return MOE_EINVAL;
    if (!aligned(x, 16) || !aligned(send_buf, 16) || !aligned(expert_x, 16) || !aligned(topk_idx, 4))
      return MOE_EINVAL;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int rrc = enqueue_routing(ctx, topk_idx, s);
  if (rrc != MOE_OK) return rrc;
  if (c.num_tokens > 0) {
    moe::StagedLayoutParams sp = {};
    sp.topk_idx = topk_idx;
    sp.slot_row = ctx->slot_row;
    sp.expert_offsets = ctx->expert_offsets;
    sp.src_offsets = ctx->src_offsets;
    sp.send_pos = ctx->send_pos;
    sp.send_dest = ctx->send_dest;
    sp.T = c.num_tokens;
    sp.K = c.top_k;
    sp.E = c.num_experts;
    sp.N = c.num_ranks;
    sp.error_word = ctx->error_word;
    if (moe::launch_staged_layout(sp, ctx->pdl != 0, s) != cudaSuccess) return MOE_ECUDA;
    // Stage 1, every source rank: x rows into its per-peer send rows.
    const int64_t row_bytes = static_cast<int64_t>(c.hidden) * 2;
    int prc = enqueue_pack(ctx, x, send_buf, send_rows, ctx->send_pos, c.num_tokens, c.top_k, row_bytes, ctx->pdl != 0,
                           true, -1,
                           s);
    if (prc != MOE_OK) return prc;
    // Stage 2, every receiver: send rows into the grouped rows.  Its source is
    // the previous kernel's output, so it is not launched early, and there is
    // nothing for an L2 prefetch to overlap.  One destination per row: the
    // 16-byte vector copy is used (measured faster on GB300 than the bulk
    // pipeline, which moves one row piece per stage cycle when K = 1).
    prc = enqueue_pack(ctx, send_buf, expert_x, expert_x_rows, ctx->send_dest, static_cast<int32_t>(pairs), 1, row_bytes,
                       false, false,
                       moe::kPackVector, s);
    if (prc != MOE_OK) return prc;
  }
  ctx->pack_timed = false;  // the event-timed pack is that of moe_dispatch_send(_fp8) only
  ctx->dense_cap = 0;
  ctx->phase = kDispatched;
  return MOE_OK;
}

MOE_API int moe_dispatch_send_quantized(moe_ctx* ctx, const void* xq, const float* x_scales, const int32_t* topk_idx,
                                        void* expert_xq, float* expert_scales, int64_t expert_rows, void* stream) {
  NvtxRange nvtx_range("moe_dispatch_send_quantized");
  if (!ctx) return MOE_EINVAL;
  if (ctx->phase != kIdle) return MOE_ESTATE;
  const moe_config& c = ctx->cfg;
  const int64_t pairs = static_cast<int64_t>(c.num_tokens) * c.top_k;
  const int64_t scale_row_bytes = static_cast<int64_t>(c.hidden / MOE_FP8_BLOCK) * 4;
  // Both rows move in 16-byte units: H a multiple of 512 (scale rows of 16*m bytes).
  if (c.hidden % MOE_FP8_BLOCK != 0 || scale_row_bytes % 16 != 0 || expert_rows < pairs) return MOE_EINVAL;
  if (c.num_tokens > 0) {
    if (!xq || !x_scales || !topk_idx || !expert_xq || !expert_scales) return MOE_EINVAL;
    if (!aligned(xq, 16) || !aligned(x_scales, 16) || !aligned(expert_xq, 16) || !aligned(expert_scales, 16) ||
        !aligned(topk_idx, 4))
      return MOE_EINVAL;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int rrc = enqueue_routing(ctx, topk_idx, s);
  if (rrc != MOE_OK) return rrc;
  if (c.num_tokens > 0) {
    // The E4M3 rows, then their scale rows: the same placement, two byte-row
    // copies (neither reads what the other writes).  Scale rows are short
    // (H/32 bytes): the 16-byte vector copy moves them with less per-row
    // overhead than the bulk pipeline (measured on GB300: DeepSeek-sized
    // layer 148.0 -> 134.6 us; doing them first was slower, 138.2 us).
    int prc = enqueue_pack(ctx, xq, expert_xq, expert_rows, ctx->slot_row, c.num_tokens, c.top_k, c.hidden,
                           ctx->pdl != 0, true,
                           -1, s);
    if (prc != MOE_OK) return prc;
    prc = enqueue_pack(ctx, x_scales, expert_scales, expert_rows, ctx->slot_row, c.num_tokens, c.top_k, scale_row_bytes,
                       ctx->pdl != 0, false, moe::kPackVector, s);
    if (prc != MOE_OK) return prc;
  }
  ctx->pack_timed = false;
  ctx->dense_cap = 0;
  ctx->phase = kDispatched;
  return MOE_OK;
}

MOE_API int moe_dispatch_send_fp8(moe_ctx* ctx, const void* x, const int32_t* topk_idx, void* expert_xq,
                                  float* expert_scales, int64_t expert_rows, void* stream) {
  NvtxRange nvtx_range("moe_dispatch_send_fp8");
  if (!ctx) return MOE_EINVAL;
  if (ctx->phase != kIdle) return MOE_ESTATE;
  const moe_config& c = ctx->cfg;
  const int64_t pairs = static_cast<int64_t>(c.num_tokens) * c.top_k;
  if (c.hidden % MOE_FP8_BLOCK != 0 || expert_rows < pairs) return MOE_EINVAL;
  // Two stages of one bf16 row must fit in shared memory.
  if (moe::pack_fp8_smem_bytes(2, c.hidden) > static_cast<size_t>(ctx->max_smem_optin)) return MOE_EINVAL;
  if (c.num_tokens > 0) {
    if (!x || !topk_idx || !expert_xq || !expert_scales) return MOE_EINVAL;
    if (!aligned(x, 16) || !aligned(expert_xq, 16) || !aligned(expert_scales, 4) || !aligned(topk_idx, 4))
      return MOE_EINVAL;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (c.num_tokens > 0 && dispatch_fp8_uses_route_pack(ctx)) {
    const bool timed = ctx->kernel_events != 0;
    if (timed && cudaEventRecord(ctx->ev[0], s) != cudaSuccess) return MOE_ECUDA;
    const int frc = enqueue_route_pack_fp8(ctx, x, topk_idx, expert_xq, expert_scales, expert_rows, s);
    if (frc != MOE_OK) return frc;
    if (timed && cudaEventRecord(ctx->ev[1], s) != cudaSuccess) return MOE_ECUDA;
    ctx->pack_timed = timed;
    ctx->dense_cap = 0;
    ctx->phase = kDispatched;
    return MOE_OK;
  }
  const int rrc = enqueue_routing(ctx, topk_idx, s);
  if (rrc != MOE_OK) return rrc;
  if (c.num_tokens > 0) {
    moe::PackFp8Params fp = {};
    fp.x = static_cast<const uint8_t*>(x);
    fp.expert_xq = static_cast<uint8_t*>(expert_xq);
    fp.expert_scales = expert_scales;
    fp.slot_row = ctx->slot_row;
    fp.error_word = ctx->error_word;
    fp.T = c.num_tokens;
    fp.K = c.top_k;
    fp.H = c.hidden;
    fp.dst_rows = expert_rows;
    // MOE_OPT_PACK_STAGES / _CTAS_PER_SM apply here too.  Automatic, K >= 4:
    // about 72 KiB of row stages per CTA, three CTAs (12 consumer warps) per
    // SM.  K < 4: each token row carries little write traffic for the
    // quantisation work it needs, so more CTAs work on tokens side by side:
    // three stages, up to eight CTAs per SM (measured on GB300, Mixtral-sized
    // layers: 8 % faster per layer than three CTAs).
    const bool few_dest = c.top_k < 4;
    int stages = ctx->pack_stages > 0 ? ctx->pack_stages
                 : few_dest         ? 3
                                    : static_cast<int>((72 * 1024) / (static_cast<int64_t>(c.hidden) * 2));
    const int maxst = moe::pack_fp8_max_stages();
    if (stages > maxst) stages = maxst;
    if (stages < 2) stages = 2;
    while (stages > 2 && moe::pack_fp8_smem_bytes(stages, c.hidden) > static_cast<size_t>(ctx->max_smem_optin))
      --stages;
    const size_t smem = moe::pack_fp8_smem_bytes(stages, c.hidden);
    int per_sm = moe::smem_ctas_per_sm(smem);
    const int want = ctx->pack_ctas_per_sm > 0 ? ctx->pack_ctas_per_sm : (few_dest ? 8 : 3);
    if (per_sm > want) per_sm = want;
    if (per_sm < 1) per_sm = 1;
    // Token queue (MOE_OPT_PACK_SCHEDULE; strided order only): automatic when a
    // CTA has more than three prologues (`stages` tokens) of work; the static
    // split otherwise, or if the queue's larger shared-memory header would not
    // fit.  Measured on GB300 (A/B, one box): Kimi-sized fp8 layer 543.1 ->
    // 520.9 us with the queue; DeepSeek-sized (9 tokens per CTA, 5 stages)
    // 139.1 -> 140.4 and Mixtral-sized 34.2 -> 35.0, so those stay static.
    if (ctx->fp8_order == 1 && ctx->pack_schedule != 0 &&
        moe::pack_fp8_smem_bytes(stages, c.hidden, true) <= static_cast<size_t>(ctx->max_smem_optin)) {
      int64_t grid = static_cast<int64_t>(grid_sms(ctx)) * per_sm;
      if (grid > c.num_tokens) grid = c.num_tokens;
      if (ctx->pack_schedule == 1 || static_cast<int64_t>(c.num_tokens) > 3 * static_cast<int64_t>(stages) * grid)
        fp.queue = ctx->queue;
    }
    const bool timed = ctx->kernel_events != 0;
    if (timed && cudaEventRecord(ctx->ev[0], s) != cudaSuccess) return MOE_ECUDA;
    if (moe::launch_dispatch_pack_fp8(fp, grid_sms(ctx), per_sm, stages, ctx->pdl != 0, ctx->fp8_order == 1, s) !=
        cudaSuccess)
      return MOE_ECUDA;
    if (timed && cudaEventRecord(ctx->ev[1], s) != cudaSuccess) return MOE_ECUDA;
    ctx->pack_timed = timed;
  }
  ctx->dense_cap = 0;
  ctx->phase = kDispatched;
  return MOE_OK;
}

MOE_API int moe_dispatch_recv(moe_ctx* ctx, moe_dispatch_layout* layout, void* stream) {
  (void)stream;
  if (!ctx || !layout) return MOE_EINVAL;
  if (ctx->phase != kDispatched) return MOE_ESTATE;
  layout->expert_counts = ctx->expert_counts;
  layout->expert_offsets = ctx->expert_offsets;
  layout->src_offsets = ctx->src_offsets;
  layout->rank_offsets = ctx->rank_offsets;
  layout->slot_row = ctx->slot_row;
  layout->row_src = ctx->row_src;
  layout->error_word = ctx->error_word;
  layout->rows = static_cast<int64_t>(ctx->cfg.num_tokens) * ctx->cfg.top_k;
  int64_t bound = 0;
  moe_recv_bound_rows(&ctx->cfg, &bound);
  layout->recv_bound_rows = bound;
  ctx->phase = kReceived;
  return MOE_OK;
}

MOE_API int moe_combine_send(moe_ctx* ctx, const void* expert_y, int64_t expert_y_rows, void* stream) {
  (void)stream;
  if (!ctx) return MOE_EINVAL;
  if (ctx->phase != kReceived) return MOE_ESTATE;
  const moe_config& c = ctx->cfg;
  if (expert_y_rows < static_cast<int64_t>(c.num_tokens) * c.top_k) return MOE_EINVAL;
  if (c.num_tokens > 0 && (!expert_y || !aligned(expert_y, 16))) return MOE_EINVAL;
  ctx->expert_y = expert_y;
  ctx->expert_y_rows = expert_y_rows;
  ctx->phase = kCombineSent;
  return MOE_OK;
}

namespace {

// Enqueues the receiver-only combine of the context's variant:
//   out[t] = bf16( fma chain over k of w[t,k] * y[table[t*K+k]] )
// with table the grouped rows (slot_row) or, for the dense all-to-all, the
// rows of the returned blocks.  MOE_OK, MOE_EINVAL or MOE_ECUDA.
int enqueue_combine(moe_ctx* ctx, const void* y, int64_t y_rows, const int32_t* table, const float* topk_w, void* out,
                    cudaStream_t cs) {
  const moe_config& c = ctx->cfg;
  moe::CombineParams cp = {};
  cp.y = static_cast<const uint8_t*>(y);
  cp.w = topk_w;
  cp.slot_row = table;
  cp.out = static_cast<uint8_t*>(out);
  cp.T = c.num_tokens;
  cp.K = c.top_k;
  cp.H = c.hidden;
  cp.y_rows = y_rows;
  cp.error_word = ctx->error_word;
  moe::CombineLaunch cl = {};
  cl.pdl = ctx->pdl != 0;
  cl.variant = combine_variant_of(ctx);
  cl.grid = 0;
  cl.sms = grid_sms(ctx);
  if (cl.variant == moe::kCombineBulk) {
    // By default the CTAs take tokens in the strided order (the leftover
    // tokens split evenly by pieces) with pieces of up to 4 KiB; measured on
    // GB300 against a contiguous range with 2 KiB pieces: DeepSeek-sized
    // layers 169.6 -> 167.6 us, Kimi-sized 700 -> 680 us, the worst case
    // 352 -> 344 us.  (The strided order with 2 KiB pieces was slower.)
    const bool strided = ctx->combine_order != 0;
    cl.shape = moe::combine_bulk_shape(c.hidden, c.top_k, ctx->combine_stages, ctx->combine_piece_bytes,
                                       ctx->max_smem_optin, strided ? 4096 : 2048);
    cl.shape.hints = ctx->cache_hints;
    cl.shape.drop_unit = ctx->test_drop_unit;
    // Token queue (MOE_OPT_COMBINE_SCHEDULE; default on, not with the
    // failure-injection hook).  Measured on GB300 (A/B, one box) against the
    // strided static order: DeepSeek-sized layer 162.7 -> 160.4 us,
    // Kimi-sized 659.2 -> 645.0, worst case 325.0 -> 318.1.  Claiming single
    // (token, piece) units instead was slower than the static order
    // (DeepSeek 164.0 -> 168.3, Kimi 661 -> 702): pieces of one token read
    // by different CTAs at once lose the row locality of one CTA streaming
    // a token's K rows piece after piece.
    cl.shape.queue = ctx->combine_schedule != 0 && ctx->test_drop_unit < 0 ? 1 : 0;
    if (cl.shape.queue && moe::combine_bulk_smem_bytes(cl.shape, c.top_k) > static_cast<size_t>(ctx->max_smem_optin))
      cl.shape.queue = 0;
    if (cl.shape.queue) cp.queue = ctx->queue + 1;
    const size_t smem = moe::combine_bulk_smem_bytes(cl.shape, c.top_k);
    if (smem > static_cast<size_t>(ctx->max_smem_optin)) return MOE_EINVAL;
    const int fit = moe::smem_ctas_per_sm(smem);
    int per_sm = ctx->combine_ctas_per_sm > 0 && ctx->combine_ctas_per_sm < fit ? ctx->combine_ctas_per_sm : fit;
    if (per_sm < 1) per_sm = 1;
    const int64_t units = static_cast<int64_t>(c.num_tokens) * cl.shape.pieces;
    int64_t grid = static_cast<int64_t>(grid_sms(ctx)) * per_sm;
    if (grid > units) grid = units;
    cl.grid = static_cast<int>(grid);
    cl.shape.strided = strided ? 1 : 0;
  }
  if (moe::launch_combine(cp, cl, cs) != cudaSuccess) return MOE_ECUDA;
  return MOE_OK;
}

}  // namespace

MOE_API int moe_combine_recv(moe_ctx* ctx, const float* topk_w, void* out, void* stream) {
  NvtxRange nvtx_range("moe_combine_recv");
  if (!ctx) return MOE_EINVAL;
  if (ctx->phase != kCombineSent) return MOE_ESTATE;
  const moe_config& c = ctx->cfg;
  if (c.num_tokens > 0) {
    if (!topk_w || !out || !aligned(topk_w, 4) || !aligned(out, 16)) return MOE_EINVAL;
    const bool timed = ctx->kernel_events != 0;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    if (timed && cudaEventRecord(ctx->ev[2], cs) != cudaSuccess) return MOE_ECUDA;
    const int rc = enqueue_combine(ctx, ctx->expert_y, ctx->expert_y_rows, ctx->slot_row, topk_w, out, cs);
    if (rc != MOE_OK) return rc;
    if (timed && cudaEventRecord(ctx->ev[3], cs) != cudaSuccess) return MOE_ECUDA;
    ctx->combine_timed = timed;
  }
  ctx->expert_y = nullptr;
  ctx->phase = kIdle;
  return MOE_OK;
}

MOE_API int moe_dense_capacity(const moe_config* cfg, int64_t* rows) {
  if (!rows) return MOE_EINVAL;
  const int rc = moe_validate_config(cfg);
  if (rc) return rc;
  const int64_t Tr = cfg->num_tokens / cfg->num_ranks;
  const int64_t L = cfg->num_experts / cfg->num_ranks;
  const int64_t cap = Tr * (cfg->top_k < L ? cfg->top_k : L);
  *rows = cap > 0 ? cap : 1;
  return MOE_OK;
}

namespace {

// Argument checks shared by the dense dispatch and combine: capacity at
// least moe_dense_capacity, row indices of N*N*capacity within int32, both
// block buffers that large and 16-byte aligned.
int check_dense_args(const moe_ctx* ctx, int64_t capacity, const void* send_buf, const void* recv_buf,
                     int64_t buf_rows) {
  const moe_config& c = ctx->cfg;
  int64_t need = 0;
  if (moe_dense_capacity(&c, &need) != MOE_OK) return MOE_EINVAL;
  if (capacity < need) return MOE_EINVAL;
  const int64_t rows = static_cast<int64_t>(c.num_ranks) * c.num_ranks * capacity;
  if (rows > INT32_MAX || buf_rows < rows) return MOE_EINVAL;
  if (c.num_tokens > 0 && (!send_buf || !recv_buf || !aligned(send_buf, 16) || !aligned(recv_buf, 16)))
    return MOE_EINVAL;
  return MOE_OK;
}

}  // namespace

MOE_API int moe_dispatch_send_dense(moe_ctx* ctx, const void* x, const int32_t* topk_idx, int64_t capacity,
                                    void* send_buf, void* recv_buf, int64_t buf_rows, void* expert_x,
                                    int64_t expert_x_rows, void* stream) {
  NvtxRange nvtx_range("moe_dispatch_send_dense");
  if (!ctx) return MOE_EINVAL;
  if (ctx->phase != kIdle) return MOE_ESTATE;
  const moe_config& c = ctx->cfg;
  const int64_t pairs = static_cast<int64_t>(c.num_tokens) * c.top_k;
  const int arc = check_dense_args(ctx, capacity, send_buf, recv_buf, buf_rows);
  if (arc != MOE_OK) return arc;
  if (expert_x_rows < pairs) return MOE_EINVAL;
  if (c.num_tokens > 0) {
    if (!x || !topk_idx || !expert_x) return MOE_EINVAL;
    if (!aligned(x, 16) || !aligned(expert_x, 16) || !aligned(topk_idx, 4)) return MOE_EINVAL;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int rrc = enqueue_routing(ctx, topk_idx, s);
  if (rrc != MOE_OK) return rrc;
  if (c.num_tokens > 0) {
    const int64_t row_bytes = static_cast<int64_t>(c.hidden) * 2;
    moe::DenseLayoutParams lp = {};
    lp.topk_idx = topk_idx;
    lp.slot_row = ctx->slot_row;
    lp.src_offsets = ctx->src_offsets;
    lp.expert_offsets = ctx->expert_offsets;
    lp.send_pos = ctx->send_pos;
    lp.recv_pos = ctx->send_dest;
    lp.T = c.num_tokens;
    lp.K = c.top_k;
    lp.E = c.num_experts;
    lp.N = c.num_ranks;
    lp.cap = capacity;
    lp.error_word = ctx->error_word;
    if (moe::launch_dense_layout(lp, ctx->num_sms, ctx->pdl != 0, s) != cudaSuccess) return MOE_ECUDA;
    // Senders: every token row to its K block rows.
    int prc = enqueue_pack(ctx, x, send_buf, buf_rows, ctx->send_pos, c.num_tokens, c.top_k, row_bytes,
                           ctx->pdl != 0, true, -1, s);
    if (prc != MOE_OK) return prc;
    // The exchange: every block whole.
    moe::DenseA2aParams ap = {};
    ap.in = static_cast<const uint8_t*>(send_buf);
    ap.out = static_cast<uint8_t*>(recv_buf);
    ap.N = c.num_ranks;
    ap.cap = capacity;
    ap.row_bytes = row_bytes;
    ap.error_word = ctx->error_word;
    if (moe::launch_dense_a2a(ap, ctx->num_sms, ctx->pdl != 0, s) != cudaSuccess) return MOE_ECUDA;
    // Receivers: block rows into the grouped rows.
    moe::RowMoveParams mp = {};
    mp.src = static_cast<const uint8_t*>(recv_buf);
    mp.dst = static_cast<uint8_t*>(expert_x);
    mp.src_row = ctx->send_dest;
    mp.dst_row = ctx->slot_row;
    mp.n = pairs;
    mp.row_bytes = row_bytes;
    mp.src_rows = buf_rows;
    mp.dst_rows = expert_x_rows;
    mp.error_word = ctx->error_word;
    if (moe::launch_row_move(mp, ctx->num_sms, ctx->pdl != 0, s) != cudaSuccess) return MOE_ECUDA;
  }
  ctx->pack_timed = false;
  ctx->phase = kDispatched;
  ctx->dense_cap = capacity;
  return MOE_OK;
}

MOE_API int moe_combine_recv_dense(moe_ctx* ctx, const float* topk_w, int64_t capacity, void* send_buf,
                                   void* recv_buf, int64_t buf_rows, void* out, void* stream) {
  NvtxRange nvtx_range("moe_combine_recv_dense");
  if (!ctx) return MOE_EINVAL;
  if (ctx->phase != kCombineSent || ctx->dense_cap == 0) return MOE_ESTATE;
  if (capacity != ctx->dense_cap) return MOE_EINVAL;
  const int arc = check_dense_args(ctx, capacity, send_buf, recv_buf, buf_rows);
  if (arc != MOE_OK) return arc;
  const moe_config& c = ctx->cfg;
  if (c.num_tokens > 0) {
    if (!topk_w || !out || !aligned(topk_w, 4) || !aligned(out, 16)) return MOE_EINVAL;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int64_t row_bytes = static_cast<int64_t>(c.hidden) * 2;
    // Each expert rank's outputs into the blocks they came in by.
    moe::RowMoveParams mp = {};
    mp.src = static_cast<const uint8_t*>(ctx->expert_y);
    mp.dst = static_cast<uint8_t*>(send_buf);
    mp.src_row = ctx->slot_row;
    mp.dst_row = ctx->send_dest;
    mp.n = static_cast<int64_t>(c.num_tokens) * c.top_k;
    mp.row_bytes = row_bytes;
    mp.src_rows = ctx->expert_y_rows;
    mp.dst_rows = buf_rows;
    mp.error_word = ctx->error_word;
    if (moe::launch_row_move(mp, ctx->num_sms, ctx->pdl != 0, s) != cudaSuccess) return MOE_ECUDA;
    // The exchange back: block r*N+s to block s*N+r, every block whole.
    moe::DenseA2aParams ap = {};
    ap.in = static_cast<const uint8_t*>(send_buf);
    ap.out = static_cast<uint8_t*>(recv_buf);
    ap.N = c.num_ranks;
    ap.cap = capacity;
    ap.row_bytes = row_bytes;
    ap.error_word = ctx->error_word;
    if (moe::launch_dense_a2a(ap, ctx->num_sms, ctx->pdl != 0, s) != cudaSuccess) return MOE_ECUDA;
    // The receiver-only combine over the returned rows.
    const int rc = enqueue_combine(ctx, recv_buf, buf_rows, ctx->send_pos, topk_w, out, s);
    if (rc != MOE_OK) return rc;
  }
  ctx->combine_timed = false;
  ctx->expert_y = nullptr;
  ctx->phase = kIdle;
  return MOE_OK;
}

MOE_API int moe_partial_rows(const moe_config* cfg, int64_t* rows) {
  if (!cfg || !rows) return MOE_EINVAL;
  const int st = moe_validate_config(cfg);
  if (st != MOE_OK) return st;
  const int32_t s = cfg->top_k < cfg->num_ranks ? cfg->top_k : cfg->num_ranks;
  *rows = static_cast<int64_t>(cfg->num_tokens) * s;
  return MOE_OK;
}

MOE_API int moe_combine_recv_two_level(moe_ctx* ctx, const float* topk_w, void* partial, int64_t partial_rows,
                                       void* out, void* stream) {
  NvtxRange nvtx_range("moe_combine_recv_two_level");
  if (!ctx) return MOE_EINVAL;
  if (ctx->phase != kCombineSent) return MOE_ESTATE;
  const moe_config& c = ctx->cfg;
  if (c.num_tokens > 0) {
    int64_t need = 0;
    moe_partial_rows(&c, &need);
    if (partial_rows < need) return MOE_EINVAL;
    if (!topk_w || !out || !partial || !aligned(topk_w, 4) || !aligned(out, 16) || !aligned(partial, 16))
      return MOE_EINVAL;
    moe::TwoLevelParams tp = {};
    tp.y = static_cast<const uint8_t*>(ctx->expert_y);
    tp.w = topk_w;
    tp.slot_row = ctx->slot_row;
    tp.rank_offsets = ctx->rank_offsets;
    tp.partial = static_cast<uint8_t*>(partial);
    tp.out = static_cast<uint8_t*>(out);
    tp.plan_row = ctx->plan_row;
    tp.plan_w = ctx->plan_w;
    tp.plan_mask = ctx->plan_mask;
    tp.T = c.num_tokens;
    tp.K = c.top_k;
    tp.H = c.hidden;
    tp.N = c.num_ranks;
    tp.y_rows = ctx->expert_y_rows;
    tp.error_word = ctx->error_word;
    if (moe::launch_combine_two_level(tp, ctx->pdl != 0, static_cast<cudaStream_t>(stream)) != cudaSuccess)
      return MOE_ECUDA;
  }
  ctx->combine_timed = false;  // the event-timed combine is that of moe_combine_recv only
  ctx->expert_y = nullptr;
  ctx->phase = kIdle;
  return MOE_OK;
}

MOE_API int moe_kernel_times(moe_ctx* ctx, float* pack_ms, float* combine_ms) {
  if (!ctx || !pack_ms || !combine_ms) return MOE_EINVAL;
  *pack_ms = -1.0f;
  *combine_ms = -1.0f;
  if (ctx->pack_timed) {
    if (cudaEventSynchronize(ctx->ev[1]) != cudaSuccess) return MOE_ECUDA;
    if (cudaEventElapsedTime(pack_ms, ctx->ev[0], ctx->ev[1]) != cudaSuccess) return MOE_ECUDA;
  }
  if (ctx->combine_timed) {
    if (cudaEventSynchronize(ctx->ev[3]) != cudaSuccess) return MOE_ECUDA;
    if (cudaEventElapsedTime(combine_ms, ctx->ev[2], ctx->ev[3]) != cudaSuccess) return MOE_ECUDA;
  }
  return MOE_OK;
}

MOE_API int moe_get_error(moe_ctx* ctx, void* stream) {
  if (!ctx) return MOE_EINVAL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t h = MOE_OK;
  if (cudaMemcpyAsync(&h, ctx->error_word, sizeof h, cudaMemcpyDeviceToHost, s) != cudaSuccess) return MOE_ECUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ECUDA;
  return h;
}

MOE_API const char* moe_strerror(int status) {
  switch (status) {
    case MOE_OK:
      return "ok";
    case MOE_EINVAL:
      return "invalid argument (null or misaligned pointer, or unsupported sizes)";
    case MOE_ESTATE:
      return "call out of order: dispatch_send -> dispatch_recv -> combine_send -> combine_recv";
    case MOE_EROUTE:
      return "expert index out of range or repeated within one token";
    case MOE_ECUDA:
      return "CUDA runtime or launch failure";
    case MOE_EBOUND:
      return "a logical rank would receive more rows than N*T/N*max(K,E/N)";
    case MOE_ECORRUPT:
      return "a routing-table entry points outside its buffer (checked build)";
    case MOE_ETIMEDOUT:
      return "a bounded wait inside a kernel gave up";
    default:
      return "unknown status";
  }
}
