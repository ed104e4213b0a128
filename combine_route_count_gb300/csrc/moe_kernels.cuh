// Internal interface between the C ABI (moe_abi.cu) and the three kernels.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>
#include <utility>

#include "moe.h"

namespace moe {

// Checked builds (compiled with -DMOE_CHECKED, libmoe_checked.so) verify every
// row index read from a routing table against the buffer it addresses before
// using it; an entry out of range sets MOE_ECORRUPT in the error word and the
// access is skipped.  In the normal build the checks are constant-false and
// compile away.
#ifdef MOE_CHECKED
constexpr bool kChecked = true;
#else
constexpr bool kChecked = false;
#endif

// ---- route_count: counts, exclusive scan, stable slot ranks (one block) ----
struct RouteCountParams {
  const int32_t* topk_idx;  // [T, K]
  int32_t T, K, E, N;
  int32_t* expert_counts;   // [E]
  int32_t* expert_offsets;  // [E+1]
  int32_t* src_offsets;     // [E*N]
  int32_t* rank_offsets;    // [N+1]
  int32_t* slot_row;        // [T*K]
  int32_t* row_src;         // [T*K]
  int32_t* error_word;      // [1]
  unsigned long long* queue;  // [2] the pack's and the combine's unit queues: set to 0 here (may be null)
};
constexpr int kRouteThreads = 1024;
// Dynamic shared memory the kernel needs for E experts.
size_t route_count_smem_bytes(int E);
// idx_vec: 4, 2 or 1 int32 per load (K % idx_vec == 0, topk_idx aligned to 4*idx_vec bytes).
cudaError_t launch_route_count(const RouteCountParams& p, int idx_vec, cudaStream_t stream);

// ---- route_local + route_finalize: the same results from many blocks --------
constexpr int kSplitThreads = 256;    // tokens per sub-chunk (one per thread)
constexpr int kMaxSplitBlocks = 128;  // chunks (blocks) at most; workspace holds kMaxSplitBlocks*E counts
struct RouteSplitParams {
  const int32_t* topk_idx;  // [T, K]
  int32_t T, K, E, N;
  int32_t chunk;            // tokens per block, a multiple of kSplitThreads
  int32_t* expert_counts;   // [E]
  int32_t* expert_offsets;  // [E+1]
  int32_t* src_offsets;     // [E*N]
  int32_t* rank_offsets;    // [N+1]
  int32_t* slot_row;        // [T*K]
  int32_t* row_src;         // [T*K]
  int32_t* error_word;      // [1]
  unsigned long long* queue;  // [2] the pack's and the combine's unit queues: set to 0 here (may be null)
  int32_t* hist;            // [blocks*E] per-chunk expert histograms
  int32_t* block_err;       // [blocks]   per-chunk routing error flags
};
size_t route_local_smem_bytes(int E);
int route_split_chunk(int T);
cudaError_t launch_route_split(const RouteSplitParams& p, int idx_vec, cudaStream_t stream);

// ---- route_cluster: the same results from one cluster of <= 16 CTAs ---------
constexpr int kClusterThreads = 1024;
constexpr int kMaxClusterCtas = 16;
struct RouteClusterParams {
  const int32_t* topk_idx;  // [T, K]
  int32_t T, K, E, N;
  int32_t chunk;            // tokens per CTA (multiple of 32)
  int32_t warps;            // warps of tokens per sub-chunk (<= 32)
  int32_t staged;           // 1: one sub-chunk per CTA, row_src staged in shared memory
  int32_t dsmem_group;      // threads per expert in the histogram exchange (power of 2, <= 16)
  int32_t* expert_counts;   // [E]
  int32_t* expert_offsets;  // [E+1]
  int32_t* src_offsets;     // [E*N]
  int32_t* rank_offsets;    // [N+1]
  int32_t* slot_row;        // [T*K]
  int32_t* row_src;         // [T*K]
  int32_t* error_word;      // [1]
  unsigned long long* queue;  // [2] the pack's and the combine's unit queues: set to 0 here (may be null)
};
size_t route_cluster_smem_bytes(int E, int warps, int staged_pairs);
// Fills chunk/warps/staged/dsmem_group of p for a cluster of `cluster` CTAs.
void route_cluster_plan(RouteClusterParams* p, int cluster, int max_smem);
void route_cluster_shape(int T, int E, int max_cluster, int* cluster, int* chunk, int* warps);
bool route_cluster_supported(const RouteClusterParams& p, int idx_vec, int cluster);
cudaError_t launch_route_cluster(const RouteClusterParams& p, int idx_vec, int cluster, cudaStream_t stream);

// ---- dispatch_pack: expert_x[slot_row[t,k]] = x[t] --------------------------
// Routing and pack in one kernel, for small layers (route_pack.cu): one CTA
// per SM computes the whole routing from topk_idx in shared memory, then
// `copy_warps` of its warps each copy units through their own stage ring.
constexpr int kRoutePackThreads = 1024;  // largest block; 256 for layers of at most 32 token words
constexpr int kRoutePackMaxPairs = 16384;     // T*K: index reads per CTA
constexpr int kRoutePackMaxMaskWords = 4096;  // E*ceil(T/32): token-mask words per CTA
struct RoutePackParams {
  const int32_t* topk_idx;  // [T, K]
  const uint8_t* x;         // [T, row_bytes]
  uint8_t* expert_x;        // [dst_rows, row_bytes]
  int32_t T, K, E, N;
  int64_t row_bytes;        // multiple of 16
  int32_t piece_bytes;      // bytes moved per unit (multiple of 16, <= row_bytes)
  int32_t pieces;           // ceil(row_bytes / piece_bytes)
  int64_t dst_rows;         // rows of expert_x (checked builds)
  int32_t* expert_counts;   // [E]
  int32_t* expert_offsets;  // [E+1]
  int32_t* src_offsets;     // [E*N]
  int32_t* rank_offsets;    // [N+1]
  int32_t* slot_row;        // [T*K]
  int32_t* row_src;         // [T*K]
  int32_t* error_word;      // [1]
  unsigned long long* queue;  // [2] the pack's and the combine's queues: set to 0 here (may be null)
};
struct RoutePackLaunch {
  int grid;        // CTAs (at most one per SM)
  int threads;     // block size: 256 or kRoutePackThreads (a multiple of 32, >= 32 * copy_warps)
  bool vec;        // rows through registers instead of stages (route_pack_vec_ok); stages unused
  int copy_warps;  // warps per CTA that copy, each a virtual pack CTA (0..8; 0: routing only)
  int stages;      // shared-memory stages per copy warp (2..route_pack_max_stages)
  int hints;   // CacheHints
  int depth;   // store groups in flight before a stage is refilled
  bool pdl;    // launch with programmatic stream serialization
};
size_t route_pack_tables_bytes(int T, int E);
size_t route_pack_smem_bytes(int T, int K, int E, int copy_warps, int stages, int piece_bytes);
int route_pack_max_stages(int copy_warps);
// Rows small and few enough per copy warp to go through registers.
bool route_pack_vec_ok(int64_t row_bytes, int64_t units_per_warp);
bool route_pack_eligible(int T, int K, int E);
cudaError_t prepare_route_pack(int max_smem_bytes);  // one-time per-device attribute setup
cudaError_t launch_route_pack(const RoutePackParams& p, const RoutePackLaunch& l, cudaStream_t stream);

// ---- route_pack_fp8: routing and the fp8 pack in one kernel (small layers) ----
struct RoutePackFp8Params {
  const int32_t* topk_idx;  // [T, K]
  const uint8_t* x;         // bf16 [T, H]
  uint8_t* expert_xq;       // e4m3 [dst_rows, H]
  float* expert_scales;     // [dst_rows, H/128]
  int32_t T, K, E, N, H;    // H % 128 == 0
  int64_t dst_rows;         // rows of expert_xq / expert_scales (checked builds)
  int32_t* expert_counts;   // [E]
  int32_t* expert_offsets;  // [E+1]
  int32_t* src_offsets;     // [E*N]
  int32_t* rank_offsets;    // [N+1]
  int32_t* slot_row;        // [T*K]
  int32_t* row_src;         // [T*K]
  int32_t* error_word;      // [1]
  unsigned long long* queue;  // [2] set to 0 here (may be null)
};
constexpr int kRoutePackFp8GroupThreads = 128;  // threads quantising one row together
size_t route_pack_fp8_smem_bytes(int T, int K, int E, int H, int groups, int stages);
int route_pack_fp8_max_stages(int groups);
cudaError_t prepare_route_pack_fp8(int max_smem_bytes);
// grid CTAs of groups * 128 threads (groups 1..8), `stages` whole-row stages per group.
cudaError_t launch_route_pack_fp8(const RoutePackFp8Params& p, int grid, int groups, int stages, bool pdl,
                                  cudaStream_t stream);

struct PackParams {
  const uint8_t* x;         // [T, row_bytes]
  uint8_t* expert_x;        // [rows, row_bytes]
  const int32_t* slot_row;  // [T*K]
  int32_t* error_word;
  int32_t T, K;
  int64_t row_bytes;        // H * 2, multiple of 16
  int32_t piece_bytes;      // bytes moved per unit (multiple of 16, <= row_bytes)
  int32_t pieces;           // ceil(row_bytes / piece_bytes)
  int64_t dst_rows;         // rows of expert_x (checked builds verify every table entry against it)
  unsigned long long* queue;  // [1] unit queue of the dynamic schedule, 0 at launch (set by routing)
};
enum PackVariant { kPackBulk = 0, kPackVector = 1 };
// L2 eviction hints on the bulk copies (bit flags, MOE_OPT_CACHE_HINTS).
enum CacheHints { kHintPackLoads = 1, kHintPackStores = 2, kHintCombineLoads = 4 };
struct PackLaunch {
  int variant;    // PackVariant
  int grid;       // CTAs
  int stages;     // bulk: shared-memory stages per CTA (2..8)
  bool pdl;       // launch with programmatic stream serialization
  int prefetch;   // bulk: 0 = off, 1 = prefetch the CTA's later rows into L2 in the prologue, 2 = same, evict-last
  int hints;      // CacheHints
  int depth;      // bulk: store groups in flight before a stage is refilled (0 = default 1)
  int prefetch_units;  // bulk: units past the prologue each CTA prefetches (-1 = all)
  bool dynamic;        // bulk: after its first `stages` units a CTA claims units from p.queue
};
size_t pack_bulk_smem_bytes(int stages, int piece_bytes);
cudaError_t prepare_pack(int max_smem_bytes);  // one-time per-device attribute setup
cudaError_t launch_dispatch_pack(const PackParams& p, const PackLaunch& l, cudaStream_t stream);

// ---- dispatch_pack_fp8: block-scaled E4M3 payload ---------------------------
struct PackFp8Params {
  const uint8_t* x;         // bf16 [T, H]
  uint8_t* expert_xq;       // e4m3 [rows, H]
  float* expert_scales;     // [rows, H/128]
  const int32_t* slot_row;  // [T*K]
  int32_t* error_word;
  int32_t T, K, H;          // H % 128 == 0
  int64_t dst_rows;         // rows of expert_xq / expert_scales (checked builds)
  unsigned long long* queue;  // [1] token queue, 0 at launch (set by routing); null: static split
};
size_t pack_fp8_smem_bytes(int stages, int H, bool queue = false);
int pack_fp8_max_stages();
// Persistent grid of up to sms x per_sm CTAs (fewer if fewer can be resident
// or T is smaller); with p.queue: each CTA's first `stages` tokens b, b+grid,
// ... then tokens claimed from the queue; else strided: CTA b packs tokens b,
// b+grid, ...; else one contiguous token range.
cudaError_t launch_dispatch_pack_fp8(const PackFp8Params& p, int sms, int per_sm, int stages, bool pdl, bool strided,
                                     cudaStream_t stream);

// ---- combine: out[t] = bf16(sum_k w[t,k] * y[slot_row[t,k]]) -----------------
struct CombineParams {
  const uint8_t* y;         // [rows, H] bf16
  const float* w;           // [T, K]
  const int32_t* slot_row;  // [T*K]
  uint8_t* out;             // [T, H] bf16
  int32_t* error_word;      // [1] bounded waits report MOE_ETIMEDOUT here
  int32_t T, K, H;
  int64_t y_rows;           // rows of y (checked builds verify slot_row against it)
  unsigned long long* queue;  // [1] unit queue of the bulk combine, 0 at launch (set by routing)
};
enum CombineVariant { kCombineBulk = 0, kCombineVector = 1 };
struct BulkCombineShape {
  int stages;          // shared-memory stages per CTA
  int piece_bytes;     // bytes of a row per unit (multiple of 16)
  int pieces;          // units per token
  int hints;           // CacheHints
  int64_t drop_unit;   // failure-injection hook: unit the producer never posts (-1: none)
  int strided;         // 1: a CTA takes tokens b, b+G, ...; 0: a contiguous unit range
  int queue;           // 1: units claimed from CombineParams::queue after the first `stages`
};
struct CombineLaunch {
  int variant;             // CombineVariant
  int grid;                // bulk: CTAs
  BulkCombineShape shape;  // bulk
  bool pdl;                // launch with programmatic stream serialization
  int sms;                 // vector: SMs the grid may spread over
};
size_t combine_bulk_smem_bytes(const BulkCombineShape& sh, int K);
// Stages and pieces of the bulk combine; piece_bytes <= 0 picks equal pieces
// of at most auto_piece_max bytes (a multiple of 16, at most 4096).
BulkCombineShape combine_bulk_shape(int H, int K, int stages, int piece_bytes, int max_smem, int auto_piece_max);
cudaError_t launch_combine(const CombineParams& p, const CombineLaunch& l, cudaStream_t stream);

// Two-stage dispatch: per-pair send rows and per-send-row grouped rows.
struct StagedLayoutParams {
  const int32_t* topk_idx;        // [T*K]
  const int32_t* slot_row;        // [T*K]
  const int32_t* expert_offsets;  // [E+1]
  const int32_t* src_offsets;     // [E*N]
  int32_t* send_pos;              // [T*K] send row of pair t*K+k (-1 after a routing error)
  int32_t* send_dest;             // [T*K] grouped row of send row j (-1 after a routing error)
  int32_t T, K, E, N;
  int32_t* error_word;            // checked builds report MOE_ECORRUPT here
};
cudaError_t launch_staged_layout(const StagedLayoutParams& p, bool pdl, cudaStream_t stream);

// Dense padded all-to-all (dense_a2a.cu): blocks of `cap` rows per
// (source rank, destination rank) pair.
struct DenseLayoutParams {
  const int32_t* topk_idx;        // [T*K]
  const int32_t* slot_row;        // [T*K] grouped row of each pair (-1 after a routing error)
  const int32_t* src_offsets;     // [E*N]
  const int32_t* expert_offsets;  // [E+1]
  int32_t* send_pos;              // [T*K] row (s*N+r)*cap+j of the pair in the send buffer, -1 if none
  int32_t* recv_pos;              // [T*K] row (r*N+s)*cap+j of the pair in the receive buffer, -1 if none
  int32_t T, K, E, N;
  int64_t cap;                    // rows per block, >= T/N * min(K, E/N)
  int32_t* error_word;            // checked builds report MOE_ECORRUPT here
};
cudaError_t launch_dense_layout(const DenseLayoutParams& p, int sms, bool pdl, cudaStream_t stream);
struct DenseA2aParams {
  const uint8_t* in;     // [N*N*cap, row_bytes]
  uint8_t* out;          // [N*N*cap, row_bytes]: block r*N+s = block s*N+r of in
  int32_t N;
  int64_t cap;
  int64_t row_bytes;     // multiple of 16
  const int32_t* error_word;  // MOE_EROUTE: nothing is copied (may be null)
};
cudaError_t launch_dense_a2a(const DenseA2aParams& p, int sms, bool pdl, cudaStream_t stream);
struct RowMoveParams {
  const uint8_t* src;
  uint8_t* dst;
  const int32_t* src_row;  // [n]
  const int32_t* dst_row;  // [n]; an entry < 0 in either table skips the row
  int64_t n;
  int64_t row_bytes;       // multiple of 16
  int64_t src_rows, dst_rows;  // buffer rows (checked builds verify the tables against them)
  int32_t* error_word;
};
cudaError_t launch_row_move(const RowMoveParams& p, int sms, bool pdl, cudaStream_t stream);

// Two-level combine (partial sums on the sending side, then on the receiver).
struct TwoLevelParams {
  const uint8_t* y;             // [rows, H] bf16
  const float* w;               // [T, K]
  const int32_t* slot_row;      // [T*K]
  const int32_t* rank_offsets;  // [N+1]
  uint8_t* partial;             // [T*min(K,N), H] bf16
  uint8_t* out;                 // [T, H] bf16
  int32_t* plan_row;            // [T*K] the token's grouped rows, sorted by (rank, k)
  float* plan_w;                // [T*K] their weights
  int32_t* plan_mask;           // [T] bit i: sorted slot i ends a rank's group (0: routing error)
  int32_t T, K, H, N;
  int64_t y_rows;               // rows of y (checked builds)
  int32_t* error_word;          // checked builds report MOE_ECORRUPT here
};
cudaError_t launch_combine_two_level(const TwoLevelParams& p, bool pdl, cudaStream_t stream);

// Raises a kernel's dynamic shared-memory limit to at least `bytes` (and, if
// asked, allows non-portable cluster sizes) on the current device.  Each
// (kernel, device) pair pays the runtime call once; later launches only look
// the pair up.
cudaError_t set_kernel_limits(const void* kernel, size_t bytes, bool nonportable_cluster = false);

// CTAs of `kernel` that can be resident on one SM with this block size and
// dynamic shared memory (0 if the query fails); cached per device.
int resident_ctas_per_sm(const void* kernel, int threads, size_t smem);

// CTAs with `smem` bytes of dynamic shared memory that fit on one SM of the
// current device (its shared memory per SM over smem plus the per-CTA
// reserve); at least 1, cached per device.
int smem_ctas_per_sm(size_t smem);

// Launch helper: plain or programmatic-dependent launch with cudaLaunchKernelEx.
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                          bool pdl, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  if (pdl) {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace moe
