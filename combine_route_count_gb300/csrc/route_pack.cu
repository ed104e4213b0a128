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
// runs P pack CTAs per SM; one routing per SM instead of P).  Steps 1-4 are
// the per-CTA routing of route_tables.cuh, shared with route_pack_fp8:
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
// CTA reaches the same decision on a malformed routing, so after a routing
// error no CTA copies anything and every slot_row entry becomes -1 (the
// combine then writes nothing).

#include <cuda_runtime.h>

#include "moe_kernels.cuh"
#include "ptx.cuh"
#include "route_tables.cuh"

namespace moe {
namespace {

constexpr int kMaxStages = 16;
constexpr int kBarBytes = 512;  // mbarriers: copy warps' stages (<= 63), then the index copy's
constexpr int kIdxBar = kBarBytes / 8 - 1;
using rtab::index_bytes;
using rtab::tables_bytes;
using rtab::wait_phase;

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
  const int T = p.T, K = p.K, E = p.E;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, W = blockDim.x >> 5;
  const bool copier = warp < copy_warps;
  // This warp's stage ring and mbarriers (copy warps only).
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem) + (copier ? warp * stages : 0);
  uint8_t* stage_buf = smem + kBarBytes + (copier ? static_cast<size_t>(warp) * stages * p.piece_bytes : 0);
  const rtab::Tables tb =
      rtab::carve_tables(smem + kBarBytes + static_cast<size_t>(copy_warps) * stages * p.piece_bytes, T, E);
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
  rtab::start_index_copy(p, sidx, idx_bar, bulk_ints, 32 * (W - 1));
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

  // 1.-4. the routing tables, the CTA's slot_row / row_src entries and (CTA 0)
  // the counts, offsets and status.
  const bool bad = __syncthreads_or(rtab::token_masks<KMAX>(sidx, tb, T, K, E));
  rtab::expert_scans(tb, E);
  rtab::write_routing(p, tb, sidx, bad);
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
        const int my_row = lane < K ? rtab::row_of(tb, t, sidx[t * K + lane]) : -1;
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
    return lane < K ? rtab::row_of(tb, tt, sidx[tt * K + lane]) : -1;
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
