// dispatch_pack: expert_x[slot_row[t, k]] = x[t] for every token t and slot k.
//
// "Enabling trillion-parameter models on AWS EFA" (Dispatch and combine):
// once the offsets are known, every token is packed into the send buffer at
// its offset.  "Efficient and portable mixture-of-experts communication"
// (Portable kernels; Dispatch): dispatch-send is parallelised over the tokens
// of a rank, and the receiver's layout is the grouped-GEMM input.  On one GPU
// the send buffer and the receive layout are the same memory, so one copy
// places each row directly ("Further improvements": shared buffers remove
// copies).
//
// Each token row is read from HBM once and written K times.  Work is split
// into units (token t, piece j of the row); CTA b takes units b, b+G, b+2G...
// (static split), or its first `stages` of those and then units claimed from
// a queue in the workspace (dispatch_pack_bulk_queue, below).
//
// Bulk variant (default): one warp per CTA drives the TMA engine.  Lane 0
// loads a piece into a shared-memory stage with cp.async.bulk (completion on
// an mbarrier), then lanes 0..K-1 each store the stage to one destination row
// with cp.async.bulk (bulk async-groups).  A stage is refilled once every
// lane's store group has finished reading it.  The first loads are issued
// before griddepcontrol.wait: token rows do not depend on route_count, so
// under programmatic dependent launch they overlap it.
//
// Vector variant: each warp copies a unit with 16-byte loads and K 16-byte
// stores per chunk, no shared memory.

#include <cuda_runtime.h>

#include "moe_kernels.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kMaxStages = 16;
constexpr int kBarBytes = 256;  // mbarriers, then the queue variant's stage_unit[kMaxStages]
constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s

__device__ __forceinline__ unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Bounded wait on an mbarrier phase.  False if it did not complete in time.
__device__ __forceinline__ bool wait_phase(uint64_t* bar, uint32_t parity) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const unsigned long long start = globaltimer();
  while (!ptx::mbar_try_wait(bar, parity)) {
    if (globaltimer() - start > kWaitLimitNs) return false;
  }
  return true;
}

// Waits until at most `depth` of this thread's bulk store groups still read
// shared memory (depth 0..7; wait_group takes an immediate).
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

__device__ __forceinline__ void report(int32_t* error_word, int status) {
  atomicCAS(error_word, MOE_OK, status);
}

__global__ void __launch_bounds__(32) dispatch_pack_bulk(PackParams p, int stages, int prefetch, int hints,
                                                          int depth, int prefetch_units) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem);
  uint8_t* stage_buf = smem + kBarBytes;
  const int lane = threadIdx.x;
  const int64_t units = static_cast<int64_t>(p.T) * p.pieces;
  const int64_t first = blockIdx.x;
  const int64_t step = gridDim.x;
  const int64_t mine = units > first ? (units - first + step - 1) / step : 0;

  if (lane == 0) {
    for (int s = 0; s < stages; ++s) ptx::mbar_init(&bars[s], 1);
    ptx::mbar_fence_init();
  }
  __syncwarp();

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

  // Token rows are ready before this grid starts: prefetch while the routing
  // kernel is still running.
  const int64_t prologue = mine < stages ? mine : stages;
  if (lane == 0)
    for (int64_t i = 0; i < prologue; ++i) issue_load(i);
  // At most prefetch_units units past the prologue (the soonest needed), so
  // that the prefetched rows fit in L2 next to the write stream.
  const int64_t pf_end =
      !prefetch ? prologue : (prefetch_units < 0 || prologue + prefetch_units > mine ? mine : prologue + prefetch_units);
  if (prefetch) {
    // The later rows of this CTA go to L2 now, while routing still runs.
    // prefetch == 2 marks them evict-last so that the write stream of this
    // kernel does not push them out before they are loaded; each piece is
    // handed back to normal priority as soon as it has been loaded.
    const uint64_t keep = prefetch == 2 ? ptx::policy_evict_last() : 0;
    for (int64_t i = prologue + lane; i < pf_end; i += 32) {
      const int64_t u = first + i * step;
      const int64_t t = u / p.pieces;
      const int j = static_cast<int>(u - t * p.pieces);
      const uint8_t* src = p.x + t * p.row_bytes + static_cast<int64_t>(j) * p.piece_bytes;
      if (prefetch == 2)
        ptx::bulk_prefetch_l2_hint(src, piece_bytes(j), keep);
      else
        ptx::bulk_prefetch_l2(src, piece_bytes(j));
    }
  }

  ptx::wait_prerequisites();  // slot_row is written by route_count

  int64_t i = 0;
  bool ok = true;
  // Destination rows are loaded one unit ahead, so that their latency is not
  // on the path of every unit (it matters when a unit has few stores).
  // Coherent loads: the table is written by the previous grid.
  auto dest_row = [&](int64_t unit_index) -> int {
    const int64_t tt = (first + unit_index * step) / p.pieces;
    return lane < p.K ? p.slot_row[tt * p.K + lane] : -1;
  };
  int next_row = mine > 0 ? dest_row(0) : -1;
  for (; i < mine; ++i) {
    const int64_t u = first + i * step;
    const int64_t t = u / p.pieces;
    const int j = static_cast<int>(u - t * p.pieces);
    const int s = static_cast<int>(i % stages);
    const int row = next_row;
    if (i + 1 < mine) next_row = dest_row(i + 1);
    // Every lane waits; the outcome is made warp-uniform so that no lane is
    // left behind at a later __syncwarp.
    const bool arrived = wait_phase(&bars[s], static_cast<uint32_t>((i / stages) & 1));
    if (!__all_sync(0xffffffffu, arrived)) {
      ok = false;
      break;
    }
    if (prefetch == 2 && i >= prologue && i < pf_end) {
      // This piece was prefetched evict-last; it is in shared memory now, so
      // hand its L2 lines back to normal priority.
      const uint8_t* src = p.x + t * p.row_bytes + static_cast<int64_t>(j) * p.piece_bytes;
      const uint32_t lines = (piece_bytes(j) + 127) / 128;
      for (uint32_t q = lane; q < lines; q += 32) ptx::l2_priority_normal(src + static_cast<size_t>(q) * 128);
    }
    int row_ok = row;
    if (kChecked && row >= 0 && row >= p.dst_rows) {
      report(p.error_word, MOE_ECORRUPT);
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
    // Refill the stage of unit r = i-depth+1 once every lane's stores of unit
    // r have read it; the store groups of the depth-1 later units stay in flight.
    const int64_t r = i - depth + 1;
    if (r >= 0 && r + stages < mine) {
      wait_reads_at_most(depth - 1);
      __syncwarp();
      if (lane == 0) issue_load(r + stages);
    }
  }
  if (!ok) {
    if (lane == 0) {
      report(p.error_word, MOE_ETIMEDOUT);
      // Loads issued so far: the prologue's [0, prologue) and, from the
      // refills of iterations up to i-1, units up to i-1-depth+1+stages.
      // Wait (bounded) for those not yet consumed before the CTA exits.
      int64_t last = prologue - 1;
      if (i - depth + stages > last) last = i - depth + stages;
      if (last > mine - 1) last = mine - 1;
      for (int64_t q = i; q <= last; ++q) wait_phase(&bars[q % stages], static_cast<uint32_t>((q / stages) & 1));
    }
    __syncwarp();
  }
  ptx::bulk_wait<0>();  // stores complete before shared memory goes away
}

// Bulk variant with a unit queue.  The static split above gives every CTA
// the same number of units, but CTAs do not progress at the same rate (their
// stores compete differently for DRAM), so some SMs finish long before the
// last.  Here CTA b still takes units b, b+G, ..., b+(stages-1)G (its
// prologue, loaded while routing runs), and the units from stages*G on are
// claimed in increasing order from a counter that the routing kernel sets to
// 0: CTAs that progress faster take more of them, the CTAs still work on a
// window of consecutive tokens, and a CTA runs out of work at most one unit
// after the others.  One claim is always in flight ahead of its use, so its
// latency overlaps a unit's copies.  stage_unit[] (shared memory) holds the
// unit loaded into each stage (-1: none, the end of this CTA's sequence).
__global__ void __launch_bounds__(32) dispatch_pack_bulk_queue(PackParams p, int stages, int prefetch, int hints,
                                                                int depth, int prefetch_units) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem);
  int64_t* stage_unit = reinterpret_cast<int64_t*>(smem + kMaxStages * sizeof(uint64_t));
  uint8_t* stage_buf = smem + kBarBytes;
  const int lane = threadIdx.x;
  const int64_t units = static_cast<int64_t>(p.T) * p.pieces;
  const int64_t G = gridDim.x;
  const int64_t static_end = static_cast<int64_t>(stages) * G;  // units [0, static_end) are split statically
  const int64_t static_units = units < static_end ? units : static_end;
  const int64_t nstatic = static_units > blockIdx.x ? (static_units - blockIdx.x + G - 1) / G : 0;

  if (lane == 0) {
    for (int s = 0; s < stages; ++s) ptx::mbar_init(&bars[s], 1);
    ptx::mbar_fence_init();
  }
  __syncwarp();

  auto piece_bytes = [&](int j) -> uint32_t {
    const int64_t left = p.row_bytes - static_cast<int64_t>(j) * p.piece_bytes;
    return static_cast<uint32_t>(left < p.piece_bytes ? left : p.piece_bytes);
  };
  const uint64_t pol = hints ? ptx::policy_evict_first() : 0;
  // Lane 0: load unit u into the stage of sequence index i.
  auto issue_load = [&](int64_t i, int64_t u) {
    const int64_t t = u / p.pieces;
    const int j = static_cast<int>(u - t * p.pieces);
    const uint32_t bytes = piece_bytes(j);
    const int s = static_cast<int>(i % stages);
    ptx::mbar_arrive_expect_tx(&bars[s], bytes);
    const uint8_t* src = p.x + t * p.row_bytes + static_cast<int64_t>(j) * p.piece_bytes;
    uint8_t* dst = stage_buf + static_cast<size_t>(s) * p.piece_bytes;
    if (hints & kHintPackLoads)
      ptx::bulk_g2s_hint(dst, src, bytes, &bars[s], pol);
    else
      ptx::bulk_g2s(dst, src, bytes, &bars[s]);
  };

  // Prologue: the static units, while routing still runs.
  if (lane == 0) {
    for (int64_t i = 0; i < stages; ++i) {
      const int64_t u = i < nstatic ? blockIdx.x + i * G : -1;
      stage_unit[i] = u;
      if (u >= 0) issue_load(i, u);
    }
  }
  // L2 prefetch of the claimed region [static_end, pf_end), spread over the
  // CTAs in the strided order (L2 is shared: which CTA claims a unit later
  // does not matter).  prefetch_units counts rounds of G units.
  int64_t pf_end = static_end;
  if (prefetch) {
    pf_end = units;
    if (prefetch_units >= 0 && static_end + static_cast<int64_t>(prefetch_units) * G < units)
      pf_end = static_end + static_cast<int64_t>(prefetch_units) * G;
    const uint64_t keep = prefetch == 2 ? ptx::policy_evict_last() : 0;
    for (int64_t u = static_end + blockIdx.x + static_cast<int64_t>(lane) * G; u < pf_end; u += 32 * G) {
      const int64_t t = u / p.pieces;
      const int j = static_cast<int>(u - t * p.pieces);
      const uint8_t* src = p.x + t * p.row_bytes + static_cast<int64_t>(j) * p.piece_bytes;
      if (prefetch == 2)
        ptx::bulk_prefetch_l2_hint(src, piece_bytes(j), keep);
      else
        ptx::bulk_prefetch_l2(src, piece_bytes(j));
    }
  }
  __syncwarp();  // stage_unit[] of the prologue is visible to every lane

  ptx::wait_prerequisites();  // slot_row, and the queue reset, come from routing

  bool claiming = units > static_end;
  unsigned long long claim = 0;
  if (lane == 0 && claiming) claim = atomicAdd(p.queue, 1ull);

  // Coherent loads: the table is written by the previous grid.
  auto dest_row = [&](int64_t u) -> int {
    const int64_t tt = u / p.pieces;
    return lane < p.K ? p.slot_row[tt * p.K + lane] : -1;
  };
  // Invariant: the stage_unit entries of sequence indices [i, issued) are
  // set; issued = stages + the refills done so far, and depth < stages, so
  // the entry of i+1 is always set when iteration i reads it.
  int64_t issued = stages;
  int64_t i = 0;
  bool ok = true;
  int64_t u_cur = stage_unit[0];
  int next_row = u_cur >= 0 ? dest_row(u_cur) : -1;
  while (u_cur >= 0) {
    const int64_t t = u_cur / p.pieces;
    const int j = static_cast<int>(u_cur - t * p.pieces);
    const int s = static_cast<int>(i % stages);
    const int row = next_row;
    const int64_t u_next = stage_unit[(i + 1) % stages];
    if (u_next >= 0) next_row = dest_row(u_next);
    const bool arrived = wait_phase(&bars[s], static_cast<uint32_t>((i / stages) & 1));
    if (!__all_sync(0xffffffffu, arrived)) {
      ok = false;
      break;
    }
    if (prefetch == 2 && u_cur >= static_end && u_cur < pf_end) {
      // Prefetched evict-last; now in shared memory: back to normal priority.
      const uint8_t* src = p.x + t * p.row_bytes + static_cast<int64_t>(j) * p.piece_bytes;
      const uint32_t lines = (piece_bytes(j) + 127) / 128;
      for (uint32_t q = lane; q < lines; q += 32) ptx::l2_priority_normal(src + static_cast<size_t>(q) * 128);
    }
    int row_ok = row;
    if (kChecked && row >= 0 && row >= p.dst_rows) {
      report(p.error_word, MOE_ECORRUPT);
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
    // Refill the stage of sequence r = i-depth+1 (its stores have read it)
    // with sequence r+stages: the claimed unit, or -1 once the queue is empty
    // (claims grow monotonically, so every later one is past the end too).
    const int64_t r = i - depth + 1;
    if (r >= 0) {
      wait_reads_at_most(depth - 1);
      __syncwarp();
      if (lane == 0) {
        int64_t u = -1;
        if (claiming) {
          const int64_t c = static_end + static_cast<int64_t>(claim);
          if (c < units) {
            u = c;
            claim = atomicAdd(p.queue, 1ull);
          } else {
            claiming = false;
          }
        }
        stage_unit[(r + stages) % stages] = u;
        if (u >= 0) issue_load(r + stages, u);
      }
      ++issued;
      claiming = __shfl_sync(0xffffffffu, claiming ? 1 : 0, 0) != 0;
      __syncwarp();
    }
    ++i;
    u_cur = stage_unit[i % stages];
  }
  if (!ok) {
    if (lane == 0) {
      report(p.error_word, MOE_ETIMEDOUT);
      // Wait (bounded) for the loads of sequences [i, issued) still in flight.
      for (int64_t q = i; q < issued; ++q)
        if (stage_unit[q % stages] >= 0) wait_phase(&bars[q % stages], static_cast<uint32_t>((q / stages) & 1));
    }
    __syncwarp();
  }
  ptx::bulk_wait<0>();  // stores complete before shared memory goes away
}

__global__ void __launch_bounds__(256) dispatch_pack_vector(PackParams p) {
  ptx::wait_prerequisites();
  const int lane = threadIdx.x & 31;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  const int64_t units = static_cast<int64_t>(p.T) * p.pieces;
  for (int64_t u = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); u < units; u += warps) {
    const int64_t t = u / p.pieces;
    const int j = static_cast<int>(u - t * p.pieces);
    int my_row = lane < p.K ? p.slot_row[t * p.K + lane] : -1;
    if (kChecked && my_row >= 0 && my_row >= p.dst_rows) {
      report(p.error_word, MOE_ECORRUPT);
      my_row = -1;
    }
    const int64_t off = static_cast<int64_t>(j) * p.piece_bytes;
    const int64_t left = p.row_bytes - off;
    const int chunks = static_cast<int>((left < p.piece_bytes ? left : p.piece_bytes) >> 4);
    const uint8_t* src = p.x + t * p.row_bytes + off;
    for (int c0 = 0; c0 < chunks; c0 += 4 * 32) {
      uint4 v[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int c = c0 + q * 32 + lane;
        if (c < chunks) v[q] = ptx::ld_stream_v4(src + static_cast<int64_t>(c) * 16);
      }
      for (int k = 0; k < p.K; ++k) {
        const int row = __shfl_sync(0xffffffffu, my_row, k);
        if (row < 0) continue;
        uint8_t* dst = p.expert_x + static_cast<int64_t>(row) * p.row_bytes + off;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int c = c0 + q * 32 + lane;
          if (c < chunks) ptx::st_v4(dst + static_cast<int64_t>(c) * 16, v[q]);
        }
      }
    }
  }
}

// Store groups kept in flight before a stage is refilled: 1..min(8, stages-1)
// (default 1: refill a stage as soon as its own stores have read it).
int store_depth(int depth, int stages) {
  if (depth < 1) depth = 1;
  if (depth > 8) depth = 8;
  if (depth > stages - 1) depth = stages - 1;
  return depth < 1 ? 1 : depth;
}

}  // namespace

size_t pack_bulk_smem_bytes(int stages, int piece_bytes) {
  return kBarBytes + static_cast<size_t>(stages) * piece_bytes;
}

cudaError_t prepare_pack(int max_smem_bytes) {
  const cudaError_t err =
      set_kernel_limits(reinterpret_cast<const void*>(dispatch_pack_bulk), static_cast<size_t>(max_smem_bytes));
  if (err != cudaSuccess) return err;
  return set_kernel_limits(reinterpret_cast<const void*>(dispatch_pack_bulk_queue),
                           static_cast<size_t>(max_smem_bytes));
}

cudaError_t launch_dispatch_pack(const PackParams& p, const PackLaunch& l, cudaStream_t stream) {
  if (l.variant == kPackVector) {
    return launch_kernel(dispatch_pack_vector, dim3(l.grid), dim3(256), 0, stream, l.pdl, p);
  }
  const int stages = l.stages < 2 ? 2 : (l.stages > kMaxStages ? kMaxStages : l.stages);
  auto* kern = l.dynamic && p.queue ? dispatch_pack_bulk_queue : dispatch_pack_bulk;
  return launch_kernel(kern, dim3(l.grid), dim3(32), pack_bulk_smem_bytes(stages, p.piece_bytes), stream, l.pdl, p,
                       stages, l.prefetch, l.hints, store_depth(l.depth, stages), l.prefetch_units);
}

}  // namespace moe
