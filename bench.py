"""Benchmark: one MoE dispatch + combine layer per step on one GB300.

A step is the whole hot path on one batch: moe_dispatch_send (routing +
dispatch_pack) -> moe_dispatch_recv -> moe_combine_send -> moe_combine_recv
(combine), on the DeepSeek-R1-decode-shaped workload by default
(T = 32 logical ranks x 128 tokens, H = 7168, E = 256, K = 8).  Inputs are
synthetic, seeded, resident in HBM; the synthetic expert outputs are made
before timing (no expert GEMM).  Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the CPU oracle on this host's cores

Under torchrun (N > 1) every rank runs an independent replica on its own
GPU: there is no cross-GPU exchange on this path.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "dispatch+combine µs/layer and achieved HBM GB/s vs GB300 peak, 1 GPU"
UNIT = "us/layer"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--workload", default="deepseek")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-workloads", action="store_true",
                    help="time only the headline workload (not the other workloads of the benchmark)")
    ap.add_argument("--buffer-sets", type=int, default=2)
    ap.add_argument("--payload", choices=["bf16", "fp8", "fp8q"], default="bf16",
                    help="dispatch payload: bf16 rows, or block-scaled fp8 rows (moe_dispatch_send_fp8)")
    ap.add_argument("--dispatch", choices=["direct", "staged"], default="direct",
                    help="rows straight to their grouped position (moe_dispatch_send), or through per-peer "
                         "send buffers and a receive shuffle (moe_dispatch_send_staged)")
    ap.add_argument("--combine", choices=["receiver", "two_level"], default="receiver",
                    help="receiver-only combine (moe_combine_recv), or partial sums on the sending side "
                         "then on the receiver (moe_combine_recv_two_level)")
    ap.add_argument("--overlap", action="store_true",
                    help="instead of the headline: how much of an independent GEMM (a shared-expert-sized "
                         "bf16 matmul, random weights) the split send/receive layer hides, per MOE_OPT_MAX_SMS, "
                         "and a two-micro-batch pipeline against the same work in sequence")
    ap.add_argument("--graph", action="store_true",
                    help="capture 16 steps (alternating the buffer sets) in a CUDA graph and replay it")
    return ap.parse_args()


def algorithmic_bytes(w, payload="bf16", partial_rows=None, staged=False, dense_cap=None):
    """Bytes a layer must move at minimum:
    dispatch reads x and writes T*K rows (bf16, or E4M3 bytes plus one float32
    scale per 128 elements); combine reads T*K bf16 rows and writes T rows;
    plus the routing metadata.  The two-level combine (partial_rows = the
    number of (token, rank) partials) also writes and reads back its partial
    rows.  The two-stage dispatch (staged) also writes every dispatched row
    to its send buffer and reads it back.  The dense padded all-to-all
    (dense_cap = rows per block) writes every dispatched row to its block,
    moves all N*N*dense_cap block rows (read and write) each way, and moves
    every dispatched row between its block and its grouped row each way."""
    T, H, K, E, N = w.T, w.H, w.K, w.E, w.N
    row = H * 2
    pairs = T * K
    out_row = row if payload == "bf16" else H + (H // 128) * 4
    in_row = H + (H // 128) * 4 if payload == "fp8q" else row  # fp8q: tokens arrive already quantised
    dispatch = T * in_row + pairs * out_row
    if staged:
        dispatch += 2 * pairs * row
    dispatch_meta = 2 * pairs * 4 + 2 * pairs * 4 + pairs * 4 + (3 * E + E * N + N + 2) * 4
    if staged:
        dispatch_meta += 4 * pairs * 4
    combine = pairs * row + T * row
    combine_meta = pairs * 4 + pairs * 4
    if dense_cap is not None:
        block_rows = N * N * dense_cap
        dispatch += 2 * block_rows * row + 2 * pairs * row
        dispatch_meta += 2 * pairs * 4 + 2 * pairs * 4
        combine += 2 * pairs * row + 2 * block_rows * row
        combine_meta += 2 * pairs * 4
    if partial_rows is not None:
        combine += 2 * partial_rows * row
        combine_meta += pairs * 4 + (N + 1) * 4
    return {"dispatch": dispatch + dispatch_meta, "combine": combine + combine_meta,
            "total": dispatch + dispatch_meta + combine + combine_meta}


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def committed_traffic(kernel: str, workload: str):
    """Per-launch DRAM bytes of `kernel` from the committed ncu summary, or
    None when the kernel source changed since it was captured: the record's
    source_sha covers its .cu file and the headers that hold only that
    kernel's device code (kernel_headers)."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except Exception:
        return None
    entry = rec.get(workload, {}).get(kernel)
    if not entry:
        return None
    h = hashlib.sha256()
    try:
        for name in [entry["source"]] + entry.get("kernel_headers", []):
            h.update(open(os.path.join(ROOT, "combine_route_count_gb300", "csrc", name), "rb").read())
    except OSError:
        return None
    return entry["dram_bytes_per_launch"] if h.hexdigest()[:16] == entry["source_sha"] else None


class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.proc = None
        self.index = index
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu=timestamp,{self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def stop(self, t0: float, t1: float):
        if self.proc is None:
            return None
        time.sleep(0.05)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        rows = []
        for line in out.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((parts[0], float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [r[1] for r in rows]
        loaded = [s for s in sm if s > 0.5 * max(sm)] or sm
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i, v in enumerate(r[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(r[2] for r in rows),
                "reasons": reasons, "samples": len(rows)}


def max_over_ranks(value: float, device) -> float:
    """The largest of every rank's value (all ranks get it); the value itself
    with one rank.  NCCL wants a device tensor, gloo a host one."""
    import torch
    import torch.distributed as dist
    if not dist.is_available() or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_us_per_layer(step_us_max: float, world_size: int) -> float:
    """Whole-job µs per layer: every replica runs one layer per step, so the
    job finishes world_size layers in the slowest rank's step time."""
    return step_us_max / max(world_size, 1)


def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def run_reference(args):
    """The CPU oracle, as it stands, on this host: each step is one oracle
    layer (dispatch + combine) over a bounded sample of the workload (the
    tokens of the first N/8 logical ranks, all experts), scaled to a full
    layer by the token ratio."""
    ws, rank, _ = dist_setup()
    if rank != 0:
        return
    import numpy as np

    import oracle
    from combine_route_count_gb300 import inputs as gen
    w = gen.BY_NAME[args.workload]
    oracle.build()
    li = gen.make_inputs(w)
    n_s = max(1, w.N // 8)
    Ts = n_s * w.tokens_per_rank
    xs, idx_s, w_s = li.x[:Ts], li.topk_idx[:Ts], li.topk_w[:Ts]
    ys = li.y[:Ts * w.K]
    for _ in range(args.warmup):
        d = oracle.dispatch(xs, idx_s, w.E, n_s)
        oracle.combine(ys, w_s, d.slot_row)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        d = oracle.dispatch(xs, idx_s, w.E, n_s)
        oracle.combine(ys, w_s, d.slot_row)
        times.append(time.perf_counter() - t0)
    scale = w.T / Ts
    us = statistics.mean(times) * 1e6 * scale
    sample = f"tokens of the first {n_s} of {w.N} logical ranks ({Ts} of {w.T} tokens) per step, x{scale:g} to a layer"
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(us, 1), "unit": UNIT, "higher_is_better": False,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(us / 1e3, 3),
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, **{k: v for k, v in w.describe().items() if k != "workload"},
                   "parallelism": "replicas" if ws > 1 else "single"},
        "cpu_baseline": {"value": round(us, 1), "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample},
        "e2e": {"value": round(us, 1), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def _time_oracle_layer(dispatch_fn, combine_fn, w, li, budget_s, max_reps):
    times = []
    t_end = time.perf_counter() + budget_s
    while len(times) < max_reps and (not times or time.perf_counter() < t_end):
        t0 = time.perf_counter()
        d = dispatch_fn(li.x, li.topk_idx, w.E, w.N)
        combine_fn(li.y, li.topk_w, d.slot_row)
        times.append(time.perf_counter() - t0)
    return statistics.mean(times) * 1e6, len(times)


def cpu_baseline(w, li, budget_s=8.0, max_reps=100):
    """The oracle on this host over the full layer, repeated: its loops
    spread over every core this process may use (OpenMP, the headline
    value), and as it stands on one core, in the same run."""
    import oracle
    oracle.build()
    threads = oracle.par_threads()
    us_par, n_par = _time_oracle_layer(oracle.dispatch_par, oracle.combine_par, w, li, budget_s, max_reps)
    us_one, n_one = _time_oracle_layer(oracle.dispatch, oracle.combine, w, li, budget_s, max_reps)
    try:
        affinity = len(os.sched_getaffinity(0))
    except AttributeError:
        affinity = None
    return {"value": round(us_par, 1), "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"full {w.name} layer (dispatch + combine) x{n_par}, the oracle's loops over {threads} "
                      f"threads (OpenMP: grouped-row copy and per-token combine in parallel)",
            "single_thread": {"value": round(us_one, 1), "unit": UNIT, "cores": 1,
                              "sample": f"full {w.name} layer x{n_one}, the oracle as it stands"},
            "host_cpus": os.cpu_count(), "host_cpus_usable": affinity}


def run_gpu(args):
    import numpy as np
    import torch

    from combine_route_count_gb300 import build as build_mod
    from combine_route_count_gb300 import inputs as gen
    from combine_route_count_gb300 import moe

    ws, rank, local = dist_setup()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    build_mod.build()
    moe.load_library()

    w = gen.BY_NAME[args.workload]
    li = gen.make_inputs(w)
    T, H, K, E, N = w.T, w.H, w.K, w.E, w.N
    rows = T * K
    stream = torch.cuda.Stream(device=dev)

    # Rotating buffer sets: consecutive steps touch different memory, and each
    # layer's working set (x, y, expert_x, out: ~1 GB at DeepSeek size) is far
    # larger than the 129 MB L2, so no step starts with its inputs in L2.
    sets = []
    with torch.cuda.stream(stream):
        x0 = torch.from_numpy(li.x.view(np.int16)).to(dev)
        idx0 = torch.from_numpy(li.topk_idx).to(dev)
        w0 = torch.from_numpy(li.topk_w).to(dev)
        y0 = torch.from_numpy(li.y.view(np.int16)).to(dev)
        if args.payload == "fp8q":
            # Already-quantised tokens: any byte pattern is a valid payload for
            # the copy, so seeded random codes and scales stand in for them.
            g = torch.Generator(device=dev)
            g.manual_seed(1234)
            xq0 = torch.randint(0, 256, (T, H), generator=g, device=dev, dtype=torch.uint8)
            xs0 = torch.rand((T, H // 128), generator=g, device=dev, dtype=torch.float32) + 1e-3
        for _ in range(args.buffer_sets):
            sets.append(dict(x=x0.clone(), idx=idx0.clone(), w=w0.clone(), y=y0.clone(),
                             xq=xq0.clone() if args.payload == "fp8q" else None,
                             xs=xs0.clone() if args.payload == "fp8q" else None,
                             expert_x=torch.empty((rows, H), dtype=torch.int16, device=dev)
                             if args.payload == "bf16" else torch.empty((rows, H), dtype=torch.uint8, device=dev),
                             expert_scales=None if args.payload == "bf16"
                             else torch.empty((rows, H // 128), dtype=torch.float32, device=dev),
                             out=torch.empty((T, H), dtype=torch.int16, device=dev),
                             partial=torch.empty((T * min(K, N), H), dtype=torch.int16, device=dev)
                             if args.combine == "two_level" else None,
                             send=torch.empty((rows, H), dtype=torch.int16, device=dev)
                             if args.dispatch == "staged" else None))
        del x0, idx0, w0, y0
    torch.cuda.synchronize(dev)
    layer = moe.MoELayer(T, H, K, E, N, device=dev)

    if args.dispatch == "staged" and args.payload != "bf16":
        raise SystemExit("--dispatch staged moves bf16 rows only")

    def dispatch(s, lay=layer):
        if args.dispatch == "staged":
            lay.dispatch_send_staged(s["x"], s["idx"], s["send"], s["expert_x"], stream)
        elif args.payload == "bf16":
            lay.dispatch_send(s["x"], s["idx"], s["expert_x"], stream)
        elif args.payload == "fp8q":
            lay.dispatch_send_quantized(s["xq"], s["xs"], s["idx"], s["expert_x"], s["expert_scales"], stream)
        else:
            lay.dispatch_send_fp8(s["x"], s["idx"], s["expert_x"], s["expert_scales"], stream)

    def combine(s, lay=layer):
        if args.combine == "receiver":
            lay.combine_recv(s["w"], s["out"], stream)
        else:
            lay.combine_recv_two_level(s["w"], s["partial"], s["out"], stream)

    def step(s):
        dispatch(s)
        layer.dispatch_recv(stream)
        layer.combine_send(s["y"], stream)
        combine(s)

    def barrier():
        if ws > 1:
            import torch.distributed as dist
            dist.barrier()

    for i in range(args.warmup):
        step(sets[i % len(sets)])
    if layer.get_error(stream) != moe.MOE_OK:
        raise RuntimeError("device reported an error during warm-up")

    run_steps = None
    if args.graph:
        # One replay = GRAPH_LAYERS steps, alternating the buffer sets; the
        # remainder of K runs as direct calls.
        graph = torch.cuda.CUDAGraph()
        per_graph = GRAPH_LAYERS - GRAPH_LAYERS % len(sets)
        with torch.cuda.graph(graph, stream=stream):
            for i in range(per_graph):
                step(sets[i % len(sets)])
        torch.cuda.synchronize(dev)

        def run_steps(k):
            with torch.cuda.stream(stream):
                for _ in range(k // per_graph):
                    graph.replay()
            for i in range(k % per_graph):
                step(sets[i % len(sets)])

    clocks = ClockSampler(torch.cuda.current_device() if ws == 1 else local).start()
    time.sleep(0.2)
    # Headline: exactly K steps between one pair of events, nothing recorded
    # inside (an event between two kernels would break their programmatic
    # dependent launch and add its own gap).
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize(dev)
    t_wall0 = time.time()
    t_start.record(stream)
    if run_steps is not None:
        run_steps(args.steps)
    else:
        for i in range(args.steps):
            step(sets[i % len(sets)])
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    t_wall1 = time.time()
    clk = clocks.stop(t_wall0, t_wall1)
    status = layer.get_error(stream)
    if status != moe.MOE_OK:
        raise RuntimeError(f"device reported status {status} in the timed region")
    total_ms = t_start.elapsed_time(t_end)
    ms_step = max_over_ranks(total_ms / args.steps, dev)  # slowest replica
    us_layer = job_us_per_layer(ms_step * 1e3, ws)

    # Warm-L2 figure (not the headline): the same steps on one buffer set, so
    # whatever of the previous step's data is still in L2 is reused.
    n_warm = min(args.steps, 500)
    torch.cuda.synchronize(dev)
    w0, w1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    w0.record(stream)
    for _ in range(n_warm):
        step(sets[0])
    w1.record(stream)
    torch.cuda.synchronize(dev)
    l2_warm_us = w0.elapsed_time(w1) / n_warm * 1e3

    # Attribution pass (not the headline).  Each dispatch_send is timed
    # between its own two events.  An event between dispatch_send and
    # combine_recv would break their programmatic dependent launch and charge
    # the launch gap to the combine, so combine_recv is timed over runs of R
    # back-to-back calls on R contexts dispatched beforehand; consecutive
    # combines overlap as the combine overlaps the pack inside the layer.
    R = 8
    ctxs = [layer] + [moe.MoELayer(T, H, K, E, N, device=dev) for _ in range(R - 1)]
    rounds = max(2, min(args.steps, 400) // R)
    d_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(R)]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    d_ms, c_ms = [], []
    torch.cuda.synchronize(dev)
    for rnd in range(rounds):
        for j, lay in enumerate(ctxs):
            s = sets[(rnd + j) % len(sets)]
            d_ev[j][0].record(stream)
            dispatch(s, lay)
            d_ev[j][1].record(stream)
            lay.dispatch_recv(stream)
            lay.combine_send(s["y"], stream)
        e0.record(stream)
        for j, lay in enumerate(ctxs):
            combine(sets[(rnd + j) % len(sets)], lay)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        if rnd > 0:  # the first round warms the extra contexts
            d_ms.extend(d_ev[j][0].elapsed_time(d_ev[j][1]) for j in range(R))
            c_ms.append(e0.elapsed_time(e1) / R)
    for lay in ctxs:
        if lay.get_error(stream) != moe.MOE_OK:
            raise RuntimeError("device reported an error in the attribution pass")
    for lay in ctxs[1:]:
        lay.close()
    disp_ms, comb_ms = d_ms, c_ms
    n_attr = len(disp_ms)

    partial_rows = None
    if args.combine == "two_level":
        ranks = np.sort(li.topk_idx // (E // N), axis=1)
        partial_rows = int(T + np.count_nonzero(np.diff(ranks, axis=1)))  # distinct ranks per token, summed
    ab = algorithmic_bytes(w, args.payload, partial_rows, args.dispatch == "staged")
    peak, peak_kind = measured_peaks()
    disp_alone_us = statistics.mean(disp_ms) * 1e3
    comb_us = statistics.mean(comb_ms) * 1e3
    # Inside the layer the pack's tail overlaps the combine's start; the
    # dispatch phase's share of the layer is what the combine leaves.
    disp_us = max(us_layer * ws - comb_us, 1e-3)
    fused = route_of(layer, moe, args.payload, args.dispatch) == 4
    pack_name = "dispatch_pack" if args.payload == "bf16" else "dispatch_pack_fp8"
    fused_name = "route_pack" if args.payload == "bf16" else "route_pack_fp8"
    kernels = {
        "dispatch_send": {"us": round(disp_us, 2), "alone_us": round(disp_alone_us, 2), "bytes": ab["dispatch"],
                          "gbs": round(ab["dispatch"] / disp_us / 1e3, 1),
                          "kernels": ([fused_name] if fused else ["route_cluster", pack_name])
                          if args.dispatch == "direct"
                          else ["route_cluster", "staged_layout", "dispatch_pack (send rows)",
                                "dispatch_pack (receive shuffle)"]},
        "combine_recv": {"us": round(comb_us, 2), "bytes": ab["combine"],
                         "gbs": round(ab["combine"] / comb_us / 1e3, 1),
                         "kernels": ["combine"] if args.combine == "receiver"
                         else ["combine_partial", "combine_reduce"]},
        "attribution": f"combine_recv over runs of {R} back-to-back calls on {R} contexts; dispatch_send = "
                       f"the layer's step time minus that (alone_us: between its own events); "
                       f"{n_attr} calls per phase",
    }
    # Kernel level: the pack and the combine kernel each between two CUDA
    # events that the library records on this stream right around its launch
    # (MOE_OPT_KERNEL_EVENTS), one layer at a time.
    kernel_us = None
    if args.dispatch == "direct" and args.combine == "receiver" and args.payload != "fp8q":
        timer = moe.MoELayer(T, H, K, E, N, device=dev, kernel_events=1)
        pk, cb = [], []
        for i in range(min(args.steps, 200) + 3):
            s = sets[i % len(sets)]
            dispatch(s, timer)
            timer.dispatch_recv(stream)
            timer.combine_send(s["y"], stream)
            combine(s, timer)
            a, b = timer.kernel_times()
            if i >= 3:
                pk.append(a)
                cb.append(b)
        if timer.get_error(stream) != moe.MOE_OK:
            raise RuntimeError("device reported an error in the kernel timing pass")
        timer.close()
        row_out = H * 2 if args.payload == "bf16" else H + (H // 128) * 4
        pack_bytes = T * H * 2 + rows * row_out + rows * 4
        comb_bytes = rows * H * 2 + T * H * 2 + rows * 8
        kernel_us = {"pack": statistics.mean(pk) * 1e3, "combine": statistics.mean(cb) * 1e3}
        kernels["dispatch_pack_kernel"] = {"us": round(kernel_us["pack"], 2), "bytes": pack_bytes,
                                           "kernel": fused_name if fused else pack_name,
                                           "gbs": round(pack_bytes / kernel_us["pack"] / 1e3, 1),
                                           "timing": f"events around the kernel launch, {len(pk)} layers"}
        kernels["combine_kernel"] = {"us": round(kernel_us["combine"], 2), "bytes": comb_bytes,
                                     "gbs": round(comb_bytes / kernel_us["combine"] / 1e3, 1),
                                     "timing": f"events around the kernel launch, {len(cb)} layers"}
    if kernel_us is not None:
        if kernel_us["combine"] >= kernel_us["pack"]:
            dom, dom_us, dom_bytes, dom_kernel = "combine", kernel_us["combine"], comb_bytes, "combine"
        else:
            dom, dom_us, dom_bytes = "dispatch_pack", kernel_us["pack"], pack_bytes
            dom_kernel = fused_name if fused else pack_name
    elif comb_us >= disp_us:
        dom, dom_us, dom_bytes = "combine", comb_us, ab["combine"]
        dom_kernel = "combine" if args.combine == "receiver" else "combine_two_level"
    else:
        dom, dom_us, dom_bytes = "route+dispatch_pack", disp_us, ab["dispatch"]
        dom_kernel = "dispatch_pack" if args.dispatch == "direct" else "dispatch_staged"
    achieved = dom_bytes / dom_us / 1e3
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "traffic": committed_traffic(dom_kernel, w.name),
                "kernel": dom, "peak_source": f"{peak_kind} hbm_gbs (copy, burst)",
                "timing": "kernel duration between CUDA events recorded around its launch" if kernel_us
                          else "phase time (see kernels.attribution)"}

    e2e = None
    if not args.no_e2e and args.payload == "bf16" and args.combine == "receiver" and args.dispatch == "direct":
        e2e = run_e2e(args, w, li, layer, stream, dev)

    workloads = None
    if not args.no_workloads and ws == 1 and args.payload == "bf16" and args.dispatch == "direct" \
            and args.combine == "receiver" and not args.graph:
        # Every workload of the benchmark in the same run; "frac" uses the
        # faster of direct calls and graph replay.
        wclocks = ClockSampler(torch.cuda.current_device()).start()
        time.sleep(0.2)
        t_w0 = time.time()
        workloads = {w.name: {"us": round(us_layer, 2), "bytes": ab["total"], "steps": args.steps,
                              "tbs": round(ab["total"] / us_layer / 1e6, 3),
                              "frac": round(ab["total"] / us_layer / 1e3 / peak, 4), "payload": "bf16",
                              "note": "the headline line"}}
        for name, payload, n in EXTRA_WORKLOADS:
            key = name if payload == "bf16" else f"{name}_{payload}"
            if key == w.name:
                continue
            workloads[key] = time_workload(name, payload, max(n, min(args.steps, 4 * n)), dev, peak)
        workloads["clocks"] = wclocks.stop(t_w0, time.time())
        workloads["method"] = ("two rotating buffer sets, one pair of CUDA events around `steps` layers; us: direct "
                               f"C-ABI calls from Python, us_graph: the same calls, {GRAPH_LAYERS} layers per CUDA "
                               "graph, replayed; us_graph_2: two layers per graph (each replay adds the graph "
                               "launch's gap); frac: algorithmic bytes / the faster of us and us_graph / measured "
                               "copy peak")

    cpu = None
    if not args.no_cpu and rank == 0:
        cpu = cpu_baseline(w, li)

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(us_layer, 2), "unit": UNIT, "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_step, 5), "higher_is_better": False,
            "scaling": "weak", "vs_baseline": None,
            "dtype": {"bf16": "bf16", "fp8": "fp8-e4m3 dispatch (quantised in the pack) / bf16 combine",
                      "fp8q": "fp8-e4m3 dispatch (tokens already quantised) / bf16 combine"}[args.payload],
            "data": "synthetic",
            "config": {"workload": w.name, **{k: v for k, v in w.describe().items() if k != "workload"},
                       "parallelism": "replicas" if ws > 1 else "single",
                       "l2": f"inputs > L2: {ab['total'] / 1e6:.0f} MB moved per layer, "
                             f"{args.buffer_sets} rotating buffer sets",
                       "launch": f"CUDA graph replay, {GRAPH_LAYERS} layers per graph" if args.graph
                                 else "direct C-ABI calls",
                       "payload": args.payload,
                       "dispatch": "direct placement" if args.dispatch == "direct"
                                   else "two-stage: per-peer send rows, then receive shuffle",
                       "pack": f"bulk (TMA), {layer.get_option(moe.MOE_OPT_PACK_STAGES) or 'auto'} stages, "
                               f"prefetch={layer.get_option(moe.MOE_OPT_PACK_PREFETCH)}, "
                               f"hints={layer.get_option(moe.MOE_OPT_CACHE_HINTS)}, PDL, "
                               f"schedule={ {-1: 'auto', 0: 'static', 1: 'queue'}[layer.get_option(moe.MOE_OPT_PACK_SCHEDULE)]}",
                       "combine": ("two-level: sending-side partial sums, "
                                   f"{partial_rows} partial rows" if args.combine == "two_level"
                                   else "bulk (TMA gather), " + ("static order" if layer.get_option(
                                       moe.MOE_OPT_COMBINE_SCHEDULE) == 0 else "token queue")
                                   if layer.get_option(moe.MOE_OPT_COMBINE_VARIANT) == 0
                                   else "vector"),
                       "routing": routing_label(layer, moe, args)},
            "l2_warm_us": round(l2_warm_us, 2),
            "achieved_gbs": round(ab["total"] / us_layer / 1e3, 1),
            "hbm_frac": round(ab["total"] / us_layer / 1e3 / (peak * ws), 4),  # per GPU
            "algorithmic_bytes_per_layer": ab["total"],
            "kernels": kernels,
            "roofline": roofline,
            "workloads": workloads,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "clocks": clk,
            "gpu_launches": (layer.kernels_per_layer() + (args.combine == "two_level")
                             + 2 * (args.dispatch == "staged") + (args.payload == "fp8q")) * args.steps,
        }
        print(json.dumps(line), flush=True)
    layer.close()
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# The other workloads of the benchmark, timed in the same run with the
# headline's method (two rotating buffer sets, one pair of CUDA events around
# K layers); the DeepSeek-sized layer also with the fp8 dispatch payload and
# through the dense padded all-to-all (the pages' comparison system).
# Steps per workload: at least ~20 ms of timed layers.
EXTRA_WORKLOADS = [("tiny", "bf16", 4000), ("mixtral", "bf16", 1000), ("kimi", "bf16", 60), ("worst", "bf16", 120),
                   ("deepseek", "fp8", 300), ("deepseek", "dense", 10)]


# Layers per CUDA graph in the graph-replay timings.
GRAPH_LAYERS = 16


def time_workload(name, payload, steps, dev, peak, warmup=10):
    """µs per layer of one workload: direct C-ABI calls (what the headline
    times) and the same calls replayed from a CUDA graph (no host work per
    layer).  Token rows and routing from the seeded generator; the
    synthetic expert outputs are drawn on the device (their values do not
    change the work)."""
    import numpy as np
    import torch

    from combine_route_count_gb300 import inputs as gen
    from combine_route_count_gb300 import moe
    w = gen.BY_NAME[name]
    li = gen.make_inputs(w, with_y=False)
    T, H, K, E, N = w.T, w.H, w.K, w.E, w.N
    stream = torch.cuda.Stream(device=dev)
    g = torch.Generator(device=dev)
    g.manual_seed(w.seed)
    layer = moe.MoELayer(T, H, K, E, N, device=dev)
    cap = layer.dense_capacity() if payload == "dense" else None
    with torch.cuda.stream(stream):
        x0 = torch.from_numpy(li.x.view(np.int16)).to(dev)
        idx0 = torch.from_numpy(li.topk_idx).to(dev)
        w0 = torch.from_numpy(li.topk_w).to(dev)
        y0 = torch.randn((T * K, H), generator=g, device=dev, dtype=torch.bfloat16).view(torch.int16)
        sets = []
        for _ in range(2):
            sets.append(dict(x=x0.clone(), idx=idx0.clone(), w=w0.clone(), y=y0.clone(),
                             ex=torch.empty((T * K, H), dtype=torch.uint8 if payload == "fp8" else torch.int16,
                                            device=dev),
                             xs=None if payload != "fp8" else torch.empty((T * K, H // 128), dtype=torch.float32,
                                                                          device=dev),
                             out=torch.empty((T, H), dtype=torch.int16, device=dev)))
        del x0, idx0, w0, y0
        # Dense padded all-to-all: one pair of block buffers (scratch) for both sets.
        blocks = None if cap is None else [torch.empty((N * N * cap, H), dtype=torch.int16, device=dev)
                                           for _ in range(2)]
    torch.cuda.synchronize(dev)

    def step(s_):
        if payload == "bf16":
            layer.dispatch_send(s_["x"], s_["idx"], s_["ex"], stream)
        elif payload == "dense":
            layer.dispatch_send_dense(s_["x"], s_["idx"], cap, blocks[0], blocks[1], s_["ex"], stream)
        else:
            layer.dispatch_send_fp8(s_["x"], s_["idx"], s_["ex"], s_["xs"], stream)
        layer.dispatch_recv(stream)
        layer.combine_send(s_["y"], stream)
        if payload == "dense":
            layer.combine_recv_dense(s_["w"], cap, blocks[0], blocks[1], s_["out"], stream)
        else:
            layer.combine_recv(s_["w"], s_["out"], stream)

    for i in range(warmup):
        step(sets[i % 2])
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    e0.record(stream)
    for i in range(steps):
        step(sets[i % 2])
    e1.record(stream)
    torch.cuda.synchronize(dev)
    us = e0.elapsed_time(e1) / steps * 1e3
    # Graph replay: GRAPH_LAYERS layers (alternating the two buffer sets) per
    # graph, as a model's graph holds many layers; and one layer per set (two
    # per graph), where every replay adds the graph launch's own gap.
    def graph_us(layers):
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            for i in range(layers):
                step(sets[i % 2])
        with torch.cuda.stream(stream):
            for _ in range(3):
                graph.replay()
        torch.cuda.synchronize(dev)
        replays = max(1, steps // layers)
        e0.record(stream)
        with torch.cuda.stream(stream):
            for _ in range(replays):
                graph.replay()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        del graph
        return e0.elapsed_time(e1) / (replays * layers) * 1e3

    us_graph = graph_us(GRAPH_LAYERS)
    us_graph_2 = graph_us(2)
    status = layer.get_error(stream)
    if status != moe.MOE_OK:
        raise RuntimeError(f"device reported status {status} timing {name}")
    v = route_of(layer, moe, "bf16" if payload == "dense" else payload, "dense" if payload == "dense" else "direct")
    routing = {1: "route_count", 2: "route_local+route_finalize", 3: "route_cluster",
               4: "route_pack (in the pack)" if payload != "fp8" else "route_pack_fp8 (in the fp8 pack)",
               5: "route_pack (one CTA)"}[v]
    layer.close()
    del sets, blocks
    torch.cuda.empty_cache()
    ab = algorithmic_bytes(w, "bf16" if payload == "dense" else payload, dense_cap=cap)["total"]
    best = min(us, us_graph)
    res = {"us": round(us, 2), "us_graph": round(us_graph, 2), "us_graph_2": round(us_graph_2, 2), "bytes": ab,
           "steps": steps,
           "tbs": round(ab / best / 1e6, 3), "frac": round(ab / best / 1e3 / peak, 4),
           "payload": "bf16" if payload == "dense" else payload, "routing": routing}
    if cap is not None:
        res.update({"exchange": "dense padded all-to-all", "capacity_rows_per_block": cap,
                    "exchanged_rows_each_way": N * N * cap, "dispatched_rows": T * K,
                    "exchange_to_sparse_rows": round(N * N * cap / (T * K), 2)})
    return res


def route_of(layer, moe, payload, dispatch="direct"):
    """The routing path of the timed dispatch (the MOE_OPT_ROUTE_VARIANT
    numbering): the context reports moe_dispatch_send's and
    moe_dispatch_send_fp8's; the other dispatch forms never route inside the
    pack."""
    if dispatch == "direct" and payload == "bf16":
        return layer.get_option(moe.MOE_OPT_ROUTE_VARIANT)
    if dispatch == "direct" and payload == "fp8":
        return layer.get_option(moe.MOE_OPT_ROUTE_VARIANT_FP8)
    v = layer.get_option(moe.MOE_OPT_ROUTE_VARIANT)
    if v == 4:
        v = 3 if layer.get_option(moe.MOE_OPT_ROUTE_CLUSTER_CTAS) > 0 else 2
    return v


def routing_label(layer, moe, args):
    """The routing kernels the timed dispatch runs."""
    v = route_of(layer, moe, args.payload, args.dispatch)
    return {1: "route_count (1 block)", 2: "route_local+route_finalize",
            3: f"route_cluster ({layer.get_option(moe.MOE_OPT_ROUTE_CLUSTER_CTAS)} CTAs)",
            4: "route_pack (routing inside the pack kernel)" if args.payload != "fp8"
            else "route_pack_fp8 (routing inside the fp8 pack kernel)",
            5: "route_pack (routing alone in one CTA)"}[v]


def run_e2e(args, w, li, layer, stream, dev):
    """The same layer through the public API with HOST buffers: every step
    uploads x, topk_idx, topk_w and the expert outputs y from pinned host
    memory, runs the four calls, and downloads out to pinned host memory.
    Uploads for step i+1 and the download of step i-1 run on their own
    streams while step i computes (two device buffer sets, event-ordered),
    so the step time is bound by the host link, not by the sum of the parts."""
    import numpy as np
    import torch
    T, H, K = w.T, w.H, w.K
    hx = torch.from_numpy(li.x.view(np.int16)).pin_memory()
    hidx = torch.from_numpy(li.topk_idx).pin_memory()
    hw = torch.from_numpy(li.topk_w).pin_memory()
    hy = torch.from_numpy(li.y.view(np.int16)).pin_memory()
    hout = torch.empty((T, H), dtype=torch.int16).pin_memory()
    bufs = [dict(x=torch.empty_like(hx, device=dev), idx=torch.empty_like(hidx, device=dev),
                 w=torch.empty_like(hw, device=dev), y=torch.empty_like(hy, device=dev),
                 ex=torch.empty((T * K, H), dtype=torch.int16, device=dev),
                 out=torch.empty((T, H), dtype=torch.int16, device=dev)) for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in (hx, hidx, hw, hy))
    d2h = hout.numel() * hout.element_size()
    s_up = torch.cuda.Stream(device=dev)
    s_down = torch.cuda.Stream(device=dev)
    up_ev = [torch.cuda.Event() for _ in range(2)]
    comp_ev = [torch.cuda.Event() for _ in range(2)]
    down_ev = [torch.cuda.Event() for _ in range(2)]

    def upload(b):
        with torch.cuda.stream(s_up):
            for name, src in (("x", hx), ("idx", hidx), ("w", hw), ("y", hy)):
                bufs[b][name].copy_(src, non_blocking=True)
        up_ev[b].record(s_up)

    def run(steps):
        upload(0)
        for i in range(steps):
            b = i % 2
            if i + 1 < steps:
                nb = (i + 1) % 2
                if i >= 1:
                    s_up.wait_event(comp_ev[nb])  # buffer nb was last read by step i-1
                upload(nb)
            stream.wait_event(up_ev[b])
            if i >= 2:
                stream.wait_event(down_ev[b])  # out[b] was last read by the download of step i-2
            B = bufs[b]
            layer.dispatch_send(B["x"], B["idx"], B["ex"], stream)
            layer.dispatch_recv(stream)
            layer.combine_send(B["y"], stream)
            layer.combine_recv(B["w"], B["out"], stream)
            comp_ev[b].record(stream)
            s_down.wait_event(comp_ev[b])
            with torch.cuda.stream(s_down):
                hout.copy_(B["out"], non_blocking=True)
            down_ev[b].record(s_down)

    steps = max(4, min(args.steps, 100))
    run(4)
    torch.cuda.synchronize(dev)
    # The host link on this machine, measured alone with the same copies: the
    # floor the end-to-end step cannot beat (uploads dominate it).  Best of
    # three runs of four uploads (one run has read a third of the link's rate).
    h2d_gbs = 0.0
    for _ in range(3):
        l0 = torch.cuda.Event(enable_timing=True)
        l1 = torch.cuda.Event(enable_timing=True)
        l0.record(s_up)
        for _ in range(4):
            upload(0)
        l1.record(s_up)
        torch.cuda.synchronize(dev)
        h2d_gbs = max(h2d_gbs, 4 * h2d / (l0.elapsed_time(l1) * 1e-3) / 1e9)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(s_up)
    s_down.wait_event(e0)
    stream.wait_event(e0)
    run(steps)
    stream.wait_event(down_ev[(steps - 1) % 2])
    e1.record(stream)
    torch.cuda.synchronize(dev)
    us = e0.elapsed_time(e1) / steps * 1e3
    if layer.get_error(stream) != 0:
        raise RuntimeError("device reported an error in the end-to-end pass")
    ok = bool(torch.equal(hout, bufs[(steps - 1) % 2]["out"].cpu()))
    return {"value": round(us, 1), "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "steps": steps, "pipelined": True, "out_matches_device": ok,
            "host_link_h2d_gbs": round(h2d_gbs, 1), "h2d_floor_us": round(h2d / h2d_gbs / 1e3, 1)}


def run_overlap(args):
    """Split send/receive halves let other work run between and beside them
    ("Efficient and portable mixture-of-experts communication", Benchmarks:
    splitting into send and receive parts can hide latency; "Enabling
    trillion-parameter models on AWS EFA", evaluation: micro-batching).  On one
    GPU the layer is HBM-bound and a bf16 GEMM is tensor-bound, so they can
    share the SMs.  Measured here, each over `steps` iterations between events:
      layer      dispatch_send..combine_recv alone;
      gemm       the independent work alone: [T, H] x [H, 4096] bf16 (the
                 gate+up projection of a DeepSeek-sized shared expert);
      serial     layer then gemm on one stream;
      overlap    layer on one stream, gemm on another, joined each step, for
                 several MOE_OPT_MAX_SMS values;
      pipeline   two micro-batches of T/2 tokens (two contexts): each
                 micro-batch's GEMM (on the T/2 tokens) runs on a second
                 stream between its dispatch and its combine, so micro-batch
                 1's dispatch overlaps micro-batch 0's GEMM; against the same
                 calls in sequence on one stream."""
    import numpy as np
    import torch

    from combine_route_count_gb300 import build as build_mod
    from combine_route_count_gb300 import inputs as gen
    from combine_route_count_gb300 import moe

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    build_mod.build()
    moe.load_library()
    w = gen.BY_NAME[args.workload]
    li = gen.make_inputs(w)
    T, H, K, E, N = w.T, w.H, w.K, w.E, w.N
    steps = max(10, min(args.steps, 200))
    sa, sb = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    x = torch.from_numpy(li.x.view(np.int16)).to(dev)
    idx = torch.from_numpy(li.topk_idx).to(dev)
    wts = torch.from_numpy(li.topk_w).to(dev)
    y = torch.from_numpy(li.y.view(np.int16)).to(dev)
    ex = torch.empty((T * K, H), dtype=torch.int16, device=dev)
    out = torch.empty((T, H), dtype=torch.int16, device=dev)
    g = torch.Generator(device=dev)
    g.manual_seed(1234)
    a_mat = torch.randn((T, H), generator=g, device=dev, dtype=torch.bfloat16)
    b_mat = torch.randn((H, 4096), generator=g, device=dev, dtype=torch.bfloat16) * (H ** -0.5)
    c_mat = torch.empty((T, 4096), device=dev, dtype=torch.bfloat16)
    layer = moe.MoELayer(T, H, K, E, N, device=dev)

    def run_layer(lay, s, xx, ii, ww, yy, ee, oo):
        lay.dispatch_send(xx, ii, ee, s)
        lay.dispatch_recv(s)
        lay.combine_send(yy, s)
        lay.combine_recv(ww, oo, s)

    def gemm(s, a=a_mat, c=c_mat):
        with torch.cuda.stream(s):
            torch.matmul(a, b_mat, out=c)

    def timed(fn, stream):
        for _ in range(3):
            fn()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1) / steps * 1e3

    def fork_join(body_a, body_b):
        ev0, ev1 = torch.cuda.Event(), torch.cuda.Event()
        ev0.record(sa)
        sb.wait_event(ev0)
        body_a()
        body_b()
        ev1.record(sb)
        sa.wait_event(ev1)

    t_layer = timed(lambda: run_layer(layer, sa, x, idx, wts, y, ex, out), sa)
    t_gemm = timed(lambda: gemm(sa), sa)
    t_serial = timed(lambda: (run_layer(layer, sa, x, idx, wts, y, ex, out), gemm(sa)), sa)
    overlap = []
    for max_sms in (0, 128, 112, 96, 76):
        layer.set_option(moe.MOE_OPT_MAX_SMS, max_sms)
        t_l = timed(lambda: run_layer(layer, sa, x, idx, wts, y, ex, out), sa)
        t_o = timed(lambda: fork_join(lambda: run_layer(layer, sa, x, idx, wts, y, ex, out), lambda: gemm(sb)), sa)
        overlap.append({"max_sms": max_sms, "layer_alone_us": round(t_l, 2), "overlap_us": round(t_o, 2),
                        "hidden_frac": round((t_l + t_gemm - t_o) / min(t_l, t_gemm), 3)})
    layer.set_option(moe.MOE_OPT_MAX_SMS, 0)
    if layer.get_error(sa) != moe.MOE_OK:
        raise RuntimeError("device reported an error in the overlap pass")

    # Two micro-batches of T/2 tokens.
    Th = T // 2
    mbs = []
    for m in range(2):
        sl = slice(m * Th, (m + 1) * Th)
        lm = moe.MoELayer(Th, H, K, E, N, device=dev)
        mbs.append(dict(layer=lm, x=x[sl].contiguous(), idx=idx[sl].contiguous(), w=wts[sl].contiguous(),
                        y=y[: Th * K].contiguous(), ex=torch.empty((Th * K, H), dtype=torch.int16, device=dev),
                        out=torch.empty((Th, H), dtype=torch.int16, device=dev), a=a_mat[sl],
                        c=torch.empty((Th, 4096), device=dev, dtype=torch.bfloat16)))

    def mb_sequential():
        for mb in mbs:
            mb["layer"].dispatch_send(mb["x"], mb["idx"], mb["ex"], sa)
            mb["layer"].dispatch_recv(sa)
            gemm(sa, mb["a"], mb["c"])
            mb["layer"].combine_send(mb["y"], sa)
            mb["layer"].combine_recv(mb["w"], mb["out"], sa)

    def mb_pipelined():
        start = torch.cuda.Event()
        start.record(sa)
        sb.wait_event(start)
        done = []
        for mb in mbs:
            mb["layer"].dispatch_send(mb["x"], mb["idx"], mb["ex"], sa)
            mb["layer"].dispatch_recv(sa)
            ev = torch.cuda.Event()
            ev.record(sa)
            sb.wait_event(ev)  # this micro-batch's GEMM needs its dispatched rows
            gemm(sb, mb["a"], mb["c"])
            e2 = torch.cuda.Event()
            e2.record(sb)
            done.append(e2)
        for mb, e2 in zip(mbs, done):
            sa.wait_event(e2)
            mb["layer"].combine_send(mb["y"], sa)
            mb["layer"].combine_recv(mb["w"], mb["out"], sa)

    t_mb_seq = timed(mb_sequential, sa)
    t_mb_pipe = timed(mb_pipelined, sa)
    for mb in mbs:
        if mb["layer"].get_error(sa) != moe.MOE_OK:
            raise RuntimeError("device reported an error in the micro-batch pass")
        mb["layer"].close()
    layer.close()
    line = {"metric": "overlap of the split dispatch/combine with an independent bf16 GEMM", "unit": "us",
            "workload": w.name, "steps": steps, "layer_us": round(t_layer, 2), "gemm_us": round(t_gemm, 2),
            "gemm": f"[{T}, {H}] x [{H}, 4096] bf16 torch.matmul on a second stream", "serial_us": round(t_serial, 2),
            "overlap": overlap,
            "micro_batches": {"sequential_us": round(t_mb_seq, 2), "pipelined_us": round(t_mb_pipe, 2),
                              "tokens_per_micro_batch": Th, "gemm_per_micro_batch": f"[{Th}, {H}] x [{H}, 4096]"}}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    elif args.overlap:
        run_overlap(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
