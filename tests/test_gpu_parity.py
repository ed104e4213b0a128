"""GPU path vs the CPU oracle, through the C ABI (libmoe.so).

Bar: dispatch outputs (grouped rows, counts, offsets, slot_row, row_src) are
compared bit for bit; the combine output is compared bit for bit against the
oracle's float32 chain (fixed top-k order, one fused multiply-add per expert,
one round-to-nearest-even), and in addition must stay within one bf16 ulp of
the double-precision sum except where the float32 sum cancels (bounded by the
float32 accumulation error, see the oracle pins).

Covers the five named workloads at full size in the launch configuration the
benchmark uses, every pack variant and launch option, ragged and degenerate
shapes, routing errors and the call-order state machine.  Guard rows around
every output catch stray writes.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

from combine_route_count_gb300 import inputs as gen  # noqa: E402

GUARD = 3
CANARY = 0x7BCD  # a bf16 bit pattern no input row is expected to hold everywhere


@pytest.fixture(scope="module")
def moe():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from combine_route_count_gb300 import build, moe as m
    build.build()
    m.load_library()
    return m


def _dev(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.view(dtype)
    return t.cuda()


def _guarded(rows, H):
    """A [GUARD + rows + GUARD, H] int16 canary buffer and its middle view."""
    big = torch.full((GUARD + rows + GUARD, H), CANARY, dtype=torch.int16, device="cuda")
    return big, big[GUARD:GUARD + rows]


def _intact(big, rows):
    v = big.cpu().numpy().view(np.uint16)
    return bool(np.all(v[:GUARD] == CANARY) and np.all(v[GUARD + rows:] == CANARY))


def run_gpu(moe, w, li, extra_rows=0, stream=None, **options):
    T, H, K, E, N = w.T, w.H, w.K, w.E, w.N
    rows = T * K
    x = _dev(li.x.view(np.int16))
    idx = _dev(li.topk_idx)
    wt = _dev(li.topk_w)
    y = _dev(li.y.view(np.int16)) if li.y is not None else torch.zeros((rows, H), dtype=torch.int16, device="cuda")
    ex_big, expert_x = _guarded(rows + extra_rows, H)
    out_big, out = _guarded(T, H)
    layer = moe.MoELayer(T, H, K, E, N, **options)
    lay = layer.layer(x, idx, wt, expert_x, y, out, stream)
    status = layer.get_error(stream)
    torch.cuda.synchronize()
    res = {k: (v.cpu().numpy() if hasattr(v, "cpu") else v) for k, v in lay.items()}
    res.update(status=status, expert_x=expert_x.cpu().numpy().view(np.uint16), out=out.cpu().numpy().view(np.uint16),
               guards_ok=_intact(ex_big, rows + extra_rows) and _intact(out_big, T), layer=layer)
    return res


_oracle_cache = {}


def oracle_of(oracle_mod, w, li):
    key = (w.name, w.T, w.H, w.K, w.E, w.N, w.index)
    if key not in _oracle_cache:
        d = oracle_mod.dispatch(li.x, li.topk_idx, w.E, w.N)
        out = oracle_mod.combine(li.y, li.topk_w, d.slot_row)
        _oracle_cache.clear()
        _oracle_cache[key] = (d, out)
    return _oracle_cache[key]


def assert_parity(res, d, out_ref, w, extra_rows=0):
    rows = w.T * w.K
    assert res["status"] == 0
    assert res["guards_ok"], "a write landed outside an output buffer"
    assert np.array_equal(res["expert_counts"], d.expert_counts)
    assert np.array_equal(res["expert_offsets"], d.expert_offsets)
    assert np.array_equal(res["rank_offsets"], d.rank_offsets)
    assert np.array_equal(res["src_offsets"], d.src_offsets)
    assert np.array_equal(res["slot_row"], d.slot_row)
    assert np.array_equal(res["row_src"], d.row_src)
    assert np.array_equal(res["expert_x"][:rows], d.expert_x[:rows])
    if extra_rows:
        assert np.all(res["expert_x"][rows:] == CANARY), "rows past T*K must stay untouched"
    assert np.array_equal(res["out"], out_ref)


@pytest.mark.parametrize("name", [w.name for w in gen.WORKLOADS])
def test_named_workload_full_size(moe, oracle_mod, name):
    w = gen.BY_NAME[name]
    li = gen.make_inputs(w)
    d, out_ref = oracle_of(oracle_mod, w, li)
    res = run_gpu(moe, w, li)
    assert_parity(res, d, out_ref, w)
    assert res["recv_bound_rows"] == w.N * w.tokens_per_rank * max(w.K, w.E // w.N)
    if name == "worst":
        recv = np.diff(res["rank_offsets"])
        assert recv[0] == res["recv_bound_rows"] == 65536 and np.all(recv[1:] == 0)
    # combine within one bf16 step of the double-precision sum wherever the
    # float32 chain does not cancel (sampled rows: the f64 oracle is slower)
    sample = np.random.default_rng(0).choice(w.T, size=min(w.T, 64), replace=False)
    sub_w = li.topk_w[sample]
    sub_slot = d.slot_row[sample]
    o64, exact, mag = oracle_mod.combine_f64(li.y, sub_w, sub_slot)
    gpu = res["out"][sample]
    step = np.abs(gpu.astype(np.int32) - o64.astype(np.int32))
    assert np.mean(step <= 1) > 0.999
    g = gen.bf16_bits_to_f32(gpu).astype(np.float64)
    ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(g), 2.0 ** -126))) - 7)
    assert np.all(np.abs(g - exact) <= w.K * 2.0 ** -24 * mag * 1.001 + 0.5 * ulp + 1e-30)


def test_identity_experts_return_the_input(moe):
    """y = expert_x (identity experts) with weights summing to one gives x."""
    w = gen.BY_NAME["deepseek"]
    li = gen.make_inputs(gen.Workload("ds-id", T=1024, H=w.H, K=w.K, E=w.E, N=8, router=w.router, index=w.index),
                         with_y=False)
    T, H, K = 1024, w.H, w.K
    x = _dev(li.x.view(np.int16))
    idx = _dev(li.topk_idx)
    wt = _dev(li.topk_w)
    expert_x = torch.empty((T * K, H), dtype=torch.int16, device="cuda")
    out = torch.empty((T, H), dtype=torch.int16, device="cuda")
    layer = moe.MoELayer(T, H, K, w.E, 8)
    layer.layer(x, idx, wt, expert_x, expert_x, out)
    assert layer.get_error() == 0
    # The chain starts from +0.0, so a -0.0 element comes back as +0.0.
    assert torch.equal(out, torch.where(x == -32768, torch.zeros_like(x), x))


PACK_OPTIONS = [
    dict(pack_variant=0, pack_stages=2),
    dict(pack_variant=0, pack_stages=8, pack_piece_bytes=2048),
    dict(pack_variant=0, pack_stages=3, pack_piece_bytes=4096 + 512, pack_ctas_per_sm=1),
    dict(pack_variant=0, pdl=0),
    dict(pack_variant=1),
    dict(pack_variant=1, pack_piece_bytes=1024, pdl=0),
    dict(route_variant=1),
    dict(route_variant=1, pdl=0, pack_variant=1),
    dict(route_variant=2),
    dict(route_variant=2, pdl=0),
    dict(combine_variant=1),
    dict(combine_variant=0, combine_stages=2, combine_piece_bytes=1024),
    dict(combine_variant=0, combine_stages=8, combine_piece_bytes=2048 + 16, combine_ctas_per_sm=1),
    dict(combine_variant=0, combine_piece_bytes=4096, pdl=0),
    dict(cache_hints=0, pack_prefetch=0),
    dict(cache_hints=5, pack_prefetch=1, pack_stages=16, pack_ctas_per_sm=1),
    dict(pack_stages=14, pack_ctas_per_sm=2, combine_stages=5),
    dict(pack_store_depth=1),
    dict(pack_store_depth=5, pack_stages=6),
    dict(combine_variant=0, combine_order=1),
    dict(combine_variant=0, combine_order=1, combine_piece_bytes=2048 + 16, combine_stages=3, combine_ctas_per_sm=3),
    dict(combine_variant=0, combine_order=0),
    dict(pack_schedule=0),
    dict(pack_schedule=1),
    dict(pack_schedule=1, pack_stages=2, pack_store_depth=1),
    dict(pack_schedule=1, pack_stages=16, pack_store_depth=8, pack_ctas_per_sm=1),
    dict(pack_schedule=1, pack_piece_bytes=2048, pack_prefetch=2),
    dict(pack_schedule=1, pack_prefetch=0, cache_hints=0, pdl=0),
    dict(pack_schedule=1, route_variant=1),
    dict(pack_schedule=1, route_variant=2),
    dict(combine_variant=0, combine_schedule=0),
    dict(combine_variant=0, combine_schedule=1),
    dict(combine_variant=0, combine_schedule=1, combine_stages=2, combine_piece_bytes=1024),
    dict(combine_variant=0, combine_schedule=1, combine_stages=8, combine_piece_bytes=2048 + 16,
         combine_ctas_per_sm=1),
    dict(combine_variant=0, combine_schedule=1, pdl=0, route_variant=1),
    dict(combine_variant=0, combine_schedule=1, pack_schedule=1, route_variant=2),
]


@pytest.mark.parametrize("opts", PACK_OPTIONS, ids=[str(o) for o in PACK_OPTIONS])
def test_launch_options_give_identical_results(moe, oracle_mod, opts):
    w = gen.custom("opts", T=2 * 1000, H=7168, K=8, E=256, N=8, router="uniform_random", seed_index=7)
    li = gen.make_inputs(w)
    d, out_ref = oracle_of(oracle_mod, w, li)
    res = run_gpu(moe, w, li, **opts)
    assert_parity(res, d, out_ref, w)


EDGE = [
    # (T, H, K, E, N, router)
    (1, 8, 1, 1, 1, "uniform_random"),          # one token, one expert, narrowest row
    (3, 24, 3, 3, 1, "uniform_random"),         # E == K, odd K (scalar index loads)
    (6, 40, 1, 6, 6, "uniform_random"),         # one token per rank, E == N
    (1000, 136, 5, 40, 4, "uniform_random"),    # ragged chunk, odd K, rows not a power of two
    (2049, 64, 2, 6, 3, "uniform_random"),      # chunks of 1024 + tail of 1
    (512, 256, 16, 64, 4, "uniform_random"),    # K = 16 (max)
    (1024, 128, 7, 1024, 8, "uniform_random"),  # E = 1024 (max): 512-token chunks
    (1540, 64, 4, 770, 2, "uniform_random"),    # E > 768 path, ragged
    (64, 8200, 2, 8, 2, "uniform_random"),      # row > 16 KiB: split into pieces
    (4096, 2056, 6, 96, 16, "uniform_random"),  # odd-ish row bytes (4112)
    (8192, 64, 8, 64, 8, "rank0_only"),         # everything to rank 0
    (40960, 16, 2, 64, 8, "uniform_random"),    # > 128 chunks of 256: 512-token chunks in the split routing
    (33024, 8, 1, 8, 4, "uniform_random"),      # chunk of 512 with a ragged last chunk
]


VARIANTS = [(0, 0, 0), (1, 1, 1), (2, 0, 0)]  # (route_variant, combine_variant, pack_variant)


@pytest.mark.parametrize("variants", VARIANTS, ids=["cluster-bulk-bulk", "single-vector-vector", "split-bulk-bulk"])
@pytest.mark.parametrize("shape", EDGE, ids=["x".join(map(str, s[:5])) for s in EDGE])
def test_edge_shapes(moe, oracle_mod, shape, variants):
    T, H, K, E, N, router = shape
    w = gen.custom("edge", T=T, H=H, K=K, E=E, N=N, router=router, seed_index=11)
    li = gen.make_inputs(w)
    d, out_ref = oracle_of(oracle_mod, w, li)
    res = run_gpu(moe, w, li, extra_rows=5, route_variant=variants[0], combine_variant=variants[1],
                  pack_variant=variants[2])
    assert_parity(res, d, out_ref, w, extra_rows=5)


def test_empty_layer(moe):
    layer = moe.MoELayer(0, 64, 2, 8, 2)
    x = torch.empty((0, 64), dtype=torch.int16, device="cuda")
    idx = torch.empty((0, 2), dtype=torch.int32, device="cuda")
    wt = torch.empty((0, 2), dtype=torch.float32, device="cuda")
    big, ex = _guarded(0, 64)
    lay = layer.layer(x, idx, wt, ex, ex, x)
    assert layer.get_error() == 0
    assert lay["expert_counts"].cpu().tolist() == [0] * 8
    assert lay["expert_offsets"].cpu().tolist() == [0] * 9
    assert lay["src_offsets"].cpu().numpy().tolist() == [[0, 0]] * 8
    assert _intact(big, 0)


@pytest.mark.parametrize("shape", EDGE, ids=["x".join(map(str, s[:5])) for s in EDGE])
def test_edge_shapes_pack_queue(moe, oracle_mod, shape):
    """The bulk pack with its unit queue forced on, at every edge shape."""
    T, H, K, E, N, router = shape
    w = gen.custom("edge", T=T, H=H, K=K, E=E, N=N, router=router, seed_index=17)
    li = gen.make_inputs(w)
    d, out_ref = oracle_of(oracle_mod, w, li)
    res = run_gpu(moe, w, li, extra_rows=2, pack_schedule=1, pack_variant=0)
    assert_parity(res, d, out_ref, w, extra_rows=2)


@pytest.mark.parametrize("shape", EDGE, ids=["x".join(map(str, s[:5])) for s in EDGE])
def test_edge_shapes_combine_queue(moe, oracle_mod, shape):
    """The bulk combine with its unit queue forced on, at every edge shape."""
    T, H, K, E, N, router = shape
    w = gen.custom("edge", T=T, H=H, K=K, E=E, N=N, router=router, seed_index=19)
    li = gen.make_inputs(w)
    d, out_ref = oracle_of(oracle_mod, w, li)
    res = run_gpu(moe, w, li, extra_rows=2, combine_variant=0, combine_schedule=1)
    assert_parity(res, d, out_ref, w, extra_rows=2)


def test_pack_queue_is_reset_every_layer(moe, oracle_mod):
    """Layers with different routings on one context, the pack's and the
    combine's queues forced on: each layer's routing resets both (a stale
    count would leave units undone), also across a routing error and with
    each routing variant."""
    T, H, K, E, N = 2048, 1024, 8, 64, 8
    layer = moe.MoELayer(T, H, K, E, N, pack_schedule=1, combine_variant=0, combine_schedule=1)
    ex = torch.empty((T * K, H), dtype=torch.int16, device="cuda")
    out = torch.empty((T, H), dtype=torch.int16, device="cuda")
    for n, route in enumerate([0, 0, 1, 2, 3, 0]):
        w = gen.custom("queue", T=T, H=H, K=K, E=E, N=N, router="uniform_random", seed_index=40 + n)
        li = gen.make_inputs(w)
        d, out_ref = oracle_of(oracle_mod, w, li)
        x, idx, wt, y = (_dev(li.x.view(np.int16)), _dev(li.topk_idx), _dev(li.topk_w), _dev(li.y.view(np.int16)))
        layer.set_option(moe.MOE_OPT_ROUTE_VARIANT, route)
        if n == 3:
            bad = li.topk_idx.copy()
            bad[7, 3] = bad[7, 2]  # a repeated expert: nothing is copied, the queue is still consumed
            bad_d = _dev(bad)
            layer.layer(x, bad_d, wt, ex, y, out)
            assert layer.get_error() == moe.MOE_EROUTE
        lay = layer.layer(x, idx, wt, ex, y, out)
        assert layer.get_error() == 0
        assert np.array_equal(lay["slot_row"].cpu().numpy(), d.slot_row)
        assert np.array_equal(ex.cpu().numpy().view(np.uint16), d.expert_x), n
        assert np.array_equal(out.cpu().numpy().view(np.uint16), out_ref), n


@pytest.mark.parametrize("shape", EDGE, ids=["x".join(map(str, s[:5])) for s in EDGE])
def test_edge_shapes_strided_combine(moe, oracle_mod, shape):
    T, H, K, E, N, router = shape
    w = gen.custom("edge", T=T, H=H, K=K, E=E, N=N, router=router, seed_index=13)
    li = gen.make_inputs(w)
    d, out_ref = oracle_of(oracle_mod, w, li)
    res = run_gpu(moe, w, li, extra_rows=3, combine_variant=0, combine_order=1)
    assert_parity(res, d, out_ref, w, extra_rows=3)


def test_non_default_stream_and_reuse(moe, oracle_mod):
    """Two layers back to back on a side stream reuse one context and workspace."""
    s = torch.cuda.Stream()
    for seed in (21, 22):
        w = gen.custom("stream", T=512, H=512, K=4, E=32, N=4, seed_index=seed)
        li = gen.make_inputs(w)
        d, out_ref = oracle_of(oracle_mod, w, li)
        with torch.cuda.stream(s):
            res = run_gpu(moe, w, li, stream=s)
        assert_parity(res, d, out_ref, w)


@pytest.mark.parametrize("variants", VARIANTS, ids=["cluster-bulk-bulk", "single-vector-vector", "split-bulk-bulk"])
@pytest.mark.parametrize("bad", ["out_of_range", "negative", "repeated"])
def test_routing_errors_write_nothing(moe, bad, variants):
    w = gen.custom("bad", T=300, H=64, K=4, E=16, N=4, seed_index=3)
    li = gen.make_inputs(w)
    idx = li.topk_idx.copy()
    if bad == "out_of_range":
        idx[123, 2] = 16
    elif bad == "negative":
        idx[7, 0] = -1
    else:
        idx[299, 3] = idx[299, 1]
    li2 = gen.LayerInputs(w, li.x, idx, li.topk_w, li.y)
    res = run_gpu(moe, w, li2, route_variant=variants[0], combine_variant=variants[1], pack_variant=variants[2])
    assert res["status"] == moe.MOE_EROUTE
    assert res["error_word"][0] == moe.MOE_EROUTE
    assert res["guards_ok"]
    assert np.all(res["expert_x"] == CANARY)
    assert np.all(res["out"] == CANARY)
    assert np.all(res["slot_row"] == -1)
    # the same context then runs a valid layer normally
    layer = res["layer"]
    T, H, K = w.T, w.H, w.K
    x = _dev(li.x.view(np.int16))
    ex = torch.empty((T * K, H), dtype=torch.int16, device="cuda")
    out = torch.empty((T, H), dtype=torch.int16, device="cuda")
    layer.layer(x, _dev(li.topk_idx), _dev(li.topk_w), ex, _dev(li.y.view(np.int16)), out)
    assert layer.get_error() == moe.MOE_OK


def test_cluster_routing_is_available_on_this_device(moe):
    """The default routing path on a GB300 is the 16-CTA cluster kernel."""
    layer = moe.MoELayer(4096, 7168, 8, 256, 32)
    assert layer.get_option(moe.MOE_OPT_ROUTE_CLUSTER_CTAS) == 16
    assert layer.get_option(moe.MOE_OPT_ROUTE_VARIANT) == moe.ROUTE_CLUSTER
    assert layer.kernels_per_layer() == 3
    layer.set_option(moe.MOE_OPT_ROUTE_VARIANT, moe.ROUTE_SPLIT)
    assert layer.kernels_per_layer() == 4


def test_layer_replays_from_a_cuda_graph(moe, oracle_mod):
    """The four calls capture into a CUDA graph (no host sync, no allocation)
    and replays give the same bits as direct calls."""
    w = gen.custom("graph", T=1024, H=1024, K=8, E=64, N=8, seed_index=9)
    li = gen.make_inputs(w)
    d, out_ref = oracle_of(oracle_mod, w, li)
    x, idx, wt, y = _dev(li.x.view(np.int16)), _dev(li.topk_idx), _dev(li.topk_w), _dev(li.y.view(np.int16))
    ex = torch.zeros((w.T * w.K, w.H), dtype=torch.int16, device="cuda")
    out = torch.zeros((w.T, w.H), dtype=torch.int16, device="cuda")
    layer = moe.MoELayer(w.T, w.H, w.K, w.E, w.N)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        layer.layer(x, idx, wt, ex, y, out, s)  # first call sets kernel attributes outside the capture
    torch.cuda.synchronize()
    ex.zero_()
    out.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        layer.layer(x, idx, wt, ex, y, out, s)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert layer.get_error() == moe.MOE_OK
    assert np.array_equal(ex.cpu().numpy().view(np.uint16), d.expert_x)
    assert np.array_equal(out.cpu().numpy().view(np.uint16), out_ref)


def test_call_order_and_argument_checks(moe):
    T, H, K, E, N = 64, 64, 2, 8, 2
    layer = moe.MoELayer(T, H, K, E, N)
    x = torch.zeros((T, H), dtype=torch.int16, device="cuda")
    idx = torch.tensor([[t % E, (t + 1) % E] for t in range(T)], dtype=torch.int32, device="cuda")
    wt = torch.full((T, K), 0.5, dtype=torch.float32, device="cuda")
    ex = torch.zeros((T * K, H), dtype=torch.int16, device="cuda")
    out = torch.zeros((T, H), dtype=torch.int16, device="cuda")
    with pytest.raises(moe.MoEError) as ei:
        layer.dispatch_recv()
    assert ei.value.code == moe.MOE_ESTATE
    with pytest.raises(moe.MoEError) as ei:
        layer.combine_recv(wt, out)
    assert ei.value.code == moe.MOE_ESTATE
    # too few rows, misaligned pointer
    with pytest.raises(moe.MoEError) as ei:
        moe.moe_dispatch_send(layer.ctx, x, idx, ex, T * K - 1)
    assert ei.value.code == moe.MOE_EINVAL
    with pytest.raises(moe.MoEError) as ei:
        moe.moe_dispatch_send(layer.ctx, x.data_ptr() + 2, idx, ex, T * K)
    assert ei.value.code == moe.MOE_EINVAL
    layer.dispatch_send(x, idx, ex)
    with pytest.raises(moe.MoEError) as ei:
        layer.dispatch_send(x, idx, ex)
    assert ei.value.code == moe.MOE_ESTATE
    layer.dispatch_recv()
    with pytest.raises(moe.MoEError) as ei:
        moe.moe_combine_send(layer.ctx, ex, T * K - 1)
    assert ei.value.code == moe.MOE_EINVAL
    layer.combine_send(ex)
    with pytest.raises(moe.MoEError) as ei:
        moe.moe_combine_recv(layer.ctx, wt, out.data_ptr() + 8)
    assert ei.value.code == moe.MOE_EINVAL
    layer.combine_recv(wt, out)
    assert layer.get_error() == moe.MOE_OK
    for opt, val in [(moe.MOE_OPT_PACK_STAGES, 1), (moe.MOE_OPT_PACK_VARIANT, 5),
                     (moe.MOE_OPT_PACK_PIECE_BYTES, 24), (moe.MOE_OPT_PACK_SCHEDULE, 2),
                     (moe.MOE_OPT_PACK_SCHEDULE, -2), (99, 0)]:
        with pytest.raises(moe.MoEError):
            layer.set_option(opt, val)
    assert layer.get_option(moe.MOE_OPT_PACK_SCHEDULE) == -1  # automatic by default
    assert layer.get_option(moe.MOE_OPT_COMBINE_SCHEDULE) == -1
    with pytest.raises(moe.MoEError):
        layer.set_option(moe.MOE_OPT_COMBINE_SCHEDULE, 3)
    layer.set_option(moe.MOE_OPT_PACK_SCHEDULE, 1)
    assert layer.get_option(moe.MOE_OPT_PACK_SCHEDULE) == 1


def test_repeat_runs_are_byte_identical(moe):
    w = gen.custom("det", T=2048, H=1024, K=8, E=64, N=8, seed_index=5)
    li = gen.make_inputs(w)
    first = run_gpu(moe, w, li)
    for _ in range(10):
        again = run_gpu(moe, w, li)
        for k in ("expert_x", "out", "slot_row", "row_src", "expert_offsets", "src_offsets"):
            assert np.array_equal(first[k], again[k]), k


def test_kernel_events_time_both_kernels_and_keep_results(moe, oracle_mod):
    w = gen.custom("timed", T=1024, H=2048, K=8, E=64, N=8, router="uniform_random", seed_index=83)
    li = gen.make_inputs(w)
    d, out_ref = oracle_of(oracle_mod, w, li)
    res = run_gpu(moe, w, li, kernel_events=1)
    assert_parity(res, d, out_ref, w)
    layer = moe.MoELayer(w.T, w.H, w.K, w.E, w.N)
    assert layer.kernel_times() == (-1.0, -1.0)  # nothing timed yet
    layer.set_option(moe.MOE_OPT_KERNEL_EVENTS, 1)
    x, idx, wt, y = (_dev(li.x.view(np.int16)), _dev(li.topk_idx), _dev(li.topk_w), _dev(li.y.view(np.int16)))
    ex = torch.zeros((w.T * w.K, w.H), dtype=torch.int16, device="cuda")
    out = torch.zeros((w.T, w.H), dtype=torch.int16, device="cuda")
    layer.layer(x, idx, wt, ex, y, out)
    pack_ms, comb_ms = layer.kernel_times()
    assert 0.0 < pack_ms < 100.0 and 0.0 < comb_ms < 100.0
    assert layer.get_error() == 0
    # The staged dispatch and the two-level combine are not timed: after them
    # the times of the earlier layer are no longer reported.
    send = torch.zeros_like(ex)
    partial = torch.zeros((layer.partial_rows(), w.H), dtype=torch.int16, device="cuda")
    layer.dispatch_send_staged(x, idx, send, ex)
    layer.dispatch_recv()
    layer.combine_send(y)
    layer.combine_recv_two_level(wt, partial, out)
    assert layer.kernel_times() == (-1.0, -1.0)
    assert layer.get_error() == 0
    with pytest.raises(moe.MoEError):
        layer.set_option(moe.MOE_OPT_KERNEL_EVENTS, 2)


ROUTE_PACK_OPTIONS = [
    dict(),
    dict(pack_stages=2, pack_store_depth=1),
    dict(pack_piece_bytes=1024, pack_ctas_per_sm=1, pack_stages=16),
    dict(pdl=0, cache_hints=0),
    dict(pack_store_depth=5, pack_stages=6, combine_variant=0, combine_schedule=1),
]
ROUTE_PACK_SHAPES = [s for s in EDGE if s[0] * s[2] <= 16384 and (s[0] + 31) // 32 * s[3] <= 4096] + [
    (4000, 4104, 4, 32, 8, "uniform_random"),   # two pieces per row, many units per CTA
    (2048, 512, 8, 64, 8, "uniform_random"),    # at both limits: T*K = 16384, E*ceil(T/32) = 4096
    (1024, 64, 4, 16, 4, "rank0_only"),         # every token to rank 0
]


@pytest.mark.parametrize("route", [4, 5], ids=["in-pack", "one-cta"])
@pytest.mark.parametrize("opts", ROUTE_PACK_OPTIONS, ids=[str(o) for o in ROUTE_PACK_OPTIONS])
@pytest.mark.parametrize("shape", ROUTE_PACK_SHAPES, ids=["x".join(map(str, s[:5])) for s in ROUTE_PACK_SHAPES])
def test_route_pack_shapes_and_options(moe, oracle_mod, shape, opts, route):
    """Routing inside the pack kernel (route variant 4), or the same routing
    alone in one CTA ahead of the pack (variant 5): every table and row
    bit-exact, nothing written outside the outputs."""
    T, H, K, E, N, router = shape
    w = gen.custom("fused", T=T, H=H, K=K, E=E, N=N, router=router, seed_index=61)
    li = gen.make_inputs(w)
    d, out_ref = oracle_of(oracle_mod, w, li)
    res = run_gpu(moe, w, li, extra_rows=4, route_variant=route, **opts)
    assert res["layer"].kernels_per_layer() == (2 if route == 4 else 3)
    assert_parity(res, d, out_ref, w, extra_rows=4)


def test_route_pack_is_the_automatic_choice_for_small_layers_only(moe):
    small = moe.MoELayer(4096, 4096, 2, 8, 8)  # Mixtral-sized
    assert small.get_option(moe.MOE_OPT_ROUTE_VARIANT) == moe.ROUTE_FUSED
    assert small.kernels_per_layer() == 2
    small.set_option(moe.MOE_OPT_PACK_SCHEDULE, 1)  # the unit queue is a two-kernel feature
    assert small.get_option(moe.MOE_OPT_ROUTE_VARIANT) == moe.ROUTE_CLUSTER
    small.set_option(moe.MOE_OPT_PACK_SCHEDULE, -1)
    small.set_option(moe.MOE_OPT_PACK_VARIANT, moe.PACK_VECTOR)
    assert small.get_option(moe.MOE_OPT_ROUTE_VARIANT) == moe.ROUTE_CLUSTER
    big = moe.MoELayer(4096, 7168, 8, 256, 32)  # DeepSeek-sized: T*K = 32768
    assert big.get_option(moe.MOE_OPT_ROUTE_VARIANT) == moe.ROUTE_CLUSTER
    with pytest.raises(moe.MoEError) as ei:
        big.set_option(moe.MOE_OPT_ROUTE_VARIANT, moe.ROUTE_FUSED)
    assert ei.value.code == moe.MOE_EINVAL
    with pytest.raises(moe.MoEError):
        small.set_option(moe.MOE_OPT_ROUTE_VARIANT, 6)


@pytest.mark.parametrize("route", [4, 5], ids=["in-pack", "one-cta"])
@pytest.mark.parametrize("bad", ["out_of_range", "negative", "repeated"])
def test_route_pack_routing_errors_write_nothing(moe, bad, route):
    w = gen.custom("bad", T=300, H=64, K=4, E=16, N=4, seed_index=3)
    li = gen.make_inputs(w)
    idx = li.topk_idx.copy()
    if bad == "out_of_range":
        idx[123, 2] = 16
    elif bad == "negative":
        idx[7, 0] = -1
    else:
        idx[299, 3] = idx[299, 1]
    li2 = gen.LayerInputs(w, li.x, idx, li.topk_w, li.y)
    res = run_gpu(moe, w, li2, route_variant=route, combine_variant=0)
    assert res["status"] == moe.MOE_EROUTE
    assert res["guards_ok"]
    assert np.all(res["expert_x"] == CANARY)
    assert np.all(res["out"] == CANARY)
    assert np.all(res["slot_row"] == -1)
    assert np.all(res["expert_counts"] == 0) and np.all(res["expert_offsets"] == 0)
    assert np.all(res["src_offsets"] == 0) and np.all(res["rank_offsets"] == 0)
    layer = res["layer"]
    T, H, K = w.T, w.H, w.K
    ex = torch.empty((T * K, H), dtype=torch.int16, device="cuda")
    out = torch.empty((T, H), dtype=torch.int16, device="cuda")
    layer.layer(_dev(li.x.view(np.int16)), _dev(li.topk_idx), _dev(li.topk_w), ex, _dev(li.y.view(np.int16)), out)
    assert layer.get_error() == moe.MOE_OK


def test_route_pack_resets_the_combine_queue_every_layer(moe, oracle_mod):
    """Layers with different routings on one context, routing inside the pack
    and the bulk combine's token queue on: the pack kernel resets the queue
    each layer, also across a routing error and a two-kernel layer."""
    T, H, K, E, N = 1024, 1024, 8, 32, 8
    layer = moe.MoELayer(T, H, K, E, N, combine_variant=0, combine_schedule=1)
    ex = torch.empty((T * K, H), dtype=torch.int16, device="cuda")
    out = torch.empty((T, H), dtype=torch.int16, device="cuda")
    for n, route in enumerate([4, 4, 3, 4, 5, 0, 5, 4]):
        w = gen.custom("queue", T=T, H=H, K=K, E=E, N=N, router="uniform_random", seed_index=70 + n)
        li = gen.make_inputs(w)
        d, out_ref = oracle_of(oracle_mod, w, li)
        x, idx, wt, y = (_dev(li.x.view(np.int16)), _dev(li.topk_idx), _dev(li.topk_w), _dev(li.y.view(np.int16)))
        layer.set_option(moe.MOE_OPT_ROUTE_VARIANT, route)
        if n == 3:
            bad = li.topk_idx.copy()
            bad[9, 5] = bad[9, 0]
            layer.layer(x, _dev(bad), wt, ex, y, out)
            assert layer.get_error() == moe.MOE_EROUTE
        lay = layer.layer(x, idx, wt, ex, y, out)
        assert layer.get_error() == 0
        assert np.array_equal(lay["slot_row"].cpu().numpy(), d.slot_row)
        assert np.array_equal(ex.cpu().numpy().view(np.uint16), d.expert_x), n
        assert np.array_equal(out.cpu().numpy().view(np.uint16), out_ref), n


UNALIGNED_SHAPES = [  # (T, H, K, E, N): T*K not a multiple of 4 for the odd ones
    (64, 256, 2, 8, 2),
    (1000, 136, 5, 40, 4),
    (3, 24, 3, 3, 1),
    (4096, 512, 8, 256, 32),
]


@pytest.mark.parametrize("route", [0, 1, 2, 3, 4, 5])
@pytest.mark.parametrize("shape", UNALIGNED_SHAPES, ids=["x".join(map(str, s)) for s in UNALIGNED_SHAPES])
def test_index_array_four_bytes_off_a_16_byte_boundary(moe, oracle_mod, shape, route):
    """topk_idx that is 4-byte aligned but not 16-byte aligned: the routing
    kernels then load every index with plain loads instead of bulk or
    16-byte vector copies; bf16 and fp8 payloads, every routing kernel."""
    T, H, K, E, N = shape
    w = gen.custom("unaligned", T=T, H=H, K=K, E=E, N=N, seed_index=131)
    li = gen.make_inputs(w)
    layer = moe.MoELayer(T, H, K, E, N)
    try:
        layer.set_option(moe.MOE_OPT_ROUTE_VARIANT, route)
    except moe.MoEError:
        pytest.skip("route variant not available for this shape")
    d, out_ref = oracle_of(oracle_mod, w, li)
    big = torch.zeros(T * K + 4, dtype=torch.int32, device="cuda")
    big[1:1 + T * K] = _dev(li.topk_idx).view(-1)
    idx = big[1:1 + T * K].view(T, K)
    assert idx.data_ptr() % 16 == 4
    x, wt, y = _dev(li.x.view(np.int16)), _dev(li.topk_w), _dev(li.y.view(np.int16))
    ex = torch.zeros((T * K, H), dtype=torch.int16, device="cuda")
    out = torch.zeros((T, H), dtype=torch.int16, device="cuda")
    lay = layer.layer(x, idx, wt, ex, y, out)
    assert layer.get_error() == moe.MOE_OK
    assert np.array_equal(lay["slot_row"].cpu().numpy(), d.slot_row)
    assert np.array_equal(lay["row_src"].cpu().numpy(), d.row_src)
    assert np.array_equal(lay["src_offsets"].cpu().numpy().reshape(-1), d.src_offsets.reshape(-1))
    assert np.array_equal(ex.cpu().numpy().view(np.uint16), d.expert_x)
    assert np.array_equal(out.cpu().numpy().view(np.uint16), out_ref)
    if H % 128 == 0:
        _, xq_ref, xs_ref = oracle_mod.dispatch_fp8(li.x, li.topk_idx, E, N)
        xq = torch.zeros((T * K, H), dtype=torch.uint8, device="cuda")
        xs = torch.zeros((T * K, H // 128), dtype=torch.float32, device="cuda")
        layer.dispatch_send_fp8(x, idx, xq, xs)
        lay = layer.dispatch_recv()
        layer.combine_send(y)
        layer.combine_recv(wt, out)
        assert layer.get_error() == moe.MOE_OK
        assert np.array_equal(lay["slot_row"].cpu().numpy(), d.slot_row)
        assert np.array_equal(xq.cpu().numpy(), xq_ref)
        assert np.array_equal(xs.cpu().numpy().view(np.uint32), xs_ref.view(np.uint32))
    layer.close()
