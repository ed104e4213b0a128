"""GPU fp8 dispatch (moe_dispatch_send_fp8) vs the CPU oracle.

Bar: the E4M3 codes and the float32 block scales of every dispatched row are
compared bit for bit with the oracle's quantisation placed by the oracle's
dispatch; counts, offsets, slot_row and row_src are the same as for the bf16
payload; the bf16 combine that follows is bit-exact as well.  Guard rows
catch stray writes.  Both forms are covered: routing kernel + fp8 pack, and
routing inside the fp8 pack (route_pack_fp8, route variant 4)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

from combine_route_count_gb300 import inputs as gen  # noqa: E402

GUARD = 2
CANARY8 = 0x5A
CANARYF = -7.25


@pytest.fixture(scope="module")
def moe():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from combine_route_count_gb300 import build, moe as m
    build.build()
    m.load_library()
    return m


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def run_fp8(moe, w, li, layer=None, **options):
    T, H, K = w.T, w.H, w.K
    rows = T * K
    xq_big = torch.full((GUARD + rows + GUARD, H), CANARY8, dtype=torch.uint8, device="cuda")
    xs_big = torch.full((GUARD + rows + GUARD, H // 128), CANARYF, dtype=torch.float32, device="cuda")
    xq, xs = xq_big[GUARD:GUARD + rows], xs_big[GUARD:GUARD + rows]
    out = torch.zeros((T, H), dtype=torch.int16, device="cuda")
    if layer is None:
        layer = moe.MoELayer(T, H, K, w.E, w.N, **options)
    layer.dispatch_send_fp8(_dev(li.x.view(np.int16)), _dev(li.topk_idx), xq, xs)
    lay = layer.dispatch_recv()
    y = _dev(li.y.view(np.int16)) if li.y is not None else torch.zeros((rows, H), dtype=torch.int16, device="cuda")
    layer.combine_send(y)
    layer.combine_recv(_dev(li.topk_w), out)
    status = layer.get_error()
    xqb, xsb = xq_big.cpu().numpy(), xs_big.cpu().numpy()
    guards = (np.all(xqb[:GUARD] == CANARY8) and np.all(xqb[GUARD + rows:] == CANARY8)
              and np.all(xsb[:GUARD] == CANARYF) and np.all(xsb[GUARD + rows:] == CANARYF))
    tables = {k: lay[k].cpu().numpy() for k in TABLES}
    return dict(status=status, xq=xqb[GUARD:GUARD + rows], xs=xsb[GUARD:GUARD + rows], guards=bool(guards),
                out=out.cpu().numpy().view(np.uint16), layer=layer, **tables)


TABLES = ("expert_counts", "expert_offsets", "src_offsets", "rank_offsets", "slot_row", "row_src")


def check(res, oracle_mod, w, li):
    d, xq_ref, xs_ref = oracle_mod.dispatch_fp8(li.x, li.topk_idx, w.E, w.N)
    assert res["status"] == 0
    assert res["guards"], "a write landed outside an output buffer"
    for key in TABLES:
        assert np.array_equal(res[key].reshape(-1), getattr(d, key).reshape(-1)), key
    assert np.array_equal(res["xq"], xq_ref)
    assert np.array_equal(res["xs"].view(np.uint32), xs_ref.view(np.uint32))
    if li.y is not None:
        assert np.array_equal(res["out"], oracle_mod.combine(li.y, li.topk_w, d.slot_row))


@pytest.mark.parametrize("pack_schedule", [-1, 0, 1])
@pytest.mark.parametrize("name", [w.name for w in gen.WORKLOADS])
def test_fp8_named_workloads(moe, oracle_mod, name, pack_schedule):
    w = gen.BY_NAME[name]
    li = gen.make_inputs(w)
    check(run_fp8(moe, w, li, pack_schedule=pack_schedule), oracle_mod, w, li)


FP8_EDGE = [
    (1, 128, 1, 1, 1),        # one token, one block
    (30, 2304, 3, 12, 3),     # 18 blocks: the last chunk pass leaves lanes idle; odd K
    (1000, 1024, 16, 64, 4),  # K = 16
    (257, 384, 2, 8, 1),      # ragged token ranges per CTA
]


def wide_range(w, li, seed=3):
    """Rows scaled over a wide dynamic range, and one all-zero block."""
    xf = gen.bf16_bits_to_f32(li.x) * np.exp(np.random.default_rng(seed).uniform(-8, 8, (w.T, 1))).astype(np.float32)
    xf[0, :128] = 0.0
    return gen.LayerInputs(w, gen.to_bf16_bits(xf), li.topk_idx, li.topk_w, li.y)


@pytest.mark.parametrize("pack_schedule", [0, 1])
@pytest.mark.parametrize("route_variant", [0, 1, 2, 3, 4])
@pytest.mark.parametrize("shape", FP8_EDGE, ids=["x".join(map(str, s)) for s in FP8_EDGE])
def test_fp8_edge_shapes(moe, oracle_mod, shape, route_variant, pack_schedule):
    T, H, K, E, N = shape
    w = gen.custom("fp8edge", T=T, H=H, K=K, E=E, N=N, seed_index=17)
    li = wide_range(w, gen.make_inputs(w))
    check(run_fp8(moe, w, li, route_variant=route_variant, pack_schedule=pack_schedule), oracle_mod, w, li)


FUSED_SHAPES = [  # (T, H, K, E, N, router): route_pack_fp8 (T*K <= 16384, E*ceil(T/32) <= 4096)
    (64, 256, 2, 8, 2, "softmax_topk"),
    (4096, 4096, 2, 8, 8, "uniform_random"),  # Mixtral-sized
    (2048, 512, 8, 64, 8, "uniform_random"),  # at both limits
    (1000, 1024, 16, 64, 4, "uniform_random"),  # K = 16
    (4000, 4096, 4, 32, 8, "uniform_random"),  # several tokens per group
    (1024, 128, 4, 16, 4, "rank0_only"),  # every token to rank 0
    (64, 7168, 8, 256, 32, "uniform_random"),  # 14 KiB rows, E = 256
    (257, 384, 2, 8, 1, "uniform_random"),  # ragged: not a multiple of the groups
    (1, 128, 1, 1, 1, "uniform_random"),
    (96, 2304, 3, 12, 3, "uniform_random"),  # odd K, 18 blocks
    (256, 16384, 2, 8, 2, "uniform_random"),  # 32 KiB rows: few stages fit
]
FUSED_OPTIONS = [
    dict(),
    dict(pack_ctas_per_sm=1, pack_stages=2),  # one group of 128 threads per CTA
    dict(pack_ctas_per_sm=8, pack_stages=2),
    dict(pack_ctas_per_sm=3, pack_stages=5),
    dict(pdl=0, max_sms=7),  # few CTAs: many tokens per group, stages refilled many times
]


@pytest.mark.parametrize("opts", FUSED_OPTIONS, ids=[str(o) for o in FUSED_OPTIONS])
@pytest.mark.parametrize("shape", FUSED_SHAPES, ids=["x".join(map(str, s[:5])) for s in FUSED_SHAPES])
def test_fp8_route_pack_shapes_and_options(moe, oracle_mod, shape, opts):
    T, H, K, E, N, router = shape
    w = gen.custom("fp8fused", T=T, H=H, K=K, E=E, N=N, router=router, seed_index=67)
    li = wide_range(w, gen.make_inputs(w), seed=5)
    check(run_fp8(moe, w, li, route_variant=4, **opts), oracle_mod, w, li)


@pytest.mark.parametrize("name", ["tiny", "mixtral", "deepseek"])
def test_fp8_contiguous_token_order(moe, oracle_mod, name):
    w = gen.BY_NAME[name]
    li = gen.make_inputs(w)
    check(run_fp8(moe, w, li, fp8_order=0), oracle_mod, w, li)


@pytest.mark.parametrize("shape", FP8_EDGE, ids=["x".join(map(str, s)) for s in FP8_EDGE])
def test_fp8_contiguous_edge_shapes(moe, oracle_mod, shape):
    T, H, K, E, N = shape
    w = gen.custom("fp8edge", T=T, H=H, K=K, E=E, N=N, seed_index=23)
    li = gen.make_inputs(w)
    check(run_fp8(moe, w, li, fp8_order=0), oracle_mod, w, li)


@pytest.mark.parametrize("pack_schedule", [0, 1])
def test_fp8_routing_error_writes_nothing(moe, pack_schedule):
    w = gen.custom("fp8bad", T=64, H=256, K=2, E=8, N=2, seed_index=19)
    li = gen.make_inputs(w)
    idx = li.topk_idx.copy()
    idx[5, 1] = 99
    res = run_fp8(moe, w, gen.LayerInputs(w, li.x, idx, li.topk_w, li.y), pack_schedule=pack_schedule)
    assert res["status"] == moe.MOE_EROUTE
    assert res["guards"]
    assert np.all(res["xq"] == CANARY8) and np.all(res["xs"] == CANARYF)


@pytest.mark.parametrize("bad", ["out_of_range", "negative", "repeated"])
def test_fp8_route_pack_routing_errors_write_nothing(moe, oracle_mod, bad):
    w = gen.custom("fp8bad", T=300, H=256, K=4, E=16, N=4, seed_index=29)
    li = gen.make_inputs(w)
    idx = li.topk_idx.copy()
    if bad == "out_of_range":
        idx[123, 2] = 16
    elif bad == "negative":
        idx[7, 0] = -1
    else:
        idx[299, 3] = idx[299, 1]
    res = run_fp8(moe, w, gen.LayerInputs(w, li.x, idx, li.topk_w, li.y), route_variant=4)
    assert res["status"] == moe.MOE_EROUTE
    assert res["guards"]
    assert np.all(res["xq"] == CANARY8) and np.all(res["xs"] == CANARYF)
    assert np.all(res["slot_row"] == -1)
    for key in ("expert_counts", "expert_offsets", "src_offsets", "rank_offsets"):
        assert np.all(res[key] == 0), key
    # The same context runs a valid layer next.
    check(run_fp8(moe, w, li, layer=res["layer"]), oracle_mod, w, li)


def test_fp8_route_pack_resets_the_combine_queue_every_layer(moe, oracle_mod):
    """fp8 layers on one context with the bulk combine's token queue on,
    routing inside the fp8 pack or in its own kernel: each layer's routing
    resets the queue, also after a routing error."""
    T, H, K, E, N = 1024, 1024, 8, 32, 8
    layer = moe.MoELayer(T, H, K, E, N, combine_variant=0, combine_schedule=1)
    for n, route in enumerate([4, 4, 3, 4, 0, 1, 4]):
        w = gen.custom("fp8queue", T=T, H=H, K=K, E=E, N=N, router="uniform_random", seed_index=80 + n)
        li = gen.make_inputs(w)
        layer.set_option(moe.MOE_OPT_ROUTE_VARIANT, route)
        if n == 3:  # a routing error in the middle
            idx = li.topk_idx.copy()
            idx[10, 1] = idx[10, 0]
            res = run_fp8(moe, w, gen.LayerInputs(w, li.x, idx, li.topk_w, li.y), layer=layer)
            assert res["status"] == moe.MOE_EROUTE
        check(run_fp8(moe, w, li, layer=layer), oracle_mod, w, li)


def test_fp8_route_pack_is_the_automatic_choice_for_small_layers_only(moe):
    small = moe.MoELayer(4096, 4096, 2, 8, 8)  # Mixtral-sized
    assert small.get_option(moe.MOE_OPT_ROUTE_VARIANT_FP8) == moe.ROUTE_FUSED
    small.set_option(moe.MOE_OPT_FP8_ORDER, 0)  # the contiguous order is a two-kernel feature
    assert small.get_option(moe.MOE_OPT_ROUTE_VARIANT_FP8) == moe.ROUTE_CLUSTER
    small.set_option(moe.MOE_OPT_FP8_ORDER, 1)
    small.set_option(moe.MOE_OPT_PACK_SCHEDULE, 1)  # so is the token queue
    assert small.get_option(moe.MOE_OPT_ROUTE_VARIANT_FP8) == moe.ROUTE_CLUSTER
    small.set_option(moe.MOE_OPT_ROUTE_VARIANT, moe.ROUTE_FUSED)  # ... unless forced
    assert small.get_option(moe.MOE_OPT_ROUTE_VARIANT_FP8) == moe.ROUTE_FUSED
    small.set_option(moe.MOE_OPT_ROUTE_VARIANT, moe.ROUTE_SINGLE)
    assert small.get_option(moe.MOE_OPT_ROUTE_VARIANT_FP8) == moe.ROUTE_SINGLE
    big = moe.MoELayer(4096, 7168, 8, 256, 32)  # DeepSeek-sized: T*K = 32768
    assert big.get_option(moe.MOE_OPT_ROUTE_VARIANT_FP8) == moe.ROUTE_CLUSTER
    odd = moe.MoELayer(64, 200, 2, 8, 2)  # rows not a multiple of the fp8 block
    assert odd.get_option(moe.MOE_OPT_ROUTE_VARIANT) == moe.ROUTE_FUSED
    assert odd.get_option(moe.MOE_OPT_ROUTE_VARIANT_FP8) in (moe.ROUTE_CLUSTER, moe.ROUTE_SPLIT)
    with pytest.raises(moe.MoEError):
        small.set_option(moe.MOE_OPT_ROUTE_VARIANT_FP8, 4)


def test_fp8_rejects_rows_not_a_multiple_of_the_block(moe):
    layer = moe.MoELayer(8, 200, 2, 4, 2)
    x = torch.zeros((8, 200), dtype=torch.int16, device="cuda")
    idx = torch.zeros((8, 2), dtype=torch.int32, device="cuda")
    xq = torch.zeros((16, 200), dtype=torch.uint8, device="cuda")
    xs = torch.zeros((16, 2), dtype=torch.float32, device="cuda")
    with pytest.raises(moe.MoEError) as ei:
        layer.dispatch_send_fp8(x, idx, xq, xs)
    assert ei.value.code == moe.MOE_EINVAL
