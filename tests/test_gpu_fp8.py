"""GPU fp8 dispatch (moe_dispatch_send_fp8) vs the CPU oracle.

Bar: the E4M3 codes and the float32 block scales of every dispatched row are
compared bit for bit with the oracle's quantisation placed by the oracle's
dispatch; counts, offsets and slot_row are the same as for the bf16 payload;
the bf16 combine that follows is bit-exact as well.  Guard rows catch stray
writes."""
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


def run_fp8(moe, w, li, **options):
    T, H, K = w.T, w.H, w.K
    rows = T * K
    xq_big = torch.full((GUARD + rows + GUARD, H), CANARY8, dtype=torch.uint8, device="cuda")
    xs_big = torch.full((GUARD + rows + GUARD, H // 128), CANARYF, dtype=torch.float32, device="cuda")
    xq, xs = xq_big[GUARD:GUARD + rows], xs_big[GUARD:GUARD + rows]
    out = torch.zeros((T, H), dtype=torch.int16, device="cuda")
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
    return dict(status=status, xq=xqb[GUARD:GUARD + rows], xs=xsb[GUARD:GUARD + rows], guards=bool(guards),
                slot_row=lay["slot_row"].cpu().numpy(), offsets=lay["expert_offsets"].cpu().numpy(),
                out=out.cpu().numpy().view(np.uint16))


def check(res, oracle_mod, w, li):
    d, xq_ref, xs_ref = oracle_mod.dispatch_fp8(li.x, li.topk_idx, w.E, w.N)
    assert res["status"] == 0
    assert res["guards"], "a write landed outside an output buffer"
    assert np.array_equal(res["slot_row"], d.slot_row)
    assert np.array_equal(res["offsets"], d.expert_offsets)
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


@pytest.mark.parametrize("pack_schedule", [0, 1])
@pytest.mark.parametrize("route_variant", [0, 1, 2])
@pytest.mark.parametrize("shape", FP8_EDGE, ids=["x".join(map(str, s)) for s in FP8_EDGE])
def test_fp8_edge_shapes(moe, oracle_mod, shape, route_variant, pack_schedule):
    T, H, K, E, N = shape
    w = gen.custom("fp8edge", T=T, H=H, K=K, E=E, N=N, seed_index=17)
    li = gen.make_inputs(w)
    # wide dynamic range across rows and an all-zero block
    xf = gen.bf16_bits_to_f32(li.x) * np.exp(np.random.default_rng(3).uniform(-8, 8, (T, 1))).astype(np.float32)
    xf[0, :128] = 0.0
    li = gen.LayerInputs(w, gen.to_bf16_bits(xf), li.topk_idx, li.topk_w, li.y)
    check(run_fp8(moe, w, li, route_variant=route_variant, pack_schedule=pack_schedule), oracle_mod, w, li)


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


def test_fp8_rejects_rows_not_a_multiple_of_the_block(moe):
    layer = moe.MoELayer(8, 200, 2, 4, 2)
    x = torch.zeros((8, 200), dtype=torch.int16, device="cuda")
    idx = torch.zeros((8, 2), dtype=torch.int32, device="cuda")
    xq = torch.zeros((16, 200), dtype=torch.uint8, device="cuda")
    xs = torch.zeros((16, 2), dtype=torch.float32, device="cuda")
    with pytest.raises(moe.MoEError) as ei:
        layer.dispatch_send_fp8(x, idx, xq, xs)
    assert ei.value.code == moe.MOE_EINVAL
