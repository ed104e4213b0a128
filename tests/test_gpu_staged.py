"""GPU two-stage dispatch (moe_dispatch_send_staged) vs the CPU oracle.

Bar: the send rows (per-peer send buffers), the grouped rows and the routing
tables are compared bit for bit with the oracle's two-stage dispatch; the
grouped rows also equal the direct dispatch's, and the combine that follows is
bit-exact.  Guard rows around both buffers catch stray writes."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

from combine_route_count_gb300 import inputs as gen  # noqa: E402

GUARD = 2
CANARY = 0x5A5A


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


def run_staged(moe, w, li, **options):
    T, H, K = w.T, w.H, w.K
    rows = T * K
    layer = moe.MoELayer(T, H, K, w.E, w.N, **options)
    sbig = torch.full((GUARD + rows + GUARD, H), CANARY, dtype=torch.int16, device="cuda")
    ebig = torch.full((GUARD + rows + GUARD, H), CANARY, dtype=torch.int16, device="cuda")
    send, ex = sbig[GUARD:GUARD + rows], ebig[GUARD:GUARD + rows]
    out = torch.zeros((T, H), dtype=torch.int16, device="cuda")
    # inputs stay referenced until the layer is done: the context keeps raw pointers
    x, idx, wts = _dev(li.x.view(np.int16)), _dev(li.topk_idx), _dev(li.topk_w)
    y = _dev(li.y.view(np.int16)) if li.y is not None else torch.zeros((max(rows, 1), H), dtype=torch.int16,
                                                                       device="cuda")
    layer.dispatch_send_staged(x, idx, send, ex)
    lay = layer.dispatch_recv()
    layer.combine_send(y)
    layer.combine_recv(wts, out)
    status = layer.get_error()
    sb, eb = sbig.cpu().numpy().view(np.uint16), ebig.cpu().numpy().view(np.uint16)
    guards = all(np.all(a[:GUARD] == CANARY) and np.all(a[GUARD + rows:] == CANARY) for a in (sb, eb))
    return dict(status=status, send=sb[GUARD:GUARD + rows], ex=eb[GUARD:GUARD + rows], guards=bool(guards),
                slot_row=lay["slot_row"].cpu().numpy(), offsets=lay["expert_offsets"].cpu().numpy(),
                out=out.cpu().numpy().view(np.uint16))


def check(res, oracle_mod, w, li):
    send, dest, ex, sr = oracle_mod.dispatch_staged(li.x, li.topk_idx, w.E, w.N)
    d = oracle_mod.dispatch(li.x, li.topk_idx, w.E, w.N)
    assert res["status"] == 0
    assert res["guards"], "a write landed outside an output buffer"
    assert np.array_equal(res["slot_row"], sr)
    assert np.array_equal(res["offsets"], d.expert_offsets)
    assert np.array_equal(res["send"], send)
    assert np.array_equal(res["ex"], ex)
    assert np.array_equal(res["ex"], d.expert_x)
    if li.y is not None:
        assert np.array_equal(res["out"], oracle_mod.combine(li.y, li.topk_w, d.slot_row))


@pytest.mark.parametrize("name", [w.name for w in gen.WORKLOADS])
def test_staged_named_workloads(moe, oracle_mod, name):
    w = gen.BY_NAME[name]
    li = gen.make_inputs(w)
    check(run_staged(moe, w, li), oracle_mod, w, li)


STAGED_EDGE = [
    (1, 8, 1, 1, 1),
    (96, 136, 3, 12, 3),
    (1000, 1024, 16, 64, 4),
    (128, 512, 8, 32, 32),
    (64, 7168, 8, 1024, 64),   # E = MOE_MAX_EXPERTS: the scan uses every thread
    (4096, 64, 2, 8, 8),       # many small rows
]


@pytest.mark.parametrize("pack_schedule", [-1, 0, 1])
@pytest.mark.parametrize("route_variant", [0, 1, 2])
@pytest.mark.parametrize("shape", STAGED_EDGE, ids=["x".join(map(str, s)) for s in STAGED_EDGE])
def test_staged_edge_shapes(moe, oracle_mod, shape, route_variant, pack_schedule):
    T, H, K, E, N = shape
    w = gen.custom("stagededge", T=T, H=H, K=K, E=E, N=N, seed_index=67)
    li = gen.make_inputs(w)
    check(run_staged(moe, w, li, route_variant=route_variant, pack_schedule=pack_schedule), oracle_mod, w, li)


def test_staged_empty_layer(moe):
    layer = moe.MoELayer(0, 64, 2, 8, 2)
    x = torch.zeros((1, 64), dtype=torch.int16, device="cuda")
    idx = torch.zeros((1, 2), dtype=torch.int32, device="cuda")
    buf = torch.zeros((1, 64), dtype=torch.int16, device="cuda")
    layer.dispatch_send_staged(x, idx, buf, buf)
    layer.dispatch_recv()
    assert layer.get_error() == 0


def test_staged_routing_error_writes_nothing(moe):
    w = gen.custom("stagedbad", T=64, H=256, K=2, E=8, N=2, seed_index=71)
    li = gen.make_inputs(w)
    idx = li.topk_idx.copy()
    idx[9] = [3, 3]
    res = run_staged(moe, w, gen.LayerInputs(w, li.x, idx, li.topk_w, li.y))
    assert res["status"] == moe.MOE_EROUTE
    assert res["guards"]
    assert np.all(res["send"] == CANARY) and np.all(res["ex"] == CANARY)


def test_staged_short_send_buffer_is_rejected(moe):
    layer = moe.MoELayer(64, 256, 2, 8, 2)
    x = torch.zeros((64, 256), dtype=torch.int16, device="cuda")
    idx = torch.tensor([[0, 1]] * 64, dtype=torch.int32, device="cuda")
    ex = torch.zeros((128, 256), dtype=torch.int16, device="cuda")
    with pytest.raises(moe.MoEError) as ei:
        layer.dispatch_send_staged(x, idx, ex[:127], ex)
    assert ei.value.code == moe.MOE_EINVAL
