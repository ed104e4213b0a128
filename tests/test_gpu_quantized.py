"""GPU dispatch of already-quantised fp8 tokens (moe_dispatch_send_quantized)
vs the CPU oracle.

Bar: the E4M3 code rows and the float32 scale rows land bit for bit where the
oracle's dispatch places the token rows (the oracle's dispatch moves 16-bit
words, so each byte row is viewed as half as many 16-bit words); counts and
offsets match the bf16 dispatch; guard rows catch stray writes."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

from combine_route_count_gb300 import inputs as gen  # noqa: E402

GUARD = 2
CANARY8 = 0xA5
CANARYF = -3.5


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


def payload(w, seed):
    """Synthetic fp8 tokens: any byte pattern is a valid payload for a copy."""
    rng = np.random.default_rng(seed)
    xq = rng.integers(0, 256, size=(w.T, w.H), dtype=np.uint8)
    xs = rng.uniform(1e-3, 1.0, size=(w.T, w.H // 128)).astype(np.float32)
    return xq, xs


def run(moe, w, li, xq, xs, **options):
    T, H, K = w.T, w.H, w.K
    rows = T * K
    qbig = torch.full((GUARD + rows + GUARD, H), CANARY8, dtype=torch.uint8, device="cuda")
    sbig = torch.full((GUARD + rows + GUARD, H // 128), CANARYF, dtype=torch.float32, device="cuda")
    eq, es = qbig[GUARD:GUARD + rows], sbig[GUARD:GUARD + rows]
    layer = moe.MoELayer(T, H, K, w.E, w.N, **options)
    dq, ds, idx = _dev(xq), _dev(xs), _dev(li.topk_idx)
    layer.dispatch_send_quantized(dq, ds, idx, eq, es)
    lay = layer.dispatch_recv()
    status = layer.get_error()
    qb, sb = qbig.cpu().numpy(), sbig.cpu().numpy()
    guards = (np.all(qb[:GUARD] == CANARY8) and np.all(qb[GUARD + rows:] == CANARY8)
              and np.all(sb[:GUARD] == CANARYF) and np.all(sb[GUARD + rows:] == CANARYF))
    return dict(status=status, q=qb[GUARD:GUARD + rows], s=sb[GUARD:GUARD + rows], guards=bool(guards),
                slot_row=lay["slot_row"].cpu().numpy(), offsets=lay["expert_offsets"].cpu().numpy())


def check(res, oracle_mod, w, li, xq, xs):
    dq = oracle_mod.dispatch(xq.view(np.uint16), li.topk_idx, w.E, w.N)
    ds = oracle_mod.dispatch(xs.view(np.uint16), li.topk_idx, w.E, w.N)
    assert res["status"] == 0
    assert res["guards"], "a write landed outside an output buffer"
    assert np.array_equal(res["slot_row"], dq.slot_row)
    assert np.array_equal(res["offsets"], dq.expert_offsets)
    assert np.array_equal(res["q"].view(np.uint16), dq.expert_x)
    assert np.array_equal(res["s"].view(np.uint16), ds.expert_x)


@pytest.mark.parametrize("pack_schedule", [-1, 1])
@pytest.mark.parametrize("name", ["mixtral", "deepseek", "kimi", "worst"])
def test_quantized_named_workloads(moe, oracle_mod, name, pack_schedule):
    w = gen.BY_NAME[name]
    li = gen.make_inputs(w, with_y=False)
    xq, xs = payload(w, 89)
    check(run(moe, w, li, xq, xs, pack_schedule=pack_schedule), oracle_mod, w, li, xq, xs)


@pytest.mark.parametrize("pack_schedule", [0, 1])
@pytest.mark.parametrize("shape", [(1, 512, 1, 1, 1), (1000, 1024, 16, 64, 4), (96, 512, 3, 12, 3)],
                         ids=["1x512x1", "1000x1024x16", "96x512x3"])
def test_quantized_edge_shapes(moe, oracle_mod, shape, pack_schedule):
    T, H, K, E, N = shape
    w = gen.custom("q", T=T, H=H, K=K, E=E, N=N, seed_index=97)
    li = gen.make_inputs(w, with_y=False)
    xq, xs = payload(w, 101)
    check(run(moe, w, li, xq, xs, pack_schedule=pack_schedule), oracle_mod, w, li, xq, xs)


def test_quantized_routing_error_writes_nothing(moe):
    w = gen.custom("qbad", T=64, H=512, K=2, E=8, N=2, seed_index=103)
    li = gen.make_inputs(w, with_y=False)
    idx = li.topk_idx.copy()
    idx[4] = [7, 7]
    xq, xs = payload(w, 107)
    res = run(moe, w, gen.LayerInputs(w, li.x, idx, li.topk_w, None), xq, xs)
    assert res["status"] == moe.MOE_EROUTE
    assert res["guards"] and np.all(res["q"] == CANARY8) and np.all(res["s"] == CANARYF)


def test_quantized_rejects_rows_that_are_not_16_byte_scale_rows(moe):
    layer = moe.MoELayer(8, 256, 2, 4, 2)  # 2 scales per row = 8 bytes
    q = torch.zeros((8, 256), dtype=torch.uint8, device="cuda")
    s = torch.zeros((8, 2), dtype=torch.float32, device="cuda")
    idx = torch.zeros((8, 2), dtype=torch.int32, device="cuda")
    with pytest.raises(moe.MoEError) as ei:
        layer.dispatch_send_quantized(q, s, idx, torch.zeros((16, 256), dtype=torch.uint8, device="cuda"),
                                      torch.zeros((16, 2), dtype=torch.float32, device="cuda"))
    assert ei.value.code == moe.MOE_EINVAL
