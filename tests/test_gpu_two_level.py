"""GPU two-level combine (moe_combine_recv_two_level) vs the CPU oracle.

Bar: the partial rows each token uses and the combined output are compared
bit for bit with the oracle's two-level combine on the same seeded inputs;
rows a token does not use keep their sentinel, and guard rows around every
output catch stray writes."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

from combine_route_count_gb300 import inputs as gen  # noqa: E402

GUARD = 2
SENTINEL = 0x7FC1  # a NaN pattern neither side writes


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


def run_two_level(moe, w, li, **options):
    T, H, K, N = w.T, w.H, w.K, w.N
    slots = min(K, N)
    layer = moe.MoELayer(T, H, K, w.E, N, **options)
    assert layer.partial_rows() == T * slots
    prow = T * slots
    pbig = torch.full((GUARD + prow + GUARD, H), SENTINEL, dtype=torch.int16, device="cuda")
    obig = torch.full((GUARD + T + GUARD, H), SENTINEL, dtype=torch.int16, device="cuda")
    partial, out = pbig[GUARD:GUARD + prow], obig[GUARD:GUARD + T]
    ex = torch.zeros((max(T * K, 1), H), dtype=torch.int16, device="cuda")
    # every device input stays referenced until the layer has finished: the
    # context keeps raw pointers (combine_send only registers expert_y)
    x, idx, y, wts = _dev(li.x.view(np.int16)), _dev(li.topk_idx), _dev(li.y.view(np.int16)), _dev(li.topk_w)
    layer.dispatch_send(x, idx, ex)
    lay = layer.dispatch_recv()
    layer.combine_send(y)
    layer.combine_recv_two_level(wts, partial, out)
    status = layer.get_error()
    pb, ob = pbig.cpu().numpy().view(np.uint16), obig.cpu().numpy().view(np.uint16)
    guards = (np.all(pb[:GUARD] == SENTINEL) and np.all(pb[GUARD + prow:] == SENTINEL)
              and np.all(ob[:GUARD] == SENTINEL) and np.all(ob[GUARD + T:] == SENTINEL))
    return dict(status=status, partial=pb[GUARD:GUARD + prow], out=ob[GUARD:GUARD + T], guards=bool(guards),
                slot_row=lay["slot_row"].cpu().numpy())


def check(res, oracle_mod, w, li):
    d = oracle_mod.dispatch(li.x, li.topk_idx, w.E, w.N)
    slots = min(w.K, w.N)
    sentinel = np.full((w.T * slots, w.H), SENTINEL, np.uint16)
    out, part, nr = oracle_mod.combine_two_level(li.y, li.topk_idx, li.topk_w, d.slot_row, w.E, w.N,
                                                 partial=sentinel)
    assert res["status"] == 0
    assert res["guards"], "a write landed outside an output buffer"
    assert np.array_equal(res["slot_row"], d.slot_row)
    assert np.array_equal(res["partial"], part)  # used rows bit-exact, unused rows untouched
    assert np.array_equal(res["out"], out)
    return nr


@pytest.mark.parametrize("name", [w.name for w in gen.WORKLOADS])
def test_two_level_named_workloads(moe, oracle_mod, name):
    w = gen.BY_NAME[name]
    li = gen.make_inputs(w)
    nr = check(run_two_level(moe, w, li), oracle_mod, w, li)
    if name == "worst":
        assert np.all(nr == 1)  # all experts on rank 0: one partial per token


TWO_LEVEL_EDGE = [
    (1, 8, 1, 1, 1),          # one token, one expert, one rank
    (64, 256, 4, 8, 1),       # one rank: partial = the single-level answer
    (96, 136, 3, 12, 3),      # odd K, H not a multiple of 32 chunks
    (1000, 1024, 16, 64, 4),  # K = 16 > N: several experts per rank
    (128, 512, 8, 32, 32),    # E = N: one expert per rank, partial = one product
    (64, 7168, 8, 1024, 64),  # many ranks, binary search over 65 offsets
]


@pytest.mark.parametrize("shape", TWO_LEVEL_EDGE, ids=["x".join(map(str, s)) for s in TWO_LEVEL_EDGE])
def test_two_level_edge_shapes(moe, oracle_mod, shape):
    T, H, K, E, N = shape
    w = gen.custom("twoleveledge", T=T, H=H, K=K, E=E, N=N, seed_index=41)
    li = gen.make_inputs(w)
    check(run_two_level(moe, w, li), oracle_mod, w, li)


def test_two_level_matches_single_level_on_one_rank(moe, oracle_mod):
    w = gen.custom("onerank", T=256, H=512, K=4, E=16, N=1, seed_index=43)
    li = gen.make_inputs(w)
    res = run_two_level(moe, w, li)
    d = oracle_mod.dispatch(li.x, li.topk_idx, w.E, w.N)
    assert np.array_equal(res["out"], oracle_mod.combine(li.y, li.topk_w, d.slot_row))


def test_two_level_routing_error_writes_nothing(moe):
    w = gen.custom("tlbad", T=64, H=256, K=2, E=8, N=2, seed_index=47)
    li = gen.make_inputs(w)
    idx = li.topk_idx.copy()
    idx[7, 0] = -3
    res = run_two_level(moe, w, gen.LayerInputs(w, li.x, idx, li.topk_w, li.y))
    assert res["status"] == moe.MOE_EROUTE
    assert res["guards"]
    assert np.all(res["partial"] == SENTINEL) and np.all(res["out"] == SENTINEL)


def test_two_level_argument_and_order_errors(moe):
    layer = moe.MoELayer(64, 256, 2, 8, 2)
    w = torch.zeros((64, 2), dtype=torch.float32, device="cuda")
    out = torch.zeros((64, 256), dtype=torch.int16, device="cuda")
    short = torch.zeros((64 * 2 - 1, 256), dtype=torch.int16, device="cuda")
    with pytest.raises(moe.MoEError) as ei:  # before dispatch: call order
        layer.combine_recv_two_level(w, short, out)
    assert ei.value.code == moe.MOE_ESTATE
    x = torch.zeros((64, 256), dtype=torch.int16, device="cuda")
    idx = torch.tensor([[0, 1]] * 64, dtype=torch.int32, device="cuda")
    ex = torch.zeros((128, 256), dtype=torch.int16, device="cuda")
    layer.dispatch_send(x, idx, ex)
    layer.dispatch_recv()
    layer.combine_send(ex)
    with pytest.raises(moe.MoEError) as ei:
        layer.combine_recv_two_level(w, short, out)
    assert ei.value.code == moe.MOE_EINVAL
    layer.combine_recv_two_level(w, torch.zeros((128, 256), dtype=torch.int16, device="cuda"), out)
    assert layer.get_error() == 0
