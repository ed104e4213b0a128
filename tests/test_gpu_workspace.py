"""Writes stay inside the caller's workspace, through the C ABI.

The workspace holds every routing table (counts, offsets, slot_row, row_src,
the error word), the send tables of the two-stage and the dense dispatch and
the plan of the two-level combine.  Each test places it between canary
bytes, drives one entry point after another on the same context (direct,
fp8, already quantised, two-stage and dense dispatch; receiver, two-level
and dense combine; a layer
with a bad expert index, which makes every kernel take its error path) and
checks that no canary byte changed and that the results still match the
oracle where they are defined."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

from combine_route_count_gb300 import inputs as gen  # noqa: E402

GUARD = 4096
CANARY = 0xA5


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


SHAPES = [
    # (T, H, K, E, N)
    (1000, 512, 5, 40, 4),
    (1024, 512, 16, 1024, 8),
    (64, 1024, 2, 8, 2),
    (3, 512, 3, 3, 1),
]


@pytest.mark.parametrize("shape", SHAPES, ids=["x".join(map(str, s)) for s in SHAPES])
def test_every_entry_point_stays_inside_the_workspace(moe, oracle_mod, shape):
    T, H, K, E, N = shape
    w = gen.custom("ws", T=T, H=H, K=K, E=E, N=N, router="uniform_random", seed_index=23)
    li = gen.make_inputs(w)
    nbytes = moe.moe_workspace_bytes(moe.make_config(T, H, K, E, N))
    big = torch.full((GUARD + nbytes + GUARD,), CANARY, dtype=torch.uint8, device="cuda")
    layer = moe.MoELayer(T, H, K, E, N, workspace=big[GUARD:GUARD + nbytes])

    def guards_intact():
        b = big.cpu().numpy()
        return bool(np.all(b[:GUARD] == CANARY) and np.all(b[GUARD + nbytes:] == CANARY))

    d = oracle_mod.dispatch(li.x, li.topk_idx, E, N)
    out_ref = oracle_mod.combine(li.y, li.topk_w, d.slot_row)
    rows = T * K
    x, idx, wt, y = _dev(li.x.view(np.int16)), _dev(li.topk_idx), _dev(li.topk_w), _dev(li.y.view(np.int16))
    ex = torch.empty((rows, H), dtype=torch.int16, device="cuda")
    out = torch.empty((T, H), dtype=torch.int16, device="cuda")

    # direct dispatch + receiver combine
    lay = layer.layer(x, idx, wt, ex, y, out)
    assert layer.get_error() == 0
    assert np.array_equal(lay["slot_row"].cpu().numpy(), d.slot_row)
    assert np.array_equal(out.cpu().numpy().view(np.uint16), out_ref)

    # fp8 dispatch
    xq = torch.empty((rows, H), dtype=torch.uint8, device="cuda")
    xs = torch.empty((rows, H // 128), dtype=torch.float32, device="cuda")
    layer.dispatch_send_fp8(x, idx, xq, xs)
    layer.dispatch_recv()
    layer.combine_send(y)
    layer.combine_recv(wt, out)
    assert layer.get_error() == 0

    # already-quantised tokens
    q, sc = oracle_mod.quantize_fp8(li.x)
    q_d, sc_d = _dev(q), _dev(sc)
    layer.dispatch_send_quantized(q_d, sc_d, idx, xq, xs)
    layer.dispatch_recv()
    layer.combine_send(y)
    layer.combine_recv(wt, out)
    assert layer.get_error() == 0
    src = d.row_src // K
    assert np.array_equal(xq.cpu().numpy(), q[src])

    # two-stage dispatch + two-level combine
    send = torch.empty_like(ex)
    partial = torch.empty((layer.partial_rows(), H), dtype=torch.int16, device="cuda")
    layer.dispatch_send_staged(x, idx, send, ex)
    layer.dispatch_recv()
    layer.combine_send(y)
    layer.combine_recv_two_level(wt, partial, out)
    assert layer.get_error() == 0
    assert np.array_equal(ex.cpu().numpy().view(np.uint16), d.expert_x)
    ref2, _, _ = oracle_mod.combine_two_level(li.y, li.topk_idx, li.topk_w, d.slot_row, E, N)
    assert np.array_equal(out.cpu().numpy().view(np.uint16), ref2)
    assert guards_intact()

    # dense padded all-to-all dispatch + combine (block tables in the workspace)
    cap = layer.dense_capacity()
    blocks = [torch.empty((N * N * cap, H), dtype=torch.int16, device="cuda") for _ in range(2)]
    layer.dispatch_send_dense(x, idx, cap, blocks[0], blocks[1], ex)
    layer.dispatch_recv()
    layer.combine_send(y)
    layer.combine_recv_dense(wt, cap, blocks[0], blocks[1], out)
    assert layer.get_error() == 0
    assert np.array_equal(ex.cpu().numpy().view(np.uint16), d.expert_x)
    assert np.array_equal(out.cpu().numpy().view(np.uint16), out_ref)
    assert guards_intact()

    # a bad expert index: every kernel takes its error path
    bad = li.topk_idx.copy()
    bad[T // 2, 0] = E
    bad_d = _dev(bad)
    layer.layer(x, bad_d, wt, ex, y, out)
    assert layer.get_error() == moe.MOE_EROUTE
    layer.dispatch_send_staged(x, bad_d, send, ex)
    layer.dispatch_recv()
    layer.combine_send(y)
    layer.combine_recv_two_level(wt, partial, out)
    assert layer.get_error() == moe.MOE_EROUTE
    layer.dispatch_send_dense(x, bad_d, cap, blocks[0], blocks[1], ex)
    layer.dispatch_recv()
    layer.combine_send(y)
    layer.combine_recv_dense(wt, cap, blocks[0], blocks[1], out)
    assert layer.get_error() == moe.MOE_EROUTE
    assert guards_intact()

    # and the context is usable again afterwards
    layer.layer(x, idx, wt, ex, y, out)
    assert layer.get_error() == 0
    assert np.array_equal(out.cpu().numpy().view(np.uint16), out_ref)
    assert guards_intact()


def test_workspace_argument_is_checked(moe):
    cfg = moe.make_config(64, 256, 2, 8, 2)
    nbytes = moe.moe_workspace_bytes(cfg)
    with pytest.raises(moe.MoEError):
        moe.MoELayer(64, 256, 2, 8, 2, workspace=torch.empty(nbytes - 256, dtype=torch.uint8, device="cuda"))
    with pytest.raises(moe.MoEError):  # not 256-byte aligned
        moe.MoELayer(64, 256, 2, 8, 2, workspace=torch.empty(nbytes + 512, dtype=torch.uint8, device="cuda")[16:])
    with pytest.raises(moe.MoEError):
        moe.MoELayer(64, 256, 2, 8, 2, workspace=torch.empty(nbytes // 4, dtype=torch.int32, device="cuda"))
