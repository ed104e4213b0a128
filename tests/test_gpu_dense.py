"""Dense padded all-to-all dispatch and combine (moe_dispatch_send_dense,
moe_combine_recv_dense) against the CPU oracle, through the C ABI.

Small shapes: the send blocks (valid rows bit for bit, padding rows left
untouched), the receive blocks (the whole buffer is the block transpose of
the send buffer), the grouped rows and the combine output, all against
oracle_dispatch_dense / oracle_combine_dense.  Full-size workloads: the
grouped rows and the combine output against the direct oracle, every pair's
send row against its token row, and the transpose on the device."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

from combine_route_count_gb300 import inputs as gen  # noqa: E402

CANARY = 0x7BCD


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


def send_positions(idx, E, N, cap):
    """Send row of every (token, slot), by numpy lexsort per (source, rank)."""
    T, K = idx.shape
    Tr, L = T // N, E // N
    t_of = np.repeat(np.arange(T), K)
    e_of = idx.reshape(-1)
    pos = np.empty(T * K, np.int64)
    for s in range(N):
        for r in range(N):
            sel = np.nonzero((t_of // Tr == s) & (e_of // L == r))[0]
            order = sel[np.lexsort((t_of[sel], e_of[sel]))]
            pos[order] = (s * N + r) * cap + np.arange(len(order))
    return pos


def run_dense(moe, w, li, cap, extra=0, **options):
    T, H, K, E, N = w.T, w.H, w.K, w.E, w.N
    rows = N * N * cap + extra
    send = torch.full((rows, H), CANARY, dtype=torch.int16, device="cuda")
    recv = torch.full((rows, H), CANARY, dtype=torch.int16, device="cuda")
    ex = torch.full((T * K + 2, H), CANARY, dtype=torch.int16, device="cuda")
    out = torch.full((T, H), CANARY, dtype=torch.int16, device="cuda")
    layer = moe.MoELayer(T, H, K, E, N, **options)
    x, idx = _dev(li.x.view(np.int16)), _dev(li.topk_idx)
    layer.dispatch_send_dense(x, idx, cap, send, recv, ex)
    lay = layer.dispatch_recv()
    y = _dev(li.y.view(np.int16))
    layer.combine_send(y)
    # The combine's blocks reuse the dispatch's buffers: keep copies first.
    send_d, recv_d = send.clone(), recv.clone()
    layer.combine_recv_dense(_dev(li.topk_w), cap, send, recv, out)
    status = layer.get_error()
    return dict(status=status, send=send_d, recv=recv_d, back_send=send, back_recv=recv, ex=ex, out=out, layer=layer,
                slot_row=lay["slot_row"].cpu().numpy())


SMALL = [  # (T, H, K, E, N)
    (64, 256, 2, 8, 2),
    (96, 24, 3, 12, 4),
    (40, 8, 4, 4, 4),
    (30, 16, 1, 6, 3),
    (512, 64, 8, 64, 8),
    (6, 40, 1, 6, 6),
    (1, 8, 1, 1, 1),
]


@pytest.mark.parametrize("extra_cap", [0, 3])
@pytest.mark.parametrize("shape", SMALL, ids=["x".join(map(str, s)) for s in SMALL])
def test_dense_matches_oracle(moe, oracle_mod, shape, extra_cap):
    T, H, K, E, N = shape
    w = gen.custom("dense", T=T, H=H, K=K, E=E, N=N, seed_index=93)
    li = gen.make_inputs(w)
    cap = moe.moe_dense_capacity(moe.make_config(T, H, K, E, N)) + extra_cap
    res = run_dense(moe, w, li, cap, extra=2)
    assert res["status"] == moe.MOE_OK
    send_ref, recv_ref, ex_ref, pos = oracle_mod.dispatch_dense(li.x, li.topk_idx, E, N, cap)
    rows = N * N * cap
    send = res["send"].cpu().numpy().view(np.uint16)
    recv = res["recv"].cpu().numpy().view(np.uint16)
    valid = np.zeros(rows + 2, bool)
    valid[pos.reshape(-1)] = True
    # Valid send rows bit for bit; padding rows and rows past the blocks untouched.
    assert np.array_equal(send[:rows][valid[:rows]], send_ref[valid[:rows]])
    assert np.all(send[~valid] == CANARY)
    # The exchange moves every block whole: the receive buffer is the block
    # transpose of the send buffer, padding included; rows past the blocks stay.
    assert np.array_equal(recv[:rows].reshape(N, N, cap, H), send[:rows].reshape(N, N, cap, H).transpose(1, 0, 2, 3))
    assert np.all(recv[rows:] == CANARY)
    p = pos.reshape(-1).astype(np.int64)
    blk, j = p // cap, p % cap
    recv_pos = ((blk % N) * N + blk // N) * cap + j
    assert np.array_equal(recv[recv_pos], recv_ref[recv_pos])
    assert np.array_equal(recv[recv_pos], li.x[np.repeat(np.arange(T), K)])
    ex = res["ex"].cpu().numpy().view(np.uint16)
    assert np.array_equal(ex[:T * K], ex_ref)
    assert np.all(ex[T * K:] == CANARY)
    out_ref, back_send_ref, back_recv_ref = oracle_mod.combine_dense(li.y, li.topk_w, res["slot_row"], pos, N, cap)
    assert np.array_equal(res["out"].cpu().numpy().view(np.uint16), out_ref)
    assert np.array_equal(out_ref, oracle_mod.combine(li.y, li.topk_w, res["slot_row"]))
    back_recv = res["back_recv"].cpu().numpy().view(np.uint16)
    assert np.array_equal(back_recv[pos.reshape(-1)], back_recv_ref[pos.reshape(-1)])


@pytest.mark.parametrize("name", ["tiny", "mixtral", "deepseek", "worst"])
def test_dense_named_workloads_full_size(moe, oracle_mod, name):
    w = gen.BY_NAME[name]
    li = gen.make_inputs(w)
    T, H, K, E, N = w.T, w.H, w.K, w.E, w.N
    cap = moe.moe_dense_capacity(moe.make_config(T, H, K, E, N))
    res = run_dense(moe, w, li, cap)
    assert res["status"] == moe.MOE_OK
    d = oracle_mod.dispatch(li.x, li.topk_idx, E, N)
    assert np.array_equal(res["ex"][:T * K].cpu().numpy().view(np.uint16), d.expert_x)
    assert np.array_equal(res["out"].cpu().numpy().view(np.uint16), oracle_mod.combine(li.y, li.topk_w, d.slot_row))
    pos = torch.from_numpy(send_positions(li.topk_idx, E, N, cap)).cuda()
    x = _dev(li.x.view(np.int16))
    tok = torch.arange(T, device="cuda").repeat_interleave(K)
    assert torch.equal(res["send"][pos], x[tok])
    rows = N * N * cap
    assert torch.equal(res["recv"][:rows].view(N, N, cap, H), res["send"][:rows].view(N, N, cap, H).transpose(0, 1))
    # The returned blocks hold every pair's expert output at its send row.
    y = _dev(li.y.view(np.int16))
    assert torch.equal(res["back_recv"][pos], y[torch.from_numpy(d.slot_row.reshape(-1).astype(np.int64)).cuda()])


def test_dense_routing_error_writes_nothing(moe):
    w = gen.custom("dense-bad", T=64, H=64, K=4, E=16, N=4, seed_index=7)
    li = gen.make_inputs(w)
    idx = li.topk_idx.copy()
    idx[17, 2] = idx[17, 0]
    li2 = gen.LayerInputs(w, li.x, idx, li.topk_w, li.y)
    cap = moe.moe_dense_capacity(moe.make_config(w.T, w.H, w.K, w.E, w.N))
    res = run_dense(moe, w, li2, cap)
    assert res["status"] == moe.MOE_EROUTE
    for key in ("send", "recv", "ex", "out"):
        assert torch.all(res[key] == CANARY), key


def test_dense_argument_and_order_checks(moe):
    T, H, K, E, N = 64, 64, 2, 8, 2
    cfg = moe.make_config(T, H, K, E, N)
    cap = moe.moe_dense_capacity(cfg)
    assert cap == 32 * 2
    layer = moe.MoELayer(T, H, K, E, N)
    x = torch.zeros((T, H), dtype=torch.int16, device="cuda")
    idx = torch.tensor([[t % E, (t + 1) % E] for t in range(T)], dtype=torch.int32, device="cuda")
    wt = torch.full((T, K), 0.5, dtype=torch.float32, device="cuda")
    ex = torch.zeros((T * K, H), dtype=torch.int16, device="cuda")
    out = torch.zeros((T, H), dtype=torch.int16, device="cuda")
    buf = torch.zeros((N * N * cap, H), dtype=torch.int16, device="cuda")
    buf2 = torch.zeros_like(buf)
    for bad_cap in (cap - 1, 0):
        with pytest.raises(moe.MoEError) as ei:
            layer.dispatch_send_dense(x, idx, bad_cap, buf, buf2, ex)
        assert ei.value.code == moe.MOE_EINVAL
    with pytest.raises(moe.MoEError) as ei:  # buffers one row short
        moe.moe_dispatch_send_dense(layer.ctx, x, idx, cap, buf, buf2, N * N * cap - 1, ex, T * K)
    assert ei.value.code == moe.MOE_EINVAL
    # The dense combine needs the dense dispatch before it.
    layer.dispatch_send(x, idx, ex)
    layer.dispatch_recv()
    layer.combine_send(ex)
    with pytest.raises(moe.MoEError) as ei:
        layer.combine_recv_dense(wt, cap, buf, buf2, out)
    assert ei.value.code == moe.MOE_ESTATE
    layer.combine_recv(wt, out)
    # ... with the same capacity.
    big = torch.zeros((N * N * (cap + 1), H), dtype=torch.int16, device="cuda")
    big2 = torch.zeros_like(big)
    layer.dispatch_send_dense(x, idx, cap + 1, big, big2, ex)
    layer.dispatch_recv()
    layer.combine_send(ex)
    with pytest.raises(moe.MoEError) as ei:
        layer.combine_recv_dense(wt, cap, big, big2, out)
    assert ei.value.code == moe.MOE_EINVAL
    layer.combine_recv_dense(wt, cap + 1, big, big2, out)
    assert layer.get_error() == moe.MOE_OK
