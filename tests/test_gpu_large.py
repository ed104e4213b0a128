"""Buffers past 4 GiB, through the C ABI, against the CPU oracle.

Every kernel addresses a row as a 64-bit byte offset (row index times row
bytes).  No buffer of the named workloads reaches 4 GiB (the largest, the
Kimi-sized grouped rows, is 1.9 GB), so a product taken in 32 bits would go
unnoticed there.  Here T = 16384 tokens of H = 34816 bf16 (68 KiB rows) with
K = 8 give 131,072 grouped rows: 9.1 GB as bf16 and 4.6 GB as fp8, so more
than half of the rows start beyond byte 2**32 of their buffer.

What is checked, on the GPU's own outputs:
  - the routing tables (counts, offsets, slot_row, row_src) bit for bit
    against the oracle's dispatch (the tables depend on topk_idx alone);
  - grouped rows: sampled rows and the last 64 rows hold x[row_src // K];
  - combine with y = the grouped rows and every weight 1/8: out == x bit for
    bit on every token (each partial sum m*v/8 of a bf16 v is exact in
    float32), except that -0.0 comes out as +0.0 (the chain starts from +0.0
    and +0.0 + -0.0 = +0.0 under round-to-nearest; the float32 normal draws
    of x hit exact zeros a few dozen times in 570M elements), and with the
    router's weights, sampled tokens against the oracle's combine;
  - the two-level combine, the two-stage dispatch, the fp8 dispatch and the
    dispatch of already-quantised tokens on the same sizes (sampled tokens
    against the oracle, or the whole buffer against the direct dispatch).
The oracle runs on the sampled tokens only: every output of a token depends
on that token's row, routing and weights alone."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

from combine_route_count_gb300 import inputs as gen  # noqa: E402

T, H, K, E, N = 16384, 34816, 8, 64, 8
ROWS = T * K


@pytest.fixture(scope="module")
def moe():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from combine_route_count_gb300 import build, moe as m
    build.build()
    m.load_library()
    return m


@pytest.fixture(scope="module")
def big(moe, oracle_mod):
    w = gen.custom("large", T=T, H=H, K=K, E=E, N=N, router="uniform_random", seed_index=101)
    li = gen.make_inputs(w, with_y=False)
    assert ROWS * H * 2 > 2 * 2**32
    # The tables depend on topk_idx only: the oracle's dispatch of 8-wide rows.
    d = oracle_mod.dispatch(np.zeros((T, 8), np.uint16), li.topk_idx, E, N)
    rng = np.random.default_rng(7)
    sample = np.unique(np.concatenate([rng.choice(T, size=40, replace=False), [0, T - 2, T - 1]]))
    x = torch.from_numpy(li.x.view(np.int16)).cuda()
    idx = torch.from_numpy(li.topk_idx).cuda()
    # What identity experts with weights summing to one return: x, with any
    # -0.0 (bf16 bits 0x8000) as +0.0.
    x_id = torch.where(x == -32768, torch.zeros_like(x), x)
    return dict(w=w, li=li, d=d, sample=sample, x=x, idx=idx, x_id=x_id)


def _rows_hold_tokens(dst, rows, src, tokens):
    r = torch.as_tensor(np.asarray(rows, np.int64), device="cuda")
    t = torch.as_tensor(np.asarray(tokens, np.int64), device="cuda")
    return torch.equal(dst.index_select(0, r), src.index_select(0, t))


def _check_grouped_rows(ex, src, d, sample):
    """Rows of the sampled tokens and the last 64 rows hold their token's row."""
    rows = np.concatenate([d.slot_row[sample].reshape(-1), np.arange(ROWS - 64, ROWS)])
    return _rows_hold_tokens(ex, rows, src, d.row_src[rows] // K)


def test_direct_dispatch_and_combine_beyond_4_gib(moe, oracle_mod, big):
    d, li, sample, x, idx = big["d"], big["li"], big["sample"], big["x"], big["idx"]
    layer = moe.MoELayer(T, H, K, E, N)
    ex = torch.empty((ROWS, H), dtype=torch.int16, device="cuda")
    out = torch.empty((T, H), dtype=torch.int16, device="cuda")
    w_eighth = torch.full((T, K), 0.125, dtype=torch.float32, device="cuda")
    layer.dispatch_send(x, idx, ex)
    lay = layer.dispatch_recv()
    layer.combine_send(ex)
    layer.combine_recv(w_eighth, out)
    assert layer.get_error() == 0
    for k in ("expert_counts", "expert_offsets", "rank_offsets", "src_offsets", "slot_row", "row_src"):
        assert np.array_equal(lay[k].cpu().numpy(), getattr(d, k)), k
    assert int(d.slot_row.max()) * H * 2 > 2**32
    assert _check_grouped_rows(ex, x, d, sample)
    assert torch.equal(out, big["x_id"]), "identity experts with weights 1/8 must return x"

    # Router weights: sampled tokens against the oracle's combine of the
    # same rows (y = the grouped rows, so y[slot_row[t, k]] = x[t]).
    wts = torch.from_numpy(li.topk_w).cuda()
    layer.dispatch_send(x, idx, ex)
    layer.dispatch_recv()
    layer.combine_send(ex)
    layer.combine_recv(wts, out)
    assert layer.get_error() == 0
    S = len(sample)
    y_sub = np.repeat(li.x[sample], K, axis=0)
    ref = oracle_mod.combine(y_sub, li.topk_w[sample], np.arange(S * K, dtype=np.int32).reshape(S, K))
    got = out.index_select(0, torch.as_tensor(sample, device="cuda")).cpu().numpy().view(np.uint16)
    assert np.array_equal(got, ref)

    # Two-level combine: partial rows past 4 GiB too.
    partial = torch.empty((layer.partial_rows(), H), dtype=torch.int16, device="cuda")
    assert layer.partial_rows() * H * 2 > 2**32
    layer.dispatch_send(x, idx, ex)
    layer.dispatch_recv()
    layer.combine_send(ex)
    layer.combine_recv_two_level(wts, partial, out)
    assert layer.get_error() == 0
    ref2, _, _ = oracle_mod.combine_two_level(y_sub, li.topk_idx[sample], li.topk_w[sample],
                                              np.arange(S * K, dtype=np.int32).reshape(S, K), E, N)
    got2 = out.index_select(0, torch.as_tensor(sample, device="cuda")).cpu().numpy().view(np.uint16)
    assert np.array_equal(got2, ref2)
    del partial

    # Two-stage dispatch: the same grouped rows through 9.1 GB of send rows.
    send = torch.empty_like(ex)
    ex2 = torch.empty_like(ex)
    layer2 = moe.MoELayer(T, H, K, E, N)
    layer2.dispatch_send_staged(x, idx, send, ex2)
    layer2.dispatch_recv()
    layer2.combine_send(ex2)
    layer2.combine_recv(w_eighth, out)
    assert layer2.get_error() == 0
    assert torch.equal(ex2, ex)
    assert torch.equal(out, big["x_id"])


def test_fp8_dispatch_beyond_4_gib(moe, oracle_mod, big):
    d, li, sample, x, idx = big["d"], big["li"], big["sample"], big["x"], big["idx"]
    layer = moe.MoELayer(T, H, K, E, N)
    xq = torch.empty((ROWS, H), dtype=torch.uint8, device="cuda")
    xs = torch.empty((ROWS, H // 128), dtype=torch.float32, device="cuda")
    assert ROWS * H > 2**32
    layer.dispatch_send_fp8(x, idx, xq, xs)
    layer.dispatch_recv()
    assert layer.get_error() == 0
    q_ref, s_ref = oracle_mod.quantize_fp8(li.x[sample])
    S = len(sample)
    for k in range(K):
        r = torch.as_tensor(d.slot_row[sample, k].astype(np.int64), device="cuda")
        assert np.array_equal(xq.index_select(0, r).cpu().numpy(), q_ref), k
        assert np.array_equal(xs.index_select(0, r).cpu().numpy().view(np.uint32), s_ref.view(np.uint32)), k
    assert S == q_ref.shape[0]

    # Already-quantised tokens: a byte copy of code rows and scale rows.
    rng = np.random.default_rng(11)
    codes = torch.from_numpy(rng.integers(0, 256, size=(T, H), dtype=np.uint8)).cuda()
    scales = torch.from_numpy(rng.random((T, H // 128), dtype=np.float32)).cuda()
    layer_q = moe.MoELayer(T, H, K, E, N)
    layer_q.dispatch_send_quantized(codes, scales, idx, xq, xs)
    layer_q.dispatch_recv()
    assert layer_q.get_error() == 0
    assert _check_grouped_rows(xq, codes, d, sample)
    assert _check_grouped_rows(xs, scales, d, sample)
