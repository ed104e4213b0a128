"""moe_dispatch_send_noalloc: dispatch for callers that cannot allocate device
memory (they cannot provide moe_ctx_create's workspace, e.g. code running
inside another framework's memory pool without an allocator handle).  Its
routing tables live in a static device array of the library.

Checked through the C ABI, bit for bit, against the CPU oracle (grouped rows,
counts, offsets) and against the existing entry point (moe_dispatch_send +
moe_dispatch_recv), on calls in a row with different shapes, so that whatever
an earlier call left in the shared static array cannot leak into a later one.
The shapes cover both chunk sizes of route_count's slot ranks (E <= 768 and
E > 768), K = 1 and K = 16, an empty layer, and a malformed routing right
after a valid call.  Collected last on purpose; it passes alone in a fresh
process as well as after the other tests.
"""
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


def _reference(moe, w, x, idx):
    """Grouped rows, counts and offsets from the workspace-based entry point."""
    layer = moe.MoELayer(w.T, w.H, w.K, w.E, w.N)
    ex = torch.empty((w.T * w.K, w.H), dtype=torch.int16, device="cuda")
    layer.dispatch_send(x, idx, ex)
    lay = layer.dispatch_recv()
    assert layer.get_error() == moe.MOE_OK
    res = (ex.clone(), lay["expert_counts"].clone(), lay["expert_offsets"].clone())
    layer.close()
    return res


def _noalloc(moe, w, x, idx, extra_rows=0):
    rows = w.T * w.K
    ex = torch.full((rows + extra_rows, w.H), CANARY, dtype=torch.int16, device="cuda")
    counts = torch.full((w.E,), -7, dtype=torch.int32, device="cuda")
    offsets = torch.full((w.E + 1,), -7, dtype=torch.int32, device="cuda")
    status = torch.full((1,), -7, dtype=torch.int32, device="cuda")
    cfg = moe.make_config(w.T, w.H, w.K, w.E, w.N)
    rc = moe.moe_dispatch_send_noalloc(cfg, x, idx, ex, ex.shape[0], counts, offsets, status)
    torch.cuda.synchronize()
    return rc, ex, counts, offsets, int(status.item())


SHAPES = [
    gen.Workload("deepseek-part", T=1024, H=7168, K=8, E=256, N=8, router="sigmoid_topk", index=2),
    gen.custom("mixed", T=3000, H=520, K=3, E=60, N=3, seed_index=41),
    gen.custom("many-experts", T=1540, H=64, K=4, E=1024, N=4, seed_index=42),  # E > 768: 16-warp chunks
    gen.custom("top-1", T=2049, H=136, K=1, E=6, N=3, seed_index=43),
    gen.custom("top-16", T=512, H=256, K=16, E=64, N=4, seed_index=44),
]


def test_noalloc_dispatch_matches_the_oracle_and_the_workspace_entry_point(moe, oracle_mod):
    for w in SHAPES:
        li = gen.make_inputs(w, with_y=False)
        d = oracle_mod.dispatch(li.x, li.topk_idx, w.E, w.N)
        x = torch.from_numpy(li.x.view(np.int16)).cuda()
        idx = torch.from_numpy(li.topk_idx).cuda()
        ref_x, ref_counts, ref_offsets = _reference(moe, w, x, idx)
        rows = w.T * w.K
        rc, ex, counts, offsets, status = _noalloc(moe, w, x, idx, extra_rows=3)
        assert rc == moe.MOE_OK and status == moe.MOE_OK, w.name
        got = ex.cpu().numpy().view(np.uint16)
        assert np.array_equal(got[:rows], d.expert_x), w.name
        assert np.all(got[rows:] == CANARY), "rows past T*K must stay untouched"
        assert np.array_equal(counts.cpu().numpy(), d.expert_counts), w.name
        assert np.array_equal(offsets.cpu().numpy(), d.expert_offsets), w.name
        assert torch.equal(ex[:rows], ref_x) and torch.equal(counts, ref_counts) and torch.equal(offsets, ref_offsets)


def test_noalloc_routing_error_after_a_valid_call_writes_nothing(moe, oracle_mod):
    w = gen.custom("bad", T=300, H=64, K=4, E=16, N=4, seed_index=3)
    li = gen.make_inputs(w, with_y=False)
    x = torch.from_numpy(li.x.view(np.int16)).cuda()
    good = torch.from_numpy(li.topk_idx).cuda()
    rc, _, counts, _, status = _noalloc(moe, w, x, good)  # fills the shared array with valid tables
    assert rc == moe.MOE_OK and status == moe.MOE_OK
    assert np.array_equal(counts.cpu().numpy(), oracle_mod.dispatch(li.x, li.topk_idx, w.E, w.N).expert_counts)
    for bad in ("out_of_range", "repeated"):
        idx = li.topk_idx.copy()
        if bad == "out_of_range":
            idx[123, 2] = 16
        else:
            idx[299, 3] = idx[299, 1]
        rc, ex, counts, offsets, status = _noalloc(moe, w, x, torch.from_numpy(idx).cuda())
        assert rc == moe.MOE_OK  # the host cannot see the indices; the device reports
        assert status == moe.MOE_EROUTE, bad
        assert np.all(counts.cpu().numpy() == 0) and np.all(offsets.cpu().numpy() == 0)
        assert np.all(ex.cpu().numpy().view(np.uint16) == CANARY), "no row may be written after a routing error"
    # and a valid call afterwards is exact again
    d = oracle_mod.dispatch(li.x, li.topk_idx, w.E, w.N)
    rc, ex, counts, offsets, status = _noalloc(moe, w, x, good)
    assert rc == moe.MOE_OK and status == moe.MOE_OK
    assert np.array_equal(ex.cpu().numpy().view(np.uint16), d.expert_x)
    assert np.array_equal(offsets.cpu().numpy(), d.expert_offsets)


def test_noalloc_empty_layer(moe):
    w = gen.custom("empty", T=0, H=64, K=2, E=8, N=2, seed_index=4)
    x = torch.empty((0, 64), dtype=torch.int16, device="cuda")
    idx = torch.empty((0, 2), dtype=torch.int32, device="cuda")
    rc, ex, counts, offsets, status = _noalloc(moe, w, x, idx, extra_rows=2)
    assert rc == moe.MOE_OK and status == moe.MOE_OK
    assert counts.cpu().tolist() == [0] * 8 and offsets.cpu().tolist() == [0] * 9
    assert np.all(ex.cpu().numpy().view(np.uint16) == CANARY)


def test_noalloc_rejects_sizes_beyond_its_static_array(moe):
    dummy = torch.zeros(16, dtype=torch.int32, device="cuda")
    too_many_pairs = moe.make_config(moe.MOE_NOALLOC_MAX_PAIRS // 8 + 8, 64, 8, 64, 8)
    assert moe.moe_dispatch_send_noalloc(too_many_pairs, dummy, dummy, dummy, 1 << 30, dummy, dummy,
                                         dummy) == moe.MOE_EINVAL
    too_many_expert_ranks = moe.make_config(1024, 64, 2, 1024, 128)
    assert moe.moe_dispatch_send_noalloc(too_many_expert_ranks, dummy, dummy, dummy, 1 << 30, dummy, dummy,
                                         dummy) == moe.MOE_EINVAL
