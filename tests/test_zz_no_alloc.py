"""moe_dispatch_send_noalloc: dispatch for callers that cannot allocate device
memory (they cannot provide moe_ctx_create's workspace, e.g. code running
inside another framework's memory pool without an allocator handle).  Its
routing tables live in a static device array of the library.

Checked through the C ABI against the existing entry point
(moe_dispatch_send + moe_dispatch_recv) bit for bit, on two calls in a row
with different shapes, so that whatever the first call left in the shared
static array cannot leak into the second.  Collected last on purpose; it
passes alone in a fresh process as well as after the other tests.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

from combine_route_count_gb300 import inputs as gen  # noqa: E402


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


def test_noalloc_dispatch_matches_the_workspace_entry_point_twice(moe):
    shapes = [
        gen.Workload("deepseek-part", T=1024, H=7168, K=8, E=256, N=8, router="sigmoid_topk", index=2),
        gen.custom("mixed", T=3000, H=520, K=3, E=60, N=3, seed_index=41),
    ]
    for w in shapes:
        li = gen.make_inputs(w, with_y=False)
        x = torch.from_numpy(li.x.view(np.int16)).cuda()
        idx = torch.from_numpy(li.topk_idx).cuda()
        ref_x, ref_counts, ref_offsets = _reference(moe, w, x, idx)

        ex = torch.full((w.T * w.K, w.H), 0x7BCD, dtype=torch.int16, device="cuda")
        counts = torch.full((w.E,), -7, dtype=torch.int32, device="cuda")
        offsets = torch.full((w.E + 1,), -7, dtype=torch.int32, device="cuda")
        status = torch.full((1,), -7, dtype=torch.int32, device="cuda")
        cfg = moe.make_config(w.T, w.H, w.K, w.E, w.N)
        rc = moe.moe_dispatch_send_noalloc(cfg, x, idx, ex, ex.shape[0], counts, offsets, status)
        assert rc == moe.MOE_OK
        torch.cuda.synchronize()
        assert int(status.item()) == moe.MOE_OK
        assert torch.equal(counts, ref_counts)
        assert torch.equal(offsets, ref_offsets)
        assert torch.equal(ex, ref_x)


def test_noalloc_rejects_sizes_beyond_its_static_array(moe):
    dummy = torch.zeros(16, dtype=torch.int32, device="cuda")
    too_many_pairs = moe.make_config(moe.MOE_NOALLOC_MAX_PAIRS // 8 + 8, 64, 8, 64, 8)
    assert moe.moe_dispatch_send_noalloc(too_many_pairs, dummy, dummy, dummy, 1 << 30, dummy, dummy,
                                         dummy) == moe.MOE_EINVAL
    too_many_expert_ranks = moe.make_config(1024, 64, 2, 1024, 128)
    assert moe.moe_dispatch_send_noalloc(too_many_expert_ranks, dummy, dummy, dummy, 1 << 30, dummy, dummy,
                                         dummy) == moe.MOE_EINVAL
