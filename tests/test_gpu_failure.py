"""Failure detection on the GPU without a fault: a lost unit in the combine.

The bulk combine's consumers wait on an mbarrier for each unit's rows with a
2 s limit.  MOE_OPT_TEST_DROP_COMBINE_UNIT makes the producer skip one unit,
as if its copies never arrived: nothing ever completes that wait, the kernel
gives up after the limit, writes MOE_ETIMEDOUT to the error word and returns
(no trap, no fault, no endless wait).  The host reads the status, and the same
context then runs a normal layer bit-exact against the oracle."""
import time

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


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def test_lost_combine_unit_times_out_and_the_context_recovers(moe, oracle_mod):
    # 2048 tokens, one 2 KiB piece per row: 2048 units over the persistent
    # grid; unit 70 is the first of its CTA's units, so both the consumers'
    # wait (for unit 70) and the producer's wait (for the stage unit 70 never
    # frees) run out.
    w = gen.custom("lost", T=2048, H=1024, K=8, E=64, N=8, seed_index=79)
    li = gen.make_inputs(w)
    layer = moe.MoELayer(w.T, w.H, w.K, w.E, w.N, combine_variant=0)
    x, idx, wts, y = _dev(li.x.view(np.int16)), _dev(li.topk_idx), _dev(li.topk_w), _dev(li.y.view(np.int16))
    ex = torch.zeros((w.T * w.K, w.H), dtype=torch.int16, device="cuda")
    out = torch.zeros((w.T, w.H), dtype=torch.int16, device="cuda")

    layer.set_option(moe.MOE_OPT_TEST_DROP_COMBINE_UNIT, 70)
    assert layer.get_option(moe.MOE_OPT_TEST_DROP_COMBINE_UNIT) == 70
    torch.cuda.synchronize()
    t0 = time.monotonic()
    layer.layer(x, idx, wts, ex, y, out)
    status = layer.get_error()
    elapsed = time.monotonic() - t0
    assert status == moe.MOE_ETIMEDOUT
    assert 1.5 < elapsed < 30.0
    assert torch.cuda.current_stream().query()  # nothing left running

    layer.set_option(moe.MOE_OPT_TEST_DROP_COMBINE_UNIT, -1)
    out.zero_()
    layer.layer(x, idx, wts, ex, y, out)
    assert layer.get_error() == moe.MOE_OK
    d = oracle_mod.dispatch(li.x, li.topk_idx, w.E, w.N)
    assert np.array_equal(ex.cpu().numpy().view(np.uint16), d.expert_x)
    assert np.array_equal(out.cpu().numpy().view(np.uint16), oracle_mod.combine(li.y, li.topk_w, d.slot_row))


def test_drop_hook_rejects_bad_values(moe):
    layer = moe.MoELayer(64, 256, 2, 8, 2)
    with pytest.raises(moe.MoEError):
        layer.set_option(moe.MOE_OPT_TEST_DROP_COMBINE_UNIT, -2)
    assert layer.get_option(moe.MOE_OPT_TEST_DROP_COMBINE_UNIT) == -1
