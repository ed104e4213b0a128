"""The all-cores CPU baseline (oracle/moe_oracle_par.cc) writes exactly what
the single-threaded oracle writes.  It is only timed by the benchmark; this
checks that the number it gives is for the same work and the same result."""
import numpy as np
import pytest

from combine_route_count_gb300 import inputs as gen

FIELDS = ("expert_x", "expert_counts", "expert_offsets", "src_offsets", "rank_offsets", "slot_row", "row_src")


def _same(oracle_mod, w, li):
    d = oracle_mod.dispatch(li.x, li.topk_idx, w.E, w.N)
    dp = oracle_mod.dispatch_par(li.x, li.topk_idx, w.E, w.N)
    for f in FIELDS:
        assert np.array_equal(getattr(d, f), getattr(dp, f)), f
    out = oracle_mod.combine(li.y, li.topk_w, d.slot_row)
    outp = oracle_mod.combine_par(li.y, li.topk_w, dp.slot_row)
    assert np.array_equal(out, outp)


def test_threads_reported(oracle_mod):
    assert oracle_mod.par_threads() >= 1


@pytest.mark.parametrize("name", ["tiny", "mixtral"])
def test_par_equals_oracle(oracle_mod, name):
    w = gen.BY_NAME[name]
    _same(oracle_mod, w, gen.make_inputs(w))


@pytest.mark.slow
def test_par_equals_oracle_deepseek(oracle_mod):
    w = gen.BY_NAME["deepseek"]
    _same(oracle_mod, w, gen.make_inputs(w))


def test_par_edge_shapes(oracle_mod):
    for T, H, K, E, N in [(0, 64, 2, 8, 2), (1, 8, 1, 1, 1), (96, 24, 3, 12, 4), (33, 16, 16, 16, 1)]:
        w = gen.custom("edge", T, H, K, E, N)
        _same(oracle_mod, w, gen.make_inputs(w))


def test_par_routing_errors(oracle_mod):
    w = gen.custom("edge", 8, 16, 2, 4, 2)
    li = gen.make_inputs(w)
    for bad in (4, -1):
        idx = li.topk_idx.copy()
        idx[3, 1] = bad
        with pytest.raises(oracle_mod.OracleError) as e:
            oracle_mod.dispatch_par(li.x, idx, w.E, w.N)
        assert e.value.code == oracle_mod.EROUTE
    idx = li.topk_idx.copy()
    idx[5, 1] = idx[5, 0]
    with pytest.raises(oracle_mod.OracleError) as e:
        oracle_mod.dispatch_par(li.x, idx, w.E, w.N)
    assert e.value.code == oracle_mod.EROUTE
