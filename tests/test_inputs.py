"""The seeded workload generator: shapes, determinism and the routing
properties each workload is meant to have."""
import numpy as np
import pytest

from combine_route_count_gb300 import inputs as gen


def _routing(w):
    rng = np.random.Generator(np.random.PCG64(w.seed))
    return gen.make_routing(w, rng)


@pytest.mark.parametrize("w", gen.WORKLOADS, ids=[w.name for w in gen.WORKLOADS])
def test_routing_shapes_and_topk_properties(w):
    idx, wt = _routing(w)
    assert idx.shape == (w.T, w.K) and idx.dtype == np.int32
    assert wt.shape == (w.T, w.K) and wt.dtype == np.float32
    assert w.T % w.N == 0 and w.E % w.N == 0
    assert idx.min() >= 0 and idx.max() < w.E
    srt = np.sort(idx, axis=1)
    assert np.all(np.diff(srt, axis=1) > 0), "experts of one token are distinct"
    assert np.all(wt > 0)
    assert np.allclose(wt.astype(np.float64).sum(axis=1), 1.0, atol=1e-6)


def test_named_sizes():
    s = {w.name: (w.T, w.H, w.K, w.E, w.N) for w in gen.WORKLOADS}
    assert s == {"tiny": (64, 256, 2, 8, 2), "mixtral": (4096, 4096, 2, 8, 8),
                 "deepseek": (4096, 7168, 8, 256, 32), "kimi": (16384, 7168, 8, 384, 64),
                 "worst": (8192, 7168, 8, 128, 16)}


def test_worst_case_routes_only_to_rank0():
    w = gen.BY_NAME["worst"]
    idx, _ = _routing(w)
    assert idx.max() < w.E // w.N
    assert np.all(np.sort(idx, axis=1) == np.arange(8))


def test_kimi_is_skewed():
    w = gen.BY_NAME["kimi"]
    idx, _ = _routing(w)
    cnt = np.bincount(idx.ravel(), minlength=w.E)
    assert cnt.max() > 8 * cnt.mean()
    # hot experts are spread over ranks, not all on one
    hot = np.argsort(-cnt)[:8]
    assert len(set((hot // (w.E // w.N)).tolist())) > 4


def test_deterministic_and_seeded():
    w = gen.custom("t", T=32, H=64, K=4, E=16, N=4)
    a = gen.make_inputs(w)
    b = gen.make_inputs(w)
    c = gen.make_inputs(w, seed=999)
    for f in ("x", "topk_idx", "topk_w", "y"):
        assert np.array_equal(getattr(a, f), getattr(b, f))
    assert not np.array_equal(a.x, c.x)
    assert a.y.shape == (32 * 4, 64)


def test_bf16_roundtrip():
    v = np.array([1.0, -2.5, 0.0, 3.140625], np.float32)
    assert np.array_equal(gen.bf16_bits_to_f32(gen.to_bf16_bits(v)), v)
