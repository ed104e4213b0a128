"""Pins for the oracle's combine, against things other than itself.

The combine is the router-weighted sum of a token's expert outputs
("Efficient and portable mixture-of-experts communication", Introduction and
Combine), accumulated only on the receiving side ("Enabling
trillion-parameter models on AWS EFA", evaluation of the prefill case).  The
oracle evaluates it as a float32 chain of fused multiply-adds in top-k order
from +0.0 and rounds once to bf16.  Pins:

* an exact rational re-evaluation of that chain (each step rounded to the
  nearest float32, ties to even, found by exact comparison among neighbours),
  then exact rounding to bf16 - catches a dropped or reordered term, a
  separately rounded multiply, a wrong start value or a wrong rounding;
* the bf16 conversion against torch's float32 -> bfloat16 (a library routine);
* closed forms: identity experts with weights summing to one return the input
  rows; a one-hot weight returns the chosen expert row; K = 1, w = 1 returns y;
* the double-precision evaluation stays within the float32 accumulation bound
  plus half a bf16 ulp of the exact sum.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

from combine_route_count_gb300 import inputs as gen


def _f32_neighbours(g: np.float32):
    return [np.nextafter(g, np.float32(-np.inf), dtype=np.float32), g,
            np.nextafter(g, np.float32(np.inf), dtype=np.float32)]


def round_fraction_to_f32(q: Fraction) -> np.float32:
    """Nearest float32 to the exact rational q, ties to the even significand."""
    g = np.float32(float(q))
    best = None
    for c in _f32_neighbours(g):
        if not np.isfinite(c):
            continue
        dist = abs(Fraction(float(c)) - q)
        key = (dist, int(np.array(c, np.float32).view(np.uint32)) & 1)
        if best is None or key < best[0]:
            best = (key, c)
    return np.float32(best[1])


def round_fraction_to_bf16_bits(q: Fraction) -> int:
    """Nearest bf16 (bit pattern) to the exact rational q, ties to even."""
    f = np.float32(float(q))
    hi16 = int(np.array(f, np.float32).view(np.uint32)) >> 16
    cands = []
    for b in (hi16 - 1, hi16, hi16 + 1):
        b &= 0xFFFF
        v = gen.bf16_bits_to_f32(np.array([b], np.uint16))[0]
        if np.isfinite(v):
            cands.append((abs(Fraction(float(v)) - q), b & 1, b))
    if q == 0:
        return 0x0000
    return min(cands)[2]


def exact_fma_chain_bf16(w_row, y_vals):
    acc = np.float32(0.0)
    for wk, yk in zip(w_row, y_vals):
        acc = round_fraction_to_f32(Fraction(float(wk)) * Fraction(float(yk)) + Fraction(float(acc)))
    return round_fraction_to_bf16_bits(Fraction(float(acc))), acc


def test_bf16_rounding_matches_torch(oracle_mod):
    rng = np.random.default_rng(7)
    vals = np.concatenate([
        rng.standard_normal(4000).astype(np.float32),
        (rng.standard_normal(1000) * 1e-30).astype(np.float32),
        (rng.standard_normal(1000) * 1e30).astype(np.float32),
        # exact ties: lower 16 bits = 0x8000 with even and odd kept halves
        (np.arange(0x3f80, 0x3f90, dtype=np.uint32) << 16 | 0x8000).view(np.float32),
        np.array([0.0, -0.0, 1.0, -1.0, 3.0e38, 1e-45], np.float32),
    ])
    want = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle_mod.float_to_bf16(float(v)) for v in vals], np.uint16)
    assert np.array_equal(got, want)


def test_double_to_bf16_is_exact_nearest(oracle_mod):
    rng = np.random.default_rng(8)
    vals = list(rng.standard_normal(3000)) + list(rng.standard_normal(200) * 1e-39) + [0.0, 1.0 + 2.0 ** -8,
                                                                                      1.0 + 3 * 2.0 ** -8]
    for v in vals:
        assert oracle_mod.double_to_bf16(float(v)) == round_fraction_to_bf16_bits(Fraction(float(v))), v


def test_fmaf_is_single_rounding(oracle_mod):
    rng = np.random.default_rng(9)
    a = rng.standard_normal(2000).astype(np.float32)
    b = rng.standard_normal(2000).astype(np.float32)
    c = rng.standard_normal(2000).astype(np.float32)
    for ai, bi, ci in zip(a, b, c):
        want = round_fraction_to_f32(Fraction(float(ai)) * Fraction(float(bi)) + Fraction(float(ci)))
        assert np.float32(oracle_mod.fmaf(float(ai), float(bi), float(ci))) == want


@pytest.mark.parametrize("seed,K", [(0, 1), (1, 2), (2, 3), (3, 8), (4, 16)])
def test_chain_matches_exact_rational_fma_chain(oracle_mod, seed, K):
    rng = np.random.default_rng(100 + seed)
    T, H = 6, 24
    rows = T * K
    y = gen.to_bf16_bits(rng.standard_normal((rows, H)).astype(np.float32))
    w = rng.random((T, K)).astype(np.float32)
    w[0] *= -1.0  # negative weights too
    slot_row = rng.permutation(rows).reshape(T, K).astype(np.int32)
    out = oracle_mod.combine(y, w, slot_row)
    yf = gen.bf16_bits_to_f32(y)
    for t in range(T):
        for h in range(H):
            bits, _ = exact_fma_chain_bf16(w[t], [yf[slot_row[t, k], h] for k in range(K)])
            assert out[t, h] == bits, (t, h)


def test_chain_start_is_positive_zero(oracle_mod):
    # w*y = -0 for every term: +0 + (-0) = +0 under round-to-nearest
    y = gen.to_bf16_bits(np.array([[-1.0, 1.0]], np.float32))
    w = np.array([[0.0]], np.float32)
    out = oracle_mod.combine(y, w, np.zeros((1, 1), np.int32))
    assert out.tolist() == [[0x0000, 0x0000]]


@pytest.mark.parametrize("name", ["tiny", "mixtral", "deepseek", "worst"])
def test_identity_experts_return_the_input(oracle_mod, name):
    wl = gen.BY_NAME[name]
    small = gen.Workload(wl.name, T=min(wl.T, 512), H=32, K=wl.K, E=wl.E, N=wl.N if min(wl.T, 512) % wl.N == 0 else 1,
                         router=wl.router, index=wl.index)
    li = gen.make_inputs(small, with_y=False)
    assert np.allclose(li.topk_w.astype(np.float64).sum(axis=1), 1.0, atol=1e-6)
    d = oracle_mod.dispatch(li.x, li.topk_idx, small.E, small.N)
    out = oracle_mod.combine(d.expert_x, li.topk_w, d.slot_row)
    assert np.array_equal(out, li.x)


def test_one_hot_weight_selects_one_expert(oracle_mod):
    rng = np.random.default_rng(5)
    T, K, H = 16, 4, 40
    y = gen.to_bf16_bits(rng.standard_normal((T * K, H)).astype(np.float32))
    slot_row = rng.permutation(T * K).reshape(T, K).astype(np.int32)
    pick = rng.integers(0, K, size=T)
    w = np.zeros((T, K), np.float32)
    w[np.arange(T), pick] = 1.0
    out = oracle_mod.combine(y, w, slot_row)
    assert np.array_equal(out, y[slot_row[np.arange(T), pick]])


def test_single_expert_unit_weight_is_a_copy(oracle_mod):
    rng = np.random.default_rng(6)
    T, H = 20, 64
    y = gen.to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    slot_row = rng.permutation(T).reshape(T, 1).astype(np.int32)
    out = oracle_mod.combine(y, np.ones((T, 1), np.float32), slot_row)
    assert np.array_equal(out, y[slot_row[:, 0]])


@pytest.mark.parametrize("name", ["tiny", "deepseek", "kimi"])
def test_double_precision_bound(oracle_mod, name):
    """|out32 - exact| <= K*2^-24*sum|w*y| (float32 chain) + half a bf16 ulp
    of the float32 result (final rounding), up to the double's own error."""
    wl = gen.BY_NAME[name]
    T = min(wl.T, 256)
    small = gen.Workload(wl.name, T=T, H=64, K=wl.K, E=wl.E, N=1, router=wl.router, index=wl.index)
    li = gen.make_inputs(small, with_y=True)
    d = oracle_mod.dispatch(li.x, li.topk_idx, small.E, 1)
    out32 = oracle_mod.combine(li.y, li.topk_w, d.slot_row)
    out64, exact, mag = oracle_mod.combine_f64(li.y, li.topk_w, d.slot_row)
    o32 = gen.bf16_bits_to_f32(out32).astype(np.float64)
    ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(o32), 2.0 ** -126))) - 7)
    bound = small.K * 2.0 ** -24 * mag * 1.001 + 0.5 * ulp + small.K * 2.0 ** -52 * mag
    assert np.all(np.abs(o32 - exact) <= bound)
    # the two evaluations round to the same bf16 almost everywhere; more than
    # one bf16 step apart only where the sum nearly cancels
    assert np.mean(out32 == out64) > 0.99
    step = np.abs(out32.astype(np.int32) - out64.astype(np.int32))
    assert np.mean(step > 1) < 1e-3
