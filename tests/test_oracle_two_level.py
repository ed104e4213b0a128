"""Pins for the oracle's two-level combine (partial sums on the sending side).

"Enabling trillion-parameter models on AWS EFA" (evaluation, prefill): DeepEP
adds up a token's expert outputs on the sending side to move less data, which
can cost precision; the pages' own kernels add only on the receiving side.
The oracle reads the sending-side form as: per rank holding some of the
token's experts, a bf16 partial = the float32 fused-multiply-add chain over
those experts in top-k order; the receiver adds the partials' float32 values in
ascending rank order and rounds once to bf16.

Pins (each ties the function to something other than itself):

* with one rank, the result is the single-level combine (already pinned);
* every partial equals the single-level combine with the weights of the other
  ranks' experts set to zero (a fused multiply-add by zero leaves a float32
  accumulator that started at +0.0 unchanged);
* the receiver's sum equals the single-level combine of the partial rows with
  unit weights (a fused multiply-add by one is a single rounded add);
* a hand-worked case where the partial's rounding changes the answer;
* the double-precision error bound on random data, and unused partial rows
  stay untouched.
"""
import numpy as np
import pytest

from combine_route_count_gb300 import inputs as gen


def ranks_of(idx, E, N):
    L = E // N
    return [sorted(set((row // L).tolist())) for row in idx]


def small_case(T=48, H=40, K=4, E=16, N=4, seed_index=31):
    w = gen.custom("twolevel", T=T, H=H, K=K, E=E, N=N, seed_index=seed_index)
    return w, gen.make_inputs(w)


def test_one_rank_is_the_single_level_combine(oracle_mod):
    w, li = small_case(E=8, N=1)
    d = oracle_mod.dispatch(li.x, li.topk_idx, w.E, w.N)
    out, part, nr = oracle_mod.combine_two_level(li.y, li.topk_idx, li.topk_w, d.slot_row, w.E, w.N)
    single = oracle_mod.combine(li.y, li.topk_w, d.slot_row)
    assert np.all(nr == 1)
    assert np.array_equal(out, single)
    assert np.array_equal(part, single)  # one slot per token: the partial is the answer


@pytest.mark.parametrize("shape", [(48, 40, 4, 16, 4), (32, 24, 8, 64, 8), (24, 16, 3, 6, 6), (16, 8, 5, 40, 2)])
def test_partials_are_masked_single_level_combines(oracle_mod, shape):
    T, H, K, E, N = shape
    w, li = small_case(T, H, K, E, N)
    d = oracle_mod.dispatch(li.x, li.topk_idx, E, N)
    out, part, nr = oracle_mod.combine_two_level(li.y, li.topk_idx, li.topk_w, d.slot_row, E, N)
    slots = min(K, N)
    L = E // N
    rk = ranks_of(li.topk_idx, E, N)
    assert nr.tolist() == [len(r) for r in rk]
    for t in range(T):
        for dd, r in enumerate(rk[t]):
            wm = np.zeros_like(li.topk_w)
            sel = (li.topk_idx[t] // L) == r
            wm[t, sel] = li.topk_w[t, sel]
            want = oracle_mod.combine(li.y, wm, d.slot_row)[t]
            assert np.array_equal(part[t * slots + dd], want), (t, dd)
    # receiver: unit-weight single-level combine over the used partial rows
    w1 = np.zeros((T, slots), np.float32)
    for t in range(T):
        w1[t, :nr[t]] = 1.0
    sr = (np.arange(T)[:, None] * slots + np.arange(slots)[None, :]).astype(np.int32)
    assert np.array_equal(out, oracle_mod.combine(part, w1, sr))


def test_hand_worked_cancellation(oracle_mod):
    """K=3, E=4, N=2 (two experts per rank); token 0 routes to experts 0, 1
    (rank 0) and 2 (rank 1), all weights 1; y rows: 1.0, 3*2^-9, -1.0.
    Receiver only: 1 + 3*2^-9 is exact in float32, minus 1 gives 3*2^-9 =
    0.005859375, a bf16 value: 0x3BC0.  Two-level: rank 0's partial
    bf16(1.005859375) rounds to 1 + 2^-7 = 0x3F81 (3/4 of a bf16 step up);
    rank 1's partial is -1.0 = 0xBF80; their sum 2^-7 gives 0x3C00: one third
    too large."""
    H = 8
    y = np.zeros((3, H), np.uint16)
    y[0, :] = 0x3F80  # 1.0
    y[1, :] = 0x3BC0  # 3 * 2^-9
    y[2, :] = 0xBF80  # -1.0
    idx = np.array([[0, 1, 2]], np.int32)
    wts = np.ones((1, 3), np.float32)
    slot_row = np.array([[0, 1, 2]], np.int32)
    single = oracle_mod.combine(y, wts, slot_row)
    out, part, nr = oracle_mod.combine_two_level(y, idx, wts, slot_row, 4, 2)
    assert np.all(single == 0x3BC0)
    assert nr.tolist() == [2]
    assert np.all(part[0] == 0x3F81) and np.all(part[1] == 0xBF80)
    assert np.all(out == 0x3C00)


def test_error_bound_and_untouched_rows(oracle_mod):
    w, li = small_case(T=64, H=96, K=8, E=64, N=16, seed_index=37)
    d = oracle_mod.dispatch(li.x, li.topk_idx, w.E, w.N)
    slots = min(w.K, w.N)
    sentinel = np.full((w.T * slots, w.H), 0x7FC1, np.uint16)  # a NaN pattern nobody writes
    out, part, nr = oracle_mod.combine_two_level(li.y, li.topk_idx, li.topk_w, d.slot_row, w.E, w.N,
                                                 partial=sentinel)
    for t in range(w.T):
        rows = part[t * slots:(t + 1) * slots]
        assert not np.any(rows[:nr[t]] == 0x7FC1)
        assert np.all(rows[nr[t]:] == 0x7FC1)
    _, exact, mag = oracle_mod.combine_f64(li.y, li.topk_w, d.slot_row)
    f = gen.bf16_bits_to_f32(out).astype(np.float64)
    pf = gen.bf16_bits_to_f32(part).astype(np.float64)
    psum = np.zeros_like(exact)
    for t in range(w.T):
        psum[t] = np.abs(pf[t * slots:t * slots + nr[t]]).sum(axis=0)
    # partial rounding (2^-8 relative each), final rounding, float32 chains
    bound = 2.0 ** -8 * psum + 2.0 ** -8 * np.abs(f) + (w.K + slots) * 2.0 ** -24 * mag * 1.01 + 1e-30
    assert np.all(np.abs(f - exact) <= bound)


def test_rejects_bad_expert_index(oracle_mod):
    w, li = small_case()
    d = oracle_mod.dispatch(li.x, li.topk_idx, w.E, w.N)
    idx = li.topk_idx.copy()
    idx[3, 1] = w.E
    with pytest.raises(oracle_mod.OracleError):
        oracle_mod.combine_two_level(li.y, idx, li.topk_w, d.slot_row, w.E, w.N)
