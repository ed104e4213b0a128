"""Pins for the oracle's two-stage dispatch (per-peer send buffers, then the
receiver's shuffle into the grouped-GEMM input).

"Enabling trillion-parameter models on AWS EFA" (dispatch and combine timing):
the sender copies tokens into contiguous per-peer send buffers at offsets
from the cumulative sum of its per-expert counts; the receiver shuffles them
into the tensor handed to the grouped GEMM.  Pins:

* each source rank's send rows equal the direct dispatch of that rank's token
  slice alone (a single-rank problem: its rows in expert, then token order);
* the shuffled result equals the direct dispatch of the whole problem;
* send_dest is a permutation, each send row's destination belongs to a token
  of that source rank, and send rows are grouped by destination rank;
* brute force over every routing of tiny problems.
"""
import itertools

import numpy as np
import pytest

from combine_route_count_gb300 import inputs as gen


@pytest.mark.parametrize("shape", [(64, 24, 2, 8, 2), (96, 16, 4, 16, 4), (32, 8, 8, 64, 8), (60, 8, 3, 6, 6),
                                   (16, 8, 1, 4, 4)])
def test_send_rows_are_per_rank_dispatches(oracle_mod, shape):
    T, H, K, E, N = shape
    w = gen.custom("staged", T=T, H=H, K=K, E=E, N=N, seed_index=53)
    li = gen.make_inputs(w, with_y=False)
    send, dest, ex, sr = oracle_mod.dispatch_staged(li.x, li.topk_idx, E, N)
    direct = oracle_mod.dispatch(li.x, li.topk_idx, E, N)
    assert np.array_equal(ex, direct.expert_x)
    assert np.array_equal(sr, direct.slot_row)
    Tr = T // N
    L = E // N
    assert np.array_equal(np.sort(dest), np.arange(T * K))
    for s in range(N):
        sl = slice(s * Tr, (s + 1) * Tr)
        alone = oracle_mod.dispatch(li.x[sl], li.topk_idx[sl], E, 1)
        rows = slice(s * Tr * K, (s + 1) * Tr * K)
        assert np.array_equal(send[rows], alone.expert_x)
        # destination rows belong to this source rank's tokens
        tok = direct.row_src[dest[rows]] // K
        assert np.all((tok >= s * Tr) & (tok < (s + 1) * Tr))
        # grouped by destination rank, ascending
        dst_rank = li.topk_idx.reshape(-1)[direct.row_src[dest[rows]]] // L
        assert np.all(np.diff(dst_rank) >= 0)


def test_brute_force_tiny(oracle_mod):
    T, H, K, E = 2, 8, 2, 4
    rng = np.random.default_rng(59)
    x = gen.to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    pairs = list(itertools.permutations(range(E), K))
    for N in (1, 2):
        for choice in itertools.product(pairs, repeat=T):
            idx = np.array(choice, np.int32)
            send, dest, ex, sr = oracle_mod.dispatch_staged(x, idx, E, N)
            direct = oracle_mod.dispatch(x, idx, E, N)
            assert np.array_equal(ex, direct.expert_x) and np.array_equal(sr, direct.slot_row)
            for j in range(T * K):
                assert np.array_equal(send[j], ex[dest[j]])


def test_rejects_bad_routes(oracle_mod):
    w = gen.custom("stagedbad", T=8, H=8, K=2, E=4, N=2, seed_index=61)
    li = gen.make_inputs(w, with_y=False)
    idx = li.topk_idx.copy()
    idx[2] = [1, 1]
    with pytest.raises(oracle_mod.OracleError):
        oracle_mod.dispatch_staged(li.x, idx, w.E, w.N)
