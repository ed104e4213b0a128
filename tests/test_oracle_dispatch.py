"""Pins for the oracle's dispatch, against things other than itself.

Dispatch has a plain definition (the method reaches it exactly): rows are
grouped by expert ("Efficient and portable mixture-of-experts communication",
Dispatch: the receiver unpacks into the grouped-GEMM input and keeps where each
row came from), counts are exchanged and their cumulative sum gives contiguous
offsets ("Enabling trillion-parameter models on AWS EFA", Dispatch and
combine; Send and receive buffers), and inside one expert rows keep the
(source rank, token) order.  That is a stable sort by expert, so:

* numpy's stable argsort (a library routine) must give the same placement;
* a brute-force loop (for each expert, for each token, for each slot) must too;
* every routing of tiny problems is enumerated;
* the invariants the pages fix hold on all five workloads: counts sum to T*K,
  placement is a bijection between (token, slot) pairs and rows, each rank
  receives at most N*T*max(R, E/N) rows (equal to the bound on rank 0 of the
  worst case), and each row is a byte copy of its token.
"""
import itertools
import os

import numpy as np
import pytest

from combine_route_count_gb300 import inputs as gen


def _small(w, H=16):
    """Same routing as workload ``w`` (routing is drawn before the rows) with
    narrow rows, to keep the CPU suite fast."""
    small = gen.Workload(w.name, T=w.T, H=H, K=w.K, E=w.E, N=w.N, router=w.router, index=w.index)
    return gen.make_inputs(small, with_y=False)


def brute_force_dispatch(idx, E, N):
    """For each expert in order, for each token in order, for each slot:
    append.  Returns (row_src, slot_row, counts, src_offsets)."""
    T, K = idx.shape
    Tr = T // N
    row_src, slot_row = [], np.full((T, K), -1, np.int64)
    counts = [0] * E
    src_off = np.zeros((E, N), np.int64)
    for e in range(E):
        for s in range(N):
            src_off[e, s] = len(row_src)
            for t in range(s * Tr, (s + 1) * Tr):
                for k in range(K):
                    if idx[t, k] == e:
                        slot_row[t, k] = len(row_src)
                        row_src.append(t * K + k)
                        counts[e] += 1
    return np.array(row_src, np.int64), slot_row, np.array(counts), src_off


def check_invariants(d, x, idx, E, N):
    T, K = idx.shape
    rows = T * K
    Tr, L = T // N, E // N
    assert d.expert_counts.sum() == rows
    assert d.expert_offsets[0] == 0 and d.expert_offsets[-1] == rows
    assert np.array_equal(np.diff(d.expert_offsets), d.expert_counts)
    # bijection: slot_row is a permutation of [0, rows) and row_src its inverse
    sr = d.slot_row.ravel().astype(np.int64)
    assert np.array_equal(np.sort(sr), np.arange(rows))
    assert np.array_equal(d.row_src[sr], np.arange(rows))
    # every row of expert e comes from a token that chose e, tokens increasing
    for e in range(E):
        a, b = d.expert_offsets[e], d.expert_offsets[e + 1]
        src = d.row_src[a:b].astype(np.int64)
        assert np.all(idx.ravel()[src] == e)
        assert np.all(np.diff(src // K) > 0)
        # src_offsets split the expert's rows by source rank
        toks = src // K
        for s in range(N):
            lo = d.src_offsets[e, s]
            hi = d.src_offsets[e, s + 1] if s + 1 < N else b
            assert a <= lo <= hi <= b
            assert np.all((toks[lo - a:hi - a] // Tr) == s)
    # per-rank receive bound
    assert np.array_equal(d.rank_offsets, d.expert_offsets[::L])
    recv = np.diff(d.rank_offsets)
    assert np.all(recv <= N * Tr * max(K, L))
    # bytes: row i is a copy of token row_src[i] // K
    if rows:
        assert np.array_equal(d.expert_x[:rows], x[d.row_src // K])


@pytest.mark.parametrize("wl", gen.WORKLOADS, ids=[w.name for w in gen.WORKLOADS])
def test_library_stable_sort_and_invariants(oracle_mod, wl):
    li = _small(wl)
    d = oracle_mod.dispatch(li.x, li.topk_idx, wl.E, wl.N)
    flat = li.topk_idx.ravel()
    order = np.argsort(flat, kind="stable")
    assert np.array_equal(d.row_src, order)
    inv = np.empty_like(order)
    inv[order] = np.arange(order.size)
    assert np.array_equal(d.slot_row.ravel(), inv)
    assert np.array_equal(d.expert_counts, np.bincount(flat, minlength=wl.E))
    assert np.array_equal(d.expert_offsets[1:], np.cumsum(np.bincount(flat, minlength=wl.E)))
    # src_offsets from per-rank histograms (numpy bincount per rank block)
    per_rank = np.stack([np.bincount(li.topk_idx[s * wl.tokens_per_rank:(s + 1) * wl.tokens_per_rank].ravel(),
                                     minlength=wl.E) for s in range(wl.N)])  # [N, E]
    before = np.cumsum(per_rank, axis=0) - per_rank                         # ranks < s
    assert np.array_equal(d.src_offsets, d.expert_offsets[:-1, None] + before.T)
    check_invariants(d, li.x, li.topk_idx, wl.E, wl.N)


def test_worst_case_reaches_the_bound(oracle_mod):
    wl = gen.BY_NAME["worst"]
    li = _small(wl)
    d = oracle_mod.dispatch(li.x, li.topk_idx, wl.E, wl.N)
    recv = np.diff(d.rank_offsets)
    bound = wl.N * wl.tokens_per_rank * max(wl.K, wl.E // wl.N)
    assert bound == 65536
    assert recv[0] == bound
    assert np.all(recv[1:] == 0)


@pytest.mark.parametrize("seed", range(6))
def test_brute_force_loops(oracle_mod, seed):
    rng = np.random.default_rng(seed)
    N = int(rng.choice([1, 2, 4]))
    T = N * int(rng.integers(1, 12))
    E = N * int(rng.integers(1, 5))
    K = int(rng.integers(1, min(E, 6) + 1))
    idx = np.stack([rng.permutation(E)[:K] for _ in range(T)]).astype(np.int32)
    x = rng.integers(0, 1 << 16, size=(T, 8), dtype=np.uint16)
    d = oracle_mod.dispatch(x, idx, E, N)
    row_src, slot_row, counts, src_off = brute_force_dispatch(idx, E, N)
    assert np.array_equal(d.row_src, row_src)
    assert np.array_equal(d.slot_row, slot_row)
    assert np.array_equal(d.expert_counts, counts)
    assert np.array_equal(d.src_offsets, src_off)
    check_invariants(d, x, idx, E, N)


def _all_routings(T, E, K):
    per_token = list(itertools.permutations(range(E), K))
    for combo in itertools.product(per_token, repeat=T):
        yield np.array(combo, dtype=np.int32).reshape(T, K)


@pytest.mark.parametrize("T,E,K,N", [(1, 2, 1, 1), (2, 3, 2, 1), (2, 4, 2, 2), (3, 4, 1, 1),
                                     (2, 4, 1, 2), (3, 3, 2, 1)])
def test_exhaustive_tiny(oracle_mod, T, E, K, N):
    if T % N:
        pytest.skip("T must split over N ranks")
    x = np.arange(T * 4, dtype=np.uint16).reshape(T, 4) * 257
    n = 0
    for idx in _all_routings(T, E, K):
        d = oracle_mod.dispatch(x, idx, E, N)
        row_src, slot_row, counts, src_off = brute_force_dispatch(idx, E, N)
        assert np.array_equal(d.row_src, row_src)
        assert np.array_equal(d.slot_row, slot_row)
        assert np.array_equal(d.src_offsets, src_off)
        check_invariants(d, x, idx, E, N)
        n += 1
    assert n > 0


def load_hand_example():
    """The hand-worked case in tests/golden/dispatch_hand_example.txt."""
    path = os.path.join(os.path.dirname(__file__), "golden", "dispatch_hand_example.txt")
    vals = {}
    for line in open(path):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, *rest = line.split()
        if key == "sizes":
            vals[key] = {kv.split("=")[0]: int(kv.split("=")[1]) for kv in rest}
        else:
            vals[key] = [int(v) for v in rest]
    return vals


def test_hand_worked_example(oracle_mod):
    g = load_hand_example()
    sz = g["sizes"]
    T, H, K, E, N = sz["T"], sz["H"], sz["K"], sz["E"], sz["N"]
    idx = np.array(g["topk_idx"], np.int32).reshape(T, K)
    x = np.array(g["x"], np.uint16).reshape(T, H)
    d = oracle_mod.dispatch(x, idx, E, N)
    assert d.expert_counts.tolist() == g["expert_counts"]
    assert d.expert_offsets.tolist() == g["expert_offsets"]
    assert d.rank_offsets.tolist() == g["rank_offsets"]
    assert d.src_offsets.ravel().tolist() == g["src_offsets"]
    assert d.slot_row.ravel().tolist() == g["slot_row"]
    assert d.row_src.tolist() == g["row_src"]
    assert d.expert_x[:, 0].tolist() == g["expert_x_col0"]


def test_empty_input(oracle_mod):
    x = np.zeros((0, 8), np.uint16)
    idx = np.zeros((0, 2), np.int32)
    d = oracle_mod.dispatch(x, idx, 4, 2)
    assert d.expert_counts.tolist() == [0] * 4
    assert d.expert_offsets.tolist() == [0] * 5
    assert d.rank_offsets.tolist() == [0] * 3


@pytest.mark.parametrize("bad", [-1, 4, 1 << 30])
def test_out_of_range_expert_is_an_error(oracle_mod, bad):
    idx = np.array([[0, 1], [2, bad]], np.int32)
    with pytest.raises(oracle_mod.OracleError) as ei:
        oracle_mod.dispatch(np.zeros((2, 8), np.uint16), idx, 4, 2)
    assert ei.value.code == oracle_mod.EROUTE


def test_repeated_expert_is_an_error(oracle_mod):
    idx = np.array([[0, 1], [3, 3]], np.int32)
    with pytest.raises(oracle_mod.OracleError) as ei:
        oracle_mod.dispatch(np.zeros((2, 8), np.uint16), idx, 4, 2)
    assert ei.value.code == oracle_mod.EROUTE


@pytest.mark.parametrize("T,E,K,N,cap", [(3, 4, 1, 2, None), (2, 3, 1, 2, None), (2, 4, 5, 1, None),
                                         (2, 4, 2, 1, 3)])
def test_bad_sizes_are_rejected(oracle_mod, T, E, K, N, cap):
    idx = np.zeros((T, K), np.int32)
    for t in range(T):
        idx[t] = np.arange(K) % max(E, 1)
    with pytest.raises(oracle_mod.OracleError) as ei:
        oracle_mod.dispatch(np.zeros((T, 8), np.uint16), idx, E, N, expert_x_rows=cap)
    assert ei.value.code == oracle_mod.EINVAL


def test_rows_past_the_filled_region_are_untouched(oracle_mod):
    li = _small(gen.BY_NAME["tiny"])
    d = oracle_mod.dispatch(li.x, li.topk_idx, 8, 2, expert_x_rows=li.x.shape[0] * 2 + 5)
    assert np.all(d.expert_x[li.x.shape[0] * 2:] == 0)
