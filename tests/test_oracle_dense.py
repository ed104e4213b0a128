"""Pins of the dense padded all-to-all oracle (oracle_dispatch_dense,
oracle_combine_dense) against things fixed independently of its loops:
the hand-worked example in tests/golden/dense_hand_example.txt, the grouped
layout of the direct dispatch (the same rows must come out), an exact block
transpose (numpy), a per-block brute force by lexsort, the receiver-only
combine (the same float32 chain on the same values), the capacity limit and
the worst case where one block is full."""
import os

import numpy as np
import pytest

from combine_route_count_gb300 import inputs as gen

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "dense_hand_example.txt")


def _golden():
    rec = {"idx": [], "send": []}
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, *vals = line.split()
        if key in ("idx", "send"):
            rec[key].append(vals)
        else:
            rec[key] = vals
    return rec


def test_hand_worked_example(oracle_mod):
    g = _golden()
    idx = np.array(g["idx"], dtype=np.int32)
    T, K, E, N, H, cap = 4, 2, 4, 2, 8, 4
    x = (np.arange(T, dtype=np.uint16)[:, None] + 1) * np.ones((1, H), np.uint16)  # row t holds t+1
    send, recv, ex, pos = oracle_mod.dispatch_dense(x, idx, E, N, cap)
    for b, rows in enumerate(g["send"]):
        for j, tok in enumerate(rows):
            want = 0 if tok == "-" else int(tok) + 1
            assert np.all(send[b * cap + j] == want), (b, j)
    for rb, sb in enumerate(int(v) for v in g["send_block_of_recv"]):
        assert np.array_equal(recv[rb * cap:(rb + 1) * cap], send[sb * cap:(sb + 1) * cap])
    assert [int(v) + 1 for v in g["grouped"]] == ex[:, 0].tolist()
    assert pos.reshape(-1).tolist() == [int(v) for v in g["send_pos"]]


def _blocks_by_lexsort(idx, E, N, cap, x):
    """Send buffer built another way: per (s, r), the pairs of source s with an
    expert on rank r, ordered by (expert, token) with numpy's lexsort."""
    T, K = idx.shape
    Tr, L = T // N, E // N
    H = x.shape[1]
    send = np.zeros((N * N * cap, H), np.uint16)
    t_of = np.repeat(np.arange(T), K)
    e_of = idx.reshape(-1)
    for s in range(N):
        for r in range(N):
            sel = np.nonzero((t_of // Tr == s) & (e_of // L == r))[0]
            order = sel[np.lexsort((t_of[sel], e_of[sel]))]
            assert len(order) <= cap
            send[(s * N + r) * cap:(s * N + r) * cap + len(order)] = x[t_of[order]]
    return send


@pytest.mark.parametrize("shape", [(64, 16, 2, 8, 2), (96, 24, 3, 12, 4), (40, 8, 4, 4, 4), (30, 16, 1, 6, 3),
                                   (64, 8, 8, 64, 8)])
def test_dense_dispatch_against_independent_forms(oracle_mod, shape):
    T, H, K, E, N = shape
    w = gen.custom("dense", T=T, H=H, K=K, E=E, N=N, seed_index=91)
    li = gen.make_inputs(w)
    cap = T // N * min(K, E // N)
    send, recv, ex, pos = oracle_mod.dispatch_dense(li.x, li.topk_idx, E, N, cap)
    d = oracle_mod.dispatch(li.x, li.topk_idx, E, N)
    # The grouped rows are those of the direct placement.
    assert np.array_equal(ex, d.expert_x)
    # The exchange is a block transpose of the whole buffer, padding included.
    blocks = send.reshape(N, N, cap, H)
    assert np.array_equal(recv.reshape(N, N, cap, H), blocks.transpose(1, 0, 2, 3))
    # Every block's rows by an independent ordering; padding stays zero.
    assert np.array_equal(send, _blocks_by_lexsort(li.topk_idx, E, N, cap, li.x))
    # The send row of every pair holds that pair's token row.
    assert np.array_equal(send[pos.reshape(-1)], li.x[np.repeat(np.arange(T), K)])
    # Combine through the padded blocks back: the receiver-only chain's bits.
    out, back_send, back_recv = oracle_mod.combine_dense(li.y, li.topk_w, d.slot_row, pos, N, cap)
    assert np.array_equal(out, oracle_mod.combine(li.y, li.topk_w, d.slot_row))
    assert np.array_equal(back_recv.reshape(N, N, cap, H), back_send.reshape(N, N, cap, H).transpose(1, 0, 2, 3))
    assert np.array_equal(back_recv[pos.reshape(-1)], li.y[d.slot_row.reshape(-1)])


def test_capacity_limit_and_a_full_block(oracle_mod):
    w = gen.custom("dense-worst", T=32, H=8, K=4, E=16, N=4, router="rank0_only", seed_index=5)
    li = gen.make_inputs(w, with_y=False)
    cap = 32 // 4 * min(4, 16 // 4)  # every token puts min(K, E/N) = 4 rows on rank 0
    with pytest.raises(oracle_mod.OracleError) as e:
        oracle_mod.dispatch_dense(li.x, li.topk_idx, 16, 4, cap - 1)
    assert e.value.code == oracle_mod.EINVAL
    send, recv, ex, pos = oracle_mod.dispatch_dense(li.x, li.topk_idx, 16, 4, cap)
    assert np.array_equal(ex, oracle_mod.dispatch(li.x, li.topk_idx, 16, 4).expert_x)
    # Block s*N+0 is full for every source; blocks to other ranks are all padding.
    per = send.reshape(4, 4, cap, 8)
    assert np.all(per[:, 0].reshape(-1, 8).any(axis=1))
    assert not per[:, 1:].any()


def test_routing_errors(oracle_mod):
    w = gen.custom("dense-bad", T=8, H=8, K=2, E=4, N=2, seed_index=6)
    li = gen.make_inputs(w, with_y=False)
    idx = li.topk_idx.copy()
    idx[3, 1] = idx[3, 0]
    with pytest.raises(oracle_mod.OracleError) as e:
        oracle_mod.dispatch_dense(li.x, idx, 4, 2, 8)
    assert e.value.code == oracle_mod.EROUTE
