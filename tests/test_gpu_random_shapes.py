"""Randomised shapes against the CPU oracle, through the C ABI.

Seeded random small configurations (logical ranks, experts per rank, top-k,
tokens per rank, hidden size), each run through every routing path the
context can take for it (automatic, single block, two kernels, cluster,
inside the pack, alone in one CTA) with random launch shapes (pack CTAs or
groups per SM, stages), for both payloads: the grouped rows, slot_row, the
fp8 codes and scales and the combine output bit for bit."""
import random

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


def _cases(seed, n):
    rng = random.Random(seed)
    out = []
    while len(out) < n:
        N = rng.choice([1, 2, 3, 4, 8, 16])
        L = rng.choice([1, 2, 3, 4, 8])
        E = N * L
        K = rng.randint(1, min(16, E))
        T = N * rng.choice([1, 3, 16, 31, 32, 33, 100, 250, 512])
        if T * K > 40000:
            continue
        H = rng.choice([128, 256, 384, 1024, 2048, 4096])
        opts = [dict(pack_ctas_per_sm=rng.randint(1, 8)) if rng.random() < 0.5 else {} for _ in range(6)]
        for o in opts:
            if rng.random() < 0.3:
                o["pack_stages"] = rng.randint(2, 8)
        out.append((T, H, K, E, N, opts))
    return out


CASES = _cases(20261202, 16)


@pytest.mark.parametrize("case", range(len(CASES)))
def test_random_shape_every_route(moe, oracle_mod, case):
    T, H, K, E, N, opts = CASES[case]
    w = gen.custom("random", T=T, H=H, K=K, E=E, N=N, seed_index=2000 + case)
    li = gen.make_inputs(w)
    d = oracle_mod.dispatch(li.x, li.topk_idx, E, N)
    out_ref = oracle_mod.combine(li.y, li.topk_w, d.slot_row)
    _, xq_ref, xs_ref = oracle_mod.dispatch_fp8(li.x, li.topk_idx, E, N)
    x, idx, wt, y = _dev(li.x.view(np.int16)), _dev(li.topk_idx), _dev(li.topk_w), _dev(li.y.view(np.int16))
    ran = 0
    for route, o in zip((0, 1, 2, 3, 4, 5), opts):
        try:
            layer = moe.MoELayer(T, H, K, E, N, route_variant=route, **o)
        except moe.MoEError:
            continue  # the path cannot run this shape (cluster not schedulable, too large for route_pack)
        ran += 1
        ex = torch.zeros((T * K, H), dtype=torch.int16, device="cuda")
        out = torch.zeros((T, H), dtype=torch.int16, device="cuda")
        lay = layer.layer(x, idx, wt, ex, y, out)
        assert layer.get_error() == moe.MOE_OK, (route, o)
        assert np.array_equal(lay["slot_row"].cpu().numpy(), d.slot_row), (route, o)
        assert np.array_equal(ex.cpu().numpy().view(np.uint16), d.expert_x), (route, o)
        assert np.array_equal(out.cpu().numpy().view(np.uint16), out_ref), (route, o)
        xq = torch.zeros((T * K, H), dtype=torch.uint8, device="cuda")
        xs = torch.zeros((T * K, H // 128), dtype=torch.float32, device="cuda")
        out.zero_()
        layer.dispatch_send_fp8(x, idx, xq, xs)
        layer.dispatch_recv()
        layer.combine_send(y)
        layer.combine_recv(wt, out)
        assert layer.get_error() == moe.MOE_OK, (route, o)
        assert np.array_equal(xq.cpu().numpy(), xq_ref), (route, o)
        assert np.array_equal(xs.cpu().numpy().view(np.uint32), xs_ref.view(np.uint32)), (route, o)
        assert np.array_equal(out.cpu().numpy().view(np.uint16), out_ref), (route, o)
        layer.close()
    assert ran >= 3  # automatic, single block and two kernels always run
