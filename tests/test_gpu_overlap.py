"""Split send/receive halves with other work in flight, and MOE_OPT_MAX_SMS.

"Efficient and portable mixture-of-experts communication" (Portable kernels,
Benchmarks): the send and receive halves are separate so that other work can
run between and beside them.  These tests interleave two contexts (two
micro-batches) on two streams with an independent bf16 GEMM on a third, and
check that every output is still bit-exact against the oracle; and that
bounding the persistent grids to fewer SMs changes nothing in the results."""
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


def _inputs(li):
    return dict(x=_dev(li.x.view(np.int16)), idx=_dev(li.topk_idx), w=_dev(li.topk_w), y=_dev(li.y.view(np.int16)))


def test_two_micro_batches_on_two_streams_with_a_gemm(moe, oracle_mod):
    w = gen.BY_NAME["deepseek"]
    mbs = []
    for m in range(2):
        wm = gen.custom(f"mb{m}", T=w.T // 2, H=w.H, K=w.K, E=w.E, N=w.N, router="sigmoid_topk", seed_index=73 + m)
        li = gen.make_inputs(wm)
        d = dict(wl=wm, li=li, layer=moe.MoELayer(wm.T, wm.H, wm.K, wm.E, wm.N), **_inputs(li),
                 ex=torch.zeros((wm.T * wm.K, wm.H), dtype=torch.int16, device="cuda"),
                 out=torch.zeros((wm.T, wm.H), dtype=torch.int16, device="cuda"),
                 stream=torch.cuda.Stream())
        mbs.append(d)
    s_gemm = torch.cuda.Stream()
    a = torch.randn((4096, 7168), device="cuda", dtype=torch.bfloat16)
    b = torch.randn((7168, 4096), device="cuda", dtype=torch.bfloat16)
    torch.cuda.synchronize()
    for _ in range(3):
        # every call of both micro-batches interleaved on the host, GEMM beside them
        with torch.cuda.stream(s_gemm):
            c = a @ b
        for mb in mbs:
            mb["layer"].dispatch_send(mb["x"], mb["idx"], mb["ex"], mb["stream"])
        for mb in mbs:
            mb["layer"].dispatch_recv(mb["stream"])
            mb["layer"].combine_send(mb["y"], mb["stream"])
        for mb in mbs:
            mb["layer"].combine_recv(mb["w"], mb["out"], mb["stream"])
    torch.cuda.synchronize()
    assert torch.isfinite(c.float()).all()
    for mb in mbs:
        wm, li = mb["wl"], mb["li"]
        assert mb["layer"].get_error(mb["stream"]) == 0
        d = oracle_mod.dispatch(li.x, li.topk_idx, wm.E, wm.N)
        assert np.array_equal(mb["ex"].cpu().numpy().view(np.uint16), d.expert_x)
        assert np.array_equal(mb["out"].cpu().numpy().view(np.uint16), oracle_mod.combine(li.y, li.topk_w, d.slot_row))


@pytest.mark.parametrize("max_sms", [1, 19, 76, 151])
def test_max_sms_keeps_results(moe, oracle_mod, max_sms):
    w = gen.BY_NAME["deepseek"]
    li = gen.make_inputs(w)
    d = oracle_mod.dispatch(li.x, li.topk_idx, w.E, w.N)
    want_out = oracle_mod.combine(li.y, li.topk_w, d.slot_row)
    for options in ({}, {"combine_variant": 0}, {"pack_variant": 0, "pack_ctas_per_sm": 1}):
        layer = moe.MoELayer(w.T, w.H, w.K, w.E, w.N, max_sms=max_sms, **options)
        assert layer.get_option(moe.MOE_OPT_MAX_SMS) == max_sms
        t = _inputs(li)
        ex = torch.zeros((w.T * w.K, w.H), dtype=torch.int16, device="cuda")
        out = torch.zeros((w.T, w.H), dtype=torch.int16, device="cuda")
        layer.layer(t["x"], t["idx"], t["w"], ex, t["y"], out)
        assert layer.get_error() == 0
        assert np.array_equal(ex.cpu().numpy().view(np.uint16), d.expert_x)
        assert np.array_equal(out.cpu().numpy().view(np.uint16), want_out)
        layer.close()


def test_max_sms_rejects_out_of_range(moe):
    layer = moe.MoELayer(64, 256, 2, 8, 2)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    with pytest.raises(moe.MoEError):
        layer.set_option(moe.MOE_OPT_MAX_SMS, sms + 1)
    with pytest.raises(moe.MoEError):
        layer.set_option(moe.MOE_OPT_MAX_SMS, -1)
    layer.set_option(moe.MOE_OPT_MAX_SMS, sms)
    assert layer.get_option(moe.MOE_OPT_MAX_SMS) == sms
