"""The checked build (libmoe_checked.so): routing-table entries verified
against their buffers before use.

In a separate process (the library is loaded once per process): a layer is
bit-exact against the oracle (the checks never fire on valid tables); then one
slot_row entry in the workspace is overwritten with T*K, one row past the
expert outputs handed to combine_send, and each combine form must report
MOE_ECORRUPT, write nothing for that token and still write every other token
bit-exact.  The fp8 dispatch runs clean and bit-exact in the checked build
too.  The expert-output buffer has guard rows after it, so the entry
points inside the allocation even if a check were missing."""
import json
import os
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = r"""
import json, sys
sys.path.insert(0, ROOT)
import numpy as np, torch
from combine_route_count_gb300 import build, inputs as gen, moe
moe.load_library(build.build(checked=True))
import oracle

SENT = 0x7FC1
w = gen.custom("checked", T=2048, H=1024, K=8, E=64, N=8, seed_index=109)
li = gen.make_inputs(w)
T, H, K, rows = w.T, w.H, w.K, w.T * w.K
d = oracle.dispatch(li.x, li.topk_idx, w.E, w.N)
ref = oracle.combine(li.y, li.topk_w, d.slot_row)
dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
x, idx, wt = dev(li.x.view(np.int16)), dev(li.topk_idx), dev(li.topk_w)
ybig = torch.zeros((rows + 4, H), dtype=torch.int16, device="cuda")
ybig[:rows] = dev(li.y.view(np.int16))
y = ybig[:rows]
res = {}
for name, opts in (("bulk", dict(combine_variant=0)), ("vector", dict(combine_variant=1)), ("two_level", {})):
    layer = moe.MoELayer(T, H, K, w.E, w.N, **opts)
    ex = torch.zeros((rows, H), dtype=torch.int16, device="cuda")
    out = torch.full((T, H), SENT, dtype=torch.int16, device="cuda")
    part = torch.zeros((layer.partial_rows(), H), dtype=torch.int16, device="cuda")
    layer.dispatch_send(x, idx, ex)
    lay = layer.dispatch_recv()
    layer.combine_send(y)
    if name == "two_level":
        layer.combine_recv_two_level(wt, part, out)
        want = oracle.combine_two_level(li.y, li.topk_idx, li.topk_w, d.slot_row, w.E, w.N)[0]
    else:
        layer.combine_recv(wt, out)
        want = ref
    clean = (layer.get_error() == 0 and np.array_equal(out.cpu().numpy().view(np.uint16), want)
             and np.array_equal(ex.cpu().numpy().view(np.uint16), d.expert_x))
    # corrupt one entry of token 5 and combine again
    out.fill_(SENT)
    layer.dispatch_send(x, idx, ex)
    lay = layer.dispatch_recv()
    lay["slot_row"].view(-1)[5 * K + 2] = rows
    layer.combine_send(y)
    if name == "two_level":
        layer.combine_recv_two_level(wt, part, out)
    else:
        layer.combine_recv(wt, out)
    status = layer.get_error()
    o = out.cpu().numpy().view(np.uint16)
    others = np.ones(T, bool)
    others[5] = False
    res[name] = dict(clean=bool(clean), status=int(status), token_untouched=bool(np.all(o[5] == SENT)),
                     others_exact=bool(np.array_equal(o[others], want[others])))
    layer.close()
# fp8 dispatch in the checked build, both forms (routing inside the fp8 pack,
# and route_cluster + the fp8 pack): bit-exact, no check fires.
_, xq_ref, xs_ref = oracle.dispatch_fp8(li.x, li.topk_idx, w.E, w.N)
for name, route in (("fp8_fused", 4), ("fp8_two_kernel", 3)):
    layer = moe.MoELayer(T, H, K, w.E, w.N, route_variant=route)
    xq = torch.zeros((rows, H), dtype=torch.uint8, device="cuda")
    xs = torch.zeros((rows, H // 128), dtype=torch.float32, device="cuda")
    layer.dispatch_send_fp8(x, idx, xq, xs)
    layer.dispatch_recv()
    layer.combine_send(y)
    out = torch.zeros((T, H), dtype=torch.int16, device="cuda")
    layer.combine_recv(wt, out)
    res[name] = dict(status=int(layer.get_error()), codes=bool(np.array_equal(xq.cpu().numpy(), xq_ref)),
                     scales=bool(np.array_equal(xs.cpu().numpy().view(np.uint32), xs_ref.view(np.uint32))),
                     out=bool(np.array_equal(out.cpu().numpy().view(np.uint16), ref)))
    layer.close()
print(json.dumps(res))
"""


def test_checked_build_detects_a_corrupt_table_entry():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from combine_route_count_gb300 import moe
    r = subprocess.run([sys.executable, "-c", SCRIPT.replace("ROOT", repr(ROOT))], capture_output=True, text=True,
                       timeout=900, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-3000:]
    res = json.loads(r.stdout.strip().splitlines()[-1])
    for name in ("fp8_fused", "fp8_two_kernel"):
        v = res.pop(name)
        assert v == dict(status=moe.MOE_OK, codes=True, scales=True, out=True), (name, v)
    for name, v in res.items():
        assert v["clean"], (name, v)
        assert v["status"] == moe.MOE_ECORRUPT, (name, v)
        assert v["token_untouched"] and v["others_exact"], (name, v)
