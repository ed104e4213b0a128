"""The C ABI on the host: the library builds, loads and exports every entry
point that include/moe.h declares; the checks that run before any CUDA call
behave as documented.  No GPU is needed."""
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def moe():
    from combine_route_count_gb300 import build, moe as m
    build.build()
    m.load_library()
    return m


def _declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if not fn.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", fn)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*(moe_[a-z0-9_]+)\s*\(", text, re.M):
            names.add(m.group(1))
    return names


def test_every_declared_symbol_is_exported(moe):
    declared = _declared_functions()
    assert declared, "no declarations found"
    assert declared == set(moe.EXPORTS)
    lib = moe.load_library()
    for name in declared:
        assert hasattr(lib, name), name
    nm = os.popen(f"nm -D --defined-only {moe.LIB_PATH}").read()
    exported = {l.split()[-1] for l in nm.splitlines() if " T " in l}
    assert declared <= exported
    # nothing else leaks out of the library
    assert {s for s in exported if s.startswith("moe")} == declared


def test_build_targets_sm103a_only():
    from combine_route_count_gb300 import build
    assert build.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]


@pytest.mark.parametrize("cfg,ok", [
    ((64, 256, 2, 8, 2), True),
    ((0, 256, 2, 8, 2), True),             # empty layer
    ((4096, 7168, 8, 256, 32), True),
    ((16384, 7168, 8, 384, 64), True),
    ((8, 8, 16, 1024, 8), True),           # limits: K = 16, E = 1024
    ((63, 256, 2, 8, 2), False),           # T % N
    ((64, 256, 2, 9, 2), False),           # E % N
    ((64, 250, 2, 8, 2), False),           # H % 8
    ((64, 256, 9, 8, 2), False),           # K > E
    ((64, 256, 17, 32, 2), False),         # K > 16
    ((64, 256, 2, 1032, 2), False),        # E > 1024
    ((64, 256, 0, 8, 2), False),
    ((-2, 256, 2, 8, 2), False),
    ((1 << 28, 256, 16, 32, 2), False),    # T*K >= 2^31
])
def test_validate_config(moe, cfg, ok):
    rc = moe.moe_validate_config(moe.make_config(*cfg))
    assert (rc == moe.MOE_OK) == ok


def test_workspace_and_bound(moe):
    cfg = moe.make_config(4096, 7168, 8, 256, 32)
    ws = moe.moe_workspace_bytes(cfg)
    assert ws % 256 == 0
    assert ws >= 4 * (2 * 4096 * 8 + 256 * 32 + 2 * 257 + 33)
    assert moe.moe_recv_bound_rows(cfg) == 32 * 128 * 8
    assert moe.moe_recv_bound_rows(moe.make_config(8192, 7168, 8, 128, 16)) == 65536
    assert moe.moe_recv_bound_rows(moe.make_config(64, 8, 2, 16, 2)) == 2 * 32 * 8   # E/N > K
    with pytest.raises(moe.MoEError) as ei:
        moe.moe_workspace_bytes(moe.make_config(63, 256, 2, 8, 2))
    assert ei.value.code == moe.MOE_EINVAL


def test_errors_detected_before_any_cuda_call(moe):
    lib = moe.load_library()
    import ctypes
    cfg = moe.make_config(64, 256, 2, 8, 2)
    h = ctypes.c_void_p(0)
    # null / short / misaligned workspace is rejected before touching the device
    assert lib.moe_ctx_create(ctypes.byref(cfg), None, 1 << 20, ctypes.byref(h)) == moe.MOE_EINVAL
    assert lib.moe_ctx_create(ctypes.byref(cfg), 256, 16, ctypes.byref(h)) == moe.MOE_EINVAL
    assert lib.moe_ctx_create(ctypes.byref(cfg), 257, 1 << 20, ctypes.byref(h)) == moe.MOE_EINVAL
    assert lib.moe_ctx_create(ctypes.byref(cfg), 256, 1 << 20, None) == moe.MOE_EINVAL
    # null context everywhere
    assert lib.moe_dispatch_send(None, None, None, None, 0, None) == moe.MOE_EINVAL
    assert lib.moe_dispatch_recv(None, None, None) == moe.MOE_EINVAL
    assert lib.moe_combine_send(None, None, 0, None) == moe.MOE_EINVAL
    assert lib.moe_combine_recv(None, None, None, None) == moe.MOE_EINVAL
    assert lib.moe_get_error(None, None) == moe.MOE_EINVAL
    assert lib.moe_ctx_set_option(None, 1, 0) == moe.MOE_EINVAL
    assert lib.moe_ctx_destroy(None) == moe.MOE_OK


def test_strerror(moe):
    for code in range(8):
        assert moe.moe_strerror(code) != "unknown status"
    assert moe.moe_strerror(99) == "unknown status"


def test_status_codes_and_options_match_the_header(moe):
    """Every MOE_E* status and MOE_OPT_* option the header defines has the
    same value in the binding."""
    import re
    text = open(os.path.join(ROOT, "include", "moe.h")).read()
    defs = dict(re.findall(r"#define (MOE_(?:OK|E[A-Z]+|OPT_[A-Z0-9_]+)) (-?\d+)", text))
    assert "MOE_ECORRUPT" in defs and "MOE_OPT_KERNEL_EVENTS" in defs
    for name, value in defs.items():
        assert getattr(moe, name) == int(value), name


def test_product_path_never_touches_the_oracle():
    """The package and the C sources do not import, link or name the oracle."""
    pkg = os.path.join(ROOT, "combine_route_count_gb300")
    for dirpath, _, files in os.walk(pkg):
        for fn in files:
            if fn.endswith((".py", ".cu", ".cuh", ".h", ".cc")):
                text = open(os.path.join(dirpath, fn)).read()
                assert "import oracle" not in text and "from oracle" not in text, fn
                assert "liboracle" not in text and "moe_oracle" not in text, fn
