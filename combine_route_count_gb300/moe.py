"""Thin ctypes binding of libmoe.so (include/moe.h).

Argument marshalling only: every step of dispatch and combine runs in the
CUDA kernels behind the C ABI.  There is no CPU fallback: if the library is
missing, every call raises.  Functions carry the C names; pointers may be
given as integers or as torch tensors (their ``data_ptr()``), streams as
integers, ``torch.cuda.Stream`` objects or ``None`` (torch's current stream).

``MoELayer`` bundles one context with its torch-allocated workspace for the
tests and the benchmark.
"""
from __future__ import annotations

import ctypes
import os
from collections.abc import Mapping
from typing import Any, Dict, Optional

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libmoe.so")

MOE_OK, MOE_EINVAL, MOE_ESTATE, MOE_EROUTE, MOE_ECUDA, MOE_EBOUND, MOE_ETIMEDOUT, MOE_ECORRUPT = range(8)
MOE_MAX_TOP_K = 16
MOE_MAX_EXPERTS = 1024
(MOE_OPT_PACK_VARIANT, MOE_OPT_PACK_STAGES, MOE_OPT_PACK_PIECE_BYTES, MOE_OPT_PACK_CTAS_PER_SM, MOE_OPT_PDL,
 MOE_OPT_ROUTE_VARIANT, MOE_OPT_ROUTE_CLUSTER_CTAS) = 1, 2, 3, 4, 5, 6, 7
ROUTE_AUTO, ROUTE_SINGLE, ROUTE_SPLIT, ROUTE_CLUSTER, ROUTE_FUSED = 0, 1, 2, 3, 4
MOE_OPT_COMBINE_VARIANT, MOE_OPT_COMBINE_STAGES, MOE_OPT_COMBINE_PIECE_BYTES, MOE_OPT_COMBINE_CTAS_PER_SM = 8, 9, 10, 11
COMBINE_BULK, COMBINE_VECTOR = 0, 1
MOE_OPT_PACK_PREFETCH = 12
MOE_OPT_CACHE_HINTS = 13
MOE_OPT_PACK_STORE_DEPTH = 14
MOE_OPT_MAX_SMS = 15
MOE_OPT_TEST_DROP_COMBINE_UNIT = 16
MOE_OPT_COMBINE_ORDER = 17
MOE_OPT_FP8_ORDER = 18
MOE_OPT_KERNEL_EVENTS = 19
MOE_OPT_PACK_SCHEDULE = 20
MOE_OPT_COMBINE_SCHEDULE = 21
MOE_OPT_ROUTE_VARIANT_FP8 = 22  # read only: the routing moe_dispatch_send_fp8 takes
PACK_BULK, PACK_VECTOR = 0, 1

# Every entry point of include/moe.h.
EXPORTS = ("moe_validate_config", "moe_workspace_bytes", "moe_recv_bound_rows", "moe_ctx_create",
           "moe_ctx_destroy", "moe_ctx_set_option", "moe_ctx_get_option", "moe_dispatch_send", "moe_dispatch_recv",
           "moe_combine_send", "moe_combine_recv", "moe_get_error", "moe_strerror",
           "moe_dispatch_send_noalloc", "moe_dispatch_send_fp8", "moe_combine_recv_two_level", "moe_partial_rows",
           "moe_dispatch_send_staged", "moe_kernel_times", "moe_dispatch_send_quantized",
           "moe_dense_capacity", "moe_dispatch_send_dense", "moe_combine_recv_dense")


class moe_config(ctypes.Structure):
    _fields_ = [("num_tokens", ctypes.c_int32), ("hidden", ctypes.c_int32), ("top_k", ctypes.c_int32),
                ("num_experts", ctypes.c_int32), ("num_ranks", ctypes.c_int32)]


class moe_dispatch_layout(ctypes.Structure):
    _fields_ = [("expert_counts", ctypes.c_void_p), ("expert_offsets", ctypes.c_void_p),
                ("src_offsets", ctypes.c_void_p), ("rank_offsets", ctypes.c_void_p),
                ("slot_row", ctypes.c_void_p), ("row_src", ctypes.c_void_p),
                ("error_word", ctypes.c_void_p), ("rows", ctypes.c_int64),
                ("recv_bound_rows", ctypes.c_int64)]


class MoEError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {moe_strerror(code)} (status {code})")
        self.code = code


_lib: Optional[ctypes.CDLL] = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Loads libmoe.so; raises if it has not been built (no fallback)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"libmoe.so is not built ({path}); run __graft_entry__.build() "
                           "or python combine_route_count_gb300/build.py")
    lib = ctypes.CDLL(path)
    P, I, I64, C = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.POINTER(moe_config)
    sig = {
        "moe_validate_config": ([C], I),
        "moe_workspace_bytes": ([C, ctypes.POINTER(ctypes.c_size_t)], I),
        "moe_recv_bound_rows": ([C, ctypes.POINTER(ctypes.c_int64)], I),
        "moe_ctx_create": ([C, P, ctypes.c_size_t, ctypes.POINTER(P)], I),
        "moe_ctx_destroy": ([P], I),
        "moe_ctx_set_option": ([P, I, I64], I),
        "moe_ctx_get_option": ([P, I, ctypes.POINTER(ctypes.c_int64)], I),
        "moe_dispatch_send": ([P, P, P, P, I64, P], I),
        "moe_dispatch_send_fp8": ([P, P, P, P, P, I64, P], I),
        "moe_dispatch_send_quantized": ([P, P, P, P, P, P, I64, P], I),
        "moe_dispatch_send_staged": ([P, P, P, P, I64, P, I64, P], I),
        "moe_dense_capacity": ([C, ctypes.POINTER(ctypes.c_int64)], I),
        "moe_dispatch_send_dense": ([P, P, P, I64, P, P, I64, P, I64, P], I),
        "moe_combine_recv_dense": ([P, P, I64, P, P, I64, P, P], I),
        "moe_dispatch_recv": ([P, ctypes.POINTER(moe_dispatch_layout), P], I),
        "moe_combine_send": ([P, P, I64, P], I),
        "moe_combine_recv": ([P, P, P, P], I),
        "moe_combine_recv_two_level": ([P, P, P, I64, P, P], I),
        "moe_partial_rows": ([C, ctypes.POINTER(ctypes.c_int64)], I),
        "moe_kernel_times": ([P, ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_float)], I),
        "moe_get_error": ([P, P], I),
        "moe_strerror": ([I], ctypes.c_char_p),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    _lib = lib
    return lib


def _ptr(x: Any) -> Optional[int]:
    if x is None:
        return None
    if hasattr(x, "data_ptr"):
        return int(x.data_ptr())
    return int(x)


def _stream(s: Any) -> Optional[int]:
    if s is None:
        import torch
        return int(torch.cuda.current_stream().cuda_stream) or None
    if hasattr(s, "cuda_stream"):
        return int(s.cuda_stream) or None
    return int(s) or None


def _check(rc: int, what: str) -> None:
    if rc != MOE_OK:
        raise MoEError(rc, what)


def make_config(T: int, H: int, K: int, E: int, N: int) -> moe_config:
    return moe_config(T, H, K, E, N)


# ---- the C entry points, same names ----------------------------------------

def moe_validate_config(cfg: moe_config) -> int:
    return load_library().moe_validate_config(ctypes.byref(cfg))


def moe_workspace_bytes(cfg: moe_config) -> int:
    n = ctypes.c_size_t(0)
    _check(load_library().moe_workspace_bytes(ctypes.byref(cfg), ctypes.byref(n)), "moe_workspace_bytes")
    return int(n.value)


def moe_recv_bound_rows(cfg: moe_config) -> int:
    n = ctypes.c_int64(0)
    _check(load_library().moe_recv_bound_rows(ctypes.byref(cfg), ctypes.byref(n)), "moe_recv_bound_rows")
    return int(n.value)


def moe_ctx_create(cfg: moe_config, workspace: Any, workspace_bytes: int) -> int:
    h = ctypes.c_void_p(0)
    _check(load_library().moe_ctx_create(ctypes.byref(cfg), _ptr(workspace), workspace_bytes, ctypes.byref(h)),
           "moe_ctx_create")
    return int(h.value)


def moe_ctx_destroy(ctx: int) -> None:
    _check(load_library().moe_ctx_destroy(ctx), "moe_ctx_destroy")


def moe_ctx_set_option(ctx: int, option: int, value: int) -> None:
    _check(load_library().moe_ctx_set_option(ctx, option, value), "moe_ctx_set_option")


def moe_ctx_get_option(ctx: int, option: int) -> int:
    v = ctypes.c_int64(0)
    _check(load_library().moe_ctx_get_option(ctx, option, ctypes.byref(v)), "moe_ctx_get_option")
    return int(v.value)


def moe_dispatch_send(ctx: int, x: Any, topk_idx: Any, expert_x: Any, expert_x_rows: int, stream: Any = None) -> None:
    _check(load_library().moe_dispatch_send(ctx, _ptr(x), _ptr(topk_idx), _ptr(expert_x), expert_x_rows,
                                            _stream(stream)), "moe_dispatch_send")


MOE_FP8_BLOCK = 128


def moe_dispatch_send_fp8(ctx: int, x: Any, topk_idx: Any, expert_xq: Any, expert_scales: Any, expert_rows: int,
                          stream: Any = None) -> None:
    _check(load_library().moe_dispatch_send_fp8(ctx, _ptr(x), _ptr(topk_idx), _ptr(expert_xq), _ptr(expert_scales),
                                                expert_rows, _stream(stream)), "moe_dispatch_send_fp8")


def moe_dispatch_send_staged(ctx: int, x: Any, topk_idx: Any, send_buf: Any, send_rows: int, expert_x: Any,
                             expert_x_rows: int, stream: Any = None) -> None:
    _check(load_library().moe_dispatch_send_staged(ctx, _ptr(x), _ptr(topk_idx), _ptr(send_buf), send_rows,
                                                   _ptr(expert_x), expert_x_rows, _stream(stream)),
           "moe_dispatch_send_staged")


def moe_dispatch_send_quantized(ctx: int, xq: Any, x_scales: Any, topk_idx: Any, expert_xq: Any, expert_scales: Any,
                                expert_rows: int, stream: Any = None) -> None:
    _check(load_library().moe_dispatch_send_quantized(ctx, _ptr(xq), _ptr(x_scales), _ptr(topk_idx), _ptr(expert_xq),
                                                      _ptr(expert_scales), expert_rows, _stream(stream)),
           "moe_dispatch_send_quantized")


def moe_dense_capacity(cfg: moe_config) -> int:
    v = ctypes.c_int64(0)
    _check(load_library().moe_dense_capacity(ctypes.byref(cfg), ctypes.byref(v)), "moe_dense_capacity")
    return int(v.value)


def moe_dispatch_send_dense(ctx: int, x: Any, topk_idx: Any, capacity: int, send_buf: Any, recv_buf: Any,
                            buf_rows: int, expert_x: Any, expert_x_rows: int, stream: Any = None) -> None:
    _check(load_library().moe_dispatch_send_dense(ctx, _ptr(x), _ptr(topk_idx), capacity, _ptr(send_buf),
                                                  _ptr(recv_buf), buf_rows, _ptr(expert_x), expert_x_rows,
                                                  _stream(stream)), "moe_dispatch_send_dense")


def moe_combine_recv_dense(ctx: int, topk_w: Any, capacity: int, send_buf: Any, recv_buf: Any, buf_rows: int,
                           out: Any, stream: Any = None) -> None:
    _check(load_library().moe_combine_recv_dense(ctx, _ptr(topk_w), capacity, _ptr(send_buf), _ptr(recv_buf),
                                                 buf_rows, _ptr(out), _stream(stream)), "moe_combine_recv_dense")


def moe_dispatch_recv(ctx: int, stream: Any = None) -> moe_dispatch_layout:
    lay = moe_dispatch_layout()
    _check(load_library().moe_dispatch_recv(ctx, ctypes.byref(lay), _stream(stream)), "moe_dispatch_recv")
    return lay


def moe_combine_send(ctx: int, expert_y: Any, expert_y_rows: int, stream: Any = None) -> None:
    _check(load_library().moe_combine_send(ctx, _ptr(expert_y), expert_y_rows, _stream(stream)), "moe_combine_send")


def moe_combine_recv(ctx: int, topk_w: Any, out: Any, stream: Any = None) -> None:
    _check(load_library().moe_combine_recv(ctx, _ptr(topk_w), _ptr(out), _stream(stream)), "moe_combine_recv")


def moe_combine_recv_two_level(ctx: int, topk_w: Any, partial: Any, partial_rows: int, out: Any,
                               stream: Any = None) -> None:
    _check(load_library().moe_combine_recv_two_level(ctx, _ptr(topk_w), _ptr(partial), partial_rows, _ptr(out),
                                                     _stream(stream)), "moe_combine_recv_two_level")


def moe_partial_rows(cfg: moe_config) -> int:
    v = ctypes.c_int64(0)
    _check(load_library().moe_partial_rows(ctypes.byref(cfg), ctypes.byref(v)), "moe_partial_rows")
    return int(v.value)


def moe_kernel_times(ctx: int):
    """(pack_ms, combine_ms) of the last kernels timed with MOE_OPT_KERNEL_EVENTS (-1: not timed)."""
    a, b = ctypes.c_float(0), ctypes.c_float(0)
    _check(load_library().moe_kernel_times(ctx, ctypes.byref(a), ctypes.byref(b)), "moe_kernel_times")
    return float(a.value), float(b.value)


def moe_get_error(ctx: int, stream: Any = None) -> int:
    return int(load_library().moe_get_error(ctx, _stream(stream)))


def moe_strerror(code: int) -> str:
    try:
        return load_library().moe_strerror(code).decode()
    except RuntimeError:
        return f"status {code}"


MOE_NOALLOC_MAX_PAIRS = 262144
MOE_NOALLOC_MAX_EXPERT_RANKS = 65536
MOE_NOALLOC_SCRATCH_BYTES = 2363648


def moe_dispatch_send_noalloc(cfg: moe_config, x: Any, topk_idx: Any, expert_x: Any, expert_x_rows: int,
                              expert_counts: Any, expert_offsets: Any, status: Any, stream: Any = None) -> int:
    """Dispatch for callers that cannot allocate device memory: the routing
    tables live in the library's static device array instead of a workspace.
    Returns the C status code (MOE_EINVAL for sizes beyond the array)."""
    fn = load_library().moe_dispatch_send_noalloc
    if fn.argtypes is None:
        P = ctypes.c_void_p
        fn.argtypes = [ctypes.POINTER(moe_config), P, P, P, ctypes.c_int64, P, P, P, P]
        fn.restype = ctypes.c_int
    return int(fn(ctypes.byref(cfg), _ptr(x), _ptr(topk_idx), _ptr(expert_x), expert_x_rows, _ptr(expert_counts),
                  _ptr(expert_offsets), _ptr(status), _stream(stream)))


# ---- convenience: one context with a torch-allocated workspace ---------------

class DispatchLayout(Mapping):
    """Read-only mapping over a moe_dispatch_layout: expert_counts [E],
    expert_offsets [E+1], src_offsets [E, N], rank_offsets [N+1],
    slot_row [T, K], row_src [T*K], error_word [1] (torch int32 views into the
    workspace), rows and recv_bound_rows (ints)."""

    _KEYS = ("expert_counts", "expert_offsets", "src_offsets", "rank_offsets", "slot_row", "row_src",
             "error_word", "rows", "recv_bound_rows")

    def __init__(self, layer: "MoELayer", lay: moe_dispatch_layout):
        self._layer, self._lay, self._cache = layer, lay, {}

    def __getitem__(self, key: str) -> Any:
        if key not in self._cache:
            self._cache[key] = self._make(key)
        return self._cache[key]

    def __iter__(self):
        return iter(self._KEYS)

    def __len__(self) -> int:
        return len(self._KEYS)

    def _make(self, key: str) -> Any:
        import torch
        lay, L = self._lay, self._layer
        if key in ("rows", "recv_bound_rows"):
            return int(getattr(lay, key))
        if key not in self._KEYS:
            raise KeyError(key)
        T, K, E, N = L.T, L.K, L.E, L.N
        n, shape = {"expert_counts": (E, None), "expert_offsets": (E + 1, None), "src_offsets": (E * N, (E, N)),
                    "rank_offsets": (N + 1, None), "slot_row": (T * K, (T, K)), "row_src": (T * K, None),
                    "error_word": (1, None)}[key]
        off = (int(getattr(lay, key)) - L.workspace.data_ptr()) // 4
        v = L.workspace.view(torch.int32)[off:off + n]
        return v.view(*shape) if shape else v


class MoELayer:
    """One dispatch+combine context on the current CUDA device.

    Allocates the workspace with torch (the library itself allocates no
    device memory), or uses the caller's `workspace` (a uint8 CUDA tensor of
    at least moe_workspace_bytes, 256-byte aligned, e.g. from a pool), and
    exposes the four calls on torch tensors:
    x bf16 [T, H], topk_idx int32 [T, K], expert_x bf16 [>= T*K, H],
    expert_y bf16 [>= T*K, H], topk_w float32 [T, K], out bf16 [T, H].
    """

    def __init__(self, T: int, H: int, K: int, E: int, N: int, device: Any = None, workspace: Any = None,
                 **options: int):
        import torch
        self.cfg = make_config(T, H, K, E, N)
        self.T, self.H, self.K, self.E, self.N = T, H, K, E, N
        nbytes = moe_workspace_bytes(self.cfg)
        if workspace is not None:
            if workspace.dtype != torch.uint8 or not workspace.is_cuda or not workspace.is_contiguous():
                raise MoEError(MOE_EINVAL, "workspace must be a contiguous uint8 CUDA tensor")
            self.device = workspace.device
        else:
            self.device = torch.device("cuda") if device is None else torch.device(device)
        with torch.cuda.device(self.device):
            if workspace is None:
                workspace = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=self.device)
            self.workspace = workspace
            self.ctx = moe_ctx_create(self.cfg, self.workspace, self.workspace.numel())
        names = {"pack_variant": MOE_OPT_PACK_VARIANT, "pack_stages": MOE_OPT_PACK_STAGES,
                 "pack_piece_bytes": MOE_OPT_PACK_PIECE_BYTES, "pack_ctas_per_sm": MOE_OPT_PACK_CTAS_PER_SM,
                 "pdl": MOE_OPT_PDL, "route_variant": MOE_OPT_ROUTE_VARIANT,
                 "combine_variant": MOE_OPT_COMBINE_VARIANT, "combine_stages": MOE_OPT_COMBINE_STAGES,
                 "combine_piece_bytes": MOE_OPT_COMBINE_PIECE_BYTES,
                 "combine_ctas_per_sm": MOE_OPT_COMBINE_CTAS_PER_SM, "pack_prefetch": MOE_OPT_PACK_PREFETCH,
                 "cache_hints": MOE_OPT_CACHE_HINTS, "pack_store_depth": MOE_OPT_PACK_STORE_DEPTH,
                 "max_sms": MOE_OPT_MAX_SMS, "combine_order": MOE_OPT_COMBINE_ORDER,
                 "fp8_order": MOE_OPT_FP8_ORDER, "kernel_events": MOE_OPT_KERNEL_EVENTS,
                 "pack_schedule": MOE_OPT_PACK_SCHEDULE, "combine_schedule": MOE_OPT_COMBINE_SCHEDULE}
        for k, v in options.items():
            moe_ctx_set_option(self.ctx, names[k], int(v))

    def close(self) -> None:
        if getattr(self, "ctx", 0):
            moe_ctx_destroy(self.ctx)
            self.ctx = 0

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def set_option(self, option: int, value: int) -> None:
        moe_ctx_set_option(self.ctx, option, value)

    def get_option(self, option: int) -> int:
        return moe_ctx_get_option(self.ctx, option)

    def kernels_per_layer(self) -> int:
        """Kernel launches of one dispatch+combine layer (T > 0)."""
        route = self.get_option(MOE_OPT_ROUTE_VARIANT)
        if route == ROUTE_FUSED:
            return 2  # route_pack, combine
        return (2 if route == ROUTE_SPLIT else 1) + 2

    def dispatch_send(self, x, topk_idx, expert_x, stream: Any = None) -> None:
        moe_dispatch_send(self.ctx, x, topk_idx, expert_x, expert_x.shape[0], stream)

    def dispatch_send_fp8(self, x, topk_idx, expert_xq, expert_scales, stream: Any = None) -> None:
        """fp8 payload: expert_xq uint8 [>= T*K, H], expert_scales float32 [>= T*K, H/128]."""
        moe_dispatch_send_fp8(self.ctx, x, topk_idx, expert_xq, expert_scales, expert_xq.shape[0], stream)

    def dispatch_send_staged(self, x, topk_idx, send_buf, expert_x, stream: Any = None) -> None:
        """Two-stage dispatch: send_buf bf16 [>= T*K, H] is caller scratch."""
        moe_dispatch_send_staged(self.ctx, x, topk_idx, send_buf, send_buf.shape[0], expert_x, expert_x.shape[0],
                                 stream)

    def dense_capacity(self) -> int:
        """Smallest block size of the dense padded all-to-all: T/N * min(K, E/N)."""
        return moe_dense_capacity(self.cfg)

    def dispatch_send_dense(self, x, topk_idx, capacity, send_buf, recv_buf, expert_x, stream: Any = None) -> None:
        """Dispatch through the dense padded all-to-all: send_buf and recv_buf
        bf16 [>= N*N*capacity, H] are caller scratch."""
        moe_dispatch_send_dense(self.ctx, x, topk_idx, capacity, send_buf, recv_buf,
                                min(send_buf.shape[0], recv_buf.shape[0]), expert_x, expert_x.shape[0], stream)

    def combine_recv_dense(self, topk_w, capacity, send_buf, recv_buf, out, stream: Any = None) -> None:
        """Combine through the dense padded all-to-all back (after dispatch_send_dense)."""
        moe_combine_recv_dense(self.ctx, topk_w, capacity, send_buf, recv_buf,
                               min(send_buf.shape[0], recv_buf.shape[0]), out, stream)

    def dispatch_send_quantized(self, xq, x_scales, topk_idx, expert_xq, expert_scales, stream: Any = None) -> None:
        """Pre-quantised payload: xq uint8 [T, H], x_scales float32 [T, H/128]."""
        moe_dispatch_send_quantized(self.ctx, xq, x_scales, topk_idx, expert_xq, expert_scales, expert_xq.shape[0],
                                    stream)

    def dispatch_recv(self, stream: Any = None) -> "DispatchLayout":
        """The dispatch layout; its arrays are torch views into the workspace,
        made on first access (the call itself only crosses the C ABI)."""
        return DispatchLayout(self, moe_dispatch_recv(self.ctx, stream))

    def combine_send(self, expert_y, stream: Any = None) -> None:
        moe_combine_send(self.ctx, expert_y, expert_y.shape[0], stream)

    def combine_recv(self, topk_w, out, stream: Any = None) -> None:
        moe_combine_recv(self.ctx, topk_w, out, stream)

    def combine_recv_two_level(self, topk_w, partial, out, stream: Any = None) -> None:
        """Two-level combine: partial bf16 [>= T*min(K,N), H] is caller scratch."""
        moe_combine_recv_two_level(self.ctx, topk_w, partial, partial.shape[0], out, stream)

    def partial_rows(self) -> int:
        return moe_partial_rows(self.cfg)

    def kernel_times(self):
        return moe_kernel_times(self.ctx)

    def get_error(self, stream: Any = None) -> int:
        return moe_get_error(self.ctx, stream)

    def layer(self, x, topk_idx, topk_w, expert_x, expert_y, out, stream: Any = None) -> "DispatchLayout":
        """dispatch_send -> dispatch_recv -> combine_send -> combine_recv."""
        self.dispatch_send(x, topk_idx, expert_x, stream)
        lay = self.dispatch_recv(stream)
        self.combine_send(expert_y, stream)
        self.combine_recv(topk_w, out, stream)
        return lay
