"""CPU oracle for MoE dispatch + combine (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library
and its binding) never imports, links or executes anything in here.

The arithmetic lives in ``moe_oracle.cc`` (plain single-threaded C++,
written from the definition of the method; the file header cites the passages
of "Efficient and portable mixture-of-experts communication" and "Enabling
trillion-parameter models on AWS EFA" it follows).  This module only compiles
it with the host compiler and marshals numpy arrays through ctypes.

Parity pins: every function here is pinned by the CPU tests
(``tests/test_oracle_*.py``) against a library stable sort, brute-force
enumeration, closed-form special cases and an exact rational FMA chain; none is
"parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.cc")
_LIB = os.path.join(_HERE, "liboracle.so")
_SELFTEST_SRC = os.path.join(_HERE, "selftest.cc")
_PAR_SRC = os.path.join(_HERE, "moe_oracle_par.cc")
_PAR_LIB = os.path.join(_HERE, "liboracle_par.so")  # the same loops over every host core (OpenMP)
SELFTEST = os.path.join(_HERE, "oracle_selftest")  # the self-test program, built by build()

OK, EINVAL, EROUTE, EBOUND = 0, 1, 3, 5

_lib: Optional[ctypes.CDLL] = None
_par: Optional[ctypes.CDLL] = None


def build(force: bool = False) -> str:
    """Compile the oracle with g++ (no fast-math, no FMA contraction, no
    -march so that x86 and Arm hosts give identical results)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["g++", "-O2", "-std=c++17", "-ffp-contract=off", "-fno-fast-math",
               "-fPIC", "-shared", "-o", tmp, _SRC]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    newest = max(os.path.getmtime(_SRC), os.path.getmtime(_SELFTEST_SRC))
    if force or not os.path.exists(SELFTEST) or os.path.getmtime(SELFTEST) < newest:
        tmp = SELFTEST + f".tmp{os.getpid()}"
        cmd = ["g++", "-O2", "-std=c++17", "-ffp-contract=off", "-fno-fast-math", "-o", tmp, _SELFTEST_SRC, _SRC]
        subprocess.run(cmd, check=True)
        os.replace(tmp, SELFTEST)
    newest = max(os.path.getmtime(_SRC), os.path.getmtime(_PAR_SRC))
    if force or not os.path.exists(_PAR_LIB) or os.path.getmtime(_PAR_LIB) < newest:
        tmp = _PAR_LIB + f".tmp{os.getpid()}"
        cmd = ["g++", "-O2", "-std=c++17", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
               "-fPIC", "-shared", "-o", tmp, _PAR_SRC]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _PAR_LIB)
    return _LIB


def _load() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        i32, i64, p = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p
        lib.oracle_dispatch.argtypes = [i32, i32, i32, i32, i32, p, p, p, i64, p, p, p, p, p, p]
        lib.oracle_dispatch.restype = ctypes.c_int
        lib.oracle_combine.argtypes = [i32, i32, i32, p, i64, p, p, p]
        lib.oracle_combine.restype = ctypes.c_int
        lib.oracle_combine_f64.argtypes = [i32, i32, i32, p, i64, p, p, p, p, p]
        lib.oracle_combine_f64.restype = ctypes.c_int
        lib.oracle_float_to_bf16.argtypes = [ctypes.c_float]
        lib.oracle_float_to_bf16.restype = ctypes.c_uint16
        lib.oracle_double_to_bf16.argtypes = [ctypes.c_double]
        lib.oracle_double_to_bf16.restype = ctypes.c_uint16
        lib.oracle_fmaf.argtypes = [ctypes.c_float, ctypes.c_float, ctypes.c_float]
        lib.oracle_fmaf.restype = ctypes.c_float
        lib.oracle_dispatch_staged.argtypes = [i32, i32, i32, i32, i32, p, p, p, p, p, p]
        lib.oracle_dispatch_staged.restype = ctypes.c_int
        lib.oracle_combine_two_level.argtypes = [i32, i32, i32, i32, i32, p, i64, p, p, p, p, p]
        lib.oracle_combine_two_level.restype = ctypes.c_int
        lib.oracle_quantize_fp8.argtypes = [i32, i32, p, p, p]
        lib.oracle_quantize_fp8.restype = ctypes.c_int
        lib.oracle_float_to_e4m3.argtypes = [ctypes.c_float]
        lib.oracle_float_to_e4m3.restype = ctypes.c_uint8
        lib.oracle_dispatch_dense.argtypes = [i32, i32, i32, i32, i32, p, p, i64, p, p, p, p]
        lib.oracle_dispatch_dense.restype = ctypes.c_int
        lib.oracle_combine_dense.argtypes = [i32, i32, i32, i32, p, i64, p, p, p, i64, p, p, p]
        lib.oracle_combine_dense.restype = ctypes.c_int
        lib.oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_to_double.restype = ctypes.c_double
        _lib = lib
    return _lib


def _load_par() -> ctypes.CDLL:
    global _par
    if _par is None:
        build()
        lib = ctypes.CDLL(_PAR_LIB)
        i32, i64, p = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p
        lib.oracle_dispatch_par.argtypes = [i32, i32, i32, i32, i32, p, p, p, i64, p, p, p, p, p, p]
        lib.oracle_dispatch_par.restype = ctypes.c_int
        lib.oracle_combine_par.argtypes = [i32, i32, i32, p, i64, p, p, p]
        lib.oracle_combine_par.restype = ctypes.c_int
        lib.oracle_par_threads.argtypes = []
        lib.oracle_par_threads.restype = ctypes.c_int
        _par = lib
    return _par


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


class OracleError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what} failed with oracle status {code}")
        self.code = code


@dataclass
class Dispatch:
    expert_x: np.ndarray        # uint16 [rows, H]
    expert_counts: np.ndarray   # int32 [E]
    expert_offsets: np.ndarray  # int32 [E+1]
    src_offsets: np.ndarray     # int32 [E, N]
    rank_offsets: np.ndarray    # int32 [N+1]
    slot_row: np.ndarray        # int32 [T, K]
    row_src: np.ndarray         # int32 [T*K]


def dispatch(x: np.ndarray, topk_idx: np.ndarray, E: int, N: int,
             expert_x_rows: Optional[int] = None) -> Dispatch:
    """Expert-grouped, stably ordered copy of the token rows plus the routing
    metadata (see ``oracle_dispatch`` in moe_oracle.cc)."""
    lib = _load()
    x = np.ascontiguousarray(x, dtype=np.uint16)
    idx = np.ascontiguousarray(topk_idx, dtype=np.int32)
    T, H = x.shape
    K = idx.shape[1] if idx.ndim == 2 else 0
    if idx.shape[0] != T:
        raise ValueError("x and topk_idx disagree on T")
    rows = T * K
    cap = rows if expert_x_rows is None else int(expert_x_rows)
    ex = np.zeros((max(cap, 0), H), dtype=np.uint16)
    out = Dispatch(ex, np.zeros(E, np.int32), np.zeros(E + 1, np.int32),
                   np.zeros((E, N), np.int32), np.zeros(N + 1, np.int32),
                   np.zeros((T, K), np.int32), np.zeros(rows, np.int32))
    rc = lib.oracle_dispatch(T, H, K, E, N, _ptr(x), _ptr(idx), _ptr(ex), cap,
                             _ptr(out.expert_counts), _ptr(out.expert_offsets),
                             _ptr(out.src_offsets), _ptr(out.rank_offsets),
                             _ptr(out.slot_row), _ptr(out.row_src))
    if rc != OK:
        raise OracleError(rc, "oracle_dispatch")
    return out


def par_threads() -> int:
    """Threads the all-cores functions (``dispatch_par``, ``combine_par``) use."""
    return int(_load_par().oracle_par_threads())


def dispatch_par(x: np.ndarray, topk_idx: np.ndarray, E: int, N: int) -> Dispatch:
    """``dispatch`` with its row copy spread over every host core
    (``oracle_dispatch_par`` in moe_oracle_par.cc); the same bytes."""
    lib = _load_par()
    x = np.ascontiguousarray(x, dtype=np.uint16)
    idx = np.ascontiguousarray(topk_idx, dtype=np.int32)
    T, H = x.shape
    K = idx.shape[1]
    rows = T * K
    out = Dispatch(np.empty((rows, H), dtype=np.uint16), np.zeros(E, np.int32), np.zeros(E + 1, np.int32),
                   np.zeros((E, N), np.int32), np.zeros(N + 1, np.int32),
                   np.zeros((T, K), np.int32), np.zeros(rows, np.int32))
    rc = lib.oracle_dispatch_par(T, H, K, E, N, _ptr(x), _ptr(idx), _ptr(out.expert_x), rows,
                                 _ptr(out.expert_counts), _ptr(out.expert_offsets),
                                 _ptr(out.src_offsets), _ptr(out.rank_offsets),
                                 _ptr(out.slot_row), _ptr(out.row_src))
    if rc != OK:
        raise OracleError(rc, "oracle_dispatch_par")
    return out


def combine_par(y: np.ndarray, topk_w: np.ndarray, slot_row: np.ndarray) -> np.ndarray:
    """``combine`` with a parallel loop over tokens (``oracle_combine_par``);
    the same bytes."""
    lib = _load_par()
    y = np.ascontiguousarray(y, dtype=np.uint16)
    w = np.ascontiguousarray(topk_w, dtype=np.float32)
    sr = np.ascontiguousarray(slot_row, dtype=np.int32)
    T, K = w.shape
    H = y.shape[1]
    out = np.empty((T, H), dtype=np.uint16)
    rc = lib.oracle_combine_par(T, H, K, _ptr(y), y.shape[0], _ptr(w), _ptr(sr), _ptr(out))
    if rc != OK:
        raise OracleError(rc, "oracle_combine_par")
    return out


def combine(y: np.ndarray, topk_w: np.ndarray, slot_row: np.ndarray) -> np.ndarray:
    """bf16 out[T, H]: float32 FMA chain over k = 0..K-1 from +0.0, one
    round-to-nearest-even to bf16."""
    lib = _load()
    y = np.ascontiguousarray(y, dtype=np.uint16)
    w = np.ascontiguousarray(topk_w, dtype=np.float32)
    sr = np.ascontiguousarray(slot_row, dtype=np.int32)
    T, K = w.shape
    H = y.shape[1]
    out = np.zeros((T, H), dtype=np.uint16)
    rc = lib.oracle_combine(T, H, K, _ptr(y), y.shape[0], _ptr(w), _ptr(sr), _ptr(out))
    if rc != OK:
        raise OracleError(rc, "oracle_combine")
    return out


def combine_f64(y: np.ndarray, topk_w: np.ndarray, slot_row: np.ndarray):
    """(bf16 out, float64 exact-ish sum, float64 sum of |w*y|) of the same
    weighted sum evaluated in double precision."""
    lib = _load()
    y = np.ascontiguousarray(y, dtype=np.uint16)
    w = np.ascontiguousarray(topk_w, dtype=np.float32)
    sr = np.ascontiguousarray(slot_row, dtype=np.int32)
    T, K = w.shape
    H = y.shape[1]
    out = np.zeros((T, H), dtype=np.uint16)
    exact = np.zeros((T, H), dtype=np.float64)
    mag = np.zeros((T, H), dtype=np.float64)
    rc = lib.oracle_combine_f64(T, H, K, _ptr(y), y.shape[0], _ptr(w), _ptr(sr), _ptr(out),
                                _ptr(exact), _ptr(mag))
    if rc != OK:
        raise OracleError(rc, "oracle_combine_f64")
    return out, exact, mag


def dispatch_staged(x: np.ndarray, topk_idx: np.ndarray, E: int, N: int):
    """Two-stage dispatch through per-peer send buffers (see
    ``oracle_dispatch_staged``).  Returns (send_buf uint16 [T*K, H], send_dest
    int32 [T*K], expert_x uint16 [T*K, H], slot_row int32 [T, K])."""
    lib = _load()
    x = np.ascontiguousarray(x, dtype=np.uint16)
    idx = np.ascontiguousarray(topk_idx, dtype=np.int32)
    T, H = x.shape
    K = idx.shape[1]
    send = np.zeros((T * K, H), np.uint16)
    dest = np.zeros(T * K, np.int32)
    ex = np.zeros((T * K, H), np.uint16)
    sr = np.zeros((T, K), np.int32)
    rc = lib.oracle_dispatch_staged(T, H, K, E, N, _ptr(x), _ptr(idx), _ptr(send), _ptr(dest), _ptr(ex), _ptr(sr))
    if rc != OK:
        raise OracleError(rc, "oracle_dispatch_staged")
    return send, dest, ex, sr


def combine_two_level(y: np.ndarray, topk_idx: np.ndarray, topk_w: np.ndarray, slot_row: np.ndarray,
                      E: int, N: int, partial: Optional[np.ndarray] = None):
    """Two-level combine with partial sums on the sending side (see
    ``oracle_combine_two_level``).  Returns (out bf16 [T, H], partial bf16
    [T*min(K,N), H], ranks_per_token int32 [T]); partial rows a token does not
    use keep the values of the ``partial`` argument (zeros if None)."""
    lib = _load()
    y = np.ascontiguousarray(y, dtype=np.uint16)
    idx = np.ascontiguousarray(topk_idx, dtype=np.int32)
    w = np.ascontiguousarray(topk_w, dtype=np.float32)
    sr = np.ascontiguousarray(slot_row, dtype=np.int32)
    T, K = w.shape
    H = y.shape[1]
    slots = min(K, N)
    part = np.zeros((T * slots, H), np.uint16) if partial is None else np.array(partial, dtype=np.uint16)
    if part.shape != (T * slots, H):
        raise ValueError("partial must be [T*min(K,N), H]")
    out = np.zeros((T, H), dtype=np.uint16)
    rc = lib.oracle_combine_two_level(T, H, K, E, N, _ptr(y), y.shape[0], _ptr(idx), _ptr(w), _ptr(sr),
                                      _ptr(part), _ptr(out))
    if rc != OK:
        raise OracleError(rc, "oracle_combine_two_level")
    L = E // N
    ranks = np.array([len(set((idx[t] // L).tolist())) for t in range(T)], np.int32)
    return out, part, ranks


def dispatch_dense(x: np.ndarray, topk_idx: np.ndarray, E: int, N: int, cap: int):
    """Dispatch through a dense padded all-to-all (see ``oracle_dispatch_dense``):
    (send_buf uint16 [N*N*cap, H], recv_buf uint16 [N*N*cap, H], expert_x
    uint16 [T*K, H], send_pos int32 [T, K]).  Both buffers start as zeros,
    so their padding rows are zero."""
    lib = _load()
    x = np.ascontiguousarray(x, dtype=np.uint16)
    idx = np.ascontiguousarray(topk_idx, dtype=np.int32)
    T, H = x.shape
    K = idx.shape[1]
    send = np.zeros((N * N * cap, H), np.uint16)
    recv = np.zeros((N * N * cap, H), np.uint16)
    ex = np.zeros((T * K, H), np.uint16)
    pos = np.zeros((T, K), np.int32)
    rc = lib.oracle_dispatch_dense(T, H, K, E, N, _ptr(x), _ptr(idx), cap, _ptr(send), _ptr(recv), _ptr(ex),
                                   _ptr(pos))
    if rc != OK:
        raise OracleError(rc, "oracle_dispatch_dense")
    return send, recv, ex, pos


def combine_dense(y: np.ndarray, topk_w: np.ndarray, slot_row: np.ndarray, send_pos: np.ndarray, N: int, cap: int):
    """Combine through the dense padded all-to-all back (see
    ``oracle_combine_dense``): (out uint16 [T, H], back_send, back_recv
    uint16 [N*N*cap, H], zero padding)."""
    lib = _load()
    y = np.ascontiguousarray(y, dtype=np.uint16)
    w = np.ascontiguousarray(topk_w, dtype=np.float32)
    sr = np.ascontiguousarray(slot_row, dtype=np.int32)
    sp = np.ascontiguousarray(send_pos, dtype=np.int32)
    T, K = w.shape
    H = y.shape[1]
    bs = np.zeros((N * N * cap, H), np.uint16)
    br = np.zeros((N * N * cap, H), np.uint16)
    out = np.zeros((T, H), np.uint16)
    rc = lib.oracle_combine_dense(T, H, K, N, _ptr(y), y.shape[0], _ptr(w), _ptr(sr), _ptr(sp), cap, _ptr(bs),
                                  _ptr(br), _ptr(out))
    if rc != OK:
        raise OracleError(rc, "oracle_combine_dense")
    return out, bs, br


def float_to_bf16(f: float) -> int:
    return int(_load().oracle_float_to_bf16(f))


def double_to_bf16(v: float) -> int:
    return int(_load().oracle_double_to_bf16(v))


def fmaf(a: float, b: float, c: float) -> float:
    return float(_load().oracle_fmaf(a, b, c))


FP8_BLOCK = 128


def quantize_fp8(x: np.ndarray):
    """Block-scaled fp8 (E4M3) payload of bf16 rows: (q uint8 [T, H],
    scales float32 [T, H/128]); see ``oracle_quantize_fp8``."""
    lib = _load()
    x = np.ascontiguousarray(x, dtype=np.uint16)
    T, H = x.shape
    q = np.zeros((T, H), dtype=np.uint8)
    sc = np.zeros((T, H // FP8_BLOCK), dtype=np.float32)
    rc = lib.oracle_quantize_fp8(T, H, _ptr(x), _ptr(q), _ptr(sc))
    if rc != OK:
        raise OracleError(rc, "oracle_quantize_fp8")
    return q, sc


def dispatch_fp8(x: np.ndarray, topk_idx: np.ndarray, E: int, N: int):
    """fp8 dispatch: the placement of ``dispatch`` applied to the quantised
    rows.  Returns (Dispatch, expert_xq uint8 [T*K, H], expert_scales
    float32 [T*K, H/128])."""
    d = dispatch(x, topk_idx, E, N)
    q, sc = quantize_fp8(x)
    src = d.row_src // max(topk_idx.shape[1], 1)
    return d, q[src], sc[src]


def float_to_e4m3(f: float) -> int:
    return int(_load().oracle_float_to_e4m3(f))


def e4m3_to_double(b: int) -> float:
    return float(_load().oracle_e4m3_to_double(b))
