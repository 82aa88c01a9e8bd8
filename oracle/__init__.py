"""CPU oracle for the MXFP4 mixture-of-experts layer (ctypes wrapper).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg are the only callers. The product library never
imports or loads it, and it shares no code with the CUDA path.

The arithmetic lives in ``moe_oracle.c`` (plain C, float64, fixed loop
orders). This module compiles it with gcc on first use and marshals numpy
arrays. Every function is pinned by ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB = os.path.join(_HERE, "libmoe_oracle.so")
_lock = threading.Lock()
_lib = None

CFLAGS = ["-O2", "-fno-fast-math", "-ffp-contract=off", "-fopenmp", "-shared", "-fPIC", "-std=c11"]


def build(force: bool = False) -> str:
    """Compile the oracle shared library (gcc, no CUDA)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", *CFLAGS, _SRC, "-o", tmp, "-lm"], check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            i32, i64, f64 = ctypes.c_int, ctypes.c_int64, ctypes.c_double
            lib.oracle_e2m1_value.argtypes = [ctypes.c_uint]
            lib.oracle_e2m1_value.restype = f64
            lib.oracle_e8m0_value.argtypes = [ctypes.c_uint]
            lib.oracle_e8m0_value.restype = f64
            lib.oracle_route.argtypes = [P, i32, i32, i32, P, P, P]
            lib.oracle_rows_capacity.argtypes = [i32, i32, i32, i32]
            lib.oracle_rows_capacity.restype = i64
            lib.oracle_permute.argtypes = [P, i32, i32, i32, i32, P, P, P, P, i64, P]
            lib.oracle_forward.argtypes = [P, P, P, P, P, P, P, i32, i32, i32, i32, i32, f64, P, i32, P]
            lib.oracle_forward_grouped.argtypes = [P, P, P, P, P, P, P, P, i32, i32, i32, i32, i32, f64, P]
            lib.oracle_max_threads.restype = i32
            _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


class OracleError(RuntimeError):
    pass


def _check(rc: int, what: str):
    if rc != 0:
        raise OracleError(f"{what}: invalid arguments (code {rc})")


def e2m1_value(code: int) -> float:
    return _load().oracle_e2m1_value(code)


def e8m0_value(s: int) -> float:
    return _load().oracle_e8m0_value(s)


def max_threads() -> int:
    return _load().oracle_max_threads()


def route(logits: np.ndarray, k: int, bitmatrix: bool = True):
    """Top-k routing. Returns (ids int32 [T,k], w float64 [T,k], bitmatrix uint32 [T, ceil(E/32)])."""
    logits = np.ascontiguousarray(logits, dtype=np.float32)
    T, E = logits.shape
    ids = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float64)
    bm = np.empty((T, (E + 31) // 32), np.uint32) if bitmatrix else None
    _check(_load().oracle_route(_ptr(logits), T, E, k, _ptr(ids), _ptr(w),
                                _ptr(bm) if bm is not None else None), "route")
    return ids, w, bm


def rows_capacity(T: int, E: int, k: int, block_m: int) -> int:
    return int(_load().oracle_rows_capacity(T, E, k, block_m))


def permute(ids: np.ndarray, E: int, block_m: int):
    """Histogram, offsets, padded offsets and the stable permutation (see moe_oracle.c)."""
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    T, k = ids.shape
    cap = rows_capacity(T, E, k, block_m)
    counts = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    padded = np.empty(E + 1, np.int32)
    r2p = np.empty(max(cap, 1), np.int32)
    p2r = np.empty(max(T * k, 1), np.int32)
    _check(_load().oracle_permute(_ptr(ids), T, E, k, block_m, _ptr(counts), _ptr(offsets),
                                  _ptr(padded), _ptr(r2p), cap, _ptr(p2r)), "permute")
    return dict(counts=counts, offsets=offsets, padded_offsets=padded,
                row_to_pair=r2p[:cap], pair_to_row=p2r[:T * k])


def forward(layer: dict, ids: np.ndarray, w: np.ndarray, tokens=None, swiglu_limit: float = 0.0):
    """Layer output (float64 [len(tokens), H]) for the listed tokens (default: all)."""
    T, H, I, E, k = layer["T"], layer["H"], layer["I"], layer["E"], layer["k"]
    tok = np.arange(T, dtype=np.int32) if tokens is None else np.ascontiguousarray(tokens, dtype=np.int32)
    y = np.empty((max(len(tok), 1), H), np.float64)
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    w = np.ascontiguousarray(w, dtype=np.float64)
    x = np.ascontiguousarray(layer["x_bits"], dtype=np.uint16)
    _check(_load().oracle_forward(
        _ptr(x), _ptr(layer["w13_q"]), _ptr(layer["w13_s"]), _ptr(layer["w2_q"]), _ptr(layer["w2_s"]),
        _ptr(ids), _ptr(w), T, H, I, E, k, float(swiglu_limit), _ptr(tok), len(tok), _ptr(y)), "forward")
    return y[:len(tok)]


def forward_grouped(layer: dict, w: np.ndarray, perm: dict, swiglu_limit: float = 0.0):
    """Grouped (permuted, padded) form of the same layer; float64 [T, H]."""
    T, H, I, E, k = layer["T"], layer["H"], layer["I"], layer["E"], layer["k"]
    y = np.empty((max(T, 1), H), np.float64)
    x = np.ascontiguousarray(layer["x_bits"], dtype=np.uint16)
    w = np.ascontiguousarray(w, dtype=np.float64)
    _check(_load().oracle_forward_grouped(
        _ptr(x), _ptr(layer["w13_q"]), _ptr(layer["w13_s"]), _ptr(layer["w2_q"]), _ptr(layer["w2_s"]),
        _ptr(w), _ptr(perm["padded_offsets"]), _ptr(perm["row_to_pair"]),
        T, H, I, E, k, float(swiglu_limit), _ptr(y)), "forward_grouped")
    return y[:T]
