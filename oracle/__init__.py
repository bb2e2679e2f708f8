"""CPU oracle for condensate-set attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The CUDA library never calls it and shares no
code with it.

The arithmetic lives in ``topo_oracle.c`` (plain C, float64 except the float32
ranking score); this file only compiles it with gcc and marshals numpy arrays.
See the header of ``topo_oracle.c`` for what each step follows on the pages
("The Condensate Theorem: Transformers are O(n), Not O(n^2)" explainers,
Technical Summary sections 2-3) and for the readings taken where they are
silent.

Parity pins: every function here is pinned by ``tests/test_oracle_pins.py``
(brute force on integer inputs, a library dense-attention routine, closed
forms and invariants); no function is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "topo_oracle.c")
_SO = os.path.join(_HERE, "libtopo_oracle.so")
_lock = threading.Lock()
_lib = None


class Params(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("Hq", ctypes.c_int32), ("Hkv", ctypes.c_int32),
                ("d", ctypes.c_int32), ("n", ctypes.c_int64), ("nq", ctypes.c_int64),
                ("kv_stride", ctypes.c_int64), ("W", ctypes.c_int32), ("k", ctypes.c_int32),
                ("scale", ctypes.c_float), ("dtype", ctypes.c_int32)]


def build(force: bool = False) -> str:
    """Compile the oracle.  -ffp-contract=off keeps every float64 sum as written;
    the float32 ranking score calls fmaf explicitly (one rounding per step)."""
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
                               "-shared", "-std=c11", "-pthread", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.orc_score_f32.restype = ctypes.c_float
            lib.orc_score_f32.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
            lib.orc_topo_attn.restype = ctypes.c_int
            lib.orc_topo_attn.argtypes = [ctypes.POINTER(Params)] + [ctypes.c_void_p] * 4 + [
                ctypes.c_int64] + [ctypes.c_void_p] * 6 + [ctypes.c_int]
            lib.orc_topo_attn_group.restype = ctypes.c_int
            lib.orc_topo_attn_group.argtypes = [ctypes.POINTER(Params)] + [ctypes.c_void_p] * 4 + [
                ctypes.c_int64] + [ctypes.c_void_p] * 2 + [ctypes.c_int]
            _lib = lib
    return _lib


def threads() -> int:
    return max(1, os.cpu_count() or 1)


def score_f32(q: np.ndarray, k: np.ndarray) -> np.float32:
    """The float32 ranking score of one query and one key (left-to-right fmaf chain)."""
    q = np.ascontiguousarray(q, dtype=np.float32)
    k = np.ascontiguousarray(k, dtype=np.float32)
    assert q.shape == k.shape and q.ndim == 1
    return np.float32(_load().orc_score_f32(q.ctypes.data, k.ctypes.data, q.size))


def make_params(B, Hq, Hkv, d, n, nq, W, k, scale, dtype, kv_stride=None) -> Params:
    return Params(B, Hq, Hkv, d, n, nq, kv_stride or n, W, k, np.float32(scale),
                  0 if dtype in ("f32", 0) else 1)


def topo_attn(P: Params, q: np.ndarray, k: np.ndarray, v: np.ndarray, rows=None,
              want=("out", "idx", "dense", "excl", "wmax", "p0"), nthreads=None) -> dict:
    """Run the oracle on rows (flat ids over [B, Hq, nq]; None = every row).

    q: [B, Hq, nq, d]; k, v: [B, Hkv, kv_stride, d]; float32 arrays, or uint16
    arrays of bfloat16 bits when P.dtype == 1.  Returns float64 arrays shaped
    [nrows, ...] (``idx`` int32 [nrows, 1+W+k]).
    """
    lib = _load()
    edt = np.float32 if P.dtype == 0 else np.uint16
    for name, a, shape in (("q", q, (P.B, P.Hq, P.nq, P.d)),
                           ("k", k, (P.B, P.Hkv, P.kv_stride, P.d)),
                           ("v", v, (P.B, P.Hkv, P.kv_stride, P.d))):
        if a.dtype != edt or tuple(a.shape) != shape or not a.flags.c_contiguous:
            raise ValueError(f"{name}: expected contiguous {edt.__name__}{shape}, got "
                             f"{a.dtype}{tuple(a.shape)}")
    if rows is None:
        nrows = P.B * P.Hq * P.nq
        rows_arr = None
    else:
        rows_arr = np.ascontiguousarray(rows, dtype=np.int64)
        nrows = rows_arr.size
        if nrows and (rows_arr.min() < 0 or rows_arr.max() >= P.B * P.Hq * P.nq):
            raise ValueError("row id out of range")
    res = {}
    cmax = 1 + P.W + P.k
    shapes = {"out": ((nrows, P.d), np.float64), "idx": ((nrows, cmax), np.int32),
              "dense": ((nrows, P.d), np.float64), "excl": ((nrows,), np.float64),
              "wmax": ((nrows,), np.float64), "p0": ((nrows,), np.float64)}
    ptrs = []
    for name in ("out", "idx", "dense", "excl", "wmax", "p0"):
        if name in want:
            shp, dt = shapes[name]
            res[name] = np.empty(shp, dtype=dt)
            ptrs.append(res[name].ctypes.data)
        else:
            ptrs.append(None)
    rc = lib.orc_topo_attn(ctypes.byref(P), q.ctypes.data, k.ctypes.data, v.ctypes.data,
                           None if rows_arr is None else rows_arr.ctypes.data, nrows,
                           *ptrs, int(nthreads or threads()))
    if rc != 0:
        raise ValueError("oracle rejected the parameters")
    return res


def topo_attn_group(P: Params, q: np.ndarray, k: np.ndarray, v: np.ndarray, rows=None,
                    want=("out", "idx"), nthreads=None) -> dict:
    """Group-shared selection (one condensate set per sequence, KV head and
    row, shared by the KV head's g query heads; the top-k ranks keys by the
    largest of the heads' float32 scores).  rows: flat ids over [B, Hkv, nq]
    (None = all).  Returns ``out`` float64 [nrows, g, d] and ``idx`` int32
    [nrows, 1+W+k]."""
    lib = _load()
    edt = np.float32 if P.dtype == 0 else np.uint16
    for name, a, shape in (("q", q, (P.B, P.Hq, P.nq, P.d)),
                           ("k", k, (P.B, P.Hkv, P.kv_stride, P.d)),
                           ("v", v, (P.B, P.Hkv, P.kv_stride, P.d))):
        if a.dtype != edt or tuple(a.shape) != shape or not a.flags.c_contiguous:
            raise ValueError(f"{name}: expected contiguous {edt.__name__}{shape}")
    g = P.Hq // P.Hkv
    if rows is None:
        nrows, rows_arr = P.B * P.Hkv * P.nq, None
    else:
        rows_arr = np.ascontiguousarray(rows, dtype=np.int64)
        nrows = rows_arr.size
        if nrows and (rows_arr.min() < 0 or rows_arr.max() >= P.B * P.Hkv * P.nq):
            raise ValueError("row id out of range")
    res = {}
    if "out" in want:
        res["out"] = np.empty((nrows, g, P.d), dtype=np.float64)
    if "idx" in want:
        res["idx"] = np.empty((nrows, 1 + P.W + P.k), dtype=np.int32)
    rc = lib.orc_topo_attn_group(ctypes.byref(P), q.ctypes.data, k.ctypes.data, v.ctypes.data,
                                 None if rows_arr is None else rows_arr.ctypes.data, nrows,
                                 res["out"].ctypes.data if "out" in res else None,
                                 res["idx"].ctypes.data if "idx" in res else None,
                                 int(nthreads or threads()))
    if rc != 0:
        raise ValueError("oracle rejected the parameters")
    return res
