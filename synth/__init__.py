"""Seeded synthetic inputs for condensate-set (topological) attention.

This module is shared by the CPU oracle's tests, the GPU parity tests and the
benchmark.  It only draws and assembles input tensors: it contains none of the
attention method's arithmetic (no scores, no selection, no softmax).

Recipe (the workloads of "The Condensate Theorem" explainer pages, Technical
Summary section 2: an anchor at position 0 that soaks up attention, a recent
window, and a few far positions with high q.k):

* Q, K, V ~ N(0, 1), element by element, from counter-based SplitMix64 +
  Box-Muller draws (see ``synth.c``), one stream per (sequence, tensor).
* One unit vector u per (sequence, KV head), drawn as N(0,1)^d normalised.
* Q += 3u on every query row (u of the row's KV head).
* Sink: K[0] += 6u for every KV head.
* Planted keys (decode and chunked-prefill workloads): per (sequence, KV head)
  P distinct positions drawn uniformly from [lo, hi); the key row there is
  replaced by 2*sqrt(d)*qbar/|qbar| + 0.3*N(0,1)^d, where qbar is the mean of
  every stored query vector that maps to that KV head in that sequence.
* Everything is evaluated in float64, rounded to float32, and for bfloat16
  workloads rounded again to bfloat16 (round-to-nearest-even).
* Rows [n, kv_stride) of K and V are filled with NaN when ``nan_tail`` is set,
  so that a kernel that reads past the causal length is caught.

bfloat16 tensors are returned as numpy ``uint16`` arrays holding the raw bits.
"""
from __future__ import annotations

import ctypes
import dataclasses
import math
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_SO = os.path.join(_HERE, "libsynth.so")
_lock = threading.Lock()
_lib = None

TAG_U, TAG_Q, TAG_K, TAG_V, TAG_POS, TAG_PLANT = 1, 2, 3, 4, 5, 6
F32, BF16 = 0, 1


def build(force: bool = False) -> str:
    """Compile ``libsynth.so`` next to its source (gcc, no fast-math)."""
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-std=c11", "-pthread",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.syn_key.restype = ctypes.c_uint64
            lib.syn_key.argtypes = [ctypes.c_uint64] * 4
            lib.syn_u64.restype = ctypes.c_uint64
            lib.syn_u64.argtypes = [ctypes.c_uint64, ctypes.c_uint64]
            lib.syn_fill_normal.restype = None
            lib.syn_fill_normal.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_int64,
                                            ctypes.c_int, ctypes.c_double, ctypes.c_double,
                                            ctypes.c_void_p, ctypes.c_int]
            lib.syn_f32_to_bf16.restype = None
            lib.syn_f32_to_bf16.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64]
            _lib = lib
    return _lib


def _threads() -> int:
    return max(1, min(64, os.cpu_count() or 1))


def normal(key: int, first: int, count: int, dtype: str = "f64") -> np.ndarray:
    """``count`` standard-normal draws of stream ``key`` starting at counter ``first``."""
    lib = _load()
    code = {"f32": 0, "bf16": 1, "f64": 2}[dtype]
    out = np.empty(count, dtype={0: np.float32, 1: np.uint16, 2: np.float64}[code])
    lib.syn_fill_normal(key, first, count, code, 0.0, 1.0, out.ctypes.data, _threads())
    return out


def key(seed: int, tag: int, a: int = 0, b: int = 0) -> int:
    return int(_load().syn_key(seed, tag, a, b))


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float values to bfloat16 (RNE); returns uint16 bits."""
    src = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(src.shape, dtype=np.uint16)
    _load().syn_f32_to_bf16(src.ctypes.data, out.ctypes.data, src.size)
    return out


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32)


@dataclasses.dataclass(frozen=True)
class Workload:
    """Shapes and generator settings of one synthetic workload."""
    name: str
    B: int
    Hq: int
    Hkv: int
    d: int
    n: int
    nq: int
    W: int
    k: int
    dtype: str = "bf16"            # "f32" or "bf16"
    seed: int = 20260211
    seq_seed_stride: int = 1000     # sequence b uses seed + b * stride
    planted: int = 0                # planted keys per (sequence, KV head)
    planted_range: str = "decode"   # "decode": [1, n-W); "all": [1, n)
    q_shift: float = 3.0
    sink: float = 6.0
    kv_stride: int = 0              # 0 -> n
    nan_tail: bool = False
    chunk: int = 0                  # prefill chunk size (0: one call)

    @property
    def scale(self) -> float:
        return float(np.float32(1.0 / math.sqrt(self.d)))

    @property
    def stride(self) -> int:
        return self.kv_stride or self.n

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five workloads, seeded 20260211 + id.
CONFIGS = {
    0: Workload("tiny causal prefill fp32 n=2048", 1, 1, 1, 64, 2048, 2048, 64, 32,
                dtype="f32", seed=20260211 + 0),
    1: Workload("decode n=32768 bf16 32/8 heads", 1, 32, 8, 128, 32768, 1, 64, 32,
                seed=20260211 + 1, planted=32),
    2: Workload("batched decode B=16 n=131072 bf16", 16, 32, 8, 128, 131072, 1, 64, 32,
                seed=20260211 + 2, planted=32),
    3: Workload("chunked prefill n=65536 bf16", 1, 32, 8, 128, 65536, 65536, 256, 32,
                seed=20260211 + 3, planted=64, planted_range="all", chunk=4096),
    4: Workload("decode n=1048576 bf16 32/8 heads", 1, 32, 8, 128, 1048576, 1, 64, 32,
                seed=20260211 + 4, planted=32),
}
PREFILL_WINDOWS = (256, 128, 64)   # the three window cases of the chunked-prefill workload


def planted_positions(w: Workload, b: int, h: int) -> np.ndarray:
    """Distinct planted positions for sequence b, KV head h (sorted)."""
    lo = 1
    hi = (w.n - w.W) if w.planted_range == "decode" else w.n
    if w.planted <= 0 or hi <= lo:
        return np.zeros(0, dtype=np.int64)
    span = hi - lo
    if span <= w.planted:
        return np.arange(lo, hi, dtype=np.int64)
    lib = _load()
    kk = key(w.seed + b * w.seq_seed_stride, TAG_POS, h)
    got, seen, t = [], set(), 0
    while len(got) < w.planted:
        x = lo + int(lib.syn_u64(kk, t) % span)
        t += 1
        if x not in seen:
            seen.add(x)
            got.append(x)
    return np.array(sorted(got), dtype=np.int64)


def make(w: Workload) -> dict:
    """Build q, k, v (numpy; bf16 as uint16 bits) and the generator metadata."""
    assert w.Hq % w.Hkv == 0
    g = w.Hq // w.Hkv
    d, n, nq, S = w.d, w.n, w.nq, w.stride
    lib = _load()
    code = F32 if w.dtype == "f32" else BF16
    npdt = np.float32 if code == F32 else np.uint16

    def store(x64: np.ndarray) -> np.ndarray:
        x32 = x64.astype(np.float32)
        return x32 if code == F32 else to_bf16_bits(x32)

    def widen(x: np.ndarray) -> np.ndarray:
        return (x if code == F32 else bf16_bits_to_f32(x)).astype(np.float64)

    q = np.empty((w.B, w.Hq, nq, d), dtype=npdt)
    k = np.empty((w.B, w.Hkv, S, d), dtype=npdt)
    v = np.empty((w.B, w.Hkv, S, d), dtype=npdt)
    u_all = np.empty((w.B, w.Hkv, d))
    planted = {}
    nt = _threads()
    for b in range(w.B):
        sb = w.seed + b * w.seq_seed_stride
        ku = key(sb, TAG_U)
        u = normal(ku, 0, w.Hkv * d).reshape(w.Hkv, d)
        u /= np.linalg.norm(u, axis=1, keepdims=True)
        u_all[b] = u
        kq = key(sb, TAG_Q)
        qn = normal(kq, 0, w.Hq * nq * d).reshape(w.Hq, nq, d)
        qn += w.q_shift * np.repeat(u, g, axis=0)[:, None, :]
        q[b] = store(qn)
        del qn
        qs = widen(q[b])                       # stored query values
        kk, kv = key(sb, TAG_K), key(sb, TAG_V)
        for h in range(w.Hkv):
            lib.syn_fill_normal(kk, h * n * d, n * d, code, 0.0, 1.0,
                                k[b, h].ctypes.data, nt)
            lib.syn_fill_normal(kv, h * n * d, n * d, code, 0.0, 1.0,
                                v[b, h].ctypes.data, nt)
            if S > n:
                fill = np.nan if w.nan_tail else 0.0
                k[b, h, n:] = store(np.full((S - n, d), fill))
                v[b, h, n:] = store(np.full((S - n, d), fill))
            row0 = normal(kk, h * n * d, d) + w.sink * u[h]
            k[b, h, 0] = store(row0)
            pos = planted_positions(w, b, h)
            planted[(b, h)] = pos
            if len(pos):
                qbar = qs[h * g:(h + 1) * g].reshape(-1, d).mean(axis=0)
                dirn = qbar / np.linalg.norm(qbar)
                kp = key(sb, TAG_PLANT, h)
                noise = normal(kp, 0, len(pos) * d).reshape(len(pos), d)
                k[b, h, pos] = store(2.0 * math.sqrt(d) * dirn[None, :] + 0.3 * noise)
    return {"q": q, "k": k, "v": v, "u": u_all, "planted": planted, "workload": w}


def widen(x: np.ndarray, dtype: str) -> np.ndarray:
    """Exact float32 view of stored values (bf16 bits widened)."""
    return x.astype(np.float32) if dtype == "f32" else bf16_bits_to_f32(x)
