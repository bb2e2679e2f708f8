"""The tensor-core accumulation bound behind exact top-k selection.

Both tensor-core scorers of the library (decode: 128 keys x 16 query columns;
prefill: 128 query columns x 256 keys) compute q . k with one chain of
tcgen05 bf16 MMAs accumulating in float32, keep every key whose score is
within 2 delta of the running k-th best, and rescore those with the exact
float32 chain.  That is only exact if, for every pair,

    |t - q.k| <= beta_d * sum_c |q_c k_c|,   beta_d = d * 2^-21,

t being the tensor-core result (the library's delta adds the float32 chain's
own bound and a factor of two on top).  This test runs the very MMA the
scorers issue -- same shared-memory layout, descriptors and instruction
descriptor, from the package's tcgen05 helpers -- on random and on
cancellation-heavy bfloat16 rows, computes the exact dot products on the host
and checks the bound, for d = 64 and 128 and both MMA shapes.  The largest
observed error, in units of 2^-24 * sum_c |q_c k_c|, is printed and, when
TOPO_TC_BOUND_OUT names a file, written there as JSON.
"""
import ctypes
import json
import os
import subprocess

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
SRC = os.path.join(HERE, "tc_bound_kernel.cu")
CSRC = os.path.join(ROOT, "dynamic_sparse_transformer_qk_b300", "csrc")
BUILD = os.path.join(HERE, "_build")
SO = os.path.join(BUILD, "libtcbound.so")
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")

_results = {}
KINDS = ["normal", "wide_range", "cancel", "one_large"]


def _lib():
    os.makedirs(BUILD, exist_ok=True)
    deps = [SRC, os.path.join(CSRC, "tc_device.cuh"), os.path.join(CSRC, "topo_device.cuh")]
    if not os.path.exists(SO) or any(os.path.getmtime(p) > os.path.getmtime(SO) for p in deps):
        tmp = SO + f".tmp{os.getpid()}"
        subprocess.check_call([NVCC, "-gencode", "arch=compute_103a,code=sm_103a", "-O3",
                               "-std=c++17", "-Xcompiler", "-fPIC", "-shared", "-I" + CSRC,
                               "-o", tmp, SRC])
        os.replace(tmp, SO)
    lib = ctypes.CDLL(SO)
    lib.tcb_run.restype = ctypes.c_int
    lib.tcb_run.argtypes = [ctypes.c_int, ctypes.c_int] + [ctypes.c_void_p] * 5
    return lib


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float64 values to bfloat16 (nearest even); uint16 bits."""
    f = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    f = (f + 0x7FFF + ((f >> 16) & 1)) >> 16
    return f.astype(np.uint16)


def widen(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def operands(kind: str, rows: int, cols: int, d: int, rng):
    """A [rows, d] and B [cols, d] as bfloat16 bits."""
    if kind == "normal":
        a = rng.standard_normal((rows, d))
        b = rng.standard_normal((cols, d))
    elif kind == "wide_range":
        # magnitudes spread over 2^-12 .. 2^12: products far apart in exponent
        a = rng.standard_normal((rows, d)) * np.exp2(rng.integers(-12, 13, (rows, d)))
        b = rng.standard_normal((cols, d)) * np.exp2(rng.integers(-12, 13, (cols, d)))
    elif kind == "cancel":
        # B rows are +-1 patterns whose second half negates the first; A rows
        # repeat x in both halves, so products cancel in pairs except one pair
        # of small entries: the exact sum is tiny next to sum |q_c k_c|
        b = rng.choice([-1.0, 1.0], size=(cols, d))
        a = np.empty((rows, d))
        half = d // 2
        x = rng.standard_normal((rows, half)) * 64.0
        a[:, :half] = x
        a[:, half:] = x
        b[:, half:] = -b[:, :half]
        a[:, half - 1] = rng.standard_normal(rows) * 2.0 ** -6
        a[:, d - 1] = rng.standard_normal(rows) * 2.0 ** -6
    elif kind == "one_large":
        # one product dominates; the others are 2^-10 .. 2^-2 of it
        a = rng.standard_normal((rows, d)) * np.exp2(rng.integers(-10, -1, (rows, d)))
        b = rng.standard_normal((cols, d))
        a[:, rng.integers(0, d)] = 2.0 ** 6
    else:
        raise ValueError(kind)
    return bf16_bits(a), bf16_bits(b)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("n", [16, 256])
@pytest.mark.parametrize("kind", KINDS)
def test_tensor_core_accumulation_within_bound(d, n, kind):
    import torch
    lib = _lib()
    rng = np.random.default_rng(1000 * d + n + KINDS.index(kind))
    beta = d * 2.0 ** -21
    worst = 0.0
    for trial in range(8):
        a, b = operands(kind, 128, n, d, rng)
        ta = torch.from_numpy(a.view(np.int16)).cuda()
        tb = torch.from_numpy(b.view(np.int16)).cuda()
        out = torch.full((128, n), float("nan"), dtype=torch.float32, device="cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        rc = lib.tcb_run(d, n, ta.data_ptr(), tb.data_ptr(), out.data_ptr(), status.data_ptr(),
                         torch.cuda.current_stream().cuda_stream)
        assert rc == 0
        torch.cuda.synchronize()
        assert int(status.item()) == 0, "MMA did not complete"
        t = out.cpu().numpy().astype(np.float64)
        af, bf = widen(a), widen(b)
        exact = af @ bf.T                 # products of bf16 are exact in float64
        mag = np.abs(af) @ np.abs(bf).T
        err = np.abs(t - exact)
        assert np.isfinite(t).all()
        ok = err <= beta * mag
        assert ok.all(), (f"{kind} d={d} n={n}: {int((~ok).sum())} pairs exceed the bound; worst "
                          f"{float((err / np.maximum(mag, 1e-300)).max()) / 2.0 ** -24:.1f} "
                          f"x 2^-24 sum|qk|")
        ratio = float(np.max(np.where(mag > 0, err / np.maximum(mag, 1e-300), 0.0)))
        worst = max(worst, ratio / 2.0 ** -24)
    _results[f"d{d}_n{n}_{kind}"] = worst
    print(f"tcgen05 accumulation d={d} n={n} {kind}: max |t - exact| = {worst:.2f} x 2^-24 "
          f"sum|q_c k_c| (bound {beta / 2.0 ** -24:.0f})")
    path = os.environ.get("TOPO_TC_BOUND_OUT")
    if path:
        with open(path, "w") as f:
            json.dump({"unit": "2^-24 * sum_c |q_c k_c|", "bound": {"64": 512, "128": 1024},
                       "max_error": _results}, f, indent=1, sort_keys=True)
