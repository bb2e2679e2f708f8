"""topo_attn_forward_noalloc: the entry point for callers that cannot allocate
device memory (plugin hosts that only hand over their input and output
buffers, serving loops that forbid cudaMalloc after start-up).  It runs the
same kernels as topo_attn_forward with its scratch in a fixed array inside the
library, so its results must match topo_attn_forward's with a caller-owned
workspace -- call after call, although every call reuses the array the
previous call left behind.

This file is collected last on purpose: the GPU test here runs after every
other test, and also passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest

import synth
import dynamic_sparse_transformer_qk_b300 as topo

TOL_F32_ABS = 1e-5
TOL_BF16_REL = 2e-3


def test_noalloc_rejects_problems_beyond_its_scratch():
    """Host-side check: a shape whose workspace exceeds the fixed array is
    refused before anything is enqueued (no GPU needed)."""
    lib = topo.load_library()
    # a 4096-row chunked-prefill call needs far more than 8 MiB of scratch
    p = topo.Params(1, 32, 8, 128, 65536, 4096, 65536, 256, 32, 0.088388, 1)
    assert lib.topo_attn_workspace_size(ctypes.byref(p)) > (8 << 20)
    fake = 0x100000  # never dereferenced: the size check comes first
    rc = lib.topo_attn_forward_noalloc(ctypes.byref(p), fake, fake, fake, fake, None, None, None)
    assert rc == -6
    assert b"scratch" in lib.topo_attn_strerror(rc)
    # argument errors are reported as by topo_attn_forward
    bad = topo.Params(1, 32, 8, 96, 4096, 1, 4096, 64, 32, 0.1, 1)
    assert lib.topo_attn_forward_noalloc(ctypes.byref(bad), fake, fake, fake, fake, None, None,
                                         None) == -2


def _close(a, b, dtype):
    a = a.double().reshape(-1, a.shape[-1])
    b = b.double().reshape(-1, b.shape[-1])
    err = (a - b).abs()
    if dtype == "f32":
        return float(err.max()) <= TOL_F32_ABS
    scale = b.abs().max(dim=1).values.clamp_min(1e-30)
    return float((err.max(dim=1).values / scale).max()) <= TOL_BF16_REL


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point_on_consecutive_calls():
    import torch
    torch.cuda.set_device(0)
    cases = [synth.CONFIGS[1],                                  # decode n=32768, bf16
             synth.CONFIGS[1].with_(n=29000, planted=16),        # another shape, same array
             synth.CONFIGS[0].with_(n=600, nq=600)]              # fp32 prefill rows
    for w in cases:
        x = synth.make(w)

        def dev(a):
            t = torch.from_numpy(np.ascontiguousarray(a))
            return (t.view(torch.bfloat16) if w.dtype == "bf16" else t).cuda()

        q, k, v = dev(x["q"]), dev(x["k"]), dev(x["v"])
        shape = (w.B, w.Hq, w.nq)
        ref_out, ref_idx, ref_excl = topo.forward(q, k, v, W=w.W, topk=w.k, n=w.n,
                                                  scale=w.scale, want_idx=True, want_excl=True,
                                                  workspace=topo.Workspace())
        for _ in range(2):  # two calls in a row on the shared array
            out = torch.full((*shape, w.d), float("nan"), device="cuda")
            idx = torch.full((*shape, 1 + w.W + w.k), -7, dtype=torch.int32, device="cuda")
            excl = torch.full(shape, float("nan"), device="cuda")
            topo.forward_noalloc(q, k, v, W=w.W, topk=w.k, n=w.n, scale=w.scale, out=out,
                                 idx=idx, excl=excl)
            torch.cuda.synchronize()
            assert torch.equal(idx, ref_idx), w.name
            assert _close(out, ref_out, w.dtype), w.name
            assert bool(((excl - ref_excl).abs() <= 1e-6 + 1e-4 * ref_excl.abs()).all()), w.name
