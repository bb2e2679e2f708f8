"""The C-ABI library: it loads, exports what the header declares, and rejects
bad arguments on the host before anything is enqueued.  No compute call is
made here (no GPU needed); every argument set below fails validation first."""
import ctypes
import os
import re

import pytest

import dynamic_sparse_transformer_qk_b300 as topo

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "topo_attn.h")


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return set(re.findall(r"\b([a-z_]+)\s*\(", text)) - {"sizeof"}


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(topo.library_path()):
        from dynamic_sparse_transformer_qk_b300 import build
        build.build()
    return topo.load_library()


def test_exports_match_header(lib):
    declared = _declared()
    assert declared == set(topo.EXPORTS)
    for name in declared:
        assert hasattr(lib, name)


def _p(**kw):
    base = dict(B=1, Hq=32, Hkv=8, d=128, n=4096, nq=1, kv_stride=4096, W=64, k=32,
                scale=0.125, dtype=1)
    base.update(kw)
    return topo.Params(**base)


def test_workspace_size(lib):
    assert lib.topo_attn_workspace_size(ctypes.byref(_p())) > 256
    assert lib.dense_attn_workspace_size(ctypes.byref(_p())) > 256
    for bad in (dict(d=96), dict(n=0), dict(nq=5000), dict(k=300), dict(Hq=30),
                dict(kv_stride=100), dict(W=0), dict(k=-1), dict(dtype=7),
                dict(scale=float("inf"))):
        assert lib.topo_attn_workspace_size(ctypes.byref(_p(**bad))) == 0, bad


def test_strerror(lib):
    for code in (0, -1, -2, -3, -4, -5):
        assert len(lib.topo_attn_strerror(code)) >= 2
    assert lib.topo_attn_strerror(12345) == b"unknown status"


FAKE = 0x100000  # aligned, never dereferenced: every call below fails validation first


@pytest.mark.parametrize("bad,code", [
    (dict(d=96), -2), (dict(k=257), -2), (dict(dtype=3), -2),
    (dict(n=0), -1), (dict(nq=4097), -1), (dict(Hq=7), -1), (dict(W=0), -1),
    (dict(kv_stride=10), -1), (dict(scale=float("nan")), -1),
])
def test_forward_rejects_bad_params(lib, bad, code):
    p = _p(**bad)
    rc = lib.topo_attn_forward(ctypes.byref(p), FAKE, FAKE, FAKE, FAKE, None, None, FAKE,
                               1 << 30, None)
    assert rc == code


def test_forward_rejects_bad_pointers(lib):
    p = _p()
    assert lib.topo_attn_forward(ctypes.byref(p), None, FAKE, FAKE, FAKE, None, None, FAKE,
                                 1 << 30, None) == -1
    assert lib.topo_attn_forward(ctypes.byref(p), FAKE, FAKE, FAKE, None, None, None, FAKE,
                                 1 << 30, None) == -1
    assert lib.topo_attn_forward(ctypes.byref(p), FAKE + 4, FAKE, FAKE, FAKE, None, None, FAKE,
                                 1 << 30, None) == -1
    assert lib.topo_attn_score_select(ctypes.byref(p), FAKE, FAKE, None, FAKE, 1 << 30,
                                      None) == -1
    assert lib.topo_attn_sparse_softmax_pv(ctypes.byref(p), FAKE, FAKE, FAKE, None, FAKE,
                                           None) == -1
    assert lib.dense_attn_forward(ctypes.byref(p), FAKE, FAKE, None, FAKE, FAKE, 1 << 30,
                                  None) == -1


def test_forward_rejects_bad_workspace(lib):
    p = _p()
    need = lib.topo_attn_workspace_size(ctypes.byref(p))
    assert lib.topo_attn_forward(ctypes.byref(p), FAKE, FAKE, FAKE, FAKE, None, None, FAKE,
                                 need - 1, None) == -3
    assert lib.topo_attn_forward(ctypes.byref(p), FAKE, FAKE, FAKE, FAKE, None, None, None,
                                 need, None) == -3
    assert lib.topo_attn_forward(ctypes.byref(p), FAKE, FAKE, FAKE, FAKE, None, None, FAKE + 16,
                                 need, None) == -3
    need_d = lib.dense_attn_workspace_size(ctypes.byref(p))
    assert lib.dense_attn_forward(ctypes.byref(p), FAKE, FAKE, FAKE, FAKE, FAKE, need_d - 1,
                                  None) == -3


def test_binding_refuses_cpu_tensors():
    import torch
    q = torch.zeros(1, 1, 1, 64)
    with pytest.raises(ValueError):
        topo.forward(q, q, q, W=4, topk=2)
