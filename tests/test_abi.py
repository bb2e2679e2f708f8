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


# ------------------------------------------------------ multi-layer step ----

def test_layer_schedule_pillars_and_window_tiers():
    """32 layers, a pillar every 16 (L/16 = 2 pillars, at 0 and 16), windows
    256 / 128 / 64 by depth third, k = 32 everywhere."""
    sch = topo.layer_schedule(32, pillar_every=16, windows=(256, 128, 64), topk=32)
    assert [l for l, s in enumerate(sch) if s["dense"]] == [0, 16]
    assert [s["W"] for s in sch] == [256] * 11 + [128] * 11 + [64] * 10
    assert all(s["topk"] == 32 for s in sch)
    ws = [s["W"] for s in sch if not s["dense"]]
    assert ws == sorted(ws, reverse=True)          # wide early, narrow late
    assert not any(s["dense"] for s in topo.layer_schedule(5, pillar_every=0))
    assert [s["W"] for s in topo.layer_schedule(3, windows=(9,))] == [9, 9, 9]


def test_layer_schedule_rejects_bad_arguments(lib):
    arr = (topo.TopoLayer * 4)()
    win = (ctypes.c_int32 * 2)(64, 32)
    a, w = ctypes.addressof(arr), ctypes.addressof(win)
    assert lib.topo_attn_layer_schedule(4, 2, w, 2, 8, a) == 0
    assert [x.dense for x in arr] == [1, 0, 1, 0] and [x.W for x in arr] == [64, 64, 32, 32]
    assert lib.topo_attn_layer_schedule(0, 2, w, 2, 8, a) == -1
    assert lib.topo_attn_layer_schedule(4, -1, w, 2, 8, a) == -1
    assert lib.topo_attn_layer_schedule(4, 2, w, 0, 8, a) == -1
    assert lib.topo_attn_layer_schedule(4, 2, w, 2, 300, a) == -1
    assert lib.topo_attn_layer_schedule(4, 2, None, 2, 8, a) == -1
    bad = (ctypes.c_int32 * 2)(64, 0)
    assert lib.topo_attn_layer_schedule(4, 2, ctypes.addressof(bad), 2, 8, a) == -1


def test_layers_forward_checks_every_layer_first(lib):
    p = _p()
    arr = (topo.TopoLayer * 3)()
    for x in arr:
        x.q = x.k = x.v = x.out = FAKE
        x.W, x.k_top, x.dense = 64, 32, 0
    arr[1].dense = 1
    a = ctypes.addressof(arr)
    need = lib.topo_attn_layers_workspace_size(ctypes.byref(p), a, 3)
    assert need >= max(lib.topo_attn_workspace_size(ctypes.byref(p)),
                       lib.dense_attn_workspace_size(ctypes.byref(p)))
    # a bad last layer: nothing is enqueued for the good ones before it
    arr[2].out = None
    assert lib.topo_attn_layers_forward(ctypes.byref(p), a, 3, FAKE, need, None) == -1
    arr[2].out = FAKE
    arr[2].k_top = 999
    assert lib.topo_attn_layers_forward(ctypes.byref(p), a, 3, FAKE, need, None) == -2
    assert lib.topo_attn_layers_workspace_size(ctypes.byref(p), a, 3) == 0
    arr[2].k_top = 32
    arr[0].reserved = 1
    assert lib.topo_attn_layers_forward(ctypes.byref(p), a, 3, FAKE, need, None) == -1
    arr[0].reserved = 0
    assert lib.topo_attn_layers_forward(ctypes.byref(p), a, 3, FAKE, need - 1, None) == -3
    assert lib.topo_attn_layers_forward(ctypes.byref(p), a, 0, FAKE, need, None) == -1
    # a pillar layer ignores W and k: a bad W there is not an error
    arr[1].W = -5
    assert lib.topo_attn_layers_workspace_size(ctypes.byref(p), a, 3) == need


def test_grouped_rejects_unsupported_shapes(lib):
    need = 1 << 30
    # float32, one head per group, prefill-sized column counts: not the grouped shapes
    for bad in (dict(dtype=0), dict(Hq=8, Hkv=8), dict(nq=64)):
        p = _p(**bad)
        rc = lib.topo_attn_forward_grouped(ctypes.byref(p), FAKE, FAKE, FAKE, FAKE, None, FAKE,
                                           need, None)
        assert rc == -2, bad
    p = _p()
    assert lib.topo_attn_forward_grouped(ctypes.byref(p), FAKE, FAKE, None, FAKE, None, FAKE,
                                         need, None) == -1


def test_compact_kv_rejects_bad_arguments(lib):
    p = _p()
    assert lib.topo_attn_compact_kv(ctypes.byref(p), FAKE, FAKE, None, FAKE, FAKE, None) == -1
    assert lib.topo_attn_compact_kv(ctypes.byref(p), FAKE, FAKE, FAKE, FAKE + 4, FAKE, None) == -1
    assert lib.topo_attn_compact_kv(ctypes.byref(_p(d=96)), FAKE, FAKE, FAKE, FAKE, FAKE,
                                    None) == -2


def test_paged_rejects_bad_arguments(lib):
    p = _p(n=4096, kv_stride=4096)
    table = FAKE
    kv = topo.PagedKV(table, None, 32, 128, 64, 0)
    assert lib.topo_attn_paged_workspace_size(ctypes.byref(p), ctypes.byref(kv)) > 0
    for bad in (dict(block_size=100), dict(block_size=64), dict(max_blocks=8),
                dict(num_blocks=0)):
        f = dict(block_table=table, seq_lens=None, max_blocks=32, block_size=128, num_blocks=64,
                 out_bf16=0)
        f.update(bad)
        kvb = topo.PagedKV(**f)
        rc = lib.topo_attn_forward_paged(ctypes.byref(p), ctypes.byref(kvb), FAKE, FAKE, FAKE,
                                         FAKE, None, FAKE, 1 << 30, None)
        assert rc == -1, bad
    # float32 and prefill-sized shapes are not the tensor-core decode shapes
    for badp in (_p(dtype=0), _p(nq=64)):
        rc = lib.topo_attn_forward_paged(ctypes.byref(badp), ctypes.byref(kv), FAKE, FAKE, FAKE,
                                         FAKE, None, FAKE, 1 << 30, None)
        assert rc == -2
    assert lib.topo_attn_forward_paged(ctypes.byref(p), None, FAKE, FAKE, FAKE, FAKE, None, FAKE,
                                       1 << 30, None) == -1
