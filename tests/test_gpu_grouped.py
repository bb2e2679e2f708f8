"""GPU parity of group-shared selection (topo_attn_forward_grouped) against
the oracle's group function: one condensate set per (sequence, KV head,
row), shared by the KV head's query heads, top-k by the largest of their
float32 scores.  Index sets bit for bit, outputs within 2e-3 row-relative
(bf16 inputs)."""
import numpy as np
import pytest
import torch

import oracle
import synth
import dynamic_sparse_transformer_qk_b300 as topo
from gpu_common import assert_out_close, device_inputs, oracle_params

pytestmark = pytest.mark.gpu

W1 = synth.CONFIGS[1]


def _grouped(w, x):
    q, k, v = device_inputs(x, w)
    out, idx = topo.forward_grouped(q, k, v, W=w.W, topk=w.k, n=w.n, scale=w.scale,
                                    want_idx=True)
    torch.cuda.synchronize()
    o = oracle.topo_attn_group(oracle_params(w), x["q"], x["k"], x["v"])
    np.testing.assert_array_equal(idx.cpu().numpy().reshape(o["idx"].shape), o["idx"])
    g = w.Hq // w.Hkv
    # out [B, Hq, nq, d] against the oracle's [B*Hkv*nq, g, d]
    got = out.cpu().numpy().reshape(w.B, w.Hkv, g, w.nq, w.d).transpose(0, 1, 3, 2, 4)
    assert_out_close(got.reshape(-1, w.d), o["out"].reshape(-1, w.d), w.dtype)
    return idx


def test_grouped_decode_32k():
    """The 32K decode workload (32/8 heads): one set per KV head."""
    _grouped(W1, synth.make(W1))


SHAPES = [
    ("g2_d64_k9", dict(d=64, Hq=4, Hkv=2, n=3000, nq=1, W=5, k=9)),
    ("g8_d128_k32", dict(Hq=16, Hkv=2, n=20000, nq=1, W=64, k=32, planted=16)),
    ("g4_k64", dict(Hq=8, Hkv=2, n=30000, nq=1, W=64, k=64, planted=32)),
    ("g2_nq2_k33", dict(Hq=4, Hkv=2, n=7000, nq=2, W=16, k=33)),
    ("g4_nq2", dict(Hq=8, Hkv=2, n=9000, nq=2, W=20, k=12)),
    ("batch3", dict(B=3, Hq=8, Hkv=2, n=12345, nq=1, W=33, k=31, planted=8)),
    ("nan_tail", dict(Hq=8, Hkv=2, n=10000, nq=1, kv_stride=10300, nan_tail=True, W=64, k=32,
                      planted=32)),
    ("short", dict(Hq=8, Hkv=2, n=150, nq=1, W=10, k=32)),
    ("wide_window", dict(d=64, Hq=4, Hkv=1, n=6000, nq=1, W=5000, k=32)),
    # 16 query heads per KV head: 16 tensor-core columns per block
    ("g16", dict(Hq=64, Hkv=4, n=15000, nq=1, W=64, k=32, planted=16)),
    ("g8_nq2", dict(d=64, Hq=16, Hkv=2, n=8000, nq=2, W=40, k=20)),
]


@pytest.mark.parametrize("name,kw", SHAPES, ids=[s[0] for s in SHAPES])
def test_grouped_shapes(name, kw):
    w = W1.with_(**kw)
    _grouped(w, synth.make(w))


def test_grouped_all_equal_keys_fall_back_exactly():
    """Every candidate ties for every head: buffers overflow, the exact rescan
    runs, and the lowest positions win."""
    w = W1.with_(Hq=4, Hkv=1, n=30000, W=10, k=32, planted=0)
    x = synth.make(w)
    x["k"][:] = x["k"][:, :, 7:8, :]
    idx = _grouped(w, x)
    assert idx[0, 0, 0, 1:33].tolist() == list(range(1, 33))


def test_grouped_equals_per_head_when_the_group_asks_one_query():
    """With the g queries of a KV head identical, the shared set is each
    head's own set and the outputs equal topo_attn_forward's."""
    w = W1.with_(n=20000)
    x = synth.make(w)
    g = w.Hq // w.Hkv
    for kvh in range(w.Hkv):
        x["q"][:, kvh * g:(kvh + 1) * g] = x["q"][:, kvh * g:kvh * g + 1]
    q, k, v = device_inputs(x, w)
    og, ig = topo.forward_grouped(q, k, v, W=w.W, topk=w.k, n=w.n, scale=w.scale, want_idx=True)
    oh, ih, _ = topo.forward(q, k, v, W=w.W, topk=w.k, n=w.n, scale=w.scale, want_idx=True)
    torch.cuda.synchronize()
    assert torch.equal(ig[:, :, None].expand(-1, -1, g, -1, -1).reshape(ih.shape), ih)
    assert torch.allclose(og, oh, rtol=0, atol=1e-6)
