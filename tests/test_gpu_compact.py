"""Condensate KV compaction (topo_attn_compact_kv): the rows each query's
condensate set names, gathered into a compact cache.  Checked bit for bit
against indexing the inputs at the oracle's sets, and for exactness of the
compact cache: the softmax over its rows reproduces the oracle's output for
the same queries."""
import numpy as np
import pytest
import torch

import oracle
import synth
import dynamic_sparse_transformer_qk_b300 as topo
from gpu_common import assert_out_close, device_inputs, oracle_params, run_oracle

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("w", [
    synth.CONFIGS[1],                                                  # decode 32K, bf16, 32/8
    synth.CONFIGS[0].with_(n=700, nq=300, Hq=4, Hkv=2, W=9, k=7),     # float32 prefill rows
    synth.CONFIGS[0].with_(dtype="bf16", n=50, nq=50, W=64, k=8),     # windows cover everything
], ids=["decode32k", "f32_rows", "wide"])
def test_compact_kv_is_the_condensate_rows_and_exact(w):
    x = synth.make(w)
    q, k, v = device_inputs(x, w)
    o = run_oracle(w, x, want=("out", "idx"))
    cmax = 1 + w.W + w.k
    idx = torch.from_numpy(o["idx"].reshape(w.B, w.Hq, w.nq, cmax)).cuda()
    ko, vo = topo.compact_kv(k, v, idx, Hq=w.Hq, n=w.n)
    torch.cuda.synchronize()
    # bit for bit: the input rows at the oracle's sets, zero rows for -1
    g = w.Hq // w.Hkv
    kin = x["k"][:, np.arange(w.Hq) // g]  # [B, Hq, S, d]
    vin = x["v"][:, np.arange(w.Hq) // g]
    ii = o["idx"].reshape(w.B, w.Hq, w.nq, cmax)
    safe = np.where(ii >= 0, ii, 0)
    bidx = np.arange(w.B)[:, None, None, None]
    hidx = np.arange(w.Hq)[None, :, None, None]
    kref = np.where((ii >= 0)[..., None], kin[bidx, hidx, safe], 0)
    vref = np.where((ii >= 0)[..., None], vin[bidx, hidx, safe], 0)
    kview = ko.view(torch.uint16) if w.dtype == "bf16" else ko
    vview = vo.view(torch.uint16) if w.dtype == "bf16" else vo
    np.testing.assert_array_equal(kview.cpu().numpy(), kref)
    np.testing.assert_array_equal(vview.cpu().numpy(), vref)
    # exactness: every query row attends over its own compact rows only
    rows = w.B * w.Hq * w.nq
    qc = q.reshape(rows, 1, 1, w.d)
    kc = ko.reshape(rows, 1, cmax, w.d)
    vc = vo.reshape(rows, 1, cmax, w.d)
    ent = np.where(ii.reshape(rows, 1, 1, cmax) >= 0, np.arange(cmax, dtype=np.int32), -1)
    out = topo.sparse_softmax_pv(qc, kc, vc, torch.from_numpy(ent).cuda(), W=cmax - 1, topk=0,
                                 n=cmax, scale=w.scale)
    torch.cuda.synchronize()
    assert_out_close(out.cpu().numpy().reshape(-1, w.d), o["out"], w.dtype)
