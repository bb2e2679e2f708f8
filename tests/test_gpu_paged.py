"""Paged KV cache, per-sequence lengths and bf16 output
(topo_attn_forward_paged), against the oracle on the equivalent contiguous
inputs: index sets bit for bit, outputs within 2e-3 row-relative (plus one
bf16 rounding, 2^-8 of the row's largest value, for bf16 outputs)."""
import numpy as np
import pytest
import torch

import oracle
import synth
import dynamic_sparse_transformer_qk_b300 as topo
from gpu_common import TOL_BF16_REL, oracle_params

pytestmark = pytest.mark.gpu

BF16_OUT_TOL = TOL_BF16_REL + 2.0 ** -8


def _bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a)).view(torch.bfloat16).cuda()


def _pool(x, w, bs, rng, spare=3):
    """Split each sequence's cache into blocks of bs keys, store them in a
    pool in a random physical order (with spare NaN blocks), and return the
    pool and the block table."""
    B, Hkv = w.B, w.Hkv
    nblk = (w.n + bs - 1) // bs
    total = B * nblk + spare
    perm = rng.permutation(total)
    kpool = np.full((total, Hkv, bs, w.d), 0x7FC0, np.uint16)  # bf16 NaN
    vpool = np.full((total, Hkv, bs, w.d), 0x7FC0, np.uint16)
    table = np.zeros((B, nblk + 2), np.int32)
    for b in range(B):
        for lb in range(nblk):
            pb = perm[b * nblk + lb]
            table[b, lb] = pb
            lo, hi = lb * bs, min((lb + 1) * bs, w.n)
            kpool[pb, :, :hi - lo] = x["k"][b, :, lo:hi]
            vpool[pb, :, :hi - lo] = x["v"][b, :, lo:hi]
    return kpool, vpool, table


def _check(got_out, got_idx, ref_out, ref_idx, tol):
    np.testing.assert_array_equal(got_idx, ref_idx)
    err = np.abs(got_out.astype(np.float64) - ref_out).max(axis=1)
    scale = np.maximum(np.abs(ref_out).max(axis=1), 1e-30)
    assert float((err / scale).max()) <= tol


@pytest.mark.parametrize("bs", [128, 256])
@pytest.mark.parametrize("out_bf16", [False, True])
def test_paged_matches_contiguous_oracle(bs, out_bf16):
    w = synth.CONFIGS[1].with_(B=2, n=20000, nq=bs // 128)  # nq 1 or 2 query rows
    x = synth.make(w)
    kpool, vpool, table = _pool(x, w, bs, np.random.default_rng(bs))
    out, idx = topo.forward_paged(_bf16(x["q"]), _bf16(kpool), _bf16(vpool), W=w.W, topk=w.k,
                                  n=w.n, block_table=torch.from_numpy(table).cuda(),
                                  scale=w.scale, out_bf16=out_bf16, want_idx=True)
    torch.cuda.synchronize()
    o = oracle.topo_attn(oracle_params(w), x["q"], x["k"], x["v"], want=("out", "idx"))
    got = out.float().cpu().numpy().reshape(-1, w.d)
    _check(got, idx.cpu().numpy().reshape(o["idx"].shape), o["out"], o["idx"],
           BF16_OUT_TOL if out_bf16 else TOL_BF16_REL)


def test_paged_with_per_sequence_lengths():
    """Three sequences of different lengths in one paged call: each against
    the oracle run on that sequence alone."""
    lens = [20000, 7777, 130]
    w = synth.CONFIGS[1].with_(B=3, n=max(lens), Hq=8, Hkv=2, planted=8)
    x = synth.make(w)
    kpool, vpool, table = _pool(x, w, 128, np.random.default_rng(5))
    out, idx = topo.forward_paged(_bf16(x["q"]), _bf16(kpool), _bf16(vpool), W=w.W, topk=w.k,
                                  n=w.n, block_table=torch.from_numpy(table).cuda(),
                                  seq_lens=torch.tensor(lens, dtype=torch.int32).cuda(),
                                  scale=w.scale, want_idx=True)
    torch.cuda.synchronize()
    go, gi = out.cpu().numpy(), idx.cpu().numpy()
    for b, nb in enumerate(lens):
        wb = w.with_(B=1, n=nb)
        xb = {"q": np.ascontiguousarray(x["q"][b:b + 1]),
              "k": np.ascontiguousarray(x["k"][b:b + 1, :, :nb]),
              "v": np.ascontiguousarray(x["v"][b:b + 1, :, :nb])}
        o = oracle.topo_attn(oracle_params(wb), xb["q"], xb["k"], xb["v"], want=("out", "idx"))
        _check(go[b].reshape(-1, w.d), gi[b].reshape(o["idx"].shape), o["out"], o["idx"],
               TOL_BF16_REL)


def test_contiguous_cache_with_bf16_output():
    w = synth.CONFIGS[1].with_(n=12000, kv_stride=12345, nan_tail=True)
    x = synth.make(w)
    out, idx = topo.forward_paged(_bf16(x["q"]), _bf16(x["k"]), _bf16(x["v"]), W=w.W, topk=w.k,
                                  n=w.n, scale=w.scale, out_bf16=True, want_idx=True)
    torch.cuda.synchronize()
    o = oracle.topo_attn(oracle_params(w), x["q"], x["k"], x["v"], want=("out", "idx"))
    _check(out.float().cpu().numpy().reshape(-1, w.d), idx.cpu().numpy().reshape(o["idx"].shape),
           o["out"], o["idx"], BF16_OUT_TOL)


def test_out_of_range_block_is_reported_not_followed():
    """A block-table entry outside the pool is read as block 0 (no access
    leaves the pool) and the device status word says so."""
    w = synth.CONFIGS[1].with_(n=5000, planted=4)
    x = synth.make(w)
    kpool, vpool, table = _pool(x, w, 128, np.random.default_rng(9))
    table[0, 3] = 10 ** 6
    ws = topo.Workspace()
    topo.forward_paged(_bf16(x["q"]), _bf16(kpool), _bf16(vpool), W=w.W, topk=w.k, n=w.n,
                       block_table=torch.from_numpy(table).cuda(), scale=w.scale, workspace=ws)
    torch.cuda.synchronize()
    assert topo.device_status(ws) == -7
    assert topo.device_status(ws) == 0  # read clears it
