"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

Index sets must match bit for bit; outputs within 1e-5 absolute (float32
inputs) or 2e-3 row-relative (bfloat16 inputs); the excluded mass within
1e-6 + 1e-4 * eps.
"""
import numpy as np
import pytest
import torch

import synth
import dynamic_sparse_transformer_qk_b300 as topo
from gpu_common import (compare, device_inputs, run_gpu, run_oracle, assert_out_close,
                        oracle_params)
import oracle

pytestmark = pytest.mark.gpu

W0 = synth.CONFIGS[0]


def _full(w, want_excl=True):
    x = synth.make(w)
    g = run_gpu(w, x, want_excl=want_excl)
    o = run_oracle(w, x, want=("out", "idx", "excl") if want_excl else ("out", "idx"))
    return compare(w, x, g, o)


# ------------------------------------------------------------- workloads ----

def test_tiny_causal_prefill_fp32():
    """n=2048 fp32 prefill, 1 head, d=64, W=64, k=32: every row."""
    _full(W0)


def test_decode_32k_bf16():
    """Single-token decode n=32768, 32/8 heads, d=128: every head."""
    _full(synth.CONFIGS[1])


@pytest.mark.parametrize("kw", [
    dict(Hq=64, Hkv=4, n=20000, planted=16),             # 16:1 GQA decode
    dict(Hq=32, Hkv=4, n=9000, nq=2, W=32, k=24),         # 8 heads x 2 rows
    dict(Hq=16, Hkv=4, n=5000, nq=3, W=48, k=32),         # 12 of 16 columns
    dict(d=64, Hq=32, Hkv=2, n=7000, nq=1, k=7, W=9),     # d = 64
], ids=["g16", "g8_nq2", "g4_nq3", "g16_d64"])
def test_decode_sixteen_columns_per_kv_head(kw):
    """Up to 16 query columns per KV head on the tensor-core decode scorer
    (the MMA's N): every row against the oracle, excluded mass included."""
    _full(synth.CONFIGS[1].with_(**kw))


def test_decode_32k_planted_keys_found():
    w = synth.CONFIGS[1]
    x = synth.make(w)
    g = run_gpu(w, x, want_excl=False)
    for h in range(w.Hq):
        top = set(g["idx"][h][1:1 + w.k].tolist())
        assert top == set(x["planted"][(0, h // 4)].tolist())


def test_batched_decode_128k_bf16():
    """B=16 sequences of n=131072: every (sequence, head)."""
    _full(synth.CONFIGS[2])


def test_million_token_decode_bf16():
    """n=1,048,576 decode, 32/8 heads: every head, plus the dense path."""
    w = synth.CONFIGS[4]
    x = synth.make(w)
    g = run_gpu(w, x, want_excl=True)
    o = run_oracle(w, x, want=("out", "idx", "excl", "dense"))
    compare(w, x, g, o)
    q, k, v = device_inputs(x, w)
    dense = topo.dense_forward(q, k, v, n=w.n, scale=w.scale)
    torch.cuda.synchronize()
    assert_out_close(dense.cpu().numpy().reshape(-1, w.d), o["dense"], w.dtype, "dense")


# ------------------------------------------------------------ edge cases ----

EDGE = [
    # name, overrides of the tiny fp32 prefill workload
    ("n1", dict(n=1, nq=1)),
    ("n2_k1", dict(n=2, nq=2, W=1, k=1)),
    ("window_covers_all", dict(n=50, nq=50, W=64, k=32)),
    ("k_zero", dict(n=300, nq=300, W=16, k=0)),
    ("k_exceeds_candidates", dict(n=90, nq=90, W=8, k=200)),
    ("ragged_tail", dict(n=1000, nq=1000, W=7, k=5)),
    ("k_256", dict(n=700, nq=700, W=3, k=256)),
    ("k_100", dict(n=700, nq=700, W=20, k=100)),
    ("k_60", dict(n=500, nq=500, W=5, k=60)),
    ("partial_rows", dict(n=777, nq=129, W=10, k=12)),
    ("decode_row", dict(n=5000, nq=1, W=64, k=32)),
    ("gqa_2", dict(n=400, nq=400, Hq=4, Hkv=2, W=9, k=7)),
    ("gqa_3", dict(n=300, nq=37, Hq=6, Hkv=2, W=9, k=7)),
    ("gqa_8_decode", dict(n=3000, nq=1, Hq=16, Hkv=2, W=33, k=31)),
    ("gqa_16_decode", dict(n=2000, nq=1, Hq=16, Hkv=1, W=5, k=9)),
    ("batch_3", dict(B=3, n=333, nq=333, Hq=2, Hkv=1, W=4, k=6)),
    ("d128_f32", dict(d=128, n=600, nq=600, W=12, k=10)),
    ("d128_f32_k200_nq8", dict(d=128, n=3000, nq=8, W=16, k=200)),
    ("d128_f32_k256_gqa", dict(d=128, n=2500, nq=2, Hq=8, Hkv=2, W=5, k=256)),
    ("kv_stride_nan_tail", dict(n=555, nq=555, kv_stride=700, nan_tail=True, W=6, k=9)),
    ("bf16_d64", dict(dtype="bf16", n=800, nq=800, W=11, k=13)),
    ("bf16_d128_gqa4", dict(dtype="bf16", d=128, Hq=8, Hkv=2, n=900, nq=900, W=16, k=16)),
    ("bf16_decode_stride", dict(dtype="bf16", d=128, Hq=32, Hkv=8, n=20000, nq=1,
                                kv_stride=20100, nan_tail=True, planted=32)),
]


@pytest.mark.parametrize("name,kw", EDGE, ids=[e[0] for e in EDGE])
def test_edge_cases(name, kw):
    _full(W0.with_(**kw))


# --------------------------------------- tensor-core scorer (bf16 decode) ----
# bf16 problems with at most 8 query columns per KV head (4 for k > 32) are
# scored on the tensor cores with exact rescoring; these shapes cover its
# column counts, both head sizes, k up to 64, short and multi-tile splits,
# several sequences and a NaN tail past the causal length.

TC_DECODE = [
    ("g4_d128_k32", dict(d=128, Hq=32, Hkv=8, n=40000, nq=1, W=64, k=32, planted=32)),
    ("g1_d64_k1", dict(d=64, Hq=2, Hkv=2, n=3000, nq=1, W=5, k=1)),
    ("g2_d128_k17", dict(d=128, Hq=4, Hkv=2, n=9000, nq=1, W=100, k=17)),
    ("g8_d128_k32", dict(d=128, Hq=16, Hkv=2, n=20000, nq=1, W=64, k=32, planted=32)),
    ("g4_d128_k64", dict(d=128, Hq=8, Hkv=2, n=30000, nq=1, W=64, k=64, planted=32)),
    ("g2_nq2_k33", dict(d=128, Hq=4, Hkv=2, n=7000, nq=2, W=16, k=33)),
    ("g2_nq3_k20", dict(d=64, Hq=4, Hkv=2, n=5000, nq=3, W=9, k=20)),
    ("short", dict(d=128, Hq=8, Hkv=2, n=150, nq=1, W=10, k=32)),
    ("one_candidate", dict(d=128, Hq=4, Hkv=1, n=66, nq=1, W=64, k=32)),
    ("batch3", dict(B=3, d=128, Hq=8, Hkv=2, n=12345, nq=1, W=33, k=31, planted=8)),
    ("nan_tail", dict(d=128, Hq=8, Hkv=2, n=10000, nq=1, kv_stride=10300, nan_tail=True,
                      W=64, k=32, planted=32)),
    ("wide_window", dict(d=64, Hq=4, Hkv=1, n=6000, nq=1, W=5000, k=32)),
    # the dependent tail kernel's staged softmax fits one CTA at W = 256 and
    # not at W = 400 (the select kernel's own tail takes over)
    ("w256_split_tail", dict(d=128, Hq=32, Hkv=8, n=30000, nq=1, W=256, k=32, planted=32)),
    ("w400_in_kernel_tail", dict(d=128, Hq=8, Hkv=2, n=20000, nq=1, W=400, k=32, planted=8)),
]


@pytest.mark.parametrize("name,kw", TC_DECODE, ids=[e[0] for e in TC_DECODE])
def test_tensor_core_decode_shapes(name, kw):
    _full(W0.with_(dtype="bf16", **kw))


@pytest.mark.parametrize("k", [1, 32, 64])
def test_tensor_core_all_equal_keys_fall_back_exactly(k):
    """Every candidate has the same score: the tensor-core survivors overflow
    their buffers and the split is rescored exactly; lowest positions win."""
    w = W0.with_(dtype="bf16", d=128, Hq=4, Hkv=1, n=30000, nq=1, W=10, k=k)
    x = synth.make(w)
    x["k"][:] = x["k"][:, :, 7:8, :]
    g = run_gpu(w, x)
    o = run_oracle(w, x)
    compare(w, x, g, o)
    for row in g["idx"]:
        assert row[1:1 + k].tolist() == list(range(1, 1 + k))


def test_tensor_core_near_ties():
    """Keys that differ in one low-order bit: tensor-core rounding cannot
    separate them, the exact rescoring must."""
    w = W0.with_(dtype="bf16", d=128, Hq=4, Hkv=1, n=20000, nq=1, W=16, k=32)
    x = synth.make(w)
    rng = np.random.default_rng(17)
    # a key along head 0's query, well above every random key's score
    q0 = synth.widen(x["q"][0, 0, 0], "bf16").astype(np.float64)
    base = synth.to_bf16_bits(2.0 * np.sqrt(w.d) * q0 / np.linalg.norm(q0))
    rows = rng.choice(np.arange(1, w.n - w.W), size=48, replace=False)
    for r in rows:
        kr = base.copy()
        c = int(rng.integers(0, w.d))
        kr[c] = np.uint16(int(kr[c]) ^ 1)  # flip the lowest mantissa bit of one element
        x["k"][0, 0, r] = kr
    g = run_gpu(w, x)
    o = run_oracle(w, x)
    compare(w, x, g, o)


# ------------------------------------------ tensor-core prefill (bf16, k <= 32)
# bf16 problems with more than 8 query columns per KV head run the chunked
# prefill path: scan on the tensor cores, exact rescoring of the survivors,
# softmax per row.  Shapes cover both head sizes, MHA and GQA up to 8, partial
# column blocks, several sequences, a NaN tail and windows longer than a tile.

TC_PREFILL = [
    ("d128_g4_full", dict(d=128, Hq=8, Hkv=2, n=1500, nq=1500, W=64, k=32, planted=16,
                          planted_range="all")),
    ("d64_g1", dict(d=64, Hq=3, Hkv=3, n=700, nq=700, W=7, k=5)),
    ("d128_g8_partial", dict(d=128, Hq=16, Hkv=2, n=2000, nq=33, W=40, k=31)),
    ("d128_b2_rows", dict(B=2, d=128, Hq=4, Hkv=2, n=3000, nq=300, W=200, k=1)),
    ("d64_k32_long_window", dict(d=64, Hq=4, Hkv=1, n=2500, nq=2500, W=300, k=32)),
    ("nan_tail", dict(d=128, Hq=8, Hkv=2, n=1000, nq=1000, kv_stride=1100, nan_tail=True,
                      W=16, k=24)),
]


@pytest.mark.parametrize("name,kw", TC_PREFILL, ids=[e[0] for e in TC_PREFILL])
def test_tensor_core_prefill_shapes(name, kw):
    _full(W0.with_(dtype="bf16", **kw))


@pytest.mark.parametrize("n,nq", [(1200, 200), (20000, 64)])
def test_tensor_core_prefill_all_equal_keys_fall_back_exactly(n, nq):
    """Every candidate ties: the column buffers overflow and the finalize step
    rescans those rows exactly; the lowest positions win.  With n = 20000 the
    first pass sees more equal tile maxima than its buffer holds (overflow
    with the cut kept)."""
    w = W0.with_(dtype="bf16", d=128, Hq=4, Hkv=1, n=n, nq=nq, W=10, k=32)
    x = synth.make(w)
    x["k"][:] = x["k"][:, :, 7:8, :]
    g = run_gpu(w, x)
    o = run_oracle(w, x)
    compare(w, x, g, o)


def test_tensor_core_prefill_near_ties():
    """Prefill rows whose top-k includes keys one mantissa bit apart along a
    query direction: the tile maxima and the cut they give must keep every
    key the exact chain ranks in."""
    w = W0.with_(dtype="bf16", d=128, Hq=8, Hkv=2, n=6000, nq=512, W=64, k=32)
    x = synth.make(w)
    rng = np.random.default_rng(7)
    q0 = synth.widen(x["q"][0, 0, 0], "bf16").astype(np.float64)
    base = synth.to_bf16_bits(2.0 * np.sqrt(w.d) * q0 / np.linalg.norm(q0))
    rows = rng.choice(np.arange(1, w.n - w.nq - w.W), size=48, replace=False)
    for r in rows:
        kr = base.copy()
        c = int(rng.integers(0, w.d))
        kr[c] = np.uint16(int(kr[c]) ^ 1)
        x["k"][0, 0, r] = kr
    g = run_gpu(w, x)
    o = run_oracle(w, x)
    compare(w, x, g, o)


# ------------------------------------------------------------------ ties ----

@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_all_equal_keys_pick_lowest_positions(dtype):
    """Every candidate ties: the lowest positions win, through many buffer
    compactions and the split merge."""
    w = W0.with_(dtype=dtype, d=128, Hq=4, Hkv=1, n=6000, nq=3, W=10, k=40)
    x = synth.make(w)
    x["k"][:] = x["k"][:, :, 7:8, :]
    g = run_gpu(w, x)
    o = run_oracle(w, x)
    compare(w, x, g, o)
    for row in g["idx"]:
        assert row[1:41].tolist() == list(range(1, 41))


def test_integer_scores_with_many_ties():
    rng = np.random.default_rng(4)
    w = W0.with_(d=64, Hq=2, Hkv=1, n=3000, nq=40, W=6, k=24)
    x = synth.make(w)
    x["q"][:] = rng.integers(-1, 2, size=x["q"].shape).astype(np.float32)
    x["k"][:] = rng.integers(-1, 2, size=x["k"].shape).astype(np.float32)
    g = run_gpu(w, x)
    o = run_oracle(w, x)
    compare(w, x, g, o)


def test_increasing_scores_stress_compaction():
    """Scores rise with position: every key beats the running threshold."""
    w = W0.with_(n=20000, nq=2, W=4, k=33)
    x = synth.make(w)
    x["q"][:] = 0.0
    x["q"][..., 0] = 1.0
    x["k"][0, 0, :, 0] = np.arange(w.n, dtype=np.float32) * 1e-3
    g = run_gpu(w, x)
    o = run_oracle(w, x)
    compare(w, x, g, o)


# ------------------------------------------------- the separate entry points

def test_score_select_and_sparse_softmax_pv():
    w = W0.with_(dtype="bf16", d=128, Hq=8, Hkv=2, n=1500, nq=40, W=20, k=24)
    x = synth.make(w)
    o = run_oracle(w, x, want=("out", "idx"))
    q, k, v = device_inputs(x, w)
    idx = topo.score_select(q, k, W=w.W, topk=w.k, n=w.n, scale=w.scale)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(idx.cpu().numpy().reshape(o["idx"].shape), o["idx"])
    # the softmax step on the oracle's own sets
    oidx = torch.from_numpy(o["idx"].reshape(idx.shape)).cuda()
    out = topo.sparse_softmax_pv(q, k, v, oidx, W=w.W, topk=w.k, n=w.n, scale=w.scale)
    torch.cuda.synchronize()
    assert_out_close(out.cpu().numpy().reshape(-1, w.d), o["out"], w.dtype)


def test_sparse_softmax_pv_ignores_out_of_range_entries():
    w = W0.with_(n=200, nq=200, W=4, k=4)
    x = synth.make(w)
    o = run_oracle(w, x, want=("out", "idx"))
    bad = o["idx"].copy()
    # -1 pads already present; add positions beyond the row and negatives
    bad[:, -1] = np.where(bad[:, -1] < 0, 10 ** 6, bad[:, -1])
    bad[:, -2] = np.where(bad[:, -2] < 0, -7, bad[:, -2])
    q, k, v = device_inputs(x, w)
    out = topo.sparse_softmax_pv(q, k, v, torch.from_numpy(bad.reshape(1, 1, w.nq, -1)).cuda(),
                                 W=w.W, topk=w.k, n=w.n, scale=w.scale)
    torch.cuda.synchronize()
    assert_out_close(out.cpu().numpy().reshape(-1, w.d), o["out"], w.dtype)


@pytest.mark.parametrize("kw", [dict(), dict(dtype="bf16", d=128, Hq=8, Hkv=2),
                                dict(n=3000, nq=1, Hq=4, Hkv=1), dict(n=1, nq=1),
                                dict(d=128, n=32768, nq=1), dict(d=128, n=5000, nq=8),
                                dict(d=128, n=4000, nq=3, Hq=8, Hkv=2),
                                # bf16 with at most 8 query columns per KV head: the
                                # tensor-core dense kernel (128-key tiles, ragged tails)
                                dict(dtype="bf16", d=128, n=5000, nq=1, Hq=32, Hkv=8),
                                dict(dtype="bf16", d=64, n=3001, nq=2, Hq=8, Hkv=2),
                                dict(dtype="bf16", d=128, n=130, nq=3, Hq=4, Hkv=2),
                                dict(dtype="bf16", d=128, n=1, nq=1, Hq=2, Hkv=2),
                                dict(dtype="bf16", d=128, n=777, nq=1, Hq=2, Hkv=2,
                                     kv_stride=1000, nan_tail=True)])
def test_dense_matches_oracle(kw):
    w = W0.with_(n=700, nq=700).with_(**kw)
    x = synth.make(w)
    o = run_oracle(w, x, want=("dense",))
    q, k, v = device_inputs(x, w)
    out = topo.dense_forward(q, k, v, n=w.n, scale=w.scale)
    torch.cuda.synchronize()
    assert_out_close(out.cpu().numpy().reshape(-1, w.d), o["dense"], w.dtype, "dense")


def test_chunked_prefill_equals_full_prefill():
    w = W0.with_(dtype="bf16", d=128, Hq=8, Hkv=2, n=4096, nq=4096, W=64, k=32, planted=16,
                 planted_range="all")
    x = synth.make(w)
    q, k, v = device_inputs(x, w)
    full_out, full_idx, _ = topo.forward(q, k, v, W=w.W, topk=w.k, n=w.n, scale=w.scale,
                                         want_idx=True)
    chunk = 1024
    for c in range(w.n // chunk):
        qc = q[:, :, c * chunk:(c + 1) * chunk].contiguous()
        out, idx, _ = topo.forward(qc, k, v, W=w.W, topk=w.k, n=(c + 1) * chunk,
                                   scale=w.scale, want_idx=True)
        torch.cuda.synchronize()
        assert torch.equal(idx, full_idx[:, :, c * chunk:(c + 1) * chunk])
        assert torch.allclose(out, full_out[:, :, c * chunk:(c + 1) * chunk], rtol=0, atol=1e-6)


def _run_chunks(w, x, keep_rows):
    """The chunked prefill (chunks of w.chunk rows through topo_attn_forward,
    idx and excluded mass on) on the device; returns idx, out and excl of the
    flat rows `keep_rows` (ids over [B=1, Hq, n])."""
    q, k, v = device_inputs(x, w)
    keep_rows = np.asarray(keep_rows)
    heads, pos = keep_rows // w.n, keep_rows % w.n
    res = {"idx": np.empty((keep_rows.size, 1 + w.W + w.k), np.int32),
           "out": np.empty((keep_rows.size, w.d), np.float32),
           "excl": np.empty(keep_rows.size, np.float32)}
    chunk = w.chunk
    for c in range(w.n // chunk):
        sel = np.nonzero((pos >= c * chunk) & (pos < (c + 1) * chunk))[0]
        if sel.size == 0:
            continue
        qc = q[:, :, c * chunk:(c + 1) * chunk].contiguous()
        out, idx, excl = topo.forward(qc, k, v, W=w.W, topk=w.k, n=(c + 1) * chunk,
                                      scale=w.scale, want_idx=True, want_excl=True)
        torch.cuda.synchronize()
        h = torch.from_numpy(heads[sel]).cuda()
        r = torch.from_numpy(pos[sel] - c * chunk).cuda()
        res["idx"][sel] = idx[0][h, r].cpu().numpy()
        res["out"][sel] = out[0][h, r].cpu().numpy()
        res["excl"][sel] = excl[0][h, r].cpu().numpy()
    return res


@pytest.mark.parametrize("W", [256, 128, 64])
def test_chunked_prefill_first_chunk_and_sampled_rows(W):
    """The chunked prefill workload (n=65536, 32/8 heads, chunks of 4096) at
    each of its windows, against the oracle: every row of every head in the
    first chunk, plus 512 seeded rows spread over all 16 chunks (32 per chunk,
    any head) -- idx bit for bit, out within 2e-3 row-relative, the excluded
    mass within 1e-6 + 1e-4 eps."""
    w = synth.CONFIGS[3].with_(W=W)
    x = synth.make(w)
    rng = np.random.default_rng(20260211 + W)
    first = (np.arange(w.Hq)[:, None] * w.n + np.arange(w.chunk)[None, :]).reshape(-1)
    sampled = []
    for c in range(w.n // w.chunk):
        hh = rng.integers(0, w.Hq, 32)
        rr = rng.choice(np.arange(c * w.chunk, (c + 1) * w.chunk), 32, replace=False)
        sampled.append(hh * w.n + rr)
    rows = np.unique(np.concatenate([first] + sampled))
    assert rows.size >= first.size + 480
    g = _run_chunks(w, x, rows)
    o = oracle.topo_attn(oracle_params(w), x["q"], x["k"], x["v"], rows=rows,
                         want=("out", "idx", "excl"))
    compare(w, x, g, o)


def test_chunked_prefill_full_size_near_ties():
    """The last 4096-row chunk of the 64K prefill (W=64) with 48 keys one
    mantissa bit apart along one query's direction: every row of that query's
    head and a seeded sample of the others must keep exactly the oracle's
    top-k, although the tensor-core scores cannot separate those keys."""
    w = synth.CONFIGS[3].with_(W=64)
    x = synth.make(w)
    rng = np.random.default_rng(31)
    p0 = w.n - w.chunk
    q0 = synth.widen(x["q"][0, 0, p0], "bf16").astype(np.float64)
    base = synth.to_bf16_bits(2.0 * np.sqrt(w.d) * q0 / np.linalg.norm(q0))
    for r in rng.choice(np.arange(1, p0 - w.W), size=48, replace=False):
        kr = base.copy()
        c = int(rng.integers(0, w.d))
        kr[c] = np.uint16(int(kr[c]) ^ 1)
        x["k"][0, 0, r] = kr
    q, k, v = device_inputs(x, w)
    qc = q[:, :, p0:].contiguous()
    out, idx, excl = topo.forward(qc, k, v, W=w.W, topk=w.k, n=w.n, scale=w.scale,
                                  want_idx=True, want_excl=True)
    torch.cuda.synchronize()
    head0 = np.arange(w.chunk)                                   # head 0: every row
    others = rng.choice(np.arange(w.chunk, w.Hq * w.chunk), 512, replace=False)
    sel = np.sort(np.concatenate([head0, others]))
    hh, rr = sel // w.chunk, sel % w.chunk
    g = {"idx": idx[0].cpu().numpy()[hh, rr], "out": out[0].cpu().numpy()[hh, rr],
         "excl": excl[0].cpu().numpy()[hh, rr]}
    o = oracle.topo_attn(oracle_params(w), x["q"], x["k"], x["v"], rows=hh * w.n + p0 + rr,
                         want=("out", "idx", "excl"))
    compare(w, x, g, o)


# ------------------------------------------------ repeatability and status --

def test_repeatable_and_workspace_reusable():
    w = synth.CONFIGS[1]
    x = synth.make(w)
    ws = topo.Workspace()
    a = run_gpu(w, x, workspace=ws)
    b = run_gpu(w, x, workspace=ws)
    c = run_gpu(w.with_(n=w.n - 1000), x, workspace=ws)  # another shape on the same workspace
    d = run_gpu(w, x, workspace=ws)
    for key in ("out", "idx", "excl"):
        assert np.array_equal(a[key], b[key]) and np.array_equal(a[key], d[key])
    assert c["idx"].shape == a["idx"].shape
    assert topo.device_status(ws) == 0
