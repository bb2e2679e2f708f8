"""Pins for the oracle's group-shared selection (one condensate set per
sequence, KV head and row, shared by the KV head's g query heads; the top-k
ranks keys by the largest of the heads' float32 scores, ties to the lower
index; each head then takes its own softmax over the shared set).

Checked against: brute force on integer inputs (float32 scores exact),
reduction to the per-head oracle where the two must agree (g = 1; all heads of
a group asking the same query), a library attention routine with the shared
set as the mask (torch SDPA in float64), and a constructed case where the max
rule decides against a sum or a single head.
"""
import numpy as np
import pytest
import torch

import oracle
import synth


def _params(B, Hq, Hkv, d, n, nq, W, k, scale, dtype="f32"):
    return oracle.make_params(B, Hq, Hkv, d, n, nq, W, k, scale, dtype)


def _brute_group_sets(qi, ki, n, nq, W, k, g):
    """Sets from exact integer scores: shat = max over the group's heads."""
    B, Hq = qi.shape[:2]
    Hkv = Hq // g
    sets = []
    for b in range(B):
        for kvh in range(Hkv):
            for r in range(nq):
                p = n - nq + r
                sc = (qi[b, kvh * g:(kvh + 1) * g, r, :] @ ki[b, kvh, :p + 1, :].T).max(axis=0)
                cand = list(range(1, p - W + 1))
                top = sorted(cand, key=lambda j: (-sc[j], j))[:k]
                s = sorted({0} | set(range(max(0, p - W + 1), p + 1)) | set(top))
                sets.append(s + [-1] * (1 + W + k - len(s)))
    return np.array(sets, np.int32)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_group_selection_matches_brute_force_on_integer_scores(dtype):
    rng = np.random.default_rng(71)
    for _ in range(25):
        g = int(rng.choice([1, 2, 4]))
        Hkv = int(rng.integers(1, 3))
        B = int(rng.integers(1, 3))
        d = int(rng.choice([4, 8]))
        n = int(rng.integers(1, 60))
        nq = int(rng.integers(1, n + 1))
        W = int(rng.integers(1, 9))
        k = int(rng.integers(0, 9))
        qi = rng.integers(-3, 4, size=(B, g * Hkv, nq, d)).astype(np.float64)
        ki = rng.integers(-3, 4, size=(B, Hkv, n, d)).astype(np.float64)
        v = rng.standard_normal((B, Hkv, n, d))
        P = _params(B, g * Hkv, Hkv, d, n, nq, W, k, 0.5, dtype)
        o = oracle.topo_attn_group(P, synth.to_bf16_bits(qi) if dtype == "bf16" else qi.astype(np.float32),
                                   synth.to_bf16_bits(ki) if dtype == "bf16" else ki.astype(np.float32),
                                   synth.to_bf16_bits(v) if dtype == "bf16" else v.astype(np.float32),
                                   want=("idx",))
        np.testing.assert_array_equal(o["idx"], _brute_group_sets(qi, ki, n, nq, W, k, g))


def test_group_of_one_is_the_per_head_selection():
    w = synth.CONFIGS[0].with_(n=400, nq=400, Hq=3, Hkv=3, W=9, k=7)
    x = synth.make(w)
    P = _params(w.B, w.Hq, w.Hkv, w.d, w.n, w.nq, w.W, w.k, w.scale)
    og = oracle.topo_attn_group(P, x["q"], x["k"], x["v"])
    oh = oracle.topo_attn(P, x["q"], x["k"], x["v"], want=("out", "idx"))
    np.testing.assert_array_equal(og["idx"], oh["idx"])
    np.testing.assert_allclose(og["out"][:, 0, :], oh["out"], rtol=0, atol=1e-13)


def test_identical_queries_in_a_group_select_like_one_head():
    w = synth.CONFIGS[0].with_(n=300, nq=40, Hq=8, Hkv=2, W=11, k=9)
    x = synth.make(w)
    g = w.Hq // w.Hkv
    for kvh in range(w.Hkv):
        x["q"][:, kvh * g:(kvh + 1) * g] = x["q"][:, kvh * g:kvh * g + 1]
    P = _params(w.B, w.Hq, w.Hkv, w.d, w.n, w.nq, w.W, w.k, w.scale)
    og = oracle.topo_attn_group(P, x["q"], x["k"], x["v"])
    oh = oracle.topo_attn(P, x["q"], x["k"], x["v"], want=("out", "idx"))
    # per-head rows are flat over [B, Hq, nq]; group rows over [B, Hkv, nq]
    for kvh in range(w.Hkv):
        for hh in range(g):
            h = kvh * g + hh
            rows_h = slice(h * w.nq, (h + 1) * w.nq)
            rows_g = slice(kvh * w.nq, (kvh + 1) * w.nq)
            np.testing.assert_array_equal(og["idx"][rows_g], oh["idx"][rows_h])
            np.testing.assert_allclose(og["out"][rows_g, hh], oh["out"][rows_h], rtol=0,
                                       atol=1e-13)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_each_head_is_softmax_over_the_shared_set(dtype):
    w = synth.CONFIGS[0].with_(dtype=dtype, n=250, nq=250, Hq=4, Hkv=2, W=7, k=5)
    x = synth.make(w)
    g = w.Hq // w.Hkv
    P = _params(w.B, w.Hq, w.Hkv, w.d, w.n, w.nq, w.W, w.k, w.scale, dtype)
    o = oracle.topo_attn_group(P, x["q"], x["k"], x["v"])
    q = torch.from_numpy(synth.widen(x["q"], dtype).astype(np.float64))
    k = torch.from_numpy(synth.widen(x["k"], dtype).astype(np.float64))
    v = torch.from_numpy(synth.widen(x["v"], dtype).astype(np.float64))
    for kvh in range(w.Hkv):
        mask = torch.zeros(w.nq, w.n, dtype=torch.bool)
        for r in range(w.nq):
            js = o["idx"][kvh * w.nq + r]
            mask[r, js[js >= 0]] = True
        for hh in range(g):
            h = kvh * g + hh
            ref = torch.nn.functional.scaled_dot_product_attention(
                q[0, h][None], k[0, kvh][None], v[0, kvh][None], attn_mask=mask[None],
                scale=w.scale)[0]
            got = o["out"][kvh * w.nq:(kvh + 1) * w.nq, hh]
            np.testing.assert_allclose(got, ref.numpy(), rtol=0, atol=1e-12)


def test_the_group_score_is_the_max_over_heads():
    """Two heads, k = 1.  Key 1 scores (10, -10) and key 2 scores (6, 6): the
    largest single score is key 1's (10), while the sum (0 vs 12) and head 1
    alone would pick key 2.  The group takes key 1."""
    d, n, W = 2, 8, 2
    q = np.zeros((1, 2, 1, d), np.float32)
    q[0, 0, 0] = [1, 0]
    q[0, 1, 0] = [0, 1]
    k = np.zeros((1, 1, n, d), np.float32)
    k[0, 0, 1] = [10, -10]
    k[0, 0, 2] = [6, 6]
    v = np.zeros_like(k)
    P = _params(1, 2, 1, d, n, 1, W, 1, 1.0)
    o = oracle.topo_attn_group(P, q, k, v, want=("idx",))
    assert o["idx"][0].tolist() == [0, 1, 6, 7]
