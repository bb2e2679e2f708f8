"""Pins for the CPU oracle, independent of the oracle's own code.

Each test checks the oracle against something the pages or the mathematics
fix: brute force on integer inputs (where float32 scores are exact), a library
dense-attention routine (torch's scaled_dot_product_attention in float64),
closed forms, invariants of the condensate set, and the set size the pages
print.  A plausible slip in the oracle (a wrong window edge, a reversed tie
rule, a dropped anchor, a transposed GQA map, an unfused score) fails one of
them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _params(B, Hq, Hkv, d, n, nq, W, k, scale, dtype="f32", kv_stride=None):
    return oracle.make_params(B, Hq, Hkv, d, n, nq, W, k, scale, dtype, kv_stride)


def _store(x, dtype):
    return x.astype(np.float32) if dtype == "f32" else synth.to_bf16_bits(x)


def _widen(x, dtype):
    return synth.widen(x, dtype).astype(np.float64)


# ---------------------------------------------------------------- the score --

def test_score_is_left_to_right_chain():
    # exact dot is 1; left-to-right float32 rounding loses the 1 against 2^24
    q = np.array([1.0, 1.0, 1.0], np.float32)
    k = np.array([2.0 ** 24, 1.0, -(2.0 ** 24)], np.float32)
    assert oracle.score_f32(q, k) == np.float32(0.0)
    # reversed order would give 1: the order is pinned, not just the value set
    assert oracle.score_f32(q[::-1].copy(), k[::-1].copy()) == np.float32(1.0)


def test_score_is_fused():
    # fma(a, a, -1) keeps 2^-24 that a separate multiply would round away
    a = np.float32(1.0 + 2.0 ** -12)
    q = np.array([1.0, a], np.float32)
    k = np.array([-1.0, a], np.float32)
    assert oracle.score_f32(q, k) == np.float32(2.0 ** -11 + 2.0 ** -24)


def test_score_starts_from_positive_zero():
    s = oracle.score_f32(np.array([-1.0], np.float32), np.array([0.0], np.float32))
    assert s == 0.0 and not math.copysign(1.0, float(s)) < 0


def test_score_within_recursive_summation_bound():
    rng = np.random.default_rng(7)
    u = 2.0 ** -24
    for d in (16, 64, 128):
        g = d * u / (1 - d * u)
        for _ in range(200):
            q = rng.standard_normal(d).astype(np.float32)
            k = rng.standard_normal(d).astype(np.float32)
            exact = float(np.dot(q.astype(np.float64), k.astype(np.float64)))
            bound = g * float(np.abs(q.astype(np.float64) * k).sum())
            assert abs(float(oracle.score_f32(q, k)) - exact) <= bound


# ----------------------------------------------------------- the selection --

def _brute_sets(qi, ki, n, nq, W, k, g):
    """Condensate sets by brute force from exact integer scores."""
    B, Hq, _, d = qi.shape
    sets = []
    for b in range(B):
        for h in range(Hq):
            for r in range(nq):
                p = n - nq + r
                s = ki[b, h // g, :p + 1] @ qi[b, h, r]
                cand = sorted(range(1, p - W + 1), key=lambda j: (-s[j], j))
                chosen = set(cand[:k]) | {0} | set(range(max(0, p - W + 1), p + 1))
                row = sorted(chosen)
                sets.append(row + [-1] * (1 + W + k - len(row)))
    return np.array(sets, dtype=np.int32)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_selection_matches_brute_force_on_integer_scores(dtype):
    rng = np.random.default_rng(11 if dtype == "f32" else 12)
    shapes = [(1, 1, 1), (2, 2, 1), (1, 4, 2), (2, 6, 3)]
    for trial in range(40):
        B, Hq, Hkv = shapes[trial % len(shapes)]
        g = Hq // Hkv
        d = int(rng.integers(1, 6))
        n = int(rng.integers(1, 41))
        nq = int(rng.choice([1, n, max(1, n // 3)]))
        W = int(rng.integers(1, 6))
        k = int(rng.choice([0, 1, 2, 3, 5, 9]))
        qi = rng.integers(-2, 3, size=(B, Hq, nq, d)).astype(np.int64)
        ki = rng.integers(-2, 3, size=(B, Hkv, n, d)).astype(np.int64)
        vi = rng.standard_normal((B, Hkv, n, d))
        P = _params(B, Hq, Hkv, d, n, nq, W, k, 0.5, dtype)
        res = oracle.topo_attn(P, _store(qi, dtype), _store(ki, dtype), _store(vi, dtype),
                               want=("idx",))
        want = _brute_sets(qi, ki, n, nq, W, k, g)
        np.testing.assert_array_equal(res["idx"], want)


def test_ties_go_to_the_lower_index():
    # all keys equal: every candidate ties, so the top-k are 1..k
    n, W, k, d = 50, 4, 6, 8
    kk = np.ones((1, 1, n, d), np.float32)
    q = np.ones((1, 1, 1, d), np.float32)
    v = np.zeros((1, 1, n, d), np.float32)
    res = oracle.topo_attn(_params(1, 1, 1, d, n, 1, W, k, 1.0), q, kk, v, want=("idx",))
    assert list(res["idx"][0]) == [0, 1, 2, 3, 4, 5, 6] + list(range(n - W, n))


def test_k_zero_is_anchor_plus_window():
    w = synth.CONFIGS[0].with_(n=300, nq=300, k=0)
    x = synth.make(w)
    P = _params(1, 1, 1, w.d, w.n, w.nq, w.W, 0, w.scale, "f32")
    idx = oracle.topo_attn(P, x["q"], x["k"], x["v"], want=("idx",))["idx"]
    for p in range(w.n):
        want = sorted({0} | set(range(max(0, p - w.W + 1), p + 1)))
        row = [j for j in idx[p] if j >= 0]
        assert row == want


def test_gqa_maps_query_head_to_its_group():
    # head h must score against KV head h // (Hq/Hkv): give each KV head one
    # distinctive planted key and check that only its own group finds it.
    Hq, Hkv, d, n, W, k = 6, 3, 4, 40, 2, 1
    kk = np.zeros((1, Hkv, n, d), np.float32)
    q = np.ones((1, Hq, 1, d), np.float32)
    for h in range(Hkv):
        kk[0, h, 5 + 7 * h] = 3.0
    res = oracle.topo_attn(_params(1, Hq, Hkv, d, n, 1, W, k, 1.0), q, kk,
                           np.zeros_like(kk), want=("idx",))
    for h in range(Hq):
        assert res["idx"][h][1] == 5 + 7 * (h // 2)


# ------------------------------------------------------ the set's structure --

def test_condensate_set_size_golden():
    gold = json.load(open(os.path.join(GOLDEN, "condensate_set_size.json")))
    W, k = gold["W"], gold["k"]
    w = synth.CONFIGS[0].with_(n=400, nq=400, W=W, k=k)
    x = synth.make(w)
    P = _params(1, 1, 1, w.d, w.n, w.nq, W, k, w.scale, "f32")
    idx = oracle.topo_attn(P, x["q"], x["k"], x["v"], want=("idx",))["idx"]
    sizes = (idx >= 0).sum(axis=1)
    assert idx.shape[1] == gold["set_size"]
    assert all(sizes[p] == min(p + 1, gold["set_size"]) for p in range(w.n))
    assert (sizes[W + k:] == gold["set_size"]).all()


def test_condensate_set_invariants():
    w = synth.CONFIGS[0].with_(n=333, nq=333, W=16, k=8)
    x = synth.make(w)
    P = _params(1, 1, 1, w.d, w.n, w.nq, w.W, w.k, w.scale, "f32")
    idx = oracle.topo_attn(P, x["q"], x["k"], x["v"], want=("idx",))["idx"]
    for p in range(w.n):
        row = idx[p]
        m = int((row >= 0).sum())
        assert (row[m:] == -1).all() and (row[:m] >= 0).all()
        c = row[:m]
        assert m == min(p + 1, 1 + w.W + w.k)
        assert (np.diff(c) > 0).all()
        assert c[0] == 0 and c[-1] == p
        assert set(range(max(0, p - w.W + 1), p + 1)) <= set(c.tolist())


# ------------------------------------------------------ softmax and outputs --

def _sdpa(q64, k64, v64, mask, scale):
    return torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q64), torch.from_numpy(k64), torch.from_numpy(v64),
        attn_mask=torch.from_numpy(mask), scale=scale).numpy()


def _expand(x, g):
    return np.repeat(x, g, axis=1)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("nq_kind", ["prefill", "decode", "partial"])
def test_dense_matches_library_attention(dtype, nq_kind):
    rng = np.random.default_rng(3)
    B, Hq, Hkv, d, n = 2, 4, 2, 16, 37
    nq = {"prefill": n, "decode": 1, "partial": 6}[nq_kind]
    q = _store(rng.standard_normal((B, Hq, nq, d)), dtype)
    k = _store(rng.standard_normal((B, Hkv, n, d)) * 2, dtype)
    v = _store(rng.standard_normal((B, Hkv, n, d)), dtype)
    scale = 0.3
    res = oracle.topo_attn(_params(B, Hq, Hkv, d, n, nq, 3, 2, scale, dtype), q, k, v,
                           want=("dense",))
    pos = np.arange(nq) + n - nq
    mask = np.arange(n)[None, :] <= pos[:, None]
    ref = _sdpa(_widen(q, dtype), _expand(_widen(k, dtype), Hq // Hkv),
                _expand(_widen(v, dtype), Hq // Hkv), mask, np.float32(scale).item())
    np.testing.assert_allclose(res["dense"], ref.reshape(-1, d), rtol=0, atol=1e-12)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_sparse_is_softmax_over_the_set(dtype):
    rng = np.random.default_rng(5)
    B, Hq, Hkv, d, n, nq, W, k = 1, 4, 1, 8, 60, 60, 5, 4
    q = _store(rng.standard_normal((B, Hq, nq, d)), dtype)
    kk = _store(rng.standard_normal((B, Hkv, n, d)) * 1.5, dtype)
    v = _store(rng.standard_normal((B, Hkv, n, d)), dtype)
    scale = 0.4
    res = oracle.topo_attn(_params(B, Hq, Hkv, d, n, nq, W, k, scale, dtype), q, kk, v,
                           want=("out", "idx"))
    idx = res["idx"].reshape(B, Hq, nq, -1)
    mask = np.zeros((B, Hq, nq, n), dtype=bool)
    for h in range(Hq):
        for r in range(nq):
            sel = idx[0, h, r]
            mask[0, h, r, sel[sel >= 0]] = True
    ref = _sdpa(_widen(q, dtype), _expand(_widen(kk, dtype), Hq // Hkv),
                _expand(_widen(v, dtype), Hq // Hkv), mask, np.float32(scale).item())
    np.testing.assert_allclose(res["out"], ref.reshape(-1, d), rtol=0, atol=1e-12)


def test_sparse_equals_dense_when_the_set_covers_the_prefix():
    w = synth.CONFIGS[0].with_(n=256, nq=256)
    x = synth.make(w)
    P = _params(1, 1, 1, w.d, w.n, w.nq, w.W, w.k, w.scale, "f32")
    res = oracle.topo_attn(P, x["q"], x["k"], x["v"], want=("out", "dense", "excl", "idx"))
    cover = 1 + w.W + w.k
    np.testing.assert_allclose(res["out"][:cover], res["dense"][:cover], rtol=0, atol=1e-12)
    assert (res["excl"][:cover] == 0).all()
    assert (res["excl"][cover:] > 0).all()
    # and against the library routine on the covered rows
    mask = np.tril(np.ones((w.n, w.n), dtype=bool))
    ref = _sdpa(_widen(x["q"], "f32"), _widen(x["k"], "f32"), _widen(x["v"], "f32"), mask,
                w.scale).reshape(-1, w.d)
    np.testing.assert_allclose(res["out"][:cover], ref[:cover], rtol=0, atol=1e-12)


def test_weights_sum_to_one():
    rng = np.random.default_rng(9)
    n, d = 80, 8
    q = rng.standard_normal((1, 2, n, d)).astype(np.float32)
    k = (rng.standard_normal((1, 1, n, d)) * 3).astype(np.float32)
    v = np.ones((1, 1, n, d), np.float32)
    res = oracle.topo_attn(_params(1, 2, 1, d, n, n, 3, 4, 0.7), q, k, v, want=("out", "dense"))
    np.testing.assert_allclose(res["out"], 1.0, rtol=0, atol=1e-13)
    np.testing.assert_allclose(res["dense"], 1.0, rtol=0, atol=1e-13)


def test_equal_scores_closed_form():
    # identical keys: dense weights are 1/(p+1) each, the sparse output is the
    # mean of V over the set, and the excluded mass counts the missing rows
    rng = np.random.default_rng(2)
    n, d, W, k = 90, 4, 7, 5
    kk = np.tile(rng.standard_normal(d).astype(np.float32), (1, 1, n, 1))
    q = rng.standard_normal((1, 1, n, d)).astype(np.float32)
    v = rng.standard_normal((1, 1, n, d)).astype(np.float32)
    res = oracle.topo_attn(_params(1, 1, 1, d, n, n, W, k, 0.5), q, kk, v)
    for p in range(n):
        c = res["idx"][p][res["idx"][p] >= 0]
        np.testing.assert_allclose(res["out"][p], v[0, 0, c].astype(np.float64).mean(0),
                                   rtol=0, atol=1e-12)
        missing = p + 1 - len(c)
        assert res["excl"][p] == pytest.approx(missing / (p + 1), abs=1e-14)
        assert res["wmax"][p] == pytest.approx(1 / (p + 1) if missing else 0.0, abs=1e-14)
        assert res["p0"][p] == pytest.approx(1 / (p + 1), abs=1e-14)


def test_sparse_dense_gap_is_bounded_by_excluded_mass():
    # o_dense = (1-eps) o_sparse + eps o_excl, so per coordinate
    # |o_sparse - o_dense| <= eps * (max_j v_jc - min_j v_jc) over the prefix
    w = synth.CONFIGS[0].with_(n=700, nq=700)
    x = synth.make(w)
    P = _params(1, 1, 1, w.d, w.n, w.nq, w.W, w.k, w.scale, "f32")
    res = oracle.topo_attn(P, x["q"], x["k"], x["v"])
    v = _widen(x["v"], "f32")[0, 0]
    for p in range(w.n):
        span = v[:p + 1].max(0) - v[:p + 1].min(0)
        gap = np.abs(res["out"][p] - res["dense"][p])
        assert (gap <= res["excl"][p] * span + 1e-12).all()
        assert res["wmax"][p] <= res["excl"][p] + 1e-15


def test_planted_keys_are_the_top_k():
    # decode n=32768, 32/8 heads: the 32 planted keys per KV head score far
    # above the random ones, so each head's top-32 is exactly the planted set
    w = synth.CONFIGS[1]
    x = synth.make(w)
    P = _params(w.B, w.Hq, w.Hkv, w.d, w.n, w.nq, w.W, w.k, w.scale, w.dtype)
    idx = oracle.topo_attn(P, x["q"], x["k"], x["v"], want=("idx",))["idx"]
    g = w.Hq // w.Hkv
    for h in range(w.Hq):
        top = set(idx[h][1:1 + w.k].tolist())
        assert top == set(x["planted"][(0, h // g)].tolist())


def test_ranking_is_decided_by_the_float32_score():
    # key 1: exact dot 1 but float32 chain 0; key 2: 0.5 either way.  The
    # selection decides in float32 (the precision the GPU ranks in), so k=1
    # picks key 2 although key 1 has the larger exact score.
    q = np.array([[[[1.0, 1.0, 1.0]]]], np.float32)
    kk = np.zeros((1, 1, 6, 3), np.float32)
    kk[0, 0, 1] = [2.0 ** 24, 1.0, -(2.0 ** 24)]
    kk[0, 0, 2] = [0.0, 0.0, 0.5]
    kk[0, 0, 3] = [0.0, 0.0, -1.0]
    res = oracle.topo_attn(_params(1, 1, 1, 3, 6, 1, 2, 1, 1.0), q, kk, np.zeros_like(kk),
                           want=("idx",))
    assert list(res["idx"][0]) == [0, 2, 4, 5]
