"""The seeded input generator: determinism, distribution and rounding."""
import numpy as np
import torch

import synth


def test_draws_do_not_depend_on_thread_count():
    key = synth.key(123, 4, 5)
    a = synth.normal(key, 10, 200_000)
    b = np.concatenate([synth.normal(key, 10, 70_000), synth.normal(key, 70_010, 130_000)])
    np.testing.assert_array_equal(a, b)


def test_normal_moments():
    x = synth.normal(synth.key(1, 2), 0, 400_000)
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1.0) < 0.01
    assert abs((x ** 3).mean()) < 0.02 and abs((x ** 4).mean() - 3.0) < 0.05


def test_bf16_rounding_matches_library():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(10000).astype(np.float32) * 100,
                        np.array([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 0.0], np.float32)])
    ours = synth.to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ours, ref)


def test_workload_recipe():
    w = synth.CONFIGS[1].with_(n=4096, kv_stride=4100, nan_tail=True)
    x = synth.make(w)
    y = synth.make(w)
    for name in ("q", "k", "v"):
        np.testing.assert_array_equal(x[name], y[name])
    k = synth.widen(x["k"], "bf16")
    assert np.isnan(k[:, :, w.n:]).all() and not np.isnan(k[:, :, :w.n]).any()
    g = w.Hq // w.Hkv
    q = synth.widen(x["q"], "bf16").astype(np.float64)
    for h in range(w.Hkv):
        pos = x["planted"][(0, h)]
        assert len(pos) == w.planted and len(set(pos.tolist())) == w.planted
        assert pos.min() >= 1 and pos.max() < w.n - w.W
        # planted rows point along the group's mean query, length ~2 sqrt(d)
        qbar = q[0, h * g:(h + 1) * g].reshape(-1, w.d).mean(0)
        rows = k[0, h, pos].astype(np.float64)
        cos = rows @ qbar / np.linalg.norm(rows, axis=1) / np.linalg.norm(qbar)
        assert (cos > 0.95).all()
        # sink row carries +6u
        assert float(k[0, h, 0].astype(np.float64) @ x["u"][0, h]) > 3.0
