"""Shared helpers of the GPU parity tests: run the CUDA path and the oracle on
the same seeded inputs and compare them under the stated tolerances."""
import numpy as np
import torch

import oracle
import synth
import dynamic_sparse_transformer_qk_b300 as topo

# output tolerances: float32 inputs absolute; bfloat16 inputs relative per row
TOL_F32_ABS = 1e-5
TOL_BF16_REL = 2e-3


def to_dev(x: np.ndarray, dtype: str) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(x))
    if dtype == "bf16":
        t = t.view(torch.bfloat16)
    return t.cuda()


def device_inputs(x: dict, w: synth.Workload):
    return to_dev(x["q"], w.dtype), to_dev(x["k"], w.dtype), to_dev(x["v"], w.dtype)


def oracle_params(w: synth.Workload, **kw):
    f = dict(B=w.B, Hq=w.Hq, Hkv=w.Hkv, d=w.d, n=w.n, nq=w.nq, W=w.W, k=w.k, scale=w.scale,
             dtype=w.dtype, kv_stride=w.stride)
    f.update(kw)
    return oracle.make_params(**f)


def run_oracle(w, x, rows=None, want=("out", "idx", "excl")):
    return oracle.topo_attn(oracle_params(w), x["q"], x["k"], x["v"], rows=rows, want=want)


def run_gpu(w, x, want_idx=True, want_excl=True, workspace=None):
    q, k, v = device_inputs(x, w)
    out, idx, excl = topo.forward(q, k, v, W=w.W, topk=w.k, n=w.n, scale=w.scale,
                                  want_idx=want_idx, want_excl=want_excl, workspace=workspace)
    torch.cuda.synchronize()
    res = {"out": out.cpu().numpy().reshape(-1, w.d)}
    if idx is not None:
        res["idx"] = idx.cpu().numpy().reshape(-1, 1 + w.W + w.k)
    if excl is not None:
        res["excl"] = excl.cpu().numpy().reshape(-1)
    return res


def assert_out_close(got: np.ndarray, ref: np.ndarray, dtype: str, what="out"):
    got = got.astype(np.float64)
    err = np.abs(got - ref)
    assert np.isfinite(got).all(), f"{what}: non-finite values"
    if dtype == "f32":
        worst = float(err.max()) if err.size else 0.0
        assert worst <= TOL_F32_ABS, f"{what}: max abs error {worst:.3e} > {TOL_F32_ABS}"
    else:
        scale = np.maximum(np.abs(ref).max(axis=1), 1e-30)
        rel = err.max(axis=1) / scale
        worst = float(rel.max()) if rel.size else 0.0
        assert worst <= TOL_BF16_REL, f"{what}: max row-relative error {worst:.3e} > {TOL_BF16_REL}"
    return worst


def assert_excl_close(got: np.ndarray, ref: np.ndarray):
    tol = 1e-6 + 1e-4 * ref
    bad = np.abs(got.astype(np.float64) - ref) > tol
    assert not bad.any(), (f"excl: {int(bad.sum())} rows off, worst "
                           f"{float(np.abs(got - ref).max()):.3e}")


def compare(w, x, g, o, rows=None):
    """g: GPU results over all rows; o: oracle results over `rows` (None = all)."""
    sel = slice(None) if rows is None else np.asarray(rows)
    if "idx" in g and "idx" in o:
        gi, oi = g["idx"][sel], o["idx"]
        if not np.array_equal(gi, oi):
            bad = np.nonzero((gi != oi).any(axis=1))[0]
            r = int(bad[0])
            raise AssertionError(f"idx differs on {len(bad)} rows; first row {r}:\n"
                                 f"gpu    {gi[r].tolist()}\noracle {oi[r].tolist()}")
    worst = assert_out_close(g["out"][sel], o["out"], w.dtype)
    if "excl" in g and "excl" in o:
        assert_excl_close(g["excl"][sel], o["excl"])
    return worst
