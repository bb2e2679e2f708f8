"""GPU parity of the multi-layer step (topo_attn_layers_forward): layer-adaptive
windows and dense pillar layers, each layer against the oracle -- the
condensate-set output for sparse layers, the dense causal output for pillars.

The pages ("Condensate Theorem" explainers, Chinese technical summary section
3, implementation strategy; Korean technical summary section 3,
layer-adaptive configuration): early layers use wider windows, later layers
leaner sets, and a few layers (e.g. L/16) keep full attention.
"""
import numpy as np
import pytest
import torch

import synth
import dynamic_sparse_transformer_qk_b300 as topo
from gpu_common import assert_out_close, device_inputs, run_oracle

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("base", [
    synth.CONFIGS[1].with_(n=12000, planted=16),                       # decode, bf16, 32/8
    synth.CONFIGS[0].with_(n=900, nq=300, Hq=4, Hkv=2),                # float32 prefill rows
], ids=["decode_bf16", "prefill_f32"])
def test_layers_forward_matches_oracle_per_layer(base):
    L = 32
    sch = topo.layer_schedule(L, pillar_every=16, windows=(256, 128, 64), topk=32)
    assert sum(s["dense"] for s in sch) == L // 16
    # every layer has its own inputs (seed per layer)
    ws = [base.with_(seed=base.seed + 101 * (l + 1)) for l in range(L)]
    xs = [synth.make(w) for w in ws]
    dev = [device_inputs(x, w) for x, w in zip(xs, ws)]
    outs = topo.layers_forward([d[0] for d in dev], [d[1] for d in dev], [d[2] for d in dev],
                               sch, n=base.n, scale=base.scale)
    torch.cuda.synchronize()
    for l, (w, x, s) in enumerate(zip(ws, xs, sch)):
        got = outs[l].cpu().numpy().reshape(-1, w.d)
        if s["dense"]:
            o = run_oracle(w, x, want=("dense",))
            assert_out_close(got, o["dense"], w.dtype, f"layer {l} (pillar)")
        else:
            o = run_oracle(w.with_(W=s["W"], k=s["topk"]), x, want=("out",))
            assert_out_close(got, o["out"], w.dtype, f"layer {l} (W={s['W']})")


def test_layers_forward_equals_single_layer_calls():
    """The multi-layer call enqueues exactly the single-layer calls: outputs
    are bit-identical to topo_attn_forward / dense_attn_forward per layer."""
    base = synth.CONFIGS[1].with_(n=9000, planted=8)
    sch = topo.layer_schedule(6, pillar_every=3, windows=(200, 50), topk=20)
    ws = [base.with_(seed=base.seed + 7 * l) for l in range(6)]
    dev = [device_inputs(synth.make(w), w) for w in ws]
    outs = topo.layers_forward([d[0] for d in dev], [d[1] for d in dev], [d[2] for d in dev],
                               sch, n=base.n, scale=base.scale)
    for (q, k, v), s, o in zip(dev, sch, outs):
        if s["dense"]:
            ref = topo.dense_forward(q, k, v, n=base.n, scale=base.scale)
        else:
            ref, _, _ = topo.forward(q, k, v, W=s["W"], topk=s["topk"], n=base.n,
                                     scale=base.scale)
        torch.cuda.synchronize()
        assert torch.equal(o, ref)
