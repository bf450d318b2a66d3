"""GPU parity of the pre-norm layer's backward (tp_layer_backward: the
forward recomputed with its state kept, the MLP block's backward, RMSNorm's
backward with the residual, the attention block's backward, RMSNorm again)
against the fp64 oracle through the C ABI.

Small layers and the full size the bench runs (4 x 2048 tokens, h 4096,
f 14336, 32 query / 8 KV heads of 128, t 8) compare every output: dX and
all seven weight gradients.  At full size the oracle runs in its composed
form (numpy matrix products, the C attention core and norms; pinned equal to
the all-C definition)."""
import numpy as np
import pytest
import torch

import megatron_tensor_transformer_colwise_gb300 as tp
import oracle
import synth
from synth import SHAPES, Shape
from gpu_util import (assert_close, dev, elementwise_excess_fraction, host64, plan_for, report,
                      sync_ok, workspace)

pytestmark = pytest.mark.gpu

NAMES = ["dX", "dWq", "dWk", "dWv", "dWo", "dW1", "dW3", "dW2"]


def run_layer_backward(s, inp, dY, accumulate=False, init=0.0):
    plan = plan_for(s)
    ws, nws = workspace(plan, tp.TP_OP_LAYER_BACKWARD)
    w = {k: dev(v) for k, v in inp.items() if k != "X"}
    f32 = dict(dtype=torch.float32, device="cuda")
    grads = {"d" + k: torch.full(tuple(v.shape), init, **f32) for k, v in w.items()}
    dX = torch.empty(s.tokens, s.hidden, dtype=torch.bfloat16, device="cuda")
    tp.tp_layer_backward(plan, dev(inp["X"]), w, dev(dY), dX, grads, accumulate, ws, nws)
    sync_ok(plan)
    out = {"dX": dX.cpu()}
    out.update({k: v.cpu() for k, v in grads.items()})
    return out


def oracle_grads(s, inp, dY):
    args = [host64(inp[k]) for k in ("X", "Wq", "Wk", "Wv", "Wo", "W1", "W3", "W2")]
    return dict(zip(NAMES, oracle.layer_backward(s.batch, s.seq, s.heads, s.kv_heads, s.head_dim,
                                                 *args, host64(dY))))


SMALL = [
    Shape("lb_small", 2, 128, 256, ffn=512, heads=4, kv_heads=2, head_dim=128, tp=2, act="swiglu",
          index=61),
    Shape("lb_replica_ragged", 1, 200, 256, ffn=320, heads=4, kv_heads=1, head_dim=128, tp=4,
          act="swiglu", index=62),
]


@pytest.mark.parametrize("s", SMALL, ids=[s.name for s in SMALL])
def test_small_layer_backward_full_output(s):
    inp = synth.workload_inputs(s)
    dY = synth.grad_output(s)
    got = run_layer_backward(s, inp, dY)
    ref = oracle_grads(s, inp, dY)
    for n in NAMES:
        assert_close(host64(got[n]), ref[n], what=f"{s.name} {n}")


def test_layer_backward_accumulates_weight_gradients():
    s = SMALL[0]
    inp = synth.workload_inputs(s)
    dY = synth.grad_output(s)
    ref = oracle_grads(s, inp, dY)
    got = run_layer_backward(s, inp, dY, accumulate=True, init=0.5)
    for n in NAMES[1:]:
        assert_close(host64(got[n]), ref[n] + 0.5, what=f"accumulate {n}")
    assert_close(host64(got["dX"]), ref["dX"], what="dX with accumulate")


def test_layer_backward_rejects_sequence_parallel_plans():
    s = SMALL[0]
    cfg = tp.make_config(tokens=s.tokens, hidden=s.hidden, ffn=s.ffn, n_heads=s.heads,
                         n_kv_heads=s.kv_heads, head_dim=s.head_dim, tp_degree=s.tp, act=s.act,
                         reduce_mode=tp.TP_REDUCE_PARTIALS, batch=s.batch, seq=s.seq,
                         sequence_parallel=1)
    plan = tp.Plan(cfg)
    bf = dict(dtype=torch.bfloat16, device="cuda")
    X = torch.zeros(s.tokens, s.hidden, **bf)
    with pytest.raises(tp.TPError) as e:
        tp.tp_layer_backward(plan, X, {}, X.clone(), X.clone(), {}, False, None, 0)
    assert e.value.code in (tp.TP_ERR_UNSUPPORTED, tp.TP_ERR_INVALID_ARG)


def test_full_size_layer_backward_full_output():
    s = SHAPES["layer"]
    inp = synth.workload_inputs(s)
    dY = synth.grad_output(s)
    got = run_layer_backward(s, inp, dY)
    W = [host64(inp[k]) for k in ("Wq", "Wk", "Wv", "Wo", "W1", "W3", "W2")]
    ref = oracle.layer_backward_composed(s.batch, s.seq, s.heads, s.kv_heads, s.head_dim,
                                         host64(inp["X"]), *W, host64(dY))
    for n, r in zip(NAMES, ref):
        g = host64(got[n])
        e = assert_close(g, r, what=f"full-size layer {n}")
        report(f"layer backward {n}", max_rel=e, frac_beyond=elementwise_excess_fraction(g, r))
