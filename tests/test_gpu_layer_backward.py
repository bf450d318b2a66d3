"""GPU parity of the pre-norm layer's backward (tp_layer_backward: the
forward recomputed with its state kept, the MLP block's backward, RMSNorm's
backward with the residual, the attention block's backward, RMSNorm again)
against the fp64 oracle through the C ABI.

Small layers and the full size the bench runs (4 x 2048 tokens, h 4096,
f 14336, 32 query / 8 KV heads of 128, t 8) compare every output: dX and
all seven weight gradients.  At full size the oracle runs in its composed
form (numpy matrix products, the C attention core and norms; pinned equal to
the all-C definition).  The sequence-parallel layer ("시퀀스 병렬화") takes
X, dY and dX in the split layout [t][batch][seq/t][h] and is compared with
oracle.layer_sp_backward."""
import numpy as np
import pytest
import torch

import megatron_tensor_transformer_colwise_gb300 as tp
import oracle
import synth
from synth import SHAPES, Shape
import full_refs
from gpu_util import (assert_close, dev, elementwise_excess_fraction, host64, plan_for, report,
                      sync_ok, workspace)

pytestmark = pytest.mark.gpu

NAMES = ["dX", "dWq", "dWk", "dWv", "dWo", "dW1", "dW3", "dW2"]


def sp_plan(s, mode=tp.TP_REDUCE_FUSED):
    return tp.Plan(tp.make_config(tokens=s.tokens, hidden=s.hidden, ffn=s.ffn, n_heads=s.heads,
                                  n_kv_heads=s.kv_heads, head_dim=s.head_dim, tp_degree=s.tp, act=s.act,
                                  reduce_mode=mode, batch=s.batch, seq=s.seq, sequence_parallel=1))


def run_layer_backward(s, inp, dY, accumulate=False, init=0.0, plan=None):
    plan = plan_for(s) if plan is None else plan
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
    Shape("lb_d64", 2, 128, 256, ffn=512, heads=8, kv_heads=2, head_dim=64, tp=4, act="swiglu", index=63),
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


def _split(x, s):
    """Token-order tensor -> the sequence-split layout (oracle's row map)."""
    return torch.from_numpy(oracle.sp_split(s.batch, s.seq, s.tp, host64(x))).to(x.dtype)


@pytest.mark.parametrize("mode", [tp.TP_REDUCE_PARTIALS, tp.TP_REDUCE_FUSED], ids=["partials", "fused"])
def test_small_sequence_parallel_layer_backward_full_output(mode):
    s = SMALL[0]
    inp = synth.workload_inputs(s)
    dY = synth.grad_output(s)
    X_sp, dY_sp = _split(inp["X"], s), _split(dY, s)
    got = run_layer_backward(s, dict(inp, X=X_sp), dY_sp, plan=sp_plan(s, mode))
    args = [host64(inp[k]) for k in ("Wq", "Wk", "Wv", "Wo", "W1", "W3", "W2")]
    ref = dict(zip(NAMES, oracle.layer_sp_backward(s.batch, s.seq, s.heads, s.kv_heads, s.head_dim, s.tp,
                                                   host64(X_sp), *args, host64(dY_sp))))
    for n in NAMES:
        assert_close(host64(got[n]), ref[n], what=f"SP {n}")
    # dX is the replicated layer's, in the split layout
    rep = run_layer_backward(s, inp, dY)
    assert torch.equal(got["dX"].view(torch.int16), _split(rep["dX"], s).view(torch.int16))


def test_full_size_layer_backward_full_output():
    s = SHAPES["layer"]
    inp, dY, ref = full_refs.layer_backward()
    got = run_layer_backward(s, inp, dY)
    for n, r in zip(NAMES, ref):
        g = host64(got[n])
        e = assert_close(g, r, what=f"full-size layer {n}")
        report(f"layer backward {n}", max_rel=e, frac_beyond=elementwise_excess_fraction(g, r))


def test_full_size_sequence_parallel_layer_backward_full_output():
    # The split layout only permutes token rows: the reference is the
    # replicated layer's backward with dX split (oracle.layer_sp_backward's
    # definition, on the cached full-size result).
    s = SHAPES["layer"]
    inp, dY, ref = full_refs.layer_backward()
    X_sp, dY_sp = _split(inp["X"], s), _split(dY, s)
    got = run_layer_backward(s, dict(inp, X=X_sp), dY_sp, plan=sp_plan(s))
    ref = [oracle.sp_split(s.batch, s.seq, s.tp, ref[0])] + list(ref[1:])
    for n, r in zip(NAMES, ref):
        g = host64(got[n])
        e = assert_close(g, r, what=f"full-size SP layer {n}")
        report(f"sp layer backward {n}", max_rel=e, frac_beyond=elementwise_excess_fraction(g, r))
