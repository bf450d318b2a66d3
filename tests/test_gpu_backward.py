"""GPU parity of the sharded MLP's backward pass against the fp64 oracle,
through the C ABI (tp_mlp_forward_train, tp_mlp_backward).

The oracle's reference is its literal t-device form: g's backward is the
identity (every shard reads the same dZ), f's backward the sum of the t
partial input gradients.  Small shapes are compared over every output;
ragged token counts, hidden sizes below one tile, and an ffn size whose
W1/W3 boundary falls inside a 256-row weight-gradient tile are included.
At the full size the bench times (8192 tokens, h 4096, f 14336, t 8) every
output is compared with the oracle's composed form (numpy matrix products;
pinned equal to the all-C definition)."""
import numpy as np
import pytest
import torch

import megatron_tensor_transformer_colwise_gb300 as tp
import oracle
import synth
from synth import Shape
from gpu_util import (assert_close, dev, elementwise_excess_fraction, host64, plan_for, report,
                      sync_ok, workspace)

pytestmark = pytest.mark.gpu


def run_backward(s, inp, dZ, saved, accumulate=False, init=0.0, want_db2=True):
    plan = plan_for(s)
    glu = s.act == "swiglu"
    M, h, f = s.tokens, s.hidden, s.ffn
    X, W1, W2 = dev(inp["X"]), dev(inp["W1"]), dev(inp["W2"])
    W3 = dev(inp["W3"]) if glu else None
    UG = None
    if saved:
        fws, nf = workspace(plan, tp.TP_OP_MLP)
        Z = torch.empty(M, h, dtype=torch.bfloat16, device="cuda")
        UG = torch.empty(M, (2 if glu else 1) * f, dtype=torch.bfloat16, device="cuda")
        tp.tp_mlp_forward_train(plan, X, W1, W3, W2, None, None, None, Z, UG, fws, nf)
    ws, nws = workspace(plan, tp.TP_OP_MLP_BACKWARD)
    f32 = dict(dtype=torch.float32, device="cuda")
    dX = torch.empty(M, h, dtype=torch.bfloat16, device="cuda")
    dW1 = torch.full((f, h), init, **f32)
    dW3 = torch.full((f, h), init, **f32) if glu else None
    dW2 = torch.full((h, f), init, **f32)
    db2 = torch.full((h,), init, **f32) if want_db2 else None
    tp.tp_mlp_backward(plan, X, W1, W3, W2, dev(dZ), UG, dX, dW1, dW3, dW2, db2, accumulate,
                       ws, nws)
    sync_ok(plan)
    out = {"dX": dX, "dW1": dW1, "dW3": dW3, "dW2": dW2, "db2": db2}
    return {k: (None if v is None else v.cpu()) for k, v in out.items()}


def oracle_grads(s, inp, dZ, t=None):
    glu = s.act == "swiglu"
    dX, dW1, dW3, dW2, db2 = oracle.mlp_backward(
        s.act, host64(inp["X"]), host64(inp["W1"]), host64(inp["W2"]), host64(dZ),
        host64(inp["W3"]) if glu else None, t=s.tp if t is None else t)
    return {"dX": dX, "dW1": dW1, "dW3": dW3, "dW2": dW2, "db2": db2}


SMALL = [
    Shape("bwd_gelu", 1, 300, 192, ffn=512, tp=4, act="gelu", index=41),
    Shape("bwd_tanh", 1, 260, 256, ffn=384, tp=2, act="gelu_tanh", index=42),
    Shape("bwd_none", 1, 129, 128, ffn=256, tp=2, act="none", index=43),
    Shape("bwd_swiglu", 1, 300, 192, ffn=512, tp=4, act="swiglu", index=44),
    # W1/W3 boundary at weight-gradient row 320 (inside a 256-row tile), t = 5
    Shape("bwd_swiglu_t5", 1, 200, 256, ffn=320, tp=5, act="swiglu", index=45),
    Shape("bwd_swiglu_multi", 1, 700, 512, ffn=1024, tp=8, act="swiglu", index=46),
]


@pytest.mark.parametrize("saved", [True, False], ids=["saved", "recompute"])
@pytest.mark.parametrize("s", SMALL, ids=[s.name for s in SMALL])
def test_small_mlp_backward_full_output(s, saved):
    inp = synth.workload_inputs(s)
    dZ = synth.grad_output(s)
    got = run_backward(s, inp, dZ, saved)
    ref = oracle_grads(s, inp, dZ)
    for k in ("dX", "dW1", "dW3", "dW2", "db2"):
        if ref[k] is None or got[k] is None:
            continue
        assert_close(host64(got[k]), ref[k], what=f"{s.name} {k}")


def test_saved_and_recomputed_pre_activations_agree():
    # dU and dG come from the same bf16 pre-activations either way, so dX,
    # dW1, dW3 are bit-identical; H differs by one rounding (the recompute
    # path writes H from the fp32 accumulator), so dW2 is only close.
    s = SMALL[3]
    inp = synth.workload_inputs(s)
    dZ = synth.grad_output(s)
    a = run_backward(s, inp, dZ, saved=True)
    b = run_backward(s, inp, dZ, saved=False)
    for k in ("dX", "dW1", "dW3", "db2"):
        assert torch.equal(a[k], b[k]), k
    assert_close(host64(a["dW2"]), host64(b["dW2"]), tol=1e-2, what="dW2")


def test_accumulate_adds_to_the_weight_gradients():
    s = SMALL[0]
    inp = synth.workload_inputs(s)
    dZ = synth.grad_output(s)
    ref = oracle_grads(s, inp, dZ)
    got = run_backward(s, inp, dZ, saved=True, accumulate=True, init=1.5)
    for k in ("dW1", "dW2", "db2"):
        assert_close(host64(got[k]), ref[k] + 1.5, what=f"accumulate {k}")
    assert_close(host64(got["dX"]), ref["dX"], what="dX with accumulate")


def test_plain_and_sharded_oracle_agree_on_gpu_inputs():
    # The GPU result is compared with the t-device oracle above; the oracle's
    # t-device and unsharded forms agree on the same bf16 inputs.
    s = SMALL[3]
    inp = synth.workload_inputs(s)
    dZ = synth.grad_output(s)
    a = oracle_grads(s, inp, dZ)
    b = oracle_grads(s, inp, dZ, t=0)
    for k in ("dX", "dW1", "dW3", "dW2", "db2"):
        assert np.abs(a[k] - b[k]).max() <= 1e-10 * np.abs(b[k]).max()


def test_bad_arguments_are_rejected_before_any_launch():
    s = SMALL[3]
    plan = plan_for(s)
    ws, nws = workspace(plan, tp.TP_OP_MLP_BACKWARD)
    M, h, f = s.tokens, s.hidden, s.ffn
    bf = dict(dtype=torch.bfloat16, device="cuda")
    X, W1, W3 = torch.zeros(M, h, **bf), torch.zeros(f, h, **bf), torch.zeros(f, h, **bf)
    W2, dZ, dX = torch.zeros(h, f, **bf), torch.zeros(M, h, **bf), torch.zeros(M, h, **bf)
    g = torch.zeros(f, h, dtype=torch.float32, device="cuda")
    g2 = torch.zeros(h, f, dtype=torch.float32, device="cuda")
    with pytest.raises(tp.TPError) as e:  # SwiGLU without dW3
        tp.tp_mlp_backward(plan, X, W1, W3, W2, dZ, None, dX, g, None, g2, None, False, ws, nws)
    assert e.value.code == tp.TP_ERR_INVALID_ARG
    with pytest.raises(tp.TPError) as e:  # workspace too small
        tp.tp_mlp_backward(plan, X, W1, W3, W2, dZ, None, dX, g, g.clone(), g2, None, False, ws,
                           nws - 256)
    assert e.value.code == tp.TP_ERR_WORKSPACE
    # f % 64 != 0 is unsupported for SwiGLU
    s2 = Shape("odd", 1, 64, 64, ffn=96, tp=2, act="swiglu", index=47)
    p2 = plan_for(s2)
    ws2, n2 = workspace(p2, tp.TP_OP_MLP_BACKWARD)
    X2, W12 = torch.zeros(64, 64, **bf), torch.zeros(96, 64, **bf)
    with pytest.raises(tp.TPError) as e:
        tp.tp_mlp_backward(p2, X2, W12, W12.clone(), torch.zeros(64, 96, **bf), X2.clone(), None,
                           X2.clone(), torch.zeros(96, 64, dtype=torch.float32, device="cuda"),
                           torch.zeros(96, 64, dtype=torch.float32, device="cuda"),
                           torch.zeros(64, 96, dtype=torch.float32, device="cuda"), None, False,
                           ws2, n2)
    assert e.value.code == tp.TP_ERR_UNSUPPORTED
    sync_ok(plan)


# The full-size MLP the layer bench runs: 8192 tokens, h 4096, f 14336, t 8.
FULL = Shape("bwd_full", 4, 2048, 4096, ffn=14336, tp=8, act="swiglu", index=48)


def test_full_size_backward_full_output():
    s = FULL
    inp = synth.workload_inputs(s)
    dZ = synth.grad_output(s)
    got = run_backward(s, inp, dZ, saved=True)
    ref = oracle.mlp_backward_composed(*(host64(inp[k]) for k in ("X", "W1", "W2")), host64(dZ),
                                       host64(inp["W3"]))
    for name, r in zip(("dX", "dW1", "dW3", "dW2", "db2"), ref):
        g = host64(got[name])
        e = assert_close(g, r, what=f"full-size {name}")
        report(f"mlp backward {name}", max_rel=e, frac_beyond=elementwise_excess_fraction(g, r))
