"""GPU parity at the edges of the configuration space, through the C ABI:
a single token, t = 1 (no sharding) and the largest t the plan accepts
(64), the attention backward at seq = 1 (where it has a closed form), and a
layer of one-token sequences.  Each is compared with the fp64 oracle."""
import numpy as np
import pytest
import torch

import megatron_tensor_transformer_colwise_gb300 as tp
import oracle
import synth
from synth import Shape
from gpu_util import assert_close, dev, host64, plan_for, sync_ok, workspace

pytestmark = pytest.mark.gpu

EDGE_MLP = [
    Shape("one_token_t64", 1, 1, 64, ffn=512, tp=64, act="gelu", index=71),
    Shape("one_token_t1", 1, 1, 128, ffn=256, tp=1, act="swiglu", index=72),
    Shape("t1", 1, 3, 96, ffn=192, tp=1, act="gelu", index=73),
    Shape("t16", 1, 17, 64, ffn=1024, tp=16, act="swiglu", index=74),
    Shape("t64_swiglu", 1, 33, 128, ffn=1024, tp=64, act="swiglu", index=75),
]


@pytest.mark.parametrize("mode", [tp.TP_REDUCE_FUSED, tp.TP_REDUCE_PARTIALS])
@pytest.mark.parametrize("s", EDGE_MLP, ids=[s.name for s in EDGE_MLP])
def test_mlp_forward_edges(s, mode):
    inp = synth.workload_inputs(s)
    plan = plan_for(s, reduce_mode=mode)
    ws, nws = workspace(plan, tp.TP_OP_MLP)
    Z = torch.empty(s.tokens, s.hidden, dtype=torch.bfloat16, device="cuda")
    P = torch.empty(s.tp, s.tokens, s.hidden, dtype=torch.float32, device="cuda") \
        if mode == tp.TP_REDUCE_PARTIALS else None
    W3 = dev(inp["W3"]) if s.act == "swiglu" else None
    tp.tp_mlp_forward(plan, dev(inp["X"]), dev(inp["W1"]), W3, dev(inp["W2"]), None, None, P, Z, ws, nws)
    sync_ok(plan)
    ref = oracle.mlp_sharded(s.act, s.tp, host64(inp["X"]), host64(inp["W1"]), host64(inp["W2"]),
                             host64(inp["W3"]) if s.act == "swiglu" else None)
    assert_close(host64(Z), ref, what=s.name)


@pytest.mark.parametrize("s", [EDGE_MLP[1], EDGE_MLP[3], EDGE_MLP[4]], ids=["one_token_t1", "t16", "t64"])
def test_mlp_backward_edges(s):
    inp = synth.workload_inputs(s)
    dZ = synth.grad_output(s)
    plan = plan_for(s)
    glu = s.act == "swiglu"
    M, h, f = s.tokens, s.hidden, s.ffn
    ws, nws = workspace(plan, tp.TP_OP_MLP_BACKWARD)
    f32 = dict(dtype=torch.float32, device="cuda")
    dX = torch.empty(M, h, dtype=torch.bfloat16, device="cuda")
    dW1, dW2 = torch.empty(f, h, **f32), torch.empty(h, f, **f32)
    dW3 = torch.empty(f, h, **f32) if glu else None
    db2 = torch.empty(h, **f32)
    tp.tp_mlp_backward(plan, dev(inp["X"]), dev(inp["W1"]), dev(inp["W3"]) if glu else None,
                       dev(inp["W2"]), dev(dZ), None, dX, dW1, dW3, dW2, db2, False, ws, nws)
    sync_ok(plan)
    ref = oracle.mlp_backward(s.act, host64(inp["X"]), host64(inp["W1"]), host64(inp["W2"]), host64(dZ),
                              host64(inp["W3"]) if glu else None, t=s.tp)
    for name, got, r in zip(("dX", "dW1", "dW3", "dW2", "db2"), (dX, dW1, dW3, dW2, db2), ref):
        if r is not None:
            assert_close(host64(got), r, what=f"{s.name} {name}")


def test_attention_backward_single_position_sequences():
    # seq = 1: each query sees only itself, P = 1, dS = 0, so dQ and dK
    # vanish and dV is the sum of dO over the group's query heads.
    s = Shape("seq1", 3, 1, 256, heads=4, kv_heads=2, head_dim=128, tp=2, act="none", index=76)
    inp = synth.workload_inputs(s)
    dOut = synth.grad_output(s)
    plan = plan_for(s)
    M, h, a, k, d = s.tokens, s.hidden, s.heads, s.kv_heads, s.head_dim
    ws, nws = workspace(plan, tp.TP_OP_ATTN_BACKWARD)
    f32 = dict(dtype=torch.float32, device="cuda")
    dX = torch.empty(M, h, dtype=torch.bfloat16, device="cuda")
    dWq, dWk = torch.empty(a * d, h, **f32), torch.empty(k * d, h, **f32)
    dWv, dWo = torch.empty(k * d, h, **f32), torch.empty(h, a * d, **f32)
    tp.tp_attn_backward(plan, dev(inp["X"]), dev(inp["Wq"]), dev(inp["Wk"]), dev(inp["Wv"]), dev(inp["Wo"]),
                        dev(dOut), None, None, None, dX, dWq, dWk, dWv, dWo, False, ws, nws)
    sync_ok(plan)
    ref = oracle.attention_backward(s.batch, s.seq, a, k, *(host64(inp[n]) for n in ("X", "Wq", "Wk", "Wv", "Wo")),
                                    host64(dOut), t=s.tp)
    rdX, rdWq, rdWk, rdWv, rdWo = ref
    assert np.abs(rdWq).max() == 0 and np.abs(rdWk).max() == 0  # the oracle's closed form
    for name, got, r in (("dX", dX, rdX), ("dWv", dWv, rdWv), ("dWo", dWo, rdWo)):
        assert_close(host64(got), r, what=f"seq1 {name}")
    # On the GPU dS = P (dP - D) is a difference of two fp32 sums of the
    # same value taken in different orders: zero up to rounding.
    scale = np.abs(rdWv).max()
    for name, got in (("dWq", dWq), ("dWk", dWk)):
        assert np.abs(host64(got)).max() <= 1e-3 * scale, f"{name} must vanish at seq = 1"


def test_layer_of_one_token_sequences():
    s = Shape("layer_seq1", 4, 1, 128, ffn=256, heads=4, kv_heads=2, head_dim=64, tp=2, act="swiglu", index=77)
    inp = synth.workload_inputs(s)
    plan = plan_for(s)
    ws, nws = workspace(plan, tp.TP_OP_LAYER)
    Y = torch.empty(s.tokens, s.hidden, dtype=torch.bfloat16, device="cuda")
    tp.tp_layer_forward(plan, dev(inp["X"]), {k: dev(v) for k, v in inp.items() if k != "X"}, Y, ws, nws)
    sync_ok(plan)
    ref = oracle.layer(s.batch, s.seq, s.heads, s.kv_heads, s.head_dim, s.tp,
                       *(host64(inp[n]) for n in ("X", "Wq", "Wk", "Wv", "Wo", "W1", "W3", "W2")), sharded=True)
    assert_close(host64(Y), ref, what="layer of one-token sequences")
