"""GPU parity of the head-sharded attention block's backward against the
fp64 oracle, through the C ABI (tp_attn_forward_train, tp_attn_backward).

Small shapes compare every output with the oracle's literal t-device form
(the same dOut to every shard; dX the sum of the shards' partials; a
replicated KV head's weight gradient the sum over the shards holding it).
They cover GQA groups of 1 to 4, KV replicas (k < t), ragged sequence
lengths (not multiples of the 64-query or 128-key blocks), sequences shorter
than one key block and several batches.  At the full size the bench runs
(4 x 2048 tokens, h 4096, 32 query / 8 KV heads of 128, t 8), two slices
the oracle computes on their own are compared: the weight gradients of one
KV group (that group's heads alone are a smaller attention block with the
same gradients there), and dX on the rows of one sequence (sequences never
attend across each other)."""
import numpy as np
import pytest
import torch

import megatron_tensor_transformer_colwise_gb300 as tp
import oracle
import synth
from synth import Shape
from gpu_util import assert_close, dev, host64, plan_for, sync_ok, workspace

pytestmark = pytest.mark.gpu


def saved_buffers(plan):
    q, o, l = tp.tp_plan_attn_saved_bytes(plan)
    u8 = dict(dtype=torch.uint8, device="cuda")
    return (torch.empty(q, **u8).view(torch.bfloat16), torch.empty(o, **u8).view(torch.bfloat16),
            torch.empty(l, **u8).view(torch.float32))


def run_backward(s, inp, dOut, saved=True, accumulate=False, init=0.0):
    plan = plan_for(s)
    M, h, a, k, d = s.tokens, s.hidden, s.heads, s.kv_heads, s.head_dim
    X, Wq, Wk, Wv, Wo = (dev(inp[n]) for n in ("X", "Wq", "Wk", "Wv", "Wo"))
    QKV = O = LSE = None
    if saved:
        QKV, O, LSE = saved_buffers(plan)
        out = torch.empty(M, h, dtype=torch.bfloat16, device="cuda")
        tp.tp_attn_forward_train(plan, X, Wq, Wk, Wv, Wo, None, None, out, QKV, O, LSE)
    ws, nws = workspace(plan, tp.TP_OP_ATTN_BACKWARD)
    f32 = dict(dtype=torch.float32, device="cuda")
    dX = torch.empty(M, h, dtype=torch.bfloat16, device="cuda")
    dWq = torch.full((a * d, h), init, **f32)
    dWk = torch.full((k * d, h), init, **f32)
    dWv = torch.full((k * d, h), init, **f32)
    dWo = torch.full((h, a * d), init, **f32)
    tp.tp_attn_backward(plan, X, Wq, Wk, Wv, Wo, dev(dOut), QKV, O, LSE, dX, dWq, dWk, dWv, dWo,
                        accumulate, ws, nws)
    sync_ok(plan)
    return {n: v.cpu() for n, v in (("dX", dX), ("dWq", dWq), ("dWk", dWk), ("dWv", dWv), ("dWo", dWo))}


def oracle_grads(s, inp, dOut):
    out = oracle.attention_backward(s.batch, s.seq, s.heads, s.kv_heads,
                                    *(host64(inp[n]) for n in ("X", "Wq", "Wk", "Wv", "Wo")),
                                    host64(dOut), t=s.tp)
    return dict(zip(("dX", "dWq", "dWk", "dWv", "dWo"), out))


SMALL = [
    Shape("ab_gqa2", 2, 128, 256, heads=4, kv_heads=2, head_dim=128, tp=2, act="none", index=51),
    Shape("ab_replica", 1, 200, 256, heads=4, kv_heads=1, head_dim=128, tp=4, act="none", index=52),
    Shape("ab_mha_ragged", 2, 192, 128, heads=2, kv_heads=2, head_dim=128, tp=2, act="none", index=53),
    Shape("ab_short_t8", 3, 40, 256, heads=8, kv_heads=8, head_dim=128, tp=8, act="none", index=54),
    Shape("ab_group4", 1, 384, 512, heads=8, kv_heads=2, head_dim=128, tp=4, act="none", index=55),
]


@pytest.mark.parametrize("s", SMALL, ids=[s.name for s in SMALL])
def test_small_attention_backward_full_output(s):
    inp = synth.workload_inputs(s)
    dOut = synth.grad_output(s)
    got = run_backward(s, inp, dOut)
    ref = oracle_grads(s, inp, dOut)
    for n in ("dX", "dWq", "dWk", "dWv", "dWo"):
        assert_close(host64(got[n]), ref[n], what=f"{s.name} {n}")


def test_recomputed_forward_state_gives_the_same_gradients():
    # With QKV, O and LSE recomputed the inputs of every kernel are the same
    # values; only the order of the fp32 dQ additions differs.
    s = SMALL[4]
    inp = synth.workload_inputs(s)
    dOut = synth.grad_output(s)
    a = run_backward(s, inp, dOut, saved=True)
    b = run_backward(s, inp, dOut, saved=False)
    for n in ("dWk", "dWv", "dWo"):
        assert torch.equal(a[n], b[n]), n
    for n in ("dX", "dWq"):
        assert_close(host64(b[n]), host64(a[n]), tol=2e-3, what=n)


def test_accumulate_adds_to_the_weight_gradients():
    s = SMALL[0]
    inp = synth.workload_inputs(s)
    dOut = synth.grad_output(s)
    ref = oracle_grads(s, inp, dOut)
    got = run_backward(s, inp, dOut, accumulate=True, init=-0.25)
    for n in ("dWq", "dWk", "dWv", "dWo"):
        assert_close(host64(got[n]), ref[n] - 0.25, what=f"accumulate {n}")
    assert_close(host64(got["dX"]), ref["dX"], what="dX with accumulate")


def test_saved_state_must_be_all_or_nothing_and_head_dim_128():
    s = SMALL[0]
    plan = plan_for(s)
    QKV, O, LSE = saved_buffers(plan)
    ws, nws = workspace(plan, tp.TP_OP_ATTN_BACKWARD)
    M, h, a, k, d = s.tokens, s.hidden, s.heads, s.kv_heads, s.head_dim
    bf = dict(dtype=torch.bfloat16, device="cuda")
    f32 = dict(dtype=torch.float32, device="cuda")
    X, dOut, dX = (torch.zeros(M, h, **bf) for _ in range(3))
    Wq, Wk, Wv = torch.zeros(a * d, h, **bf), torch.zeros(k * d, h, **bf), torch.zeros(k * d, h, **bf)
    Wo = torch.zeros(h, a * d, **bf)
    grads = (torch.zeros(a * d, h, **f32), torch.zeros(k * d, h, **f32), torch.zeros(k * d, h, **f32),
             torch.zeros(h, a * d, **f32))
    with pytest.raises(tp.TPError) as e:
        tp.tp_attn_backward(plan, X, Wq, Wk, Wv, Wo, dOut, QKV, None, LSE, dX, *grads, False, ws, nws)
    assert e.value.code == tp.TP_ERR_INVALID_ARG
    s64 = Shape("ab_d64", 1, 64, 128, heads=2, kv_heads=2, head_dim=64, tp=2, act="none", index=56)
    p64 = plan_for(s64)
    ws64, n64 = workspace(p64, tp.TP_OP_ATTN_BACKWARD)
    with pytest.raises(tp.TPError) as e:
        tp.tp_attn_backward(p64, torch.zeros(64, 128, **bf), torch.zeros(128, 128, **bf),
                            torch.zeros(128, 128, **bf), torch.zeros(128, 128, **bf),
                            torch.zeros(128, 128, **bf), torch.zeros(64, 128, **bf), None, None, None,
                            torch.zeros(64, 128, **bf), torch.zeros(128, 128, **f32),
                            torch.zeros(128, 128, **f32), torch.zeros(128, 128, **f32),
                            torch.zeros(128, 128, **f32), False, ws64, n64)
    assert e.value.code == tp.TP_ERR_UNSUPPORTED
    sync_ok(plan)


# The layer's attention block at full size (the configuration the bench times).
FULL = Shape("ab_full", 4, 2048, 4096, heads=32, kv_heads=8, head_dim=128, tp=8, act="none", index=57)


def test_full_size_attention_backward_slices():
    s = FULL
    inp = synth.workload_inputs(s)
    dOut = synth.grad_output(s)
    got = run_backward(s, inp, dOut)
    a, k, d = s.heads, s.kv_heads, s.head_dim
    G = a // k
    X, Wq, Wk, Wv, Wo = (host64(inp[n]) for n in ("X", "Wq", "Wk", "Wv", "Wo"))
    dO64 = host64(dOut)
    # (1) KV group 0 alone: query heads 0..G-1 and KV head 0.
    qr = slice(0, G * d)
    _, rWq, rWk, rWv, rWo = oracle.attention_backward_composed(
        s.batch, s.seq, G, 1, X, Wq[qr], Wk[:d], Wv[:d], Wo[:, qr], dO64)
    assert_close(host64(got["dWq"])[qr], rWq, what="full-size dWq, group 0")
    assert_close(host64(got["dWk"])[:d], rWk, what="full-size dWk, head 0")
    assert_close(host64(got["dWv"])[:d], rWv, what="full-size dWv, head 0")
    assert_close(host64(got["dWo"])[:, qr], rWo, what="full-size dWo, group 0")
    # (2) dX on the rows of the last sequence: that sequence alone.
    rows = slice((s.batch - 1) * s.seq, s.batch * s.seq)
    rdX = oracle.attention_backward_composed(1, s.seq, a, k, X[rows], Wq, Wk, Wv, Wo, dO64[rows])[0]
    assert_close(host64(got["dX"])[rows], rdX, what="full-size dX, last sequence")
