"""GPU parity of the head-sharded attention block's backward against the
fp64 oracle, through the C ABI (tp_attn_forward_train, tp_attn_backward).

Small shapes compare every output with the oracle's literal t-device form
(the same dOut to every shard; dX the sum of the shards' partials; a
replicated KV head's weight gradient the sum over the shards holding it).
They cover head dimensions 64 and 128, GQA groups of 1 to 4, KV replicas
(k < t), ragged sequence lengths (not multiples of the 64-query or 128-key
blocks), sequences shorter than one key block and several batches.  At the
full size the bench runs (4 x 2048 tokens, h 4096, 32 query / 8 KV heads of
128, t 8) every output is compared with the oracle's composed form (numpy
projections, the C attention core; pinned equal to the all-C form)."""
import numpy as np
import pytest
import torch

import megatron_tensor_transformer_colwise_gb300 as tp
import oracle
import synth
from synth import Shape
from gpu_util import (assert_close, dev, elementwise_excess_fraction, host64, plan_for, report, sync_ok,
                      workspace)

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
    # head dimension 64
    Shape("ab_d64_gqa2", 2, 128, 256, heads=8, kv_heads=4, head_dim=64, tp=2, act="none", index=58),
    Shape("ab_d64_replica_ragged", 1, 200, 256, heads=4, kv_heads=1, head_dim=64, tp=4, act="none", index=59),
    Shape("ab_d64_group4_multi", 2, 320, 512, heads=16, kv_heads=4, head_dim=64, tp=4, act="none", index=60),
    Shape("ab_d64_short_t8", 3, 40, 256, heads=8, kv_heads=8, head_dim=64, tp=8, act="none", index=61),
]


@pytest.mark.parametrize("s", SMALL, ids=[s.name for s in SMALL])
def test_small_attention_backward_full_output(s):
    inp = synth.workload_inputs(s)
    dOut = synth.grad_output(s)
    got = run_backward(s, inp, dOut)
    ref = oracle_grads(s, inp, dOut)
    for n in ("dX", "dWq", "dWk", "dWv", "dWo"):
        assert_close(host64(got[n]), ref[n], what=f"{s.name} {n}")


# Long sequences: a 128-key block's CTA loops over up to 64 causal 64-query
# blocks per query head (the full-size case has 32), and 3000 tokens end in
# ragged query and key blocks at d = 64.
LONG = [
    Shape("ab_long_seq", 1, 4096, 256, heads=4, kv_heads=1, head_dim=128, tp=2, act="none", index=66),
    Shape("ab_d64_long_seq_ragged", 1, 3000, 256, heads=4, kv_heads=2, head_dim=64, tp=2, act="none", index=67),
]


@pytest.mark.parametrize("s", LONG, ids=[s.name for s in LONG])
def test_long_sequence_attention_backward_full_output(s):
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


def test_saved_state_must_be_all_or_nothing():
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
    sync_ok(plan)


def test_head_dim_64_recomputed_forward_state_gives_the_same_gradients():
    s = SMALL[7]
    inp = synth.workload_inputs(s)
    dOut = synth.grad_output(s)
    a = run_backward(s, inp, dOut, saved=True)
    b = run_backward(s, inp, dOut, saved=False)
    for n in ("dWk", "dWv", "dWo"):
        assert torch.equal(a[n], b[n]), n
    for n in ("dX", "dWq"):
        assert_close(host64(b[n]), host64(a[n]), tol=2e-3, what=n)


# The layer's attention block at full size (the configuration the bench times).
FULL = Shape("ab_full", 4, 2048, 4096, heads=32, kv_heads=8, head_dim=128, tp=8, act="none", index=57)


def test_full_size_attention_backward_full_output():
    s = FULL
    inp = synth.workload_inputs(s)
    dOut = synth.grad_output(s)
    got = run_backward(s, inp, dOut)
    ref = oracle.attention_backward_composed(s.batch, s.seq, s.heads, s.kv_heads,
                                             *(host64(inp[n]) for n in ("X", "Wq", "Wk", "Wv", "Wo")),
                                             host64(dOut))
    for n, r in zip(("dX", "dWq", "dWk", "dWv", "dWo"), ref):
        g = host64(got[n])
        e = assert_close(g, r, what=f"full-size {n}")
        report(f"attn backward {n}", max_rel=e, frac_beyond=elementwise_excess_fraction(g, r))
