"""GPU parity of the whole blocks (sharded MLP, head-sharded attention, the
layer) against the fp64 oracle, through the C ABI.

Small shapes and the workloads' full sizes (the configuration the bench
times: FUSED reduction) are compared element by element over the whole
output.  At full size the oracle runs in its composed form (numpy matrix
products; pinned equal to the all-C definitions).  The layer is checked on y
and on the blocks' own contribution y - x (see
gpu_util.assert_layer_contribution_close)."""
import numpy as np
import pytest
import torch

import megatron_tensor_transformer_colwise_gb300 as tp
import oracle
import synth
from synth import SHAPES, Shape
import full_refs
from gpu_util import (assert_close, assert_layer_contribution_close, dev, elementwise_excess_fraction,
                      host64, plan_for, report, sync_ok, workspace)

pytestmark = pytest.mark.gpu

MODES = [tp.TP_REDUCE_FUSED, tp.TP_REDUCE_PARTIALS]


def run_mlp(s, inp, mode, partial_dtype=tp.TP_F32, bias=None, residual=None):
    plan = plan_for(s, reduce_mode=mode, partial_dtype=partial_dtype)
    ws, nws = workspace(plan, tp.TP_OP_MLP)
    Z = torch.empty(s.tokens, s.hidden, dtype=torch.bfloat16, device="cuda")
    P = None
    if mode == tp.TP_REDUCE_PARTIALS:
        dt = torch.float32 if partial_dtype == tp.TP_F32 else torch.bfloat16
        P = torch.empty(s.tp, s.tokens, s.hidden, dtype=dt, device="cuda")
    W3 = dev(inp["W3"]) if s.act == "swiglu" else None
    tp.tp_mlp_forward(plan, dev(inp["X"]), dev(inp["W1"]), W3, dev(inp["W2"]), bias, residual, P,
                      Z, ws, nws)
    sync_ok(plan)
    return host64(Z)


# ---------------------------------------------------------------- MLP

def test_worked_example_shapes_through_the_bf16_path():
    # The page's worked example (b=4, h=16, t=4, seed 0) rounded to bf16 and
    # run through the GPU path; compared with the oracle on the same values.
    w = synth.worked_example()
    s = SHAPES["worked"]
    inp = {"X": w["X"].to(torch.bfloat16), "W1": w["A"].T.contiguous().to(torch.bfloat16),
           "W2": w["B"].T.contiguous().to(torch.bfloat16)}
    for mode in MODES:
        Z = run_mlp(s, inp, mode)
        ref = oracle.mlp("gelu", host64(inp["X"]), host64(inp["W1"]), host64(inp["W2"]))
        assert_close(Z, ref, what="worked example")
        # and the oracle's own sharded form agrees with its unsharded one
        refs = oracle.mlp_sharded("gelu", 4, host64(inp["X"]), host64(inp["W1"]), host64(inp["W2"]))
        assert np.abs(refs - ref).max() < 1e-12 * np.abs(ref).max()


@pytest.mark.parametrize("act", ["gelu", "swiglu", "gelu_tanh"])
@pytest.mark.parametrize("mode", MODES)
def test_small_mlp_full_output(act, mode):
    s = Shape("m", 1, 300, 192, ffn=800, tp=4, act=act, index=21)
    inp = synth.workload_inputs(s)
    Z = run_mlp(s, inp, mode)
    w3 = host64(inp["W3"]) if act == "swiglu" else None
    ref = oracle.mlp_sharded(act, s.tp, host64(inp["X"]), host64(inp["W1"]), host64(inp["W2"]), w3)
    assert_close(Z, ref, what=f"mlp {act}")


def test_mlp_bias_and_residual_added_once():
    s = Shape("m", 1, 130, 64, ffn=256, tp=4, act="gelu", index=22)
    inp = synth.workload_inputs(s)
    bias = synth.normal_bf16((s.hidden,), 1.0, 5)
    res = synth.normal_bf16((s.tokens, s.hidden), 1.0, 6)
    ref = oracle.mlp("gelu", host64(inp["X"]), host64(inp["W1"]), host64(inp["W2"]))
    ref = ref + host64(bias)[None, :] + host64(res)
    for mode in MODES:
        Z = run_mlp(s, inp, mode, bias=dev(bias), residual=dev(res))
        assert_close(Z, ref, what="mlp + bias + residual")


def test_mlp_bf16_partials_mode():
    s = Shape("m", 1, 257, 256, ffn=1024, tp=8, act="swiglu", index=23)
    inp = synth.workload_inputs(s)
    Z = run_mlp(s, inp, tp.TP_REDUCE_PARTIALS, partial_dtype=tp.TP_BF16)
    ref = oracle.mlp("swiglu", host64(inp["X"]), host64(inp["W1"]), host64(inp["W2"]),
                     host64(inp["W3"]))
    assert_close(Z, ref, what="mlp bf16 partials")


@pytest.mark.parametrize("name", ["gpt_mlp", "llama_mlp"])
def test_full_size_mlp_full_output(name):
    s = SHAPES[name]
    inp = synth.workload_inputs(s)
    Z = run_mlp(s, inp, tp.TP_REDUCE_FUSED)
    w3 = host64(inp["W3"]) if s.act == "swiglu" else None
    if name == "gpt_mlp":   # 34 GFLOP: the plain C loops
        ref = oracle.mlp(s.act, host64(inp["X"]), host64(inp["W1"]), host64(inp["W2"]), w3)
    else:
        ref = oracle.mlp_composed(s.act, host64(inp["X"]), host64(inp["W1"]), host64(inp["W2"]), w3)
    e = assert_close(Z, ref, what=f"{name} full output")
    report(f"{name} forward", max_rel=e, frac_beyond=elementwise_excess_fraction(Z, ref))


# ---------------------------------------------------------------- attention

def run_attn(s, inp, mode, residual=None):
    plan = plan_for(s, reduce_mode=mode)
    ws, nws = workspace(plan, tp.TP_OP_ATTN)
    out = torch.empty(s.tokens, s.hidden, dtype=torch.bfloat16, device="cuda")
    P = torch.empty(s.tp, s.tokens, s.hidden, dtype=torch.float32, device="cuda") \
        if mode == tp.TP_REDUCE_PARTIALS else None
    tp.tp_attn_forward(plan, dev(inp["X"]), dev(inp["Wq"]), dev(inp["Wk"]), dev(inp["Wv"]),
                       dev(inp["Wo"]), residual, P, out, ws, nws)
    sync_ok(plan)
    return host64(out)


@pytest.mark.parametrize("a,k,t,d", [(8, 2, 4, 64), (8, 8, 4, 128), (8, 1, 8, 128), (4, 4, 2, 64)])
@pytest.mark.parametrize("mode", MODES)
def test_small_attention_block_full_output(a, k, t, d, mode):
    s = Shape("a", 2, 150, 256, heads=a, kv_heads=k, head_dim=d, tp=t, act="none", index=24)
    inp = synth.workload_inputs(s)
    out = run_attn(s, inp, mode)
    ref = oracle.attention_sharded(s.batch, s.seq, a, k, d, t, *(host64(inp[n]) for n in
                                                                  ("X", "Wq", "Wk", "Wv", "Wo")))
    assert_close(out, ref, what="attention block")


def test_attention_block_residual():
    s = Shape("a", 1, 96, 128, heads=4, kv_heads=2, head_dim=64, tp=2, act="none", index=25)
    inp = synth.workload_inputs(s)
    res = synth.normal_bf16((s.tokens, s.hidden), 1.0, 9)
    ref = oracle.attention(s.batch, s.seq, 4, 2, 64, *(host64(inp[n]) for n in
                                                       ("X", "Wq", "Wk", "Wv", "Wo"))) + host64(res)
    for mode in MODES:
        assert_close(run_attn(s, inp, mode, residual=dev(res)), ref, what="attention + residual")


def test_full_size_attention_full_output():
    s = SHAPES["attn"]
    inp = synth.workload_inputs(s)
    out = run_attn(s, inp, tp.TP_REDUCE_FUSED)
    ref = oracle.attention_composed(s.batch, s.seq, s.heads, s.kv_heads, s.head_dim,
                                    *(host64(inp[n]) for n in ("X", "Wq", "Wk", "Wv", "Wo")))
    e = assert_close(out, ref, what="attention block full output")
    report("attn forward", max_rel=e, frac_beyond=elementwise_excess_fraction(out, ref))


# ---------------------------------------------------------------- layer

def run_layer(s, inp, mode):
    plan = plan_for(s, reduce_mode=mode)
    ws, nws = workspace(plan, tp.TP_OP_LAYER)
    Y = torch.empty(s.tokens, s.hidden, dtype=torch.bfloat16, device="cuda")
    wd = {k: dev(v) for k, v in inp.items() if k != "X"}
    tp.tp_layer_forward(plan, dev(inp["X"]), wd, Y, ws, nws)
    sync_ok(plan)
    return host64(Y)


# h = 200 leaves a partial last k-block in the GEMMs over h (their loads past
# column 200 read zeros) and a row of 25 16-byte vectors for the pass that
# takes the row statistics of x (FUSED folds the norm into the GEMMs).
@pytest.mark.parametrize("s", [Shape("l", 2, 140, 256, ffn=768, heads=8, kv_heads=2, head_dim=64, tp=4,
                                     act="swiglu", index=26),
                               Shape("l_ragged_k", 2, 130, 200, ffn=384, heads=4, kv_heads=2, head_dim=64,
                                     tp=2, act="swiglu", index=29)], ids=["h256", "h200"])
@pytest.mark.parametrize("mode", MODES)
def test_small_layer_full_output(mode, s):
    inp = synth.workload_inputs(s)
    Y = run_layer(s, inp, mode)
    ref = oracle.layer(s.batch, s.seq, s.heads, s.kv_heads, s.head_dim, s.tp,
                       *(host64(inp[n]) for n in ("X", "Wq", "Wk", "Wv", "Wo", "W1", "W3", "W2")),
                       sharded=True)
    assert_close(Y, ref, what="layer")
    # The residual stream dominates y; check the block contributions too.
    X = host64(inp["X"])
    xn = oracle.rmsnorm(X)
    h1 = X + oracle.attention_sharded(s.batch, s.seq, s.heads, s.kv_heads, s.head_dim, s.tp, xn,
                                      *(host64(inp[n]) for n in ("Wq", "Wk", "Wv", "Wo")))
    assert_layer_contribution_close(Y, ref, X, h1, what=f"layer contribution ({mode})")


@pytest.mark.parametrize("s", [Shape("l_det", 2, 300, 640, ffn=1280, heads=10, kv_heads=2, head_dim=64, tp=2,
                                     act="swiglu", index=27), SHAPES["layer"]], ids=["small", "full"])
def test_layer_forward_is_bit_reproducible(s):
    # Every sum on the path runs in a fixed order (the folded norm's row
    # statistics are per-slice partials summed by the consumer, not atomics),
    # so two runs give the same bits.
    inp = synth.workload_inputs(s)
    Y1 = run_layer(s, inp, tp.TP_REDUCE_FUSED)
    Y2 = run_layer(s, inp, tp.TP_REDUCE_FUSED)
    assert np.array_equal(Y1, Y2)


def test_layer_chain_without_syncs_matches_synced_chain():
    # Eight full-size layer steps, each step's output the next step's input,
    # sharing one workspace.  Launched back to back on one stream, the next
    # kernel may start its prologue under the previous kernel's tail
    # (programmatic dependent launch); every kernel touches global memory
    # only after the previous one has completed.  The same chain with a
    # synchronize after every step must give the same bits.
    s = SHAPES["layer"]
    inp = synth.workload_inputs(s)
    plan = plan_for(s)
    ws, nws = workspace(plan, tp.TP_OP_LAYER)
    wd = {k: dev(v) for k, v in inp.items() if k != "X"}
    steps = 8

    def chain(sync_each):
        xs = [dev(inp["X"])]
        for _ in range(steps):
            y = torch.empty(s.tokens, s.hidden, dtype=torch.bfloat16, device="cuda")
            tp.tp_layer_forward(plan, xs[-1], wd, y, ws, nws)
            if sync_each:
                torch.cuda.synchronize()
            xs.append(y)
        sync_ok(plan)
        return xs[1:]

    free = chain(False)
    synced = chain(True)
    for k in range(steps):
        assert torch.equal(free[k].view(torch.int16), synced[k].view(torch.int16)), f"step {k}"
    assert torch.isfinite(free[-1].float()).all()


def test_layer_forward_replays_from_a_cuda_graph():
    # The library launches only on the caller's stream, so the layer can be
    # captured once and replayed; the replay gives the eager result's bits.
    s = Shape("l_graph", 2, 128, 256, ffn=512, heads=4, kv_heads=2, head_dim=64, tp=2, act="swiglu",
              index=28)
    inp = synth.workload_inputs(s)
    plan = plan_for(s)
    ws, nws = workspace(plan, tp.TP_OP_LAYER)
    Xd = dev(inp["X"])
    wd = {k: dev(v) for k, v in inp.items() if k != "X"}
    Y = torch.empty(s.tokens, s.hidden, dtype=torch.bfloat16, device="cuda")
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        tp.tp_layer_forward(plan, Xd, wd, Y, ws, nws, side)
    torch.cuda.synchronize()
    eager = Y.clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        tp.tp_layer_forward(plan, Xd, wd, Y, ws, nws, side)
    Y.zero_()
    torch.cuda.synchronize()
    with torch.cuda.stream(side):
        g.replay()
    sync_ok(plan)
    assert torch.equal(Y.view(torch.int16), eager.view(torch.int16))


def test_full_size_layer_full_output():
    s = SHAPES["layer"]
    inp, ref, h1 = full_refs.layer_forward()
    Y = run_layer(s, inp, tp.TP_REDUCE_FUSED)
    e = assert_close(Y, ref, what="layer full output")
    X = host64(inp["X"])
    c = assert_layer_contribution_close(Y, ref, X, h1, what="layer full output contribution")
    report("layer forward", max_rel=e, contribution=c,
           frac_beyond=elementwise_excess_fraction(Y, ref))
