"""GPU parity of sequence parallelism (sequence-split norm region, all-gather
entry, reduce-scatter exit) against the fp64 oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import megatron_tensor_transformer_colwise_gb300 as tp
import oracle
import synth
from synth import SHAPES, Shape
import full_refs
from gpu_util import (assert_close, assert_layer_contribution_close, bf16_bits, dev,
                      elementwise_excess_fraction, host64, plan_for, report, sync_ok, workspace)

pytestmark = pytest.mark.gpu


def _perm(batch, seq, t):
    return [oracle.sp_row(batch, seq, t, b, pos) for b in range(batch) for pos in range(seq)]


@pytest.mark.parametrize("batch,seq,t,h", [(2, 256, 8, 128), (3, 96, 4, 64), (1, 10, 2, 512)])
def test_all_gather_bit_exact(batch, seq, t, h):
    sp = synth.normal_bf16((batch * seq, h), 1.0, 71)
    full = torch.empty_like(sp, device="cuda")
    tp.tp_sp_all_gather(dev(sp), batch, seq, t, h, full)
    sync_ok()
    want = oracle.sp_all_gather(batch, seq, t, host64(sp))
    assert np.array_equal(bf16_bits(full), oracle.round_bf16_bits(want).reshape(want.shape))


@pytest.mark.parametrize("dtype", [tp.TP_F32, tp.TP_BF16])
def test_reduce_scatter_integer_bit_exact_and_fused_norm(dtype):
    batch, seq, t, h = 2, 64, 4, 256
    P = synth.integer_bf16((t, batch * seq, h), -40, 40, 72)
    res = synth.integer_bf16((batch * seq, h), -5, 5, 73)
    out = torch.empty(batch * seq, h, dtype=torch.bfloat16, device="cuda")
    xn = torch.empty_like(out)
    Pd = dev(P.float() if dtype == tp.TP_F32 else P)
    tp.tp_sp_reduce_scatter(Pd, dtype, t, batch, seq, h, dev(res), out, xn, 1e-5)
    sync_ok()
    want = oracle.sp_reduce_scatter(batch, seq, t, host64(P)) + host64(res)
    assert np.array_equal(bf16_bits(out), oracle.round_bf16_bits(want).reshape(want.shape))
    assert_close(host64(xn), oracle.rmsnorm(host64(out), 1e-5), tol=1e-2, what="fused local norm")


SP_MODES = [tp.TP_REDUCE_PARTIALS, tp.TP_REDUCE_FUSED]


def _run_sp_layer(s, inp, mode=tp.TP_REDUCE_PARTIALS):
    cfg = tp.make_config(tokens=s.tokens, hidden=s.hidden, ffn=s.ffn, n_heads=s.heads,
                         n_kv_heads=s.kv_heads, head_dim=s.head_dim, tp_degree=s.tp, act=s.act,
                         reduce_mode=mode, batch=s.batch, seq=s.seq, sequence_parallel=1)
    plan = tp.Plan(cfg)
    ws, nws = workspace(plan, tp.TP_OP_LAYER)
    perm = _perm(s.batch, s.seq, s.tp)
    X_sp = torch.empty_like(inp["X"])
    X_sp[perm] = inp["X"]
    Y_sp = torch.empty(s.tokens, s.hidden, dtype=torch.bfloat16, device="cuda")
    tp.tp_layer_forward(plan, dev(X_sp), {k: dev(v) for k, v in inp.items() if k != "X"}, Y_sp, ws, nws)
    sync_ok(plan)
    return X_sp, host64(Y_sp), perm


# FUSED mode: the reduce-scatter is the rowwise GEMM's sum over shards in
# TMEM, written into the split layout; PARTIALS mode sums the partials.
@pytest.mark.parametrize("mode", SP_MODES, ids=["partials", "fused"])
def test_small_sequence_parallel_layer(mode):
    s = Shape("sp", 2, 128, 256, ffn=768, heads=8, kv_heads=2, head_dim=64, tp=4, act="swiglu",
              index=27)
    inp = synth.workload_inputs(s)
    X_sp, Y_sp, perm = _run_sp_layer(s, inp, mode)
    ref = oracle.layer_sp(s.batch, s.seq, s.heads, s.kv_heads, s.head_dim, s.tp, host64(X_sp),
                          *(host64(inp[n]) for n in ("Wq", "Wk", "Wv", "Wo", "W1", "W3", "W2")))
    assert_close(Y_sp, ref, what="sequence-parallel layer")
    # The blocks' own contribution, with the residual stream h1 of the same
    # layer in the split layout (token row r sits at row perm[r]).
    X = host64(inp["X"])
    h1 = X + oracle.attention_sharded(s.batch, s.seq, s.heads, s.kv_heads, s.head_dim, s.tp,
                                      oracle.rmsnorm(X),
                                      *(host64(inp[n]) for n in ("Wq", "Wk", "Wv", "Wo")))
    h1_sp = np.empty_like(h1)
    h1_sp[perm] = h1
    assert_layer_contribution_close(Y_sp, ref, host64(X_sp), h1_sp, what="SP layer contribution")


@pytest.mark.parametrize("mode", SP_MODES, ids=["partials", "fused"])
def test_full_size_sequence_parallel_layer_full_output(mode):
    # The split layout is a permutation of the token rows, so the SP layer's
    # output, read back in token order, is the replicated layer's.
    s = SHAPES["layer"]
    inp, ref, h1 = full_refs.layer_forward()
    X_sp, Y_sp, perm = _run_sp_layer(s, inp, mode)
    got = Y_sp[perm]
    e = assert_close(got, ref, what="SP layer full output")
    c = assert_layer_contribution_close(got, ref, host64(inp["X"]), h1,
                                        what="SP layer full output contribution")
    report(f"sp layer forward ({'fused' if mode == tp.TP_REDUCE_FUSED else 'partials'})", max_rel=e,
           contribution=c, frac_beyond=elementwise_excess_fraction(got, ref))
