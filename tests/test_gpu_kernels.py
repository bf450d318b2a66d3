"""GPU parity of each kernel of the path against the fp64 oracle, through the
C ABI.  Sizes span several tiles with ragged tails (M not a multiple of 128,
N not a multiple of 256, K per shard not a multiple of 64) and the oracle
finishes them in seconds."""
import numpy as np
import pytest
import torch

import megatron_tensor_transformer_colwise_gb300 as tp
import oracle
import synth
from synth import Shape
from gpu_util import (assert_close, bf16_bits, dev, host64, plan_for, rel_err, sync_ok,
                            workspace)

pytestmark = pytest.mark.gpu


# ---------------------------------------------------------------- g reduce

@pytest.mark.parametrize("t", [1, 2, 3, 4, 8])
@pytest.mark.parametrize("dtype", [tp.TP_F32, tp.TP_BF16])
def test_reduce_integer_partials_bit_exact(t, dtype):
    M, h = 37, 264
    P = synth.integer_bf16((t, M, h), -60, 60, 100 + t)
    bias = synth.integer_bf16((h,), -5, 5, 7)
    res = synth.integer_bf16((M, h), -20, 20, 8)
    Pd = dev(P.float() if dtype == tp.TP_F32 else P)
    out = torch.empty(M, h, dtype=torch.bfloat16, device="cuda")
    tp.tp_reduce_partials(Pd, dtype, t, M * h, h, dev(bias), dev(res), out)
    sync_ok()
    ref = oracle.reduce(host64(P), host64(bias), host64(res))
    assert np.array_equal(bf16_bits(out), oracle.round_bf16_bits(ref).reshape(M, h))


def test_reduce_bias_added_once_and_optional_operands():
    t, M, h = 4, 16, 64
    P = torch.zeros(t, M, h, dtype=torch.float32)
    bias = synth.integer_bf16((h,), 1, 3, 9)
    out = torch.empty(M, h, dtype=torch.bfloat16, device="cuda")
    tp.tp_reduce_partials(dev(P), tp.TP_F32, t, M * h, h, dev(bias), None, out)
    sync_ok()
    assert torch.equal(out.cpu(), bias.expand(M, h))     # bias once, not t times
    tp.tp_reduce_partials(dev(P + 1.0), tp.TP_F32, t, M * h, h, None, None, out)
    sync_ok()
    assert torch.equal(out.cpu().float(), torch.full((M, h), float(t)))


def test_reduce_random_fp32_within_tolerance_large_ragged():
    t, M, h = 8, 1001, 1032
    g = torch.Generator().manual_seed(3)
    P = torch.randn(t, M, h, generator=g)
    res = synth.normal_bf16((M, h), 1.0, 4)
    out = torch.empty(M, h, dtype=torch.bfloat16, device="cuda")
    tp.tp_reduce_partials(dev(P), tp.TP_F32, t, M * h, h, None, dev(res), out)
    sync_ok()
    ref = oracle.reduce(P.double().numpy(), None, host64(res))
    assert_close(host64(out), ref, tol=1e-2, what="reduce")
    # Also: elementwise within bf16 rounding of the fp32 sum.
    assert np.abs(host64(out) - ref).max() <= 2.0 ** -7 * np.abs(ref).max()


def test_reduce_rejects_bad_arguments():
    P = torch.zeros(4, 8, 64, device="cuda")
    out = torch.empty(8, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(tp.TPError) as e:
        tp.tp_reduce_partials(P, tp.TP_F32, 4, 8 * 64, 60, None, None, out)    # h % 8
    assert e.value.code == tp.TP_ERR_INVALID_ARG
    with pytest.raises(tp.TPError) as e:
        tp.tp_reduce_partials(P.data_ptr() + 4, tp.TP_F32, 4, 8 * 64, 64, None, None, out)
    assert e.value.code == tp.TP_ERR_INVALID_ARG                              # misaligned


# ---------------------------------------------------------------- RMSNorm

def test_rmsnorm_matches_oracle_and_constant_rows():
    M, h = 67, 4096
    x = synth.normal_bf16((M, h), 1.0, 21)
    x[5] = 0.75                                     # constant row: c / sqrt(c^2 + eps)
    y = torch.empty_like(x, device="cuda")
    tp.tp_rmsnorm(dev(x), M, h, 1e-5, y)
    sync_ok()
    ref = oracle.rmsnorm(host64(x), 1e-5)
    assert_close(host64(y), ref, tol=1e-2, what="rmsnorm")
    assert np.abs(host64(y)[5] - 0.75 / np.sqrt(0.75 ** 2 + 1e-5)).max() < 1e-2


# ---------------------------------------------------------------- colwise

SMALL_MLP = Shape("small_mlp", 1, 300, 192, ffn=800, tp=4, act="gelu", index=11)


@pytest.mark.parametrize("act", ["none"])
def test_colwise_integer_bit_exact(act):
    s = SMALL_MLP
    inp = synth.workload_inputs(s, integer=(-2, 2))
    plan = plan_for(s, act=act)
    Y = torch.empty(s.tokens, s.ffn, dtype=torch.bfloat16, device="cuda")
    tp.tp_colwise_forward(plan, dev(inp["X"]), dev(inp["W1"]), None, Y)
    sync_ok(plan)
    ref = oracle.linear(host64(inp["X"]), host64(inp["W1"]))   # exact integers
    assert np.array_equal(bf16_bits(Y), oracle.round_bf16_bits(ref).reshape(ref.shape))


@pytest.mark.parametrize("act", ["gelu", "gelu_tanh", "swiglu"])
def test_colwise_activation_within_tolerance(act):
    s = Shape("c", 1, 300, 192, ffn=800, tp=4, act=act, index=12)
    inp = synth.workload_inputs(s)
    plan = plan_for(s)
    Y = torch.empty(s.tokens, s.ffn, dtype=torch.bfloat16, device="cuda")
    W3 = dev(inp["W3"]) if act == "swiglu" else None
    tp.tp_colwise_forward(plan, dev(inp["X"]), dev(inp["W1"]), W3, Y)
    sync_ok(plan)
    X, W1 = host64(inp["X"]), host64(inp["W1"])
    U = oracle.linear(X, W1)
    if act == "swiglu":
        G = oracle.linear(X, host64(inp["W3"]))
        ref = np.vectorize(oracle.silu)(U) * G
    elif act == "gelu":
        ref = np.vectorize(oracle.gelu_erf)(U)
    else:
        ref = np.vectorize(oracle.gelu_tanh)(U)
    assert_close(host64(Y), ref, what=f"colwise {act}")


@pytest.mark.parametrize("act", ["gelu", "gelu_tanh", "swiglu"])
def test_colwise_activation_pointwise_accuracy(act):
    # X = I: every pre-activation is exactly one bf16 weight (N(0, 3^2),
    # so both tails are covered), and every output is act(u) rounded once
    # to bf16.  It must lie within half a bf16 ulp of the exact value plus
    # the activation's own error in fp32 (the erf form is good to 7e-8 |u|
    # in exact arithmetic; the SFU exp2 and reciprocal add a few fp32 ulps).
    M = K = 256
    f, t = 512, 4
    X = torch.eye(M, dtype=torch.bfloat16)
    W1 = synth.normal_bf16((f, K), 3.0, 9001)
    W3 = synth.normal_bf16((f, K), 3.0, 9002) if act == "swiglu" else None
    cfg = tp.make_config(tokens=M, hidden=K, ffn=f, tp_degree=t, act=act)
    plan = tp.Plan(cfg)
    Y = torch.empty(M, f, dtype=torch.bfloat16, device="cuda")
    tp.tp_colwise_forward(plan, dev(X), dev(W1), dev(W3) if W3 is not None else None, Y)
    sync_ok(plan)
    U = host64(W1).T  # U[m][n] = W1[n][m]
    fn = {"gelu": oracle.gelu_erf, "gelu_tanh": oracle.gelu_tanh, "swiglu": oracle.silu}[act]
    ref = np.vectorize(fn)(U)
    if act == "swiglu":
        ref = ref * host64(W3).T
    got = host64(Y)
    mag = np.abs(ref)
    ulp = np.where(mag > 0, 2.0 ** (np.floor(np.log2(np.where(mag > 0, mag, 1.0))) - 7), 0.0)
    bound = 0.5 * ulp + 1e-6 * mag + 4e-7 * np.abs(U)
    excess = np.abs(got - ref) - bound
    i = np.unravel_index(np.argmax(excess), excess.shape)
    assert excess.max() <= 0, f"{act}: u={U[i]} got {got[i]} ref {ref[i]}"


# ---------------------------------------------------------------- rowwise

# SMALL_MLP runs the narrow (128-column) rowwise tiles, which a problem of
# at most one wave of them gets; the ragged 2500 x 1000 one has more tiles
# and runs the 256-column tiles.
ROW_SHAPES = [SMALL_MLP, Shape("row_wide", 1, 2500, 1000, ffn=800, tp=4, act="gelu", index=15)]


@pytest.mark.parametrize("mode", [tp.TP_REDUCE_FUSED, tp.TP_REDUCE_PARTIALS])
@pytest.mark.parametrize("s", ROW_SHAPES, ids=["narrow", "wide_ragged"])
def test_rowwise_integer_bit_exact(s, mode):
    t, M, h, f = s.tp, s.tokens, s.hidden, s.ffn
    Y = synth.integer_bf16((M, f), -2, 2, 31)
    W2 = synth.integer_bf16((h, f), -2, 2, 32)
    res = synth.integer_bf16((M, h), -3, 3, 33)
    bias = synth.integer_bf16((h,), -3, 3, 34)
    plan = plan_for(s, reduce_mode=mode)
    Z = torch.empty(M, h, dtype=torch.bfloat16, device="cuda")
    P = torch.empty(t, M, h, dtype=torch.float32, device="cuda")
    tp.tp_rowwise_forward(plan, dev(Y), dev(W2), dev(bias), dev(res), P, Z)
    sync_ok(plan)
    w = f // t
    parts = np.stack([oracle.linear(host64(Y)[:, i * w:(i + 1) * w], host64(W2)[:, i * w:(i + 1) * w])
                      for i in range(t)])
    if mode == tp.TP_REDUCE_PARTIALS:
        assert np.array_equal(P.cpu().double().numpy(), parts)      # each shard's Partial()
    else:
        ref = oracle.reduce(parts, host64(bias), host64(res))
        assert np.array_equal(bf16_bits(Z), oracle.round_bf16_bits(ref).reshape(M, h))


def test_rowwise_bf16_partials():
    s = SMALL_MLP
    t, M, h, f = s.tp, s.tokens, s.hidden, s.ffn
    Y = synth.integer_bf16((M, f), -2, 2, 41)
    W2 = synth.integer_bf16((h, f), -1, 1, 42)
    plan = plan_for(s, reduce_mode=tp.TP_REDUCE_PARTIALS, partial_dtype=tp.TP_BF16)
    P = torch.empty(t, M, h, dtype=torch.bfloat16, device="cuda")
    tp.tp_rowwise_forward(plan, dev(Y), dev(W2), None, None, P, None)
    sync_ok(plan)
    w = f // t
    parts = np.stack([oracle.linear(host64(Y)[:, i * w:(i + 1) * w], host64(W2)[:, i * w:(i + 1) * w])
                      for i in range(t)])   # exact integers up to 400; both sides round them to bf16
    assert np.array_equal(bf16_bits(P).reshape(-1), oracle.round_bf16_bits(parts.reshape(-1)))


# ---------------------------------------------------------------- QKV + attention

SMALL_ATTN = Shape("small_attn", 2, 200, 256, heads=8, kv_heads=2, head_dim=64, tp=4, act="none",
                   index=13)


def _qkv_ref(s, inp):
    """Oracle Q_i | K_i | V_i column blocks, built from its own shard maps."""
    X = host64(inp["X"])
    a, k, d, t = s.heads, s.kv_heads, s.head_dim, s.tp
    ap, kvn = a // t, oracle.shard_kv_count(k, t)
    blocks = []
    for i in range(t):
        kv0 = oracle.shard_kv_first(k, t, i)
        blocks.append(oracle.linear(X, host64(inp["Wq"])[i * ap * d:(i + 1) * ap * d]))
        blocks.append(oracle.linear(X, host64(inp["Wk"])[kv0 * d:(kv0 + kvn) * d]))
        blocks.append(oracle.linear(X, host64(inp["Wv"])[kv0 * d:(kv0 + kvn) * d]))
    return np.concatenate(blocks, axis=1)


# The QKV GEMM runs clusters of two CTA pairs over pairs of 256-column
# tiles; (6, 2, 2, 64) and (4, 4, 4, 64) have an odd tile count (3, ragged),
# so one pair's tile of the last unit lies past the matrix.
@pytest.mark.parametrize("a,k,t,d", [(8, 2, 4, 64), (8, 8, 4, 128), (4, 1, 4, 128), (8, 4, 2, 64),
                                     (6, 2, 2, 64), (4, 4, 4, 64)])
def test_qkv_integer_bit_exact(a, k, t, d):
    s = Shape("q", 2, 150, 192, heads=a, kv_heads=k, head_dim=d, tp=t, act="none", index=14)
    inp = synth.workload_inputs(s, integer=(-2, 2))
    plan = plan_for(s)
    kvn = oracle.shard_kv_count(k, t)
    W = (a // t + 2 * kvn) * d
    QKV = torch.empty(s.tokens, t * W, dtype=torch.bfloat16, device="cuda")
    tp.tp_qkv_forward(plan, dev(inp["X"]), dev(inp["Wq"]), dev(inp["Wk"]), dev(inp["Wv"]), QKV)
    sync_ok(plan)
    ref = _qkv_ref(s, inp)
    assert np.array_equal(bf16_bits(QKV), oracle.round_bf16_bits(ref).reshape(ref.shape))


# The (8, 512, 32, 8, 8) case has 1024 work items (query tiles x heads x
# sequences) and (8, 512, 24, 8, 8) 768, over twice as many as the kernel's
# persistent grid holds on GB300, so every CTA runs several items back to
# back; (6, 1000, 16, 4, 4) adds a ragged last query tile and key block to
# that, and (1, 1, ...) is a one-token sequence.  The 8192- and 5000-token
# sequences give items of up to 64 key blocks (the layer's have 16), so the
# K/V rings and S buffers wrap many times within one item; 5000 also ends
# in a ragged tile at d = 64.
@pytest.mark.parametrize("batch,seq,a,k,t,d", [(2, 200, 8, 2, 4, 64), (1, 130, 4, 4, 2, 128),
                                               (3, 64, 8, 1, 8, 128), (1, 1, 4, 2, 2, 64),
                                               (2, 257, 16, 8, 8, 128), (8, 512, 32, 8, 8, 128),
                                               (4, 700, 8, 2, 2, 128), (6, 1000, 16, 4, 4, 128),
                                               (8, 512, 24, 8, 8, 128), (1, 1, 4, 2, 2, 128),
                                               (1, 8192, 4, 1, 2, 128), (1, 5000, 4, 2, 2, 64)])
def test_attention_core_vs_oracle(batch, seq, a, k, t, d):
    s = Shape("ac", batch, seq, 64, heads=a, kv_heads=k, head_dim=d, tp=t, act="none", index=15)
    plan = plan_for(s)
    kvn = oracle.shard_kv_count(k, t)
    ap = a // t
    W = (ap + 2 * kvn) * d
    M = batch * seq
    # Q for all heads and K, V per KV head; each shard's block gets its query
    # heads and a copy of every KV head it holds (replicas when k < t).
    Qh = synth.normal_bf16((M, a * d), 1.0, 51)
    Kh = synth.normal_bf16((M, k * d), 1.0, 52)
    Vh = synth.normal_bf16((M, k * d), 1.0, 53)
    QKV = torch.empty(M, t * W, dtype=torch.bfloat16)
    for i in range(t):
        kv0 = oracle.shard_kv_first(k, t, i)
        QKV[:, i * W:i * W + ap * d] = Qh[:, i * ap * d:(i + 1) * ap * d]
        QKV[:, i * W + ap * d:i * W + (ap + kvn) * d] = Kh[:, kv0 * d:(kv0 + kvn) * d]
        QKV[:, i * W + (ap + kvn) * d:(i + 1) * W] = Vh[:, kv0 * d:(kv0 + kvn) * d]
    O = torch.empty(M, a * d, dtype=torch.bfloat16, device="cuda")
    QKVd = dev(QKV)
    tp.tp_attn_core_forward(plan, QKVd, O)
    sync_ok(plan)
    # A second run gives the same bits: the warps' hand-offs leave no race.
    O2 = torch.empty_like(O)
    tp.tp_attn_core_forward(plan, QKVd, O2)
    sync_ok(plan)
    assert torch.equal(O.view(torch.int16), O2.view(torch.int16)), "attention core is not deterministic"
    Q, K, V = host64(Qh), host64(Kh), host64(Vh)
    ref = oracle.attention_core(batch, seq, a, k, d, Q, K, V)
    assert_close(host64(O), ref, what="attention core")
    # First token of every sequence attends only to itself: O = V exactly
    # (up to bf16 rounding of the same value).
    for b in range(batch):
        m = b * seq
        for j in range(a):
            g = oracle.q_head_kv(a, k, j)
            assert np.abs(host64(O)[m, j * d:(j + 1) * d] - V[m, g * d:(g + 1) * d]).max() <= 1e-2


# ---------------------------------------------------------------- failure detection

def test_bounded_wait_reports_timeout_and_context_survives():
    s = SMALL_MLP
    plan = plan_for(s)
    assert tp.tp_get_device_status(plan) == tp.TP_OK
    tp.tp_selftest_wait_timeout(plan, 2_000_000)    # 2 ms limit on a barrier nobody arrives at
    torch.cuda.synchronize()
    assert tp.tp_get_device_status(plan) == tp.TP_ERR_DEVICE_TIMEOUT
    assert tp.tp_get_device_status(plan) == tp.TP_OK   # cleared by the read
    # The context is still usable.
    x = torch.ones(4, 64, dtype=torch.bfloat16, device="cuda")
    y = torch.empty_like(x)
    tp.tp_rmsnorm(x, 4, 64, 0.0, y)
    sync_ok(plan)
    assert torch.allclose(y.float().cpu(), torch.ones(4, 64))
