"""Pins of the fp64 CPU oracle to facts fixed outside the oracle itself.

Each test ties one oracle routine to something independent of it: the worked
example and the statements of the itwiki page "텐서 병렬화" (Tensor
parallelism), closed forms, exact integer arithmetic, special cases that reduce
to a library routine (scipy, numpy, torch fp64), or brute force on tiny sizes.
The cases are chosen so that a plausible slip in the oracle (a dropped term, a
wrong sign or index, a transposed operand, a mis-grouped KV head) fails one.
"""
import json
import math
import os

import numpy as np
import pytest
import scipy.special as sp
import torch
import torch.nn.functional as F

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def f64(t):
    return t.detach().double().numpy()


# ---------------------------------------------------------------- scalars

@pytest.mark.parametrize("x", [-6.0, -2.5, -1.0, -0.3, 0.0, 0.2, 1.0, 3.7, 8.0])
def test_gelu_erf_is_x_times_normal_cdf(x):
    # x * Phi(x) with Phi from scipy's ndtr (independent implementation).
    assert oracle.gelu_erf(x) == pytest.approx(x * sp.ndtr(x), rel=1e-13, abs=1e-15)
    # Phi(x) + Phi(-x) = 1  =>  gelu(x) - gelu(-x) = x.
    assert oracle.gelu_erf(x) - oracle.gelu_erf(-x) == pytest.approx(x, abs=1e-13)


def test_gelu_tanh_close_to_exact_but_distinct():
    xs = np.linspace(-6, 6, 241)
    diff = np.array([oracle.gelu_tanh(x) - oracle.gelu_erf(x) for x in xs])
    assert np.abs(diff).max() < 1e-3          # the approximation's known accuracy
    assert np.abs(diff).max() > 1e-5          # ... and it is a different function
    assert oracle.gelu_tanh(0.0) == 0.0


@pytest.mark.parametrize("x", [-9.0, -1.5, -0.1, 0.0, 0.4, 2.0, 11.0])
def test_silu_is_x_times_logistic(x):
    assert oracle.silu(x) == pytest.approx(x * sp.expit(x), rel=1e-13, abs=1e-15)
    assert oracle.silu(x) - oracle.silu(-x) == pytest.approx(x, abs=1e-12)


def test_round_bf16_matches_torch_rounding():
    vals = np.array([0.0, 1.0, -1.0, 1.00390625, 1.005859375, 257.0, 259.0, 3.0e38, -7.25,
                     1e-3, 65535.0, 33.0, 513.0, 1027.0])
    want = torch.tensor(vals, dtype=torch.float32).to(torch.bfloat16).view(torch.int16)
    want = want.numpy().astype(np.uint16)
    assert np.array_equal(oracle.round_bf16_bits(vals), want)


# ---------------------------------------------------------------- linear / MLP

def test_linear_integer_inputs_exact():
    rng = np.random.default_rng(5)
    X = rng.integers(-3, 4, size=(7, 13))
    W = rng.integers(-3, 4, size=(11, 13))
    Y = oracle.linear(X, W)
    assert np.array_equal(Y, (X @ W.T).astype(np.float64))   # X W^T, not W X or X W


def test_worked_example_identity_holds_as_the_page_states():
    g = json.load(open(os.path.join(GOLDEN, "worked_example.json")))
    w = synth.worked_example()
    X, A, B = (w[k].numpy() for k in "XAB")
    assert X.shape == (g["b"], g["h"]) and A.shape == (g["h"], 4 * g["h"])
    t = g["t"]
    # fp32, the page's own precision: sum_i GeLU(X A_i) B_i vs GeLU(XA)B.
    ref32 = oracle.mlp_worked_f32(False, t, X, A, B)
    out32 = oracle.mlp_worked_f32(True, t, X, A, B)
    assert np.allclose(out32, ref32, atol=g["atol"], rtol=g["rtol"]) == g["expect_allclose"]
    # fp64: the identity is exact up to rounding.
    ref = oracle.mlp("gelu", X, A.T, B.T)
    out = oracle.mlp_sharded("gelu", t, X, A.T, B.T)
    assert np.abs(out - ref).max() <= 1e-12 * np.abs(ref).max()
    # The textbook unsharded MLP via torch fp64 (library gelu, matmul).
    Xt, At, Bt = (torch.from_numpy(v).double() for v in (X, A, B))
    tref = F.gelu(Xt @ At) @ Bt
    assert np.abs(ref - tref.numpy()).max() <= 1e-12 * np.abs(ref).max()
    # The fp32 restatement tracks fp64 to fp32 rounding.
    assert np.abs(ref32 - ref).max() < 1e-3


def test_worked_example_partials_are_the_per_device_products():
    w = synth.worked_example()
    X, A, B = (w[k].double() for k in "XAB")
    Z, P = oracle.mlp_sharded("gelu", 4, X.numpy(), A.T.numpy(), B.T.numpy(), want_partials=True)
    # Device i holds A.chunk(4, dim=1)[i] and B.chunk(4, dim=0)[i] (torch's chunk).
    for i, (Ai, Bi) in enumerate(zip(A.chunk(4, dim=1), B.chunk(4, dim=0))):
        want = (F.gelu(X @ Ai) @ Bi).numpy()
        assert np.abs(P[i] - want).max() < 1e-12
    assert np.abs(P.sum(0) - Z).max() < 1e-12


def test_rowwise_split_before_gelu_is_not_an_identity():
    # The page: GeLU(X1 A1 + X2 A2) != GeLU(X1 A1) + GeLU(X2 A2), so a rowwise A
    # would need a sync before the nonlinearity.
    w = synth.worked_example()
    X, A, B = (w[k].numpy().astype(np.float64) for k in "XAB")
    gelu = np.vectorize(oracle.gelu_erf)
    ref = oracle.mlp("gelu", X, A.T, B.T)
    for parts in (2, 4):
        Xs = np.split(X, parts, axis=1)
        As = np.split(A, parts, axis=0)
        pre = [oracle.linear(Xi, Ai.T) for Xi, Ai in zip(Xs, As)]
        wrong = sum(gelu(p) for p in pre)
        right = gelu(sum(pre))
        assert np.abs(wrong - right).max() > 1e-2
        # With the sync before GeLU the rowwise split is exact again.
        assert np.abs(oracle.linear(right, B.T) - ref).max() < 1e-12 * np.abs(ref).max() * 10


@pytest.mark.parametrize("act", ["gelu", "gelu_tanh", "swiglu", "none"])
def test_mlp_unsharded_matches_textbook_torch(act):
    torch.manual_seed(3)
    M, h, f = 9, 24, 40
    X = torch.randn(M, h, dtype=torch.float64)
    W1 = torch.randn(f, h, dtype=torch.float64) * 0.3
    W3 = torch.randn(f, h, dtype=torch.float64) * 0.3
    W2 = torch.randn(h, f, dtype=torch.float64) * 0.3
    U = X @ W1.T
    if act == "gelu":
        H = F.gelu(U)
    elif act == "gelu_tanh":
        H = F.gelu(U, approximate="tanh")
    elif act == "swiglu":
        H = F.silu(U) * (X @ W3.T)
    else:
        H = U
    want = (H @ W2.T).numpy()
    got = oracle.mlp(act, X.numpy(), W1.numpy(), W2.numpy(), W3.numpy() if act == "swiglu" else None)
    assert np.abs(got - want).max() <= 1e-12 * max(1.0, np.abs(want).max())


@pytest.mark.parametrize("act", ["gelu", "swiglu", "gelu_tanh"])
@pytest.mark.parametrize("t", [1, 2, 4, 8])
def test_mlp_sharded_equals_unsharded(act, t):
    torch.manual_seed(10 + t)
    M, h, f = 6, 16, 64
    X = torch.randn(M, h, dtype=torch.float64)
    W1 = torch.randn(f, h, dtype=torch.float64) * 0.5
    W3 = torch.randn(f, h, dtype=torch.float64) * 0.5
    W2 = torch.randn(h, f, dtype=torch.float64) * 0.5
    w3 = W3.numpy() if act == "swiglu" else None
    ref = oracle.mlp(act, X.numpy(), W1.numpy(), W2.numpy(), w3)
    out = oracle.mlp_sharded(act, t, X.numpy(), W1.numpy(), W2.numpy(), w3)
    assert np.abs(out - ref).max() <= 1e-12 * np.abs(ref).max()


def test_mlp_sharded_identity_activation_is_exact_integer_product():
    X = synth.integer_bf16((5, 32), -2, 2, 1).double().numpy()
    W1 = synth.integer_bf16((48, 32), -2, 2, 2).double().numpy()
    W2 = synth.integer_bf16((32, 48), -2, 2, 3).double().numpy()
    Z = oracle.mlp_sharded("none", 4, X, W1, W2)
    Xi, W1i, W2i = (v.astype(np.int64) for v in (X, W1, W2))
    assert np.array_equal(Z, ((Xi @ W1i.T) @ W2i.T).astype(np.float64))


def test_mlp_sharded_rejects_uneven_chunks():
    X = np.zeros((2, 8))
    with pytest.raises(oracle.OracleError) as e:
        oracle.mlp_sharded("gelu", 3, X, np.zeros((16, 8)), np.zeros((8, 16)))
    assert e.value.code == oracle.ERR_NOT_DIVISIBLE


# ---------------------------------------------------------------- attention

def _qkv(batch, seq, a, k, d, seed):
    g = torch.Generator().manual_seed(seed)
    M = batch * seq
    Q = torch.randn(M, a * d, generator=g, dtype=torch.float64)
    K = torch.randn(M, k * d, generator=g, dtype=torch.float64)
    V = torch.randn(M, k * d, generator=g, dtype=torch.float64)
    return Q, K, V


def _torch_attention(batch, seq, a, k, d, Q, K, V):
    q = Q.view(batch, seq, a, d).transpose(1, 2)
    kk = K.view(batch, seq, k, d).transpose(1, 2).repeat_interleave(a // k, dim=1)
    vv = V.view(batch, seq, k, d).transpose(1, 2).repeat_interleave(a // k, dim=1)
    o = F.scaled_dot_product_attention(q, kk, vv, is_causal=True)
    return o.transpose(1, 2).reshape(batch * seq, a * d)


@pytest.mark.parametrize("batch,seq,a,k,d", [(1, 7, 4, 4, 8), (2, 9, 8, 2, 4), (3, 5, 6, 1, 16)])
def test_attention_core_matches_torch_sdpa(batch, seq, a, k, d):
    Q, K, V = _qkv(batch, seq, a, k, d, 7)
    got = oracle.attention_core(batch, seq, a, k, d, Q.numpy(), K.numpy(), V.numpy())
    want = _torch_attention(batch, seq, a, k, d, Q, K, V).numpy()
    assert np.abs(got - want).max() < 1e-12


def test_attention_closed_forms():
    a, k, d = 4, 2, 8
    # seq = 1: a token attends only to itself -> O = V of its KV head.
    Q, K, V = _qkv(3, 1, a, k, d, 1)
    O = oracle.attention_core(3, 1, a, k, d, Q.numpy(), K.numpy(), V.numpy())
    for j in range(a):
        g = j // (a // k)
        assert np.allclose(O[:, j * d:(j + 1) * d], V.numpy()[:, g * d:(g + 1) * d], atol=1e-15)
    # First position of every sequence -> O = V[0] of that sequence.
    batch, seq = 2, 6
    Q, K, V = _qkv(batch, seq, a, k, d, 2)
    O = oracle.attention_core(batch, seq, a, k, d, Q.numpy(), K.numpy(), V.numpy())
    for b in range(batch):
        m = b * seq
        for j in range(a):
            g = j // (a // k)
            assert np.allclose(O[m, j * d:(j + 1) * d], V.numpy()[m, g * d:(g + 1) * d], atol=1e-15)
    # All keys equal -> uniform weights over the causal prefix: O[p] = mean(V[0..p]).
    K = torch.ones_like(K)
    O = oracle.attention_core(batch, seq, a, k, d, Q.numpy(), K.numpy(), V.numpy())
    Vn = V.numpy()
    for b in range(batch):
        for p in range(seq):
            m = b * seq + p
            for j in range(a):
                g = j // (a // k)
                want = Vn[b * seq:m + 1, g * d:(g + 1) * d].mean(0)
                assert np.allclose(O[m, j * d:(j + 1) * d], want, atol=1e-13)


def test_attention_heads_are_independent():
    # Heads 4..7 (which read KV head 1 of 2) computed alone equal that slice.
    batch, seq, a, k, d = 2, 8, 8, 2, 4
    Q, K, V = _qkv(batch, seq, a, k, d, 3)
    full = oracle.attention_core(batch, seq, a, k, d, Q.numpy(), K.numpy(), V.numpy())
    sub = oracle.attention_core(batch, seq, 4, 1, d, Q.numpy()[:, 4 * d:], K.numpy()[:, d:],
                                V.numpy()[:, d:])
    assert np.array_equal(sub, full[:, 4 * d:])
    # Sequences do not see each other: changing sequence 1 leaves sequence 0 alone.
    K2, V2 = K.clone(), V.clone()
    K2[seq:] += 1.0
    V2[seq:] -= 2.0
    alt = oracle.attention_core(batch, seq, a, k, d, Q.numpy(), K2.numpy(), V2.numpy())
    assert np.array_equal(alt[:seq], full[:seq])
    assert not np.allclose(alt[seq:], full[seq:])


@pytest.mark.parametrize("a,k,t", [(8, 8, 4), (8, 2, 4), (8, 2, 8), (8, 4, 2), (4, 1, 4), (6, 3, 3)])
def test_attention_sharded_equals_unsharded(a, k, t):
    batch, seq, h, d = 2, 5, 12, 4
    g = torch.Generator().manual_seed(a * 100 + k * 10 + t)
    X = torch.randn(batch * seq, h, generator=g, dtype=torch.float64)
    Wq = torch.randn(a * d, h, generator=g, dtype=torch.float64) * 0.4
    Wk = torch.randn(k * d, h, generator=g, dtype=torch.float64) * 0.4
    Wv = torch.randn(k * d, h, generator=g, dtype=torch.float64) * 0.4
    Wo = torch.randn(h, a * d, generator=g, dtype=torch.float64) * 0.4
    ref, O = oracle.attention(batch, seq, a, k, d, X, Wq, Wk, Wv, Wo, want_O=True)
    out, P = oracle.attention_sharded(batch, seq, a, k, d, t, X, Wq, Wk, Wv, Wo, want_partials=True)
    assert np.abs(out - ref).max() <= 1e-12 * np.abs(ref).max()
    # Device i's partial is its head block of O times its column block of Wo.
    cols = a * d // t
    for i in range(t):
        want = O[:, i * cols:(i + 1) * cols] @ Wo.numpy()[:, i * cols:(i + 1) * cols].T
        assert np.abs(P[i] - want).max() < 1e-12
    # The unsharded block against torch (library projections + sdpa).
    tq, tk, tv = X @ Wq.T, X @ Wk.T, X @ Wv.T
    tO = _torch_attention(batch, seq, a, k, d, tq, tk, tv)
    assert np.abs(ref - (tO @ Wo.T).numpy()).max() < 1e-12


def test_attention_rows_match_full_block():
    batch, seq, h, a, k, d = 2, 9, 16, 4, 2, 4
    g = torch.Generator().manual_seed(11)
    X = torch.randn(batch * seq, h, generator=g, dtype=torch.float64)
    Ws = [torch.randn(s, h, generator=g, dtype=torch.float64) * 0.3
          for s in (a * d, k * d, k * d)]
    Wo = torch.randn(h, a * d, generator=g, dtype=torch.float64) * 0.3
    full = oracle.attention(batch, seq, a, k, d, X, *Ws, Wo)
    rows = [0, 4, 8, 9, 17, 13]
    part = oracle.attention_rows(batch, seq, a, k, d, X, *Ws, Wo, rows)
    assert np.abs(part - full[rows]).max() < 1e-13


# ---------------------------------------------------------------- plan

def _read_map(name):
    rows = []
    for line in open(os.path.join(GOLDEN, name)):
        line = line.strip()
        if line and not line.startswith("#"):
            rows.append(tuple(int(v) for v in line.split()))
    return rows


@pytest.mark.parametrize("name,a,k,t", [("head_map_a32_k8_t8.txt", 32, 8, 8),
                                        ("head_map_a8_k2_t4.txt", 8, 2, 4)])
def test_head_maps_match_golden(name, a, k, t):
    for shard, q0, nq, kv0, nkv in _read_map(name):
        heads = [j for j in range(a) if oracle.q_head_shard(a, t, j) == shard]
        assert heads == list(range(q0, q0 + nq))
        assert oracle.shard_kv_first(k, t, shard) == kv0
        assert oracle.shard_kv_count(k, t) == nkv
        # every query head of the shard reads a KV head the shard holds
        for j in heads:
            assert kv0 <= oracle.q_head_kv(a, k, j) < kv0 + nkv


@pytest.mark.parametrize("h,f,a,k,d,t,want", [
    (4096, 14336, 32, 8, 128, 8, oracle.OK),
    (1024, 4096, 0, 0, 0, 4, oracle.OK),
    (16, 64, 0, 0, 0, 4, oracle.OK),
    (4096, 14336, 32, 8, 128, 3, oracle.ERR_NOT_DIVISIBLE),   # t does not divide a or f
    (64, 60, 8, 8, 8, 8, oracle.ERR_NOT_DIVISIBLE),            # t does not divide f
    (64, 64, 12, 4, 8, 8, oracle.ERR_NOT_DIVISIBLE),           # t does not divide a
    (64, 64, 8, 3, 8, 4, oracle.ERR_NOT_DIVISIBLE),            # k does not divide a
    (64, 64, 16, 8, 8, 16, oracle.OK),                         # k < t, k | t: replicas
    (64, 64, 24, 6, 8, 4, oracle.ERR_NOT_DIVISIBLE),           # k >= t but t does not divide k
    (64, 48, 24, 3, 8, 6, oracle.OK),                          # k < t, k | t: replicas
    (64, 48, 24, 4, 8, 6, oracle.ERR_NOT_DIVISIBLE),           # k < t but k does not divide t
    (0, 64, 8, 8, 8, 8, oracle.ERR_INVALID),
    (64, 64, 8, 8, 8, 0, oracle.ERR_INVALID),
])
def test_plan_check(h, f, a, k, d, t, want):
    assert oracle.plan_check(h, f, a, k, d, t) == want


# ---------------------------------------------------------------- g, norm, layer

def test_reduce_exact_and_bias_added_once():
    P = synth.integer_bf16((4, 6, 8), -50, 50, 9).double().numpy()
    bias = synth.integer_bf16((8,), -3, 3, 10).double().numpy()
    res = synth.integer_bf16((6, 8), -9, 9, 11).double().numpy()
    out = oracle.reduce(P, bias, res)
    Pi = P.astype(np.int64)
    assert np.array_equal(out, (Pi.sum(0) + bias.astype(np.int64) + res.astype(np.int64)))
    plain = oracle.reduce(P)
    assert np.array_equal(out - plain - res, np.broadcast_to(bias, (6, 8)))  # once, not t times


def test_rmsnorm_closed_forms():
    eps = 1e-5
    for c in (0.0, 0.5, -3.0, 7.0):
        x = np.full((2, 10), c)
        y = oracle.rmsnorm(x, eps)
        assert np.allclose(y, c / math.sqrt(c * c + eps), rtol=1e-14, atol=0)
    g = torch.Generator().manual_seed(4)
    x = torch.randn(5, 32, generator=g, dtype=torch.float64) * 3
    want = F.rms_norm(x, (32,), eps=eps).numpy()
    assert np.abs(oracle.rmsnorm(x.numpy(), eps) - want).max() < 1e-13


def _small_layer(seed, batch=2, seq=6, h=16, a=4, k=2, d=4, f=32):
    g = torch.Generator().manual_seed(seed)
    r = lambda *s: torch.randn(*s, generator=g, dtype=torch.float64)
    X = r(batch * seq, h)
    Wq, Wk, Wv = r(a * d, h) * 0.3, r(k * d, h) * 0.3, r(k * d, h) * 0.3
    Wo = r(h, a * d) * 0.3
    W1, W3, W2 = r(f, h) * 0.3, r(f, h) * 0.3, r(h, f) * 0.3
    return (batch, seq, a, k, d), X, (Wq, Wk, Wv, Wo, W1, W3, W2)


def test_layer_reduces_to_residual_when_output_projections_vanish():
    dims, X, (Wq, Wk, Wv, Wo, W1, W3, W2) = _small_layer(1)
    Y = oracle.layer(*dims, 2, X, Wq, Wk, Wv, torch.zeros_like(Wo), W1, W3, torch.zeros_like(W2))
    assert np.array_equal(Y, X.numpy())


def test_layer_matches_composed_torch_reference_and_sharded_form():
    dims, X, W = _small_layer(2)
    batch, seq, a, k, d = dims
    Wq, Wk, Wv, Wo, W1, W3, W2 = W
    eps = 1e-5
    xn = F.rms_norm(X, (X.shape[1],), eps=eps)
    att = _torch_attention(batch, seq, a, k, d, xn @ Wq.T, xn @ Wk.T, xn @ Wv.T) @ Wo.T
    h1 = X + att
    hn = F.rms_norm(h1, (X.shape[1],), eps=eps)
    want = (h1 + (F.silu(hn @ W1.T) * (hn @ W3.T)) @ W2.T).numpy()
    Y = oracle.layer(*dims, 2, X, *W)
    assert np.abs(Y - want).max() < 1e-12
    for t in (2, 4):
        Ys = oracle.layer(*dims, t, X, *W, sharded=True)
        assert np.abs(Ys - Y).max() < 1e-12
    rows = [0, 5, 6, 11, 7]
    Yr = oracle.layer_rows(*dims, X, *W, rows)
    assert np.abs(Yr - Y[rows]).max() < 1e-12


# ---------------------------------------------------------------- packed projections

def test_packed_shard_rows_match_golden_and_differ_from_contiguous():
    for line in open(os.path.join(GOLDEN, "packed_gate_up_f4_t2.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        left, right = line.split("|")
        shard, *rows = (int(v) for v in left.split())
        contiguous = [int(v) for v in right.split()]
        got = oracle.packed_shard_rows([4, 4], 2, shard).tolist()
        assert got == rows
        assert got != contiguous


def test_packed_blocks_must_divide_individually():
    assert oracle.packed_check([8, 8], 4) == oracle.OK
    assert oracle.packed_check([6, 2], 4) == oracle.ERR_NOT_DIVISIBLE   # sum 8 divides, blocks do not
    assert oracle.packed_check([3072, 3072, 3072, 9216, 9216], 4) == oracle.OK
    assert oracle.packed_check([3072, 3072, 3072, 9216, 9216], 5) == oracle.ERR_NOT_DIVISIBLE


@pytest.mark.parametrize("t", [1, 2, 4])
def test_packed_gate_up_per_block_equals_unpacked_and_contiguous_does_not(t):
    torch.manual_seed(21 + t)
    M, h, f = 5, 16, 32
    X = torch.randn(M, h, dtype=torch.float64)
    Wg = torch.randn(f, h, dtype=torch.float64) * 0.5
    Wu = torch.randn(f, h, dtype=torch.float64) * 0.5
    W2 = torch.randn(h, f, dtype=torch.float64) * 0.5
    Wgu = torch.cat([Wg, Wu], 0)
    ref = oracle.mlp("swiglu", X.numpy(), Wg.numpy(), W2.numpy(), Wu.numpy())
    good = oracle.mlp_packed_gate_up(True, t, X.numpy(), Wgu.numpy(), W2.numpy())
    assert np.abs(good - ref).max() <= 1e-12 * np.abs(ref).max()
    bad = oracle.mlp_packed_gate_up(False, t, X.numpy(), Wgu.numpy(), W2.numpy())
    if t == 1:
        assert np.abs(bad - ref).max() <= 1e-12 * np.abs(ref).max()   # nothing to mix at t = 1
    else:
        assert np.abs(bad - ref).max() > 1e-2 * np.abs(ref).max()     # runs, but wrong


# ---------------------------------------------------------------- vocabulary parallelism

@pytest.mark.parametrize("t", [1, 2, 4, 8])
def test_vocab_parallel_embedding_is_the_gather(t):
    rng = np.random.default_rng(31 + t)
    v, h = 64, 12
    E = rng.normal(size=(v, h))
    ids = rng.integers(0, v, size=40).astype(np.int32)
    ids[[3, 7]] = [-1, v]              # no device owns these ids
    out = oracle.embedding_vocab_parallel(t, ids, E)
    want = np.where(((ids >= 0) & (ids < v))[:, None], E[np.clip(ids, 0, v - 1)], 0.0)
    assert np.array_equal(out, want)


def test_cross_entropy_matches_torch_and_closed_forms():
    rng = np.random.default_rng(5)
    z = rng.normal(size=(9, 40)) * 4
    lab = rng.integers(0, 40, size=9).astype(np.int32)
    lab[2] = -100
    got = oracle.cross_entropy(z, lab)
    want = F.cross_entropy(torch.tensor(z), torch.tensor(lab, dtype=torch.long),
                           reduction="none", ignore_index=-100).numpy()
    assert np.abs(got - want).max() < 1e-12
    # equal logits: every class has probability 1/v
    assert np.allclose(oracle.cross_entropy(np.zeros((3, 40)), np.array([0, 5, 39], np.int32)),
                       np.log(40.0), atol=1e-14)
    # a huge margin on the label: loss -> 0; on another class: loss -> margin
    zz = np.zeros((2, 10))
    zz[0, 3] = 50.0
    zz[1, 4] = 50.0
    l2 = oracle.cross_entropy(zz, np.array([3, 3], np.int32))
    assert l2[0] == pytest.approx(9 * np.exp(-50.0), abs=1e-18)
    assert l2[1] == pytest.approx(50.0, rel=1e-12)


@pytest.mark.parametrize("t", [1, 2, 4, 5, 8])
def test_vocab_parallel_cross_entropy_equals_plain(t):
    rng = np.random.default_rng(40 + t)
    M, v = 11, 40
    z = rng.normal(size=(M, v)) * 6
    lab = rng.integers(0, v, size=M).astype(np.int32)
    lab[0] = -100
    plain = oracle.cross_entropy(z, lab)
    par, st = oracle.cross_entropy_vocab_parallel(t, z, lab, want_stats=True)
    assert np.abs(par - plain).max() < 1e-12
    # Only 3 numbers per token and device cross devices; their max is the row max.
    assert st.shape == (3, t, M)
    assert np.array_equal(st[0].max(0), z.max(1))
    w = v // t
    owner = lab // w
    for m in range(1, M):
        assert st[2, owner[m], m] == z[m, lab[m]]
        assert np.count_nonzero(st[2, :, m]) <= 1


# ---------------------------------------------------------------- sequence parallelism

def test_sp_layout_matches_golden():
    for line in open(os.path.join(GOLDEN, "sp_layout_b2_s4_t2.txt")):
        line = line.strip()
        if line and not line.startswith("#"):
            b, pos, row = (int(v) for v in line.split())
            assert oracle.sp_row(2, 4, 2, b, pos) == row


@pytest.mark.parametrize("batch,seq,t", [(2, 4, 2), (3, 8, 4), (1, 6, 3), (2, 8, 1)])
def test_sp_all_gather_inverts_the_split_and_reduce_scatter_sums(batch, seq, t):
    rng = np.random.default_rng(batch * 100 + seq * 10 + t)
    h = 5
    full = rng.normal(size=(batch * seq, h))
    sp = np.empty_like(full)
    for b in range(batch):
        for pos in range(seq):
            sp[oracle.sp_row(batch, seq, t, b, pos)] = full[b * seq + pos]
    assert np.array_equal(oracle.sp_all_gather(batch, seq, t, sp), full)
    P = rng.integers(-9, 10, size=(t, batch * seq, h)).astype(np.float64)
    red = oracle.sp_reduce_scatter(batch, seq, t, P)
    S = P.sum(0)
    for b in range(batch):
        for pos in range(seq):
            assert np.array_equal(red[oracle.sp_row(batch, seq, t, b, pos)], S[b * seq + pos])


@pytest.mark.parametrize("t", [1, 2, 4])
def test_sp_layer_equals_replicated_layer_in_the_split_layout(t):
    dims, X, W = _small_layer(7, batch=2, seq=8, h=16, a=4, k=2, d=4, f=32)
    batch, seq, a, k, d = dims
    Y = oracle.layer(*dims, t, X, *W, sharded=True)
    perm = [oracle.sp_row(batch, seq, t, b, pos) for b in range(batch) for pos in range(seq)]
    X_sp = np.empty_like(X.numpy())
    X_sp[perm] = X.numpy()
    Y_sp = oracle.layer_sp(batch, seq, a, k, d, t, X_sp, *W)
    assert np.abs(Y_sp[perm] - Y).max() < 1e-12


# ---------------------------------------------------------------- backward

def _autograd_mlp(act, X, W1, W2, W3, dZ, b2):
    X, W1, W2, b2 = (v.clone().requires_grad_(True) for v in (X, W1, W2, b2))
    W3 = W3.clone().requires_grad_(True) if act == "swiglu" else None
    U = X @ W1.T
    if act == "gelu":
        H = F.gelu(U)
    elif act == "gelu_tanh":
        H = F.gelu(U, approximate="tanh")
    elif act == "swiglu":
        H = F.silu(U) * (X @ W3.T)
    else:
        H = U
    Z = H @ W2.T + b2
    Z.backward(dZ)
    return X.grad, W1.grad, (W3.grad if W3 is not None else None), W2.grad, b2.grad


@pytest.mark.parametrize("act", ["gelu", "gelu_tanh", "swiglu", "none"])
def test_mlp_backward_matches_torch_autograd(act):
    g = torch.Generator().manual_seed(61)
    M, h, f = 7, 12, 24
    X = torch.randn(M, h, generator=g, dtype=torch.float64)
    W1 = torch.randn(f, h, generator=g, dtype=torch.float64) * 0.4
    W3 = torch.randn(f, h, generator=g, dtype=torch.float64) * 0.4
    W2 = torch.randn(h, f, generator=g, dtype=torch.float64) * 0.4
    dZ = torch.randn(M, h, generator=g, dtype=torch.float64)
    b2 = torch.randn(h, generator=g, dtype=torch.float64)
    want = _autograd_mlp(act, X, W1, W2, W3, dZ, b2)
    got = oracle.mlp_backward(act, X, W1, W2, dZ, W3 if act == "swiglu" else None)
    for name, a, b in zip(("dX", "dW1", "dW3", "dW2", "db2"), got, want):
        if b is None:
            continue
        assert np.abs(a - b.numpy()).max() < 1e-12 * max(1.0, np.abs(b.numpy()).max()), name


def test_mlp_backward_central_differences():
    # d(sum dZ * Z)/dW1[n][j] by central differences of the oracle's forward.
    g = torch.Generator().manual_seed(62)
    M, h, f = 3, 4, 8
    X = torch.randn(M, h, generator=g, dtype=torch.float64).numpy()
    W1 = (torch.randn(f, h, generator=g, dtype=torch.float64) * 0.5).numpy()
    W3 = (torch.randn(f, h, generator=g, dtype=torch.float64) * 0.5).numpy()
    W2 = (torch.randn(h, f, generator=g, dtype=torch.float64) * 0.5).numpy()
    dZ = torch.randn(M, h, generator=g, dtype=torch.float64).numpy()
    _, dW1, dW3, _, _ = oracle.mlp_backward("swiglu", X, W1, W2, dZ, W3)
    eps = 1e-6
    for (n, j) in [(0, 0), (3, 2), (7, 3)]:
        for W, dW in ((W1, dW1), (W3, dW3)):
            Wp, Wm = W.copy(), W.copy()
            Wp[n, j] += eps
            Wm[n, j] -= eps
            args_p = (X, Wp, W2, W3) if W is W1 else (X, W1, W2, Wp)
            args_m = (X, Wm, W2, W3) if W is W1 else (X, W1, W2, Wm)
            Lp = (oracle.mlp("swiglu", *args_p) * dZ).sum()
            Lm = (oracle.mlp("swiglu", *args_m) * dZ).sum()
            assert (Lp - Lm) / (2 * eps) == pytest.approx(dW[n, j], rel=1e-6, abs=1e-9)


@pytest.mark.parametrize("act", ["gelu", "swiglu"])
@pytest.mark.parametrize("t", [1, 2, 4])
def test_mlp_backward_sharded_equals_plain(act, t):
    g = torch.Generator().manual_seed(63 + t)
    M, h, f = 6, 8, 32
    X = torch.randn(M, h, generator=g, dtype=torch.float64).numpy()
    W1 = (torch.randn(f, h, generator=g, dtype=torch.float64) * 0.4).numpy()
    W3 = (torch.randn(f, h, generator=g, dtype=torch.float64) * 0.4).numpy()
    W2 = (torch.randn(h, f, generator=g, dtype=torch.float64) * 0.4).numpy()
    dZ = torch.randn(M, h, generator=g, dtype=torch.float64).numpy()
    w3 = W3 if act == "swiglu" else None
    plain = oracle.mlp_backward(act, X, W1, W2, dZ, w3)
    *shard, P = oracle.mlp_backward(act, X, W1, W2, dZ, w3, t=t, want_partials=True)
    for a, b in zip(plain, shard):
        if a is not None:
            assert np.abs(a - b).max() < 1e-12 * max(1.0, np.abs(a).max())
    assert np.abs(P.sum(0) - plain[0]).max() < 1e-12   # f backward: dX = sum of the t partials


def _torch_gqa_attention(batch, seq, a, k, Q, K, V):
    """Causal GQA attention by torch ops, for autograd pins."""
    M = batch * seq
    d = Q.shape[1] // a
    q = Q.reshape(batch, seq, a, d).transpose(1, 2)                  # b a s d
    kk = K.reshape(batch, seq, k, d).transpose(1, 2).repeat_interleave(a // k, dim=1)
    vv = V.reshape(batch, seq, k, d).transpose(1, 2).repeat_interleave(a // k, dim=1)
    s = q @ kk.transpose(-1, -2) / math.sqrt(d)
    mask = torch.ones(seq, seq, dtype=torch.bool).triu(1)
    s = s.masked_fill(mask, float("-inf"))
    o = torch.softmax(s, dim=-1) @ vv
    return o.transpose(1, 2).reshape(M, a * d)


def test_attention_core_backward_matches_torch_autograd():
    g = torch.Generator().manual_seed(71)
    batch, seq, a, k, d = 2, 5, 4, 2, 3
    M = batch * seq
    Q, K, V = (torch.randn(M, n * d, generator=g, dtype=torch.float64).requires_grad_(True)
               for n in (a, k, k))
    dO = torch.randn(M, a * d, generator=g, dtype=torch.float64)
    _torch_gqa_attention(batch, seq, a, k, Q, K, V).backward(dO)
    got = oracle.attention_core_backward(batch, seq, a, k, Q.detach(), K.detach(), V.detach(), dO)
    for name, x, ref in zip(("dQ", "dK", "dV"), got, (Q.grad, K.grad, V.grad)):
        assert np.abs(x - ref.numpy()).max() < 1e-12, name


def test_attention_core_backward_single_position_closed_form():
    # seq = 1: every query attends only to itself, P = 1, so dS = 0:
    # dQ = dK = 0 and dV = the sum of dO over the query heads of the group.
    g = torch.Generator().manual_seed(72)
    batch, a, k, d = 3, 4, 2, 5
    Q, K, V = (torch.randn(batch, n * d, generator=g, dtype=torch.float64) for n in (a, k, k))
    dO = torch.randn(batch, a * d, generator=g, dtype=torch.float64).numpy()
    dQ, dK, dV = oracle.attention_core_backward(batch, 1, a, k, Q, K, V, dO)
    assert np.abs(dQ).max() == 0 and np.abs(dK).max() == 0
    want = dO.reshape(batch, k, a // k, d).sum(2).reshape(batch, k * d)
    assert np.abs(dV - want).max() < 1e-15


def test_attention_block_backward_matches_torch_autograd():
    g = torch.Generator().manual_seed(73)
    batch, seq, h, a, k, d = 2, 4, 6, 4, 2, 2
    M = batch * seq
    X = torch.randn(M, h, generator=g, dtype=torch.float64).requires_grad_(True)
    Wq = (torch.randn(a * d, h, generator=g, dtype=torch.float64) * 0.5).requires_grad_(True)
    Wk = (torch.randn(k * d, h, generator=g, dtype=torch.float64) * 0.5).requires_grad_(True)
    Wv = (torch.randn(k * d, h, generator=g, dtype=torch.float64) * 0.5).requires_grad_(True)
    Wo = (torch.randn(h, a * d, generator=g, dtype=torch.float64) * 0.5).requires_grad_(True)
    dOut = torch.randn(M, h, generator=g, dtype=torch.float64)
    out = _torch_gqa_attention(batch, seq, a, k, X @ Wq.T, X @ Wk.T, X @ Wv.T) @ Wo.T
    out.backward(dOut)
    got = oracle.attention_backward(batch, seq, a, k, *(w.detach() for w in (X, Wq, Wk, Wv, Wo)), dOut)
    for name, x, ref in zip(("dX", "dWq", "dWk", "dWv", "dWo"), got,
                            (X.grad, Wq.grad, Wk.grad, Wv.grad, Wo.grad)):
        assert np.abs(x - ref.numpy()).max() < 1e-12 * max(1.0, ref.abs().max().item()), name


@pytest.mark.parametrize("a,k,t", [(4, 2, 2), (4, 2, 4), (4, 4, 2), (8, 2, 4), (4, 1, 2), (2, 1, 1)])
def test_attention_backward_sharded_equals_plain(a, k, t):
    # k < t exercises KV replicas: their weight gradients are summed.
    g = torch.Generator().manual_seed(74 + 10 * a + k + t)
    batch, seq, h, d = 2, 3, 8, 2
    M = batch * seq
    X = torch.randn(M, h, generator=g, dtype=torch.float64).numpy()
    W = [(torch.randn(n, m, generator=g, dtype=torch.float64) * 0.5).numpy()
         for n, m in ((a * d, h), (k * d, h), (k * d, h), (h, a * d))]
    dOut = torch.randn(M, h, generator=g, dtype=torch.float64).numpy()
    plain = oracle.attention_backward(batch, seq, a, k, X, *W, dOut)
    *shard, P = oracle.attention_backward(batch, seq, a, k, X, *W, dOut, t=t, want_partials=True)
    for x, y in zip(plain, shard):
        assert np.abs(x - y).max() < 1e-12 * max(1.0, np.abs(x).max())
    assert np.abs(P.sum(0) - plain[0]).max() < 1e-12 * max(1.0, np.abs(plain[0]).max())


def test_attention_backward_composed_equals_c_form():
    # The large-size composition (numpy projections + C attention core) is
    # the same definition as the all-C block backward.
    g = torch.Generator().manual_seed(81)
    batch, seq, h, a, k, d = 2, 6, 8, 4, 2, 3
    M = batch * seq
    X = torch.randn(M, h, generator=g, dtype=torch.float64).numpy()
    W = [(torch.randn(n, m, generator=g, dtype=torch.float64) * 0.5).numpy()
         for n, m in ((a * d, h), (k * d, h), (k * d, h), (h, a * d))]
    dOut = torch.randn(M, h, generator=g, dtype=torch.float64).numpy()
    a1 = oracle.attention_backward(batch, seq, a, k, X, *W, dOut)
    a2 = oracle.attention_backward_composed(batch, seq, a, k, X, *W, dOut)
    for x, y in zip(a1, a2):
        assert np.abs(x - y).max() < 1e-12 * max(1.0, np.abs(x).max())


def test_rmsnorm_backward_matches_torch_autograd():
    g = torch.Generator().manual_seed(91)
    x = torch.randn(5, 12, generator=g, dtype=torch.float64).requires_grad_(True)
    up = torch.randn(5, 12, generator=g, dtype=torch.float64)
    y = x * torch.rsqrt(x.pow(2).mean(-1, keepdim=True) + 1e-5)
    y.backward(up)
    got = oracle.rmsnorm_backward(x.detach(), up)
    assert np.abs(got - x.grad.numpy()).max() < 1e-13


def _torch_layer(batch, seq, a, k, X, Wq, Wk, Wv, Wo, W1, W3, W2, eps=1e-5):
    rms = lambda v: v * torch.rsqrt(v.pow(2).mean(-1, keepdim=True) + eps)
    xn1 = rms(X)
    h1 = X + _torch_gqa_attention(batch, seq, a, k, xn1 @ Wq.T, xn1 @ Wk.T, xn1 @ Wv.T) @ Wo.T
    xn2 = rms(h1)
    return h1 + (F.silu(xn2 @ W1.T) * (xn2 @ W3.T)) @ W2.T


def test_layer_backward_matches_torch_autograd():
    g = torch.Generator().manual_seed(92)
    batch, seq, h, a, k, d, f = 2, 5, 8, 4, 2, 2, 16
    M = batch * seq
    X = torch.randn(M, h, generator=g, dtype=torch.float64).requires_grad_(True)
    shapes = [(a * d, h), (k * d, h), (k * d, h), (h, a * d), (f, h), (f, h), (h, f)]
    W = [(torch.randn(*s, generator=g, dtype=torch.float64) * 0.4).requires_grad_(True) for s in shapes]
    dY = torch.randn(M, h, generator=g, dtype=torch.float64)
    _torch_layer(batch, seq, a, k, X, *W).backward(dY)
    got = oracle.layer_backward(batch, seq, a, k, d, X.detach(), *(w.detach() for w in W), dY)
    want = [X.grad] + [w.grad for w in W]
    names = ["dX", "dWq", "dWk", "dWv", "dWo", "dW1", "dW3", "dW2"]
    for n, x, ref in zip(names, got, want):
        assert np.abs(x - ref.numpy()).max() < 1e-11 * max(1.0, ref.abs().max().item()), n
    comp = oracle.layer_backward_composed(batch, seq, a, k, d, X.detach(), *(w.detach() for w in W), dY)
    for n, x, y in zip(names, got, comp):
        assert np.abs(x - y).max() < 1e-11 * max(1.0, np.abs(x).max()), n + " (composed)"


# ---------------------------------------------------------------- composed forms (full-size checks)

def test_composed_forward_forms_equal_the_c_forms():
    # The full-size parity tests use the numpy-matmul compositions; at small
    # sizes they equal the all-C definitions for every activation, the
    # attention block and the layer (and the layer's residual stream h1).
    g = torch.Generator().manual_seed(93)
    batch, seq, h, a, k, d, f = 2, 9, 16, 4, 2, 4, 40
    M = batch * seq
    X = torch.randn(M, h, generator=g, dtype=torch.float64).numpy()
    rnd = lambda n, m: (torch.randn(n, m, generator=g, dtype=torch.float64) * 0.4).numpy()
    W1, W3, W2 = rnd(f, h), rnd(f, h), rnd(h, f)
    Wq, Wk, Wv, Wo = rnd(a * d, h), rnd(k * d, h), rnd(k * d, h), rnd(h, a * d)
    for act in ("gelu", "gelu_tanh", "swiglu", "none"):
        w3 = W3 if act == "swiglu" else None
        want = oracle.mlp(act, X, W1, W2, w3)
        got = oracle.mlp_composed(act, X, W1, W2, w3)
        assert np.abs(got - want).max() < 1e-12 * np.abs(want).max(), act
    want = oracle.attention(batch, seq, a, k, d, X, Wq, Wk, Wv, Wo)
    got = oracle.attention_composed(batch, seq, a, k, d, X, Wq, Wk, Wv, Wo)
    assert np.abs(got - want).max() < 1e-12 * np.abs(want).max()
    want = oracle.layer(batch, seq, a, k, d, 2, X, Wq, Wk, Wv, Wo, W1, W3, W2)
    got, h1 = oracle.layer_composed(batch, seq, a, k, d, X, Wq, Wk, Wv, Wo, W1, W3, W2, want_h1=True)
    assert np.abs(got - want).max() < 1e-12 * np.abs(want).max()
    h1_want = X + oracle.attention(batch, seq, a, k, d, oracle.rmsnorm(X), Wq, Wk, Wv, Wo)
    assert np.abs(h1 - h1_want).max() < 1e-12 * np.abs(h1_want).max()
    with pytest.raises(ValueError):
        oracle.mlp_composed("relu", X, W1, W2)


def test_composed_mlp_backward_equals_c_form():
    g = torch.Generator().manual_seed(94)
    M, h, f = 11, 12, 20
    X = torch.randn(M, h, generator=g, dtype=torch.float64).numpy()
    rnd = lambda n, m: (torch.randn(n, m, generator=g, dtype=torch.float64) * 0.5).numpy()
    W1, W3, W2 = rnd(f, h), rnd(f, h), rnd(h, f)
    dZ = torch.randn(M, h, generator=g, dtype=torch.float64).numpy()
    want = oracle.mlp_backward("swiglu", X, W1, W2, dZ, W3)
    got = oracle.mlp_backward_composed(X, W1, W2, dZ, W3)
    for n, x, y in zip(("dX", "dW1", "dW3", "dW2", "db2"), want, got):
        assert np.abs(x - y).max() < 1e-12 * max(1.0, np.abs(x).max()), n


def _torch_to_split(Y, batch, seq, t):
    """Token-order [batch seq][h] -> sequence-split [t][batch][seq/t][h], by
    its definition: shard i holds positions [i seq/t, (i+1) seq/t) of every
    sequence ("시퀀스 병렬화")."""
    h = Y.shape[1]
    return Y.reshape(batch, t, seq // t, h).permute(1, 0, 2, 3).reshape(batch * seq, h)


def _torch_from_split(Y_sp, batch, seq, t):
    h = Y_sp.shape[1]
    return Y_sp.reshape(t, batch, seq // t, h).permute(1, 0, 2, 3).reshape(batch * seq, h)


def test_sequence_parallel_layer_backward_matches_torch_autograd():
    # The split-layout layer: gather X_sp into token order, run the layer,
    # split the output.  Autograd through that composition gives dX_sp and
    # the weight gradients; the oracle's form must equal it, and its weight
    # gradients must equal the replicated layer's.
    g = torch.Generator().manual_seed(95)
    batch, seq, t, h, a, k, d, f = 2, 8, 4, 8, 4, 2, 2, 16
    M = batch * seq
    X_sp = torch.randn(M, h, generator=g, dtype=torch.float64).requires_grad_(True)
    shapes = [(a * d, h), (k * d, h), (k * d, h), (h, a * d), (f, h), (f, h), (h, f)]
    W = [(torch.randn(*s, generator=g, dtype=torch.float64) * 0.4).requires_grad_(True) for s in shapes]
    dY_sp = torch.randn(M, h, generator=g, dtype=torch.float64)
    Y_sp = _torch_to_split(_torch_layer(batch, seq, a, k, _torch_from_split(X_sp, batch, seq, t), *W), batch, seq, t)
    Y_sp.backward(dY_sp)
    got = oracle.layer_sp_backward(batch, seq, a, k, d, t, X_sp.detach(), *(w.detach() for w in W), dY_sp)
    want = [X_sp.grad] + [w.grad for w in W]
    names = ["dX", "dWq", "dWk", "dWv", "dWo", "dW1", "dW3", "dW2"]
    for n, x, ref in zip(names, got, want):
        assert np.abs(x - ref.numpy()).max() < 1e-11 * max(1.0, ref.abs().max().item()), n
    # the split of a token-order tensor is the inverse of the all-gather
    Z = torch.randn(M, h, generator=g, dtype=torch.float64)
    assert np.array_equal(oracle.sp_split(batch, seq, t, Z), _torch_to_split(Z, batch, seq, t).numpy())
    comp = oracle.layer_sp_backward(batch, seq, a, k, d, t, X_sp.detach(), *(w.detach() for w in W), dY_sp,
                                    composed=True)
    for n, x, y in zip(names, got, comp):
        assert np.abs(x - y).max() < 1e-11 * max(1.0, np.abs(x).max()), n + " (composed)"
