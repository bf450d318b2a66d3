"""ctypes binding of the fp64 CPU oracle (``tp_oracle.c``).

TEST INFRASTRUCTURE.  Only the test-suite, ``__graft_entry__.smoke()`` and the
bench's CPU-baseline leg may import this package.  It is independent of the
CUDA path: it shares no code with it and never imports it.

Inputs are numpy arrays (converted to contiguous float64); results are float64
numpy arrays.  Layouts follow the C source: row-major, weights ``W[out, in]``.
Each wrapper cites the passage its C routine follows (see ``tp_oracle.c``).
"""
from __future__ import annotations

import ctypes as C
import os
from typing import Optional, Sequence

import numpy as np

from . import build as _build

OK = 0
ERR_INVALID = 1
ERR_NOT_DIVISIBLE = 2
ERR_NOMEM = 3

ACT = {"gelu": 0, "gelu_tanh": 1, "swiglu": 2, "none": 3}

_lib = None
_D = C.POINTER(C.c_double)
_F = C.POINTER(C.c_float)
_I64 = C.c_int64


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = C.CDLL(path)
        sig = {
            "tpo_num_threads": (C.c_int, []),
            "tpo_gelu_erf": (C.c_double, [C.c_double]),
            "tpo_gelu_tanh": (C.c_double, [C.c_double]),
            "tpo_silu": (C.c_double, [C.c_double]),
            "tpo_round_bf16": (C.c_uint16, [C.c_double]),
            "tpo_linear": (None, [_D, _I64, _D, _I64, _I64, _I64, _I64, _D, _I64]),
            "tpo_mlp": (C.c_int, [C.c_int, _I64, _I64, _I64, _D, _D, _D, _D, _D]),
            "tpo_mlp_sharded": (C.c_int, [C.c_int, _I64, _I64, _I64, _I64, _D, _D, _D, _D, _D, _D]),
            "tpo_mlp_worked_f32": (C.c_int, [C.c_int, _I64, _I64, _I64, _I64, _F, _F, _F, _F]),
            "tpo_plan_check": (C.c_int, [_I64] * 6),
            "tpo_q_head_shard": (_I64, [_I64] * 3),
            "tpo_q_head_kv": (_I64, [_I64] * 3),
            "tpo_shard_kv_first": (_I64, [_I64] * 3),
            "tpo_shard_kv_count": (_I64, [_I64] * 2),
            "tpo_attention_core": (C.c_int, [_I64] * 5 + [_D, _I64, _D, _D, _I64, _D, _I64]),
            "tpo_attention": (C.c_int, [_I64] * 6 + [_D] * 7),
            "tpo_attention_sharded": (C.c_int, [_I64] * 7 + [_D] * 7),
            "tpo_reduce": (C.c_int, [_I64] * 3 + [_D] * 4),
            "tpo_rmsnorm": (C.c_int, [_I64, _I64, C.c_double, _D, _D]),
            "tpo_layer": (C.c_int, [_I64] * 8 + [C.c_int, C.c_double] + [_D] * 9),
            "tpo_layer_rows": (C.c_int, [_I64] * 7 + [C.c_double] + [_D] * 8
                               + [_I64, C.POINTER(C.c_int64), _D]),
            "tpo_attention_rows": (C.c_int, [_I64] * 6 + [_D] * 5
                                   + [_I64, C.POINTER(C.c_int64), _D]),
            "tpo_packed_shard_rows": (C.c_int, [C.POINTER(C.c_int64), _I64, _I64, _I64,
                                                C.POINTER(C.c_int64)]),
            "tpo_mlp_packed_gate_up": (C.c_int, [C.c_int] + [_I64] * 4 + [_D] * 4),
            "tpo_embedding_vocab_parallel": (C.c_int, [_I64] * 4 + [C.POINTER(C.c_int32), _D, _D]),
            "tpo_cross_entropy": (C.c_int, [_I64, _I64, _D, C.POINTER(C.c_int32), _D]),
            "tpo_cross_entropy_vocab_parallel": (C.c_int, [_I64] * 3 + [_D, C.POINTER(C.c_int32),
                                                                        _D, _D]),
            "tpo_sp_row": (_I64, [_I64] * 5),
            "tpo_sp_all_gather": (C.c_int, [_I64] * 4 + [_D, _D]),
            "tpo_sp_reduce_scatter": (C.c_int, [_I64] * 4 + [_D, _D]),
            "tpo_layer_sp": (C.c_int, [_I64] * 8 + [C.c_double] + [_D] * 9),
            "tpo_mlp_backward": (C.c_int, [C.c_int] + [_I64] * 3 + [_D] * 10),
            "tpo_rmsnorm_backward": (C.c_int, [_I64, _I64, C.c_double, _D, _D, _D]),
            "tpo_layer_backward": (C.c_int, [_I64] * 7 + [C.c_double] + [_D] * 17),
            "tpo_attention_core_backward": (C.c_int, [_I64] * 5 + [_D, _I64, _D, _D, _I64, _D, _I64, _D, _D, _D]),
            "tpo_attention_backward": (C.c_int, [_I64] * 6 + [_D] * 11),
            "tpo_attention_backward_sharded": (C.c_int, [_I64] * 7 + [_D] * 12),
            "tpo_mlp_backward_sharded": (C.c_int, [C.c_int] + [_I64] * 4 + [_D] * 11),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


class OracleError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} returned {code}")
        self.code = code


def _d(a) -> np.ndarray:
    if a is None:
        return None
    if hasattr(a, "detach"):  # torch tensor -> float64 numpy (exact widening of bf16/fp32)
        a = a.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(a, dtype=np.float64)


def _p(a):
    return None if a is None else a.ctypes.data_as(_D)


def _check(fn, rc):
    if rc != OK:
        raise OracleError(fn, rc)


def num_threads() -> int:
    return lib().tpo_num_threads()


def gelu_erf(x: float) -> float:
    return lib().tpo_gelu_erf(float(x))


def gelu_tanh(x: float) -> float:
    return lib().tpo_gelu_tanh(float(x))


def silu(x: float) -> float:
    return lib().tpo_silu(float(x))


def round_bf16_bits(values) -> np.ndarray:
    """bf16 bit patterns (uint16) of values, round-to-nearest-even."""
    v = np.asarray(values, dtype=np.float64).ravel()
    L = lib()
    return np.array([L.tpo_round_bf16(float(x)) for x in v], dtype=np.uint16)


def linear(X, W) -> np.ndarray:
    """Y = X W^T."""
    X, W = _d(X), _d(W)
    M, K = X.shape
    N = W.shape[0]
    Y = np.empty((M, N))
    lib().tpo_linear(_p(X), K, _p(W), W.shape[1], M, N, K, _p(Y), N)
    return Y


def mlp(act: str, X, W1, W2, W3=None) -> np.ndarray:
    """Unsharded MLP: act(X W1^T [(.) X W3^T]) W2^T."""
    X, W1, W2, W3 = _d(X), _d(W1), _d(W2), _d(W3)
    M, h = X.shape
    f = W1.shape[0]
    Z = np.empty((M, h))
    _check("tpo_mlp", lib().tpo_mlp(ACT[act], M, h, f, _p(X), _p(W1), _p(W3), _p(W2), _p(Z)))
    return Z


def mlp_sharded(act: str, t: int, X, W1, W2, W3=None, want_partials: bool = False):
    """Literal t-shard MLP: sum_i act(X W1_i^T [(.) X W3_i^T]) W2_i^T."""
    X, W1, W2, W3 = _d(X), _d(W1), _d(W2), _d(W3)
    M, h = X.shape
    f = W1.shape[0]
    Z = np.empty((M, h))
    P = np.empty((t, M, h)) if want_partials else None
    _check("tpo_mlp_sharded", lib().tpo_mlp_sharded(ACT[act], M, h, f, t, _p(X), _p(W1), _p(W3),
                                                     _p(W2), _p(P), _p(Z)))
    return (Z, P) if want_partials else Z


def mlp_worked_f32(sharded: bool, t: int, X, A, B) -> np.ndarray:
    """fp32 restatement of the page's worked example (A[h,f], B[f,h])."""
    X = np.ascontiguousarray(X, dtype=np.float32)
    A = np.ascontiguousarray(A, dtype=np.float32)
    B = np.ascontiguousarray(B, dtype=np.float32)
    b, h = X.shape
    f = A.shape[1]
    Z = np.empty((b, h), dtype=np.float32)
    _check("tpo_mlp_worked_f32", lib().tpo_mlp_worked_f32(
        1 if sharded else 0, b, h, f, t, X.ctypes.data_as(_F), A.ctypes.data_as(_F),
        B.ctypes.data_as(_F), Z.ctypes.data_as(_F)))
    return Z


def plan_check(h: int, f: int, a: int, k: int, d: int, t: int) -> int:
    return lib().tpo_plan_check(h, f, a, k, d, t)


def q_head_shard(a: int, t: int, j: int) -> int:
    return lib().tpo_q_head_shard(a, t, j)


def q_head_kv(a: int, k: int, j: int) -> int:
    return lib().tpo_q_head_kv(a, k, j)


def shard_kv_first(k: int, t: int, i: int) -> int:
    return lib().tpo_shard_kv_first(k, t, i)


def shard_kv_count(k: int, t: int) -> int:
    return lib().tpo_shard_kv_count(k, t)


def attention_core(batch: int, seq: int, a: int, k: int, d: int, Q, K, V) -> np.ndarray:
    """Causal GQA attention core: Q[M, a d], K/V[M, k d] -> O[M, a d]."""
    Q, K, V = _d(Q), _d(K), _d(V)
    M = batch * seq
    O = np.empty((M, a * d))
    _check("tpo_attention_core", lib().tpo_attention_core(
        batch, seq, a, k, d, _p(Q), Q.shape[1], _p(K), _p(V), K.shape[1], _p(O), a * d))
    return O


def attention(batch: int, seq: int, a: int, k: int, d: int, X, Wq, Wk, Wv, Wo,
              want_O: bool = False):
    """Unsharded attention block: (causal GQA attn of X Wq^T, X Wk^T, X Wv^T) Wo^T."""
    X, Wq, Wk, Wv, Wo = map(_d, (X, Wq, Wk, Wv, Wo))
    M, h = X.shape
    out = np.empty((M, h))
    O = np.empty((M, a * d)) if want_O else None
    _check("tpo_attention", lib().tpo_attention(batch, seq, h, a, k, d, _p(X), _p(Wq), _p(Wk),
                                                _p(Wv), _p(Wo), _p(O), _p(out)))
    return (out, O) if want_O else out


def attention_sharded(batch: int, seq: int, a: int, k: int, d: int, t: int, X, Wq, Wk, Wv, Wo,
                      want_partials: bool = False):
    """Literal head-sharded attention block, out = sum_i O_i Wo_i^T."""
    X, Wq, Wk, Wv, Wo = map(_d, (X, Wq, Wk, Wv, Wo))
    M, h = X.shape
    out = np.empty((M, h))
    P = np.empty((t, M, h)) if want_partials else None
    _check("tpo_attention_sharded", lib().tpo_attention_sharded(
        batch, seq, h, a, k, d, t, _p(X), _p(Wq), _p(Wk), _p(Wv), _p(Wo), _p(P), _p(out)))
    return (out, P) if want_partials else out


def reduce(partials, bias=None, residual=None) -> np.ndarray:
    """g forward: sum_i partials[i] (+ bias once) (+ residual)."""
    P = _d(partials)
    t = P.shape[0]
    h = P.shape[-1]
    n = int(np.prod(P.shape[1:]))
    b, r = _d(bias), _d(residual)
    out = np.empty(P.shape[1:])
    _check("tpo_reduce", lib().tpo_reduce(t, n, h, _p(P), _p(b), _p(r), _p(out)))
    return out


def rmsnorm(x, eps: float = 1e-5) -> np.ndarray:
    x = _d(x)
    M, h = x.shape
    y = np.empty_like(x)
    _check("tpo_rmsnorm", lib().tpo_rmsnorm(M, h, float(eps), _p(x), _p(y)))
    return y


def layer(batch: int, seq: int, a: int, k: int, d: int, t: int, X, Wq, Wk, Wv, Wo, W1, W3, W2,
          sharded: bool = False, eps: float = 1e-5) -> np.ndarray:
    """Pre-norm layer: h1 = x + Attn(RMSNorm(x)); y = h1 + SwiGLU-MLP(RMSNorm(h1))."""
    X, Wq, Wk, Wv, Wo, W1, W3, W2 = map(_d, (X, Wq, Wk, Wv, Wo, W1, W3, W2))
    M, h = X.shape
    f = W1.shape[0]
    Y = np.empty((M, h))
    _check("tpo_layer", lib().tpo_layer(batch, seq, h, a, k, d, f, t, 1 if sharded else 0,
                                        float(eps), _p(X), _p(Wq), _p(Wk), _p(Wv), _p(Wo),
                                        _p(W1), _p(W3), _p(W2), _p(Y)))
    return Y


def _rows(rows: Sequence[int]):
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    return r, r.ctypes.data_as(C.POINTER(C.c_int64))


def layer_rows(batch: int, seq: int, a: int, k: int, d: int, X, Wq, Wk, Wv, Wo, W1, W3, W2,
               rows: Sequence[int], eps: float = 1e-5) -> np.ndarray:
    """The layer's output at chosen token rows only (exact same definition)."""
    X, Wq, Wk, Wv, Wo, W1, W3, W2 = map(_d, (X, Wq, Wk, Wv, Wo, W1, W3, W2))
    h = X.shape[1]
    f = W1.shape[0]
    r, rp = _rows(rows)
    Y = np.empty((len(r), h))
    _check("tpo_layer_rows", lib().tpo_layer_rows(batch, seq, h, a, k, d, f, float(eps), _p(X),
                                                  _p(Wq), _p(Wk), _p(Wv), _p(Wo), _p(W1),
                                                  _p(W3), _p(W2), len(r), rp, _p(Y)))
    return Y


def attention_rows(batch: int, seq: int, a: int, k: int, d: int, X, Wq, Wk, Wv, Wo,
                   rows: Sequence[int]) -> np.ndarray:
    """The attention block's output at chosen token rows only."""
    X, Wq, Wk, Wv, Wo = map(_d, (X, Wq, Wk, Wv, Wo))
    h = X.shape[1]
    r, rp = _rows(rows)
    out = np.empty((len(r), h))
    _check("tpo_attention_rows", lib().tpo_attention_rows(batch, seq, h, a, k, d, _p(X), _p(Wq),
                                                          _p(Wk), _p(Wv), _p(Wo), len(r), rp,
                                                          _p(out)))
    return out


def packed_shard_rows(blocks: Sequence[int], t: int, i: int) -> np.ndarray:
    """Rows of a packed weight device i holds under per-block sharding."""
    b = np.ascontiguousarray(np.asarray(blocks, dtype=np.int64))
    out = np.empty(max(1, int(sum(int(x) // max(t, 1) for x in blocks))), dtype=np.int64)
    rc = lib().tpo_packed_shard_rows(b.ctypes.data_as(C.POINTER(C.c_int64)), len(b), t, i,
                                     out.ctypes.data_as(C.POINTER(C.c_int64)))
    _check("tpo_packed_shard_rows", rc)
    return out[: sum(int(x) // t for x in blocks)]


def packed_check(blocks: Sequence[int], t: int) -> int:
    """OK, or ERR_NOT_DIVISIBLE when any packed block does not divide by t."""
    b = np.ascontiguousarray(np.asarray(blocks, dtype=np.int64))
    return lib().tpo_packed_shard_rows(b.ctypes.data_as(C.POINTER(C.c_int64)), len(b), t, 0, None)


def mlp_packed_gate_up(per_block: bool, t: int, X, Wgu, W2) -> np.ndarray:
    """SwiGLU MLP from a packed [gate; up] weight, sharded per block (correct)
    or by contiguous rows of the packed tensor (the misplacement)."""
    X, Wgu, W2 = _d(X), _d(Wgu), _d(W2)
    M, h = X.shape
    f = Wgu.shape[0] // 2
    Z = np.empty((M, h))
    _check("tpo_mlp_packed_gate_up", lib().tpo_mlp_packed_gate_up(
        1 if per_block else 0, M, h, f, t, _p(X), _p(Wgu), _p(W2), _p(Z)))
    return Z


def _i32(a):
    if hasattr(a, "detach"):
        a = a.detach().to("cpu").numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def embedding_vocab_parallel(t: int, ids, E) -> np.ndarray:
    """Sum over devices of the masked partial lookups of a vocab-split E[v][h]."""
    ids, E = _i32(ids).ravel(), _d(E)
    v, h = E.shape
    out = np.empty((len(ids), h))
    _check("tpo_embedding_vocab_parallel", lib().tpo_embedding_vocab_parallel(
        len(ids), v, h, t, ids.ctypes.data_as(C.POINTER(C.c_int32)), _p(E), _p(out)))
    return out


def cross_entropy(logits, labels) -> np.ndarray:
    """Per-token log-sum-exp minus the label's logit (ignore index -100 -> 0)."""
    z, lab = _d(logits), _i32(labels).ravel()
    M, v = z.shape
    loss = np.empty(M)
    _check("tpo_cross_entropy", lib().tpo_cross_entropy(
        M, v, _p(z), lab.ctypes.data_as(C.POINTER(C.c_int32)), _p(loss)))
    return loss


def cross_entropy_vocab_parallel(t: int, logits, labels, want_stats: bool = False):
    """loss_parallel: per-device (max, sum, target) exchanged, then combined."""
    z, lab = _d(logits), _i32(labels).ravel()
    M, v = z.shape
    loss = np.empty(M)
    st = np.empty((3, t, M)) if want_stats else None
    _check("tpo_cross_entropy_vocab_parallel", lib().tpo_cross_entropy_vocab_parallel(
        M, v, t, _p(z), lab.ctypes.data_as(C.POINTER(C.c_int32)), _p(st), _p(loss)))
    return (loss, st) if want_stats else loss


def sp_row(batch: int, seq: int, t: int, b: int, pos: int) -> int:
    """Row of token (b, pos) in the sequence-split layout [t][batch][s/t]."""
    return lib().tpo_sp_row(batch, seq, t, b, pos)


def sp_all_gather(batch: int, seq: int, t: int, sp) -> np.ndarray:
    sp = _d(sp)
    h = sp.shape[1]
    full = np.empty_like(sp)
    _check("tpo_sp_all_gather", lib().tpo_sp_all_gather(batch, seq, t, h, _p(sp), _p(full)))
    return full


def sp_reduce_scatter(batch: int, seq: int, t: int, partials) -> np.ndarray:
    P = _d(partials)
    h = P.shape[-1]
    out = np.empty((batch * seq, h))
    _check("tpo_sp_reduce_scatter", lib().tpo_sp_reduce_scatter(batch, seq, t, h, _p(P), _p(out)))
    return out


def layer_sp(batch: int, seq: int, a: int, k: int, d: int, t: int, X_sp, Wq, Wk, Wv, Wo, W1, W3,
             W2, eps: float = 1e-5) -> np.ndarray:
    """Sequence-parallel pre-norm layer; X_sp and the result in [t][batch][s/t][h]."""
    X, Wq, Wk, Wv, Wo, W1, W3, W2 = map(_d, (X_sp, Wq, Wk, Wv, Wo, W1, W3, W2))
    M, h = X.shape
    f = W1.shape[0]
    Y = np.empty((M, h))
    _check("tpo_layer_sp", lib().tpo_layer_sp(batch, seq, h, a, k, d, f, t, float(eps), _p(X),
                                              _p(Wq), _p(Wk), _p(Wv), _p(Wo), _p(W1), _p(W3),
                                              _p(W2), _p(Y)))
    return Y


def mlp_backward(act: str, X, W1, W2, dZ, W3=None, t: int = 0, want_partials: bool = False):
    """Gradients (dX, dW1, dW3, dW2, db2) of the MLP given dZ (db2: of a bias
    added once to Z); t > 0 uses the literal t-device form (g backward =
    identity, f backward = all-reduce)."""
    X, W1, W2, dZ, W3 = map(_d, (X, W1, W2, dZ, W3))
    M, h = X.shape
    f = W1.shape[0]
    dX = np.empty((M, h))
    dW1 = np.empty((f, h))
    dW3 = np.empty((f, h)) if act == "swiglu" else None
    dW2 = np.empty((h, f))
    db2 = np.empty(h)
    if t:
        P = np.empty((t, M, h)) if want_partials else None
        _check("tpo_mlp_backward_sharded", lib().tpo_mlp_backward_sharded(
            ACT[act], M, h, f, t, _p(X), _p(W1), _p(W3), _p(W2), _p(dZ), _p(P), _p(dX), _p(dW1),
            _p(dW3), _p(dW2), _p(db2)))
        out = (dX, dW1, dW3, dW2, db2)
        return out + (P,) if want_partials else out
    _check("tpo_mlp_backward", lib().tpo_mlp_backward(
        ACT[act], M, h, f, _p(X), _p(W1), _p(W3), _p(W2), _p(dZ), _p(dX), _p(dW1), _p(dW3), _p(dW2),
        _p(db2)))
    return dX, dW1, dW3, dW2, db2


def attention_core_backward(batch: int, seq: int, a: int, k: int, Q, K, V, dO):
    """(dQ, dK, dV) of the causal GQA attention core; Q, dO [M][a d], K, V [M][k d]."""
    Q, K, V, dO = map(_d, (Q, K, V, dO))
    d = Q.shape[1] // a
    dQ, dK, dV = np.empty_like(Q), np.empty_like(K), np.empty_like(V)
    _check("tpo_attention_core_backward", lib().tpo_attention_core_backward(
        batch, seq, a, k, d, _p(Q), Q.shape[1], _p(K), _p(V), K.shape[1], _p(dO), dO.shape[1],
        _p(dQ), _p(dK), _p(dV)))
    return dQ, dK, dV


def attention_backward(batch: int, seq: int, a: int, k: int, X, Wq, Wk, Wv, Wo, dOut, t: int = 0,
                       want_partials: bool = False):
    """(dX, dWq, dWk, dWv, dWo) of the attention block given dOut; t > 0 uses
    the literal t-device form (same dOut per device, dX = sum of partials,
    replicated KV-head gradients summed)."""
    X, Wq, Wk, Wv, Wo, dOut = map(_d, (X, Wq, Wk, Wv, Wo, dOut))
    M, h = X.shape
    d = Wq.shape[0] // a
    dX = np.empty((M, h))
    dWq, dWk, dWv, dWo = (np.empty_like(w) for w in (Wq, Wk, Wv, Wo))
    if t:
        P = np.empty((t, M, h)) if want_partials else None
        _check("tpo_attention_backward_sharded", lib().tpo_attention_backward_sharded(
            batch, seq, h, a, k, d, t, _p(X), _p(Wq), _p(Wk), _p(Wv), _p(Wo), _p(dOut), _p(P),
            _p(dX), _p(dWq), _p(dWk), _p(dWv), _p(dWo)))
        out = (dX, dWq, dWk, dWv, dWo)
        return out + (P,) if want_partials else out
    _check("tpo_attention_backward", lib().tpo_attention_backward(
        batch, seq, h, a, k, d, _p(X), _p(Wq), _p(Wk), _p(Wv), _p(Wo), _p(dOut), _p(dX), _p(dWq),
        _p(dWk), _p(dWv), _p(dWo)))
    return dX, dWq, dWk, dWv, dWo


def attention_backward_composed(batch: int, seq: int, a: int, k: int, X, Wq, Wk, Wv, Wo, dOut):
    """The plain attention-block backward of tpo_attention_backward, composed
    for large sizes: the projections are library matmuls (numpy, fp64) and
    the attention core forward and backward are the C oracle's.  Same
    definition, same order of steps; returns (dX, dWq, dWk, dWv, dWo)."""
    X, Wq, Wk, Wv, Wo, dOut = map(_d, (X, Wq, Wk, Wv, Wo, dOut))
    d = Wq.shape[0] // a
    Q, K, V = X @ Wq.T, X @ Wk.T, X @ Wv.T
    O = attention_core(batch, seq, a, k, d, Q, K, V)
    dO = dOut @ Wo
    dWo = dOut.T @ O
    dQ, dK, dV = attention_core_backward(batch, seq, a, k, Q, K, V, dO)
    dX = dQ @ Wq + dK @ Wk + dV @ Wv
    return dX, dQ.T @ X, dK.T @ X, dV.T @ X, dWo


def rmsnorm_backward(x, g, eps: float = 1e-5) -> np.ndarray:
    """dL/dx of the unit-gain RMSNorm at x for the upstream g."""
    x, g = _d(x), _d(g)
    out = np.zeros_like(x)
    _check("tpo_rmsnorm_backward", lib().tpo_rmsnorm_backward(x.shape[0], x.shape[1], eps, _p(x), _p(g), _p(out)))
    return out


def layer_backward(batch: int, seq: int, a: int, k: int, d: int, X, Wq, Wk, Wv, Wo, W1, W3, W2, dY,
                   eps: float = 1e-5):
    """(dX, dWq, dWk, dWv, dWo, dW1, dW3, dW2) of the pre-norm SwiGLU layer."""
    X, Wq, Wk, Wv, Wo, W1, W3, W2, dY = map(_d, (X, Wq, Wk, Wv, Wo, W1, W3, W2, dY))
    M, h = X.shape
    f = W1.shape[0]
    outs = [np.empty((M, h))] + [np.empty_like(w) for w in (Wq, Wk, Wv, Wo, W1, W3, W2)]
    _check("tpo_layer_backward", lib().tpo_layer_backward(
        batch, seq, h, a, k, d, f, eps, _p(X), _p(Wq), _p(Wk), _p(Wv), _p(Wo), _p(W1), _p(W3), _p(W2),
        _p(dY), *(_p(o) for o in outs)))
    return tuple(outs)


def layer_backward_composed(batch: int, seq: int, a: int, k: int, d: int, X, Wq, Wk, Wv, Wo, W1, W3,
                            W2, dY, eps: float = 1e-5):
    """tpo_layer_backward's steps for large sizes: numpy matmuls for the
    projections and the MLP, the C oracle for the attention core and the norms."""
    X, Wq, Wk, Wv, Wo, W1, W3, W2, dY = map(_d, (X, Wq, Wk, Wv, Wo, W1, W3, W2, dY))
    xn1 = rmsnorm(X, eps)
    Q, K, V = xn1 @ Wq.T, xn1 @ Wk.T, xn1 @ Wv.T
    h1 = X + attention_core(batch, seq, a, k, d, Q, K, V) @ Wo.T
    xn2 = rmsnorm(h1, eps)
    U, G = xn2 @ W1.T, xn2 @ W3.T
    s = 1.0 / (1.0 + np.exp(-U))
    H = U * s * G
    dH = dY @ W2
    dU = dH * G * s * (1.0 + U * (1.0 - s))
    dG = dH * U * s
    dxn2 = dU @ W1 + dG @ W3
    grads_mlp = (dU.T @ xn2, dG.T @ xn2, dY.T @ H)
    dh1 = dY + rmsnorm_backward(h1, dxn2, eps)
    dxn1, dWq, dWk, dWv, dWo = attention_backward_composed(batch, seq, a, k, xn1, Wq, Wk, Wv, Wo, dh1)
    dX = dh1 + rmsnorm_backward(X, dxn1, eps)
    return (dX, dWq, dWk, dWv, dWo) + grads_mlp


# ---------------------------------------------------------------- composed forms for full sizes
#
# The same definitions as tpo_mlp, tpo_attention, tpo_layer and
# tpo_mlp_backward, with every matrix product taken by numpy's matmul (a
# library primitive used as a step) instead of the plain loops, so that the
# workloads' full sizes (up to 8192 tokens x 14336 ffn) finish in seconds
# rather than minutes.  The attention core and the norms stay in the C
# routines.  Each form is pinned to its all-C counterpart at small sizes.

def _act_np(act: str, U, G=None):
    """The activation step of "MLP" ("텐서 병렬화"), elementwise in fp64."""
    if act == "gelu":
        from scipy.special import erf
        return 0.5 * U * (1.0 + erf(U / np.sqrt(2.0)))
    if act == "gelu_tanh":
        c = np.sqrt(2.0 / np.pi)
        return 0.5 * U * (1.0 + np.tanh(c * (U + 0.044715 * U * U * U)))
    if act == "swiglu":
        return U / (1.0 + np.exp(-U)) * G
    if act == "none":
        return U
    raise ValueError(f"unknown activation {act!r}; valid: gelu, gelu_tanh, swiglu, none")


def mlp_composed(act: str, X, W1, W2, W3=None) -> np.ndarray:
    """Unsharded MLP of tpo_mlp ("MLP": Z = act(X W1^T [(.) X W3^T]) W2^T),
    matrix products by numpy."""
    X, W1, W2, W3 = _d(X), _d(W1), _d(W2), _d(W3)
    U = X @ W1.T
    G = X @ W3.T if act == "swiglu" else None
    return _act_np(act, U, G) @ W2.T


def attention_composed(batch: int, seq: int, a: int, k: int, d: int, X, Wq, Wk, Wv, Wo) -> np.ndarray:
    """Unsharded attention block of tpo_attention ("셀프 어텐션"): projections
    by numpy, the causal GQA core by tpo_attention_core."""
    X, Wq, Wk, Wv, Wo = map(_d, (X, Wq, Wk, Wv, Wo))
    O = attention_core(batch, seq, a, k, d, X @ Wq.T, X @ Wk.T, X @ Wv.T)
    return O @ Wo.T


def layer_composed(batch: int, seq: int, a: int, k: int, d: int, X, Wq, Wk, Wv, Wo, W1, W3, W2,
                   eps: float = 1e-5, want_h1: bool = False):
    """Pre-norm layer of tpo_layer ("통신 연산 f와 g": norm and residual
    replicated): h1 = x + Attn(RMSNorm(x)), y = h1 + SwiGLU-MLP(RMSNorm(h1)).
    With want_h1, also returns the residual stream h1."""
    X = _d(X)
    h1 = X + attention_composed(batch, seq, a, k, d, rmsnorm(X, eps), Wq, Wk, Wv, Wo)
    Y = h1 + mlp_composed("swiglu", rmsnorm(h1, eps), W1, W2, W3)
    return (Y, h1) if want_h1 else Y


def mlp_backward_composed(X, W1, W2, dZ, W3):
    """(dX, dW1, dW3, dW2, db2) of the SwiGLU MLP given dZ, the steps of
    tpo_mlp_backward with the matrix products by numpy:
      U = X W1^T, G = X W3^T, H = SiLU(U) (.) G, Z = H W2^T (+ b2)
      dH = dZ W2, dU = dH (.) G (.) SiLU'(U), dG = dH (.) SiLU(U)
      dX = dU W1 + dG W3, dW1 = dU^T X, dW3 = dG^T X, dW2 = dZ^T H,
      db2 = sum over tokens of dZ."""
    X, W1, W2, dZ, W3 = map(_d, (X, W1, W2, dZ, W3))
    U, G = X @ W1.T, X @ W3.T
    s = 1.0 / (1.0 + np.exp(-U))
    H = U * s * G
    dH = dZ @ W2
    dU = dH * G * s * (1.0 + U * (1.0 - s))
    dG = dH * U * s
    return (dU @ W1 + dG @ W3, dU.T @ X, dG.T @ X, dZ.T @ H, dZ.sum(axis=0))


def sp_split(batch: int, seq: int, t: int, full) -> np.ndarray:
    """A token-order tensor [batch seq][h] in the sequence-split layout
    [t][batch][seq/t][h] (row of token (b, pos) from tpo_sp_row)."""
    full = _d(full)
    out = np.empty_like(full)
    rows = [sp_row(batch, seq, t, b, pos) for b in range(batch) for pos in range(seq)]
    out[rows] = full
    return out


def layer_sp_backward(batch: int, seq: int, a: int, k: int, d: int, t: int, X_sp, Wq, Wk, Wv, Wo, W1, W3, W2,
                      dY_sp, eps: float = 1e-5, composed: bool = False):
    """(dX_sp, dWq, dWk, dWv, dWo, dW1, dW3, dW2) of the sequence-parallel
    pre-norm layer ("텐서 병렬화", "시퀀스 병렬화"): X_sp, dY_sp and dX_sp in
    the split layout [t][batch][seq/t][h].  The forward's all-gather of each
    block's input has a reduce-scatter as its backward and its reduce-scatter
    an all-gather, so: dY is all-gathered, the layer's backward runs on the
    token-order tensors (the replicated layer's, whose dX already holds the
    shards' sum), and dX is scattered into the split layout.  composed: use
    layer_backward_composed (numpy matrix products) for large sizes."""
    X = sp_all_gather(batch, seq, t, X_sp)
    dY = sp_all_gather(batch, seq, t, dY_sp)
    fn = layer_backward_composed if composed else layer_backward
    out = fn(batch, seq, a, k, d, X, Wq, Wk, Wv, Wo, W1, W3, W2, dY, eps=eps)
    return (sp_split(batch, seq, t, out[0]),) + tuple(out[1:])
