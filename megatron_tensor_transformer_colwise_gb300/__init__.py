"""Python binding of libtp.so, the sm_103a tensor-parallel block library.

Argument marshalling only: every function here forwards to the ``extern "C"``
entry point of the same name declared in ``include/tp.h``; all compute runs
in the library's CUDA kernels.  Tensors are passed as device pointers
(``tensor.data_ptr()``), streams as ``cudaStream_t`` handles (default: torch's
current stream).  PyTorch is used only for memory and streams.

There is no CPU path: if the library cannot be loaded, every call raises.
"""
from __future__ import annotations

import ctypes as C
import os
from typing import Optional

from . import _build

__all__ = [
    "TPError", "TPConfig", "TPLayerWeights", "Plan", "lib", "build",
    "TP_OK", "TP_ERR_INVALID_ARG", "TP_ERR_NOT_DIVISIBLE", "TP_ERR_UNSUPPORTED",
    "TP_ERR_WORKSPACE", "TP_ERR_CUDA", "TP_ERR_DEVICE_TIMEOUT",
    "TP_ACT_GELU_ERF", "TP_ACT_GELU_TANH", "TP_ACT_SWIGLU", "TP_ACT_NONE",
    "TP_REDUCE_FUSED", "TP_REDUCE_PARTIALS", "TP_F32", "TP_BF16",
    "TP_OP_MLP", "TP_OP_ATTN", "TP_OP_LAYER", "TP_OP_MLP_BACKWARD", "TP_OP_ATTN_BACKWARD",
    "TP_OP_LAYER_BACKWARD", "TPLayerGrads",
    "TP_TABLE_FFN_SHARDS", "TP_TABLE_Q_HEAD_SHARD", "TP_TABLE_Q_HEAD_KV",
    "TP_TABLE_SHARD_KV", "TP_TABLE_QKV_COLUMNS",
    "tp_plan_create", "tp_plan_destroy", "tp_config_check", "tp_config_shard_table",
    "tp_plan_workspace_bytes", "tp_plan_shard_table", "tp_get_device_status", "tp_last_error",
    "tp_reduce_partials", "tp_rmsnorm", "tp_colwise_forward", "tp_rowwise_forward",
    "tp_mlp_forward", "tp_mlp_forward_noalloc", "tp_qkv_forward", "tp_attn_core_forward", "tp_attn_forward",
    "tp_layer_forward", "tp_layer_forward_traced", "tp_selftest_wait_timeout",
    "tp_packed_shard_table", "tp_packed_colwise_forward", "tp_vocab_embedding_forward",
    "tp_vocab_logits_forward", "tp_vocab_parallel_cross_entropy", "tp_sp_all_gather",
    "tp_sp_reduce_scatter", "tp_mlp_forward_train", "tp_mlp_backward", "tp_plan_attn_saved_bytes",
    "tp_attn_forward_train", "tp_attn_backward", "tp_layer_backward", "EXPORTED",
]

TP_OK = 0
TP_ERR_INVALID_ARG = 1
TP_ERR_NOT_DIVISIBLE = 2
TP_ERR_UNSUPPORTED = 3
TP_ERR_WORKSPACE = 4
TP_ERR_CUDA = 5
TP_ERR_DEVICE_TIMEOUT = 6

TP_ACT_GELU_ERF, TP_ACT_GELU_TANH, TP_ACT_SWIGLU, TP_ACT_NONE = 0, 1, 2, 3
TP_REDUCE_FUSED, TP_REDUCE_PARTIALS = 0, 1
TP_F32, TP_BF16 = 0, 1
(TP_OP_MLP, TP_OP_ATTN, TP_OP_LAYER, TP_OP_MLP_BACKWARD, TP_OP_ATTN_BACKWARD,
 TP_OP_LAYER_BACKWARD) = range(6)
(TP_TABLE_FFN_SHARDS, TP_TABLE_Q_HEAD_SHARD, TP_TABLE_Q_HEAD_KV, TP_TABLE_SHARD_KV,
 TP_TABLE_QKV_COLUMNS) = range(5)

ACT_BY_NAME = {"gelu": TP_ACT_GELU_ERF, "gelu_tanh": TP_ACT_GELU_TANH, "swiglu": TP_ACT_SWIGLU,
               "none": TP_ACT_NONE}


class TPError(RuntimeError):
    """A TP_ERR_* return code with the library's message."""

    def __init__(self, fn: str, code: int, message: str):
        super().__init__(f"{fn} failed with code {code}: {message}")
        self.code = code
        self.fn = fn


class TPConfig(C.Structure):
    _fields_ = [
        ("tokens", C.c_int64),
        ("batch", C.c_int32), ("seq", C.c_int32),
        ("hidden", C.c_int32), ("ffn", C.c_int32),
        ("n_heads", C.c_int32), ("n_kv_heads", C.c_int32), ("head_dim", C.c_int32),
        ("tp_degree", C.c_int32), ("act", C.c_int32), ("reduce_mode", C.c_int32),
        ("partial_dtype", C.c_int32), ("rms_eps", C.c_float),
        ("sequence_parallel", C.c_int32),
    ]


class TPLayerWeights(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in ("Wq", "Wk", "Wv", "Wo", "W1", "W3", "W2")]


class TPLayerGrads(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in ("dWq", "dWk", "dWv", "dWo", "dW1", "dW3", "dW2")]


_VP = C.c_void_p
_SIGS = {
    "tp_plan_create": [C.POINTER(TPConfig), C.POINTER(C.c_void_p)],
    "tp_config_check": [C.POINTER(TPConfig)],
    "tp_config_shard_table": [C.POINTER(TPConfig), C.c_int, C.POINTER(C.c_int32), C.c_int64,
                              C.POINTER(C.c_int64)],
    "tp_plan_destroy": [_VP],
    "tp_plan_workspace_bytes": [_VP, C.c_int, C.POINTER(C.c_size_t)],
    "tp_plan_shard_table": [_VP, C.c_int, C.POINTER(C.c_int32), C.c_int64, C.POINTER(C.c_int64)],
    "tp_get_device_status": [_VP, _VP],
    "tp_reduce_partials": [_VP, C.c_int, C.c_int32, C.c_int64, C.c_int32, _VP, _VP, _VP, _VP],
    "tp_rmsnorm": [_VP, C.c_int64, C.c_int32, C.c_float, _VP, _VP],
    "tp_colwise_forward": [_VP, _VP, _VP, _VP, _VP, _VP],
    "tp_rowwise_forward": [_VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP],
    "tp_mlp_forward": [_VP] * 10 + [C.c_size_t, _VP],
    "tp_mlp_forward_noalloc": [_VP] * 9,
    "tp_mlp_forward_train": [_VP] * 11 + [C.c_size_t, _VP],
    "tp_mlp_backward": [_VP] * 12 + [C.c_int, _VP, C.c_size_t, _VP],
    "tp_plan_attn_saved_bytes": [_VP] + [C.POINTER(C.c_size_t)] * 3,
    "tp_attn_forward_train": [_VP] * 13,
    "tp_attn_backward": [_VP] * 15 + [C.c_int, _VP, C.c_size_t, _VP],
    "tp_layer_backward": [_VP] * 6 + [C.c_int, _VP, C.c_size_t, _VP],
    "tp_qkv_forward": [_VP] * 7,
    "tp_attn_core_forward": [_VP] * 4,
    "tp_attn_forward": [_VP] * 10 + [C.c_size_t, _VP],
    "tp_layer_forward": [_VP, _VP, C.POINTER(TPLayerWeights), _VP, _VP, C.c_size_t, _VP],
    "tp_layer_forward_traced": [_VP, _VP, C.POINTER(TPLayerWeights), _VP, _VP, C.c_size_t, _VP,
                                C.POINTER(C.c_void_p), C.c_int],
    "tp_selftest_wait_timeout": [_VP, C.c_uint64, _VP],
    "tp_packed_shard_table": [C.POINTER(C.c_int64), C.c_int32, C.c_int32, C.POINTER(C.c_int32),
                              C.c_int64, C.POINTER(C.c_int64)],
    "tp_packed_colwise_forward": [_VP, C.c_int64, C.c_int32, _VP, C.POINTER(C.c_int64), C.c_int32,
                                  C.c_int32, _VP, _VP],
    "tp_vocab_embedding_forward": [_VP, C.c_int64, _VP, C.c_int64, C.c_int32, C.c_int32, _VP, _VP],
    "tp_vocab_logits_forward": [_VP, C.c_int64, C.c_int32, _VP, C.c_int64, C.c_int32, _VP, _VP],
    "tp_vocab_parallel_cross_entropy": [_VP, C.c_int64, C.c_int64, C.c_int32, _VP, _VP, _VP, _VP],
    "tp_sp_all_gather": [_VP, C.c_int32, C.c_int32, C.c_int32, C.c_int32, _VP, _VP],
    "tp_sp_reduce_scatter": [_VP, C.c_int, C.c_int32, C.c_int32, C.c_int32, C.c_int32, _VP, _VP, _VP,
                             C.c_float, _VP],
}
EXPORTED = tuple(sorted(list(_SIGS) + ["tp_last_error"]))

_lib = None


def build(force: bool = False) -> str:
    """Compile libtp.so for sm_103a (in-tree)."""
    return _build.build(force=force)


def lib():
    """Load libtp.so (building it first if it is missing or stale)."""
    global _lib
    if _lib is None:
        path = _build.LIB
        if _build.needs_build():
            path = _build.build()
        L = C.CDLL(path)
        for name, args in _SIGS.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = C.c_int
        L.tp_last_error.argtypes = []
        L.tp_last_error.restype = C.c_char_p
        _lib = L
    return _lib


def tp_last_error() -> str:
    return lib().tp_last_error().decode("utf-8", "replace")


def _call(name: str, *args) -> None:
    rc = getattr(lib(), name)(*args)
    if rc != TP_OK:
        raise TPError(name, rc, tp_last_error())


def _p(x) -> Optional[int]:
    """Device pointer of a tensor (or an int / None)."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _s(stream) -> Optional[int]:
    if stream is None:
        import torch  # streams come from torch: plumbing only
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def make_config(tokens: int, hidden: int, ffn: int = 0, n_heads: int = 0, n_kv_heads: int = 0,
                head_dim: int = 0, tp_degree: int = 1, act="gelu", reduce_mode: int = TP_REDUCE_FUSED,
                partial_dtype: int = TP_F32, rms_eps: float = 1e-5, batch: int = 1,
                seq: Optional[int] = None, sequence_parallel: int = 0) -> TPConfig:
    if isinstance(act, str):
        act = ACT_BY_NAME[act]
    if seq is None:
        seq = tokens // max(batch, 1)
    return TPConfig(tokens, batch, seq, hidden, ffn, n_heads, n_kv_heads, head_dim, tp_degree, act,
                    reduce_mode, partial_dtype, rms_eps, sequence_parallel)


class Plan:
    """Owner of a tp_plan_t handle; destroyed with the object."""

    def __init__(self, cfg: TPConfig):
        h = C.c_void_p()
        _call("tp_plan_create", C.byref(cfg), C.byref(h))
        self.handle = h
        self.cfg = cfg

    @property
    def _as_parameter_(self):
        return self.handle

    def close(self):
        if self.handle:
            lib().tp_plan_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def tp_plan_create(cfg: TPConfig) -> Plan:
    return Plan(cfg)


def tp_plan_destroy(plan: Plan) -> None:
    plan.close()


def tp_config_check(cfg: TPConfig) -> int:
    """Host-only validation; returns the TP_* code (does not raise)."""
    return lib().tp_config_check(C.byref(cfg))


def _table(fn, target, which: int):
    n = C.c_int64(0)
    lib_fn = getattr(lib(), fn)
    rc = lib_fn(target, which, None, 0, C.byref(n))
    if rc not in (TP_OK, TP_ERR_INVALID_ARG) or (rc != TP_OK and n.value == 0):
        raise TPError(fn, rc, tp_last_error())
    buf = (C.c_int32 * max(n.value, 1))()
    _call(fn, target, which, buf, n.value, C.byref(n))
    return [buf[i] for i in range(n.value)]


def tp_config_shard_table(cfg: TPConfig, which: int):
    return _table("tp_config_shard_table", C.byref(cfg), which)


def tp_plan_shard_table(plan: Plan, which: int):
    return _table("tp_plan_shard_table", plan.handle, which)


def tp_plan_workspace_bytes(plan: Plan, op: int) -> int:
    n = C.c_size_t(0)
    _call("tp_plan_workspace_bytes", plan.handle, op, C.byref(n))
    return n.value


def tp_get_device_status(plan: Plan, stream=None) -> int:
    """TP_OK or TP_ERR_DEVICE_TIMEOUT (returned, not raised)."""
    return lib().tp_get_device_status(plan.handle, _s(stream))


def tp_reduce_partials(partials, partial_dtype: int, t: int, n: int, h: int, bias, residual, out,
                       stream=None) -> None:
    _call("tp_reduce_partials", _p(partials), partial_dtype, t, n, h, _p(bias), _p(residual),
          _p(out), _s(stream))


def tp_rmsnorm(x, rows: int, h: int, eps: float, y, stream=None) -> None:
    _call("tp_rmsnorm", _p(x), rows, h, eps, _p(y), _s(stream))


def tp_colwise_forward(plan: Plan, X, W1, W3, Y, stream=None) -> None:
    _call("tp_colwise_forward", plan.handle, _p(X), _p(W1), _p(W3), _p(Y), _s(stream))


def tp_rowwise_forward(plan: Plan, Y, W2, bias, residual, partials, Z, stream=None) -> None:
    _call("tp_rowwise_forward", plan.handle, _p(Y), _p(W2), _p(bias), _p(residual), _p(partials),
          _p(Z), _s(stream))


def tp_mlp_forward(plan: Plan, X, W1, W3, W2, b2, residual, partials, Z, workspace,
                   ws_bytes: int, stream=None) -> None:
    _call("tp_mlp_forward", plan.handle, _p(X), _p(W1), _p(W3), _p(W2), _p(b2), _p(residual),
          _p(partials), _p(Z), _p(workspace), ws_bytes, _s(stream))


def tp_mlp_forward_noalloc(plan: Plan, X, W1, W3, W2, b2, residual, Z, stream=None) -> None:
    """tp_mlp_forward with its scratch in the library's built-in device array
    (no workspace argument; nothing is allocated by the call)."""
    _call("tp_mlp_forward_noalloc", plan.handle, _p(X), _p(W1), _p(W3), _p(W2), _p(b2),
          _p(residual), _p(Z), _s(stream))


def tp_mlp_forward_train(plan: Plan, X, W1, W3, W2, b2, residual, partials, Z, UG, workspace,
                         ws_bytes: int, stream=None) -> None:
    """tp_mlp_forward that also writes the pre-activations UG its backward reads."""
    _call("tp_mlp_forward_train", plan.handle, _p(X), _p(W1), _p(W3), _p(W2), _p(b2),
          _p(residual), _p(partials), _p(Z), _p(UG), _p(workspace), ws_bytes, _s(stream))


def tp_mlp_backward(plan: Plan, X, W1, W3, W2, dZ, UG, dX, dW1, dW3, dW2, db2, accumulate: bool,
                    workspace, ws_bytes: int, stream=None) -> None:
    """Gradients of the sharded MLP (UG None: pre-activations recomputed)."""
    _call("tp_mlp_backward", plan.handle, _p(X), _p(W1), _p(W3), _p(W2), _p(dZ), _p(UG), _p(dX),
          _p(dW1), _p(dW3), _p(dW2), _p(db2), 1 if accumulate else 0, _p(workspace), ws_bytes,
          _s(stream))


def tp_plan_attn_saved_bytes(plan: Plan):
    """(qkv, o, lse) byte sizes of what tp_attn_forward_train saves."""
    q, o, l = C.c_size_t(), C.c_size_t(), C.c_size_t()
    _call("tp_plan_attn_saved_bytes", plan.handle, C.byref(q), C.byref(o), C.byref(l))
    return q.value, o.value, l.value


def tp_attn_forward_train(plan: Plan, X, Wq, Wk, Wv, Wo, residual, partials, out, QKV, O, LSE,
                          stream=None) -> None:
    """tp_attn_forward that keeps QKV, O and the softmax statistics LSE."""
    _call("tp_attn_forward_train", plan.handle, _p(X), _p(Wq), _p(Wk), _p(Wv), _p(Wo),
          _p(residual), _p(partials), _p(out), _p(QKV), _p(O), _p(LSE), _s(stream))


def tp_attn_backward(plan: Plan, X, Wq, Wk, Wv, Wo, dOut, QKV, O, LSE, dX, dWq, dWk, dWv, dWo,
                     accumulate: bool, workspace, ws_bytes: int, stream=None) -> None:
    """Gradients of the head-sharded attention block (QKV/O/LSE None: recomputed)."""
    _call("tp_attn_backward", plan.handle, _p(X), _p(Wq), _p(Wk), _p(Wv), _p(Wo), _p(dOut),
          _p(QKV), _p(O), _p(LSE), _p(dX), _p(dWq), _p(dWk), _p(dWv), _p(dWo),
          1 if accumulate else 0, _p(workspace), ws_bytes, _s(stream))


def tp_qkv_forward(plan: Plan, X, Wq, Wk, Wv, QKV, stream=None) -> None:
    _call("tp_qkv_forward", plan.handle, _p(X), _p(Wq), _p(Wk), _p(Wv), _p(QKV), _s(stream))


def tp_attn_core_forward(plan: Plan, QKV, O, stream=None) -> None:
    _call("tp_attn_core_forward", plan.handle, _p(QKV), _p(O), _s(stream))


def tp_attn_forward(plan: Plan, X, Wq, Wk, Wv, Wo, residual, partials, out, workspace,
                    ws_bytes: int, stream=None) -> None:
    _call("tp_attn_forward", plan.handle, _p(X), _p(Wq), _p(Wk), _p(Wv), _p(Wo), _p(residual),
          _p(partials), _p(out), _p(workspace), ws_bytes, _s(stream))


def tp_layer_forward(plan: Plan, X, weights: dict, Y, workspace, ws_bytes: int,
                     stream=None) -> None:
    w = TPLayerWeights(*[_p(weights.get(k)) for k in ("Wq", "Wk", "Wv", "Wo", "W1", "W3", "W2")])
    _call("tp_layer_forward", plan.handle, _p(X), C.byref(w), _p(Y), _p(workspace), ws_bytes,
          _s(stream))


def tp_layer_backward(plan: Plan, X, weights: dict, dY, dX, grads: dict, accumulate: bool, workspace,
                      ws_bytes: int, stream=None) -> None:
    """Backward of the pre-norm layer (forward recomputed): dX and the fp32
    weight gradients in ``grads`` (keys dWq, dWk, dWv, dWo, dW1, dW3, dW2)."""
    w = TPLayerWeights(*[_p(weights.get(k)) for k in ("Wq", "Wk", "Wv", "Wo", "W1", "W3", "W2")])
    g = TPLayerGrads(*[_p(grads.get(k)) for k in ("dWq", "dWk", "dWv", "dWo", "dW1", "dW3", "dW2")])
    _call("tp_layer_backward", plan.handle, _p(X), C.byref(w), _p(dY), _p(dX), C.byref(g),
          1 if accumulate else 0, _p(workspace), ws_bytes, _s(stream))


def layer_weights(weights: dict) -> TPLayerWeights:
    return TPLayerWeights(*[_p(weights.get(k)) for k in ("Wq", "Wk", "Wv", "Wo", "W1", "W3", "W2")])


def tp_layer_forward_traced(plan: Plan, X, weights, Y, workspace, ws_bytes: int, events,
                            stream=None) -> None:
    """``events``: sequence of cudaEvent_t handles (ints) recorded at kernel boundaries."""
    w = weights if isinstance(weights, TPLayerWeights) else layer_weights(weights)
    arr = (C.c_void_p * len(events))(*events)
    _call("tp_layer_forward_traced", plan.handle, _p(X), C.byref(w), _p(Y), _p(workspace),
          ws_bytes, _s(stream), arr, len(events))


def tp_selftest_wait_timeout(plan: Plan, timeout_ns: int, stream=None) -> None:
    _call("tp_selftest_wait_timeout", plan.handle, timeout_ns, _s(stream))


def _blocks(blocks):
    arr = (C.c_int64 * len(blocks))(*[int(b) for b in blocks])
    return arr, len(blocks)


def tp_packed_shard_table(blocks, t: int):
    """[(first packed row, rows)] per shard and block, flattened."""
    arr, nb = _blocks(blocks)
    n = C.c_int64(0)
    rc = lib().tp_packed_shard_table(arr, nb, t, None, 0, C.byref(n))
    if rc not in (TP_OK, TP_ERR_INVALID_ARG) or n.value == 0:
        raise TPError("tp_packed_shard_table", rc, tp_last_error())
    buf = (C.c_int32 * n.value)()
    _call("tp_packed_shard_table", arr, nb, t, buf, n.value, C.byref(n))
    return [buf[i] for i in range(n.value)]


def tp_packed_colwise_forward(X, M: int, h: int, W, blocks, t: int, Y, stream=None) -> None:
    arr, nb = _blocks(blocks)
    _call("tp_packed_colwise_forward", _p(X), M, h, _p(W), arr, nb, t, _p(Y), _s(stream))


def tp_vocab_embedding_forward(ids, M: int, E, v: int, h: int, t: int, out, stream=None) -> None:
    _call("tp_vocab_embedding_forward", _p(ids), M, _p(E), v, h, t, _p(out), _s(stream))


def tp_vocab_logits_forward(H, M: int, h: int, W, v: int, t: int, logits, stream=None) -> None:
    _call("tp_vocab_logits_forward", _p(H), M, h, _p(W), v, t, _p(logits), _s(stream))


def tp_vocab_parallel_cross_entropy(logits, M: int, v: int, t: int, labels, stats, loss,
                                    stream=None) -> None:
    _call("tp_vocab_parallel_cross_entropy", _p(logits), M, v, t, _p(labels), _p(stats), _p(loss),
          _s(stream))


def tp_sp_all_gather(sp, batch: int, seq: int, t: int, h: int, full, stream=None) -> None:
    _call("tp_sp_all_gather", _p(sp), batch, seq, t, h, _p(full), _s(stream))


def tp_sp_reduce_scatter(partials, partial_dtype: int, t: int, batch: int, seq: int, h: int,
                         residual_sp, out_sp, xn_sp=None, eps: float = 1e-5, stream=None) -> None:
    _call("tp_sp_reduce_scatter", _p(partials), partial_dtype, t, batch, seq, h, _p(residual_sp),
          _p(out_sp), _p(xn_sp), eps, _s(stream))
