"""Helpers shared by the GPU parity tests (not a test module).

The parity bar for floating point: max |gpu - ref| / max |ref| <= 2e-2 over
the compared tensor (bf16 inputs, fp32 accumulation, bf16 outputs), with ref
the fp64 oracle on the same bf16-rounded inputs.  Integer-valued work is
compared bit-exactly.
"""
import numpy as np
import torch

import megatron_tensor_transformer_colwise_gb300 as tp

REL_TOL = 2e-2


def dev(x: torch.Tensor) -> torch.Tensor:
    return x.contiguous().to("cuda")


def host64(x: torch.Tensor) -> np.ndarray:
    return x.detach().to("cpu").double().numpy()


def rel_err(got, ref) -> float:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    scale = np.abs(ref).max()
    if scale == 0:
        return float(np.abs(got).max())
    return float(np.abs(got - ref).max() / scale)


def assert_close(got, ref, tol=REL_TOL, what=""):
    e = rel_err(got, ref)
    assert np.isfinite(np.asarray(got, dtype=np.float64)).all(), f"{what}: non-finite output"
    assert e <= tol, f"{what}: max rel err {e:.3e} > {tol:.1e}"
    return e


def bf16_bits(x: torch.Tensor) -> np.ndarray:
    return x.detach().to("cpu").view(torch.int16).numpy().astype(np.uint16)


def plan_for(shape, reduce_mode=tp.TP_REDUCE_FUSED, partial_dtype=tp.TP_F32, act=None):
    cfg = tp.make_config(tokens=shape.tokens, hidden=shape.hidden, ffn=shape.ffn,
                         n_heads=shape.heads, n_kv_heads=shape.kv_heads, head_dim=shape.head_dim,
                         tp_degree=shape.tp, act=act if act is not None else shape.act,
                         reduce_mode=reduce_mode, partial_dtype=partial_dtype, batch=shape.batch,
                         seq=shape.seq)
    return tp.Plan(cfg)


def workspace(plan, op):
    n = tp.tp_plan_workspace_bytes(plan, op)
    return torch.empty(max(n, 16), dtype=torch.uint8, device="cuda"), n


def sync_ok(plan=None):
    torch.cuda.synchronize()
    if plan is not None:
        assert tp.tp_get_device_status(plan) == tp.TP_OK, tp.tp_last_error()


def half_ulp_bf16(v) -> np.ndarray:
    """Half a bf16 unit in the last place at |v| (8 significant bits):
    2^(floor(log2 |v|) - 8); 0 at v = 0."""
    a = np.abs(np.asarray(v, dtype=np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, np.exp2(e - 8), 0.0)


def assert_layer_contribution_close(Y, ref, X, h1, tol=REL_TOL, what=""):
    """The blocks' own contribution to a pre-norm layer's output, y - x, at
    the parity tolerance.

    The layer's output y and its residual stream h1 are stored in bf16, and
    |y| ~ |x| ~ N(0, 1) is up to ~10x the blocks' contribution.  Each of the
    two stores rounds by up to half a bf16 ulp of its value, and an h1
    rounding passes into y through the residual connection unchanged (the
    MLP's response to it is a few percent of it).  Those two storage errors are
    taken off elementwise, bounded by half an ulp at max(|y|, |ref|) and at
    |h1|; what is left, the arithmetic of the blocks, must be within tol of
    max |ref - x|.  On an exact computation whose y and h1 are only rounded
    to bf16, the plain (y - x) metric already reads ~2.7e-2 at h = 256, and
    this one ~4e-4."""
    got = np.asarray(Y, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    scale = np.abs(ref - X).max()
    storage = half_ulp_bf16(np.maximum(np.abs(got), np.abs(ref))) + half_ulp_bf16(h1)
    excess = np.maximum(np.abs(got - ref) - storage, 0.0).max() / scale
    assert excess <= tol, f"{what}: block contribution error {excess:.3e} > {tol:.1e}"
    return excess


def elementwise_excess_fraction(got, ref, rel=2e-2, rms_frac=1e-3) -> float:
    """Fraction of elements with |got - ref| > rel * |ref| + rms_frac * rms(ref)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    rms = np.sqrt(np.mean(ref * ref))
    return float(np.mean(np.abs(got - ref) > rel * np.abs(ref) + rms_frac * rms))


def report(what: str, **numbers):
    """Append one parity record (JSON line) to the file named by the
    TP_PARITY_REPORT environment variable, when it is set."""
    import json
    import os
    path = os.environ.get("TP_PARITY_REPORT")
    if path:
        with open(path, "a") as fh:
            fh.write(json.dumps({"what": what, **{k: float(v) for k, v in numbers.items()}}) + "\n")
