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
