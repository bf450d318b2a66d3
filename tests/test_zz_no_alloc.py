"""The allocation-free MLP entry point, tp_mlp_forward_noalloc.

It serves callers that cannot allocate device memory when they call (a
framework whose memory manager owns the GPU, a plugin with no allocator
handle, a latency-critical loop that cannot afford cudaMalloc's implicit
synchronisation): its scratch lives in the library's built-in device array
instead of a caller workspace.  Checked here through the C ABI against
tp_mlp_forward (which takes a workspace) and against the fp64 oracle on two
calls in a row, within the parity tolerance of the other tests, in both
reduction modes; and a plan
whose scratch does not fit the built-in array is refused before any launch.

This file is collected last so that a run stopping at the first failure has
already run every other test; it also passes on its own in a fresh process.
"""
import numpy as np
import pytest
import torch

import megatron_tensor_transformer_colwise_gb300 as tp
import oracle
import synth
from synth import SHAPES
from gpu_util import assert_close, dev, host64, plan_for, sync_ok, workspace

pytestmark = pytest.mark.gpu


def _with_workspace(plan, s, inp, b2, res, mode):
    ws, nws = workspace(plan, tp.TP_OP_MLP)
    Z = torch.empty(s.tokens, s.hidden, dtype=torch.bfloat16, device="cuda")
    P = (torch.empty(s.tp, s.tokens, s.hidden, dtype=torch.float32, device="cuda")
         if mode == tp.TP_REDUCE_PARTIALS else None)
    W3 = inp.get("W3")
    tp.tp_mlp_forward(plan, inp["X"], inp["W1"], W3, inp["W2"], b2, res, P, Z, ws, nws)
    sync_ok(plan)
    return host64(Z)


@pytest.mark.parametrize("mode", [tp.TP_REDUCE_FUSED, tp.TP_REDUCE_PARTIALS])
@pytest.mark.parametrize("name", ["gpt_mlp", "small_swiglu"])
def test_noalloc_matches_workspace_entry_point_on_two_calls(name, mode):
    if name == "gpt_mlp":
        s = SHAPES["gpt_mlp"]      # scratch: 16 MiB (FUSED), 48 MiB (PARTIALS)
    else:
        s = synth.Shape("nz", 1, 333, 256, ffn=1024, tp=8, act="swiglu", index=60)
    plan = plan_for(s, reduce_mode=mode)
    for call in range(2):          # two calls in a row, different inputs
        inp = {k: dev(v) for k, v in synth.workload_inputs(s, seed_base=7000 + 100 * call).items()}
        b2 = dev(synth.normal_bf16((s.hidden,), 1.0, 7050 + call)) if call == 1 else None
        res = dev(synth.normal_bf16((s.tokens, s.hidden), 1.0, 7060 + call))
        Z = torch.full((s.tokens, s.hidden), float("nan"), dtype=torch.bfloat16, device="cuda")
        tp.tp_mlp_forward_noalloc(plan, inp["X"], inp["W1"], inp.get("W3"), inp["W2"], b2, res, Z)
        sync_ok(plan)
        got = host64(Z)
        want = _with_workspace(plan, s, inp, b2, res, mode)
        assert np.isfinite(got).all()
        assert_close(got, want, what=f"noalloc call {call}")
        # The block's own contribution (without the residual) agrees as well.
        assert_close(got - host64(res), want - host64(res), what=f"noalloc call {call} minus residual")
        # And both agree with the oracle on the same bf16 inputs.
        w3 = host64(inp["W3"]) if "W3" in inp else None
        ref = oracle.mlp(s.act, host64(inp["X"]), host64(inp["W1"]), host64(inp["W2"]), w3)
        if b2 is not None:
            ref = ref + host64(b2)[None, :]
        assert_close(got, ref + host64(res), what=f"noalloc call {call} vs oracle")


def test_noalloc_refuses_scratch_beyond_the_builtin_array():
    s = SHAPES["llama_mlp"]        # colwise output alone is 4096 x 14336 bf16 = 112 MiB
    plan = plan_for(s)
    X = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(tp.TPError) as e:
        tp.tp_mlp_forward_noalloc(plan, X, X, X, X, None, None, X)
    assert e.value.code == tp.TP_ERR_WORKSPACE
    assert "scratch" in str(e.value)
