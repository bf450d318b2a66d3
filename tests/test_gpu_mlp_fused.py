"""GPU parity of the one-launch sharded MLP (tp_mlp_forward in FUSED mode on
problems too small to fill the GPU with two GEMMs).

One persistent launch runs the colwise tiles of H = act(X W1^T), then each
m-block's rowwise tiles of Z in K pieces of t / pieces shards, each piece
starting as soon as the H columns it reads are stored; with several pieces,
the last piece of a tile to arrive sums the fp32 partials in piece order
("텐서 병렬화", "MLP": Z = sum_i GeLU(X A_i) B_i).  The shapes below make
the plan choose 1, 2, 4 and 8 pieces; the piece count is read back from the
workspace size (the partials take pieces x M x h fp32).  Integer-valued
inputs with no activation are exact in fp32, so those runs are compared
bit for bit."""
import numpy as np
import pytest
import torch

import megatron_tensor_transformer_colwise_gb300 as tp
import oracle
import synth
from synth import Shape
from gpu_util import assert_close, bf16_bits, dev, host64, plan_for, sync_ok, workspace

pytestmark = pytest.mark.gpu


def _pieces(plan, s):
    """Pieces of the one-launch MLP, from the workspace size (0: two GEMMs)."""
    n = tp.tp_plan_workspace_bytes(plan, tp.TP_OP_MLP)
    y = -(-s.tokens * s.ffn * 2 // 256) * 256
    rest = n - y
    if rest == 0:
        return 0
    part = s.tokens * s.hidden * 4
    for p in (8, 4, 2):
        if rest >= -(-p * part // 256) * 256:
            return p
    return 1


def _run(s, inp, bias=None, residual=None):
    plan = plan_for(s)
    ws, nws = workspace(plan, tp.TP_OP_MLP)
    Z = torch.full((s.tokens, s.hidden), float("nan"), dtype=torch.bfloat16, device="cuda")
    tp.tp_mlp_forward(plan, dev(inp["X"]), dev(inp["W1"]), None, dev(inp["W2"]), bias, residual, None, Z,
                      ws, nws)
    sync_ok(plan)
    return plan, Z


# (tokens, hidden, ffn, t) -> pieces the plan takes on GB300's 152 SMs.
SHAPES = [
    ((300, 192, 800, 4), 2),    # ragged m-block, h below one tile, shard edges inside n-tiles
    ((130, 64, 256, 4), 1),
    ((256, 256, 8192, 4), 4),
    ((256, 256, 16384, 8), 8),
    ((520, 128, 2048, 8), None),
]


@pytest.mark.parametrize("dims,want", SHAPES, ids=[f"{m}x{h}x{f}_t{t}" for (m, h, f, t), _ in SHAPES])
def test_integer_inputs_bit_exact(dims, want):
    M, h, f, t = dims
    s = Shape("fz", 1, M, h, ffn=f, tp=t, act="none", index=80)
    inp = synth.workload_inputs(s, integer=(-1, 1))
    plan, Z = _run(s, inp)
    got = _pieces(plan, s)
    assert got >= 1, "expected the one-launch path"
    if want is not None:
        assert got == want
    ref = oracle.mlp("none", host64(inp["X"]), host64(inp["W1"]), host64(inp["W2"]))
    # |H| <= h <= 256 is exact in bf16 and every sum is an exact fp32 integer.
    assert np.abs(ref).max() < 2 ** 24
    assert np.array_equal(bf16_bits(Z), oracle.round_bf16_bits(ref).reshape(ref.shape))


@pytest.mark.parametrize("act", ["gelu", "gelu_tanh"])
@pytest.mark.parametrize("dims,want", SHAPES[:4], ids=[f"{m}x{h}x{f}_t{t}" for (m, h, f, t), _ in SHAPES[:4]])
def test_gelu_with_bias_and_residual(dims, want, act):
    M, h, f, t = dims
    s = Shape("fg", 1, M, h, ffn=f, tp=t, act=act, index=81)
    inp = synth.workload_inputs(s)
    bias = synth.normal_bf16((h,), 1.0, 8101)
    res = synth.normal_bf16((M, h), 1.0, 8102)
    plan, Z = _run(s, inp, dev(bias), dev(res))
    assert _pieces(plan, s) == want
    ref = oracle.mlp_sharded(act, t, host64(inp["X"]), host64(inp["W1"]), host64(inp["W2"]))
    assert_close(host64(Z), ref + host64(bias)[None, :] + host64(res), what=f"{act} z + bias + residual")
    # the block's own part, without the residual
    plan2, Z2 = _run(s, inp)
    assert_close(host64(Z2), ref, what=f"{act} z")


def test_two_runs_give_the_same_bits():
    # The pieces' partials are summed in piece order whichever arrives last.
    s = Shape("fd", 1, 1000, 256, ffn=8192, tp=4, act="gelu", index=82)
    inp = synth.workload_inputs(s)
    _, Z1 = _run(s, inp)
    _, Z2 = _run(s, inp)
    assert torch.equal(Z1.view(torch.int16), Z2.view(torch.int16))
    ref = oracle.mlp("gelu", host64(inp["X"]), host64(inp["W1"]), host64(inp["W2"]))
    assert_close(host64(Z1), ref, what="gelu z")


def test_gpt_shape_takes_the_one_launch_path():
    s = synth.SHAPES["gpt_mlp"]
    plan = plan_for(s)
    assert _pieces(plan, s) == 2
    # The layer-sized and Llama-sized MLPs keep the two-GEMM path.
    assert _pieces(plan_for(synth.SHAPES["llama_mlp"]), synth.SHAPES["llama_mlp"]) == 0
