"""GPU parity of packed projections (one Linear packing several logical
blocks, each sharded on its own) against the fp64 oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import megatron_tensor_transformer_colwise_gb300 as tp
import oracle
import synth
from synth import Shape
from gpu_util import assert_close, bf16_bits, dev, host64, plan_for, sync_ok, workspace

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("blocks,t,h,M", [
    ([128, 128, 128, 384, 384], 2, 192, 300),     # Q, K, V, gate, up with an MLP ratio of 3
    ([256, 256], 4, 128, 257),                     # gate, up
    ([64, 128, 192], 1, 64, 130),
])
def test_packed_colwise_integer_bit_exact(blocks, t, h, M):
    n = sum(blocks)
    X = synth.integer_bf16((M, h), -2, 2, 301)
    W = synth.integer_bf16((n, h), -2, 2, 302)
    Y = torch.empty(M, n, dtype=torch.bfloat16, device="cuda")
    tp.tp_packed_colwise_forward(dev(X), M, h, dev(W), blocks, t, Y)
    sync_ok()
    # Shard i's column block = X times the packed rows it holds (oracle map).
    rows = np.concatenate([oracle.packed_shard_rows(blocks, t, i) for i in range(t)])
    ref = oracle.linear(host64(X), host64(W)[rows])
    assert np.array_equal(bf16_bits(Y), oracle.round_bf16_bits(ref).reshape(ref.shape))


def test_packed_colwise_rejects_unsupported_widths():
    X = torch.zeros(8, 64, dtype=torch.bfloat16, device="cuda")
    W = torch.zeros(96, 64, dtype=torch.bfloat16, device="cuda")
    Y = torch.zeros(8, 96, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(tp.TPError) as e:
        tp.tp_packed_colwise_forward(X, 8, 64, W, [48, 48], 2, Y)   # 24 rows per shard
    assert e.value.code == tp.TP_ERR_UNSUPPORTED
    with pytest.raises(tp.TPError) as e:
        tp.tp_packed_colwise_forward(X, 8, 64, W, [72, 24], 4, Y)   # 72 / 4 ok, 24 / 4 ok, 18 not 64
    assert e.value.code in (tp.TP_ERR_UNSUPPORTED, tp.TP_ERR_NOT_DIVISIBLE)


@pytest.mark.parametrize("mode", [tp.TP_REDUCE_FUSED, tp.TP_REDUCE_PARTIALS])
def test_mlp_from_packed_gate_up_weight(mode):
    # A packed [gate; up] weight goes to the SwiGLU MLP by pointer offsets.
    s = Shape("pk", 1, 300, 192, ffn=512, tp=4, act="swiglu", index=31)
    inp = synth.workload_inputs(s)
    Wgu = torch.cat([inp["W1"], inp["W3"]], 0).contiguous()
    plan = plan_for(s, reduce_mode=mode)
    ws, nws = workspace(plan, tp.TP_OP_MLP)
    Z = torch.empty(s.tokens, s.hidden, dtype=torch.bfloat16, device="cuda")
    P = torch.empty(s.tp, s.tokens, s.hidden, dtype=torch.float32, device="cuda")
    Wd = dev(Wgu)
    W3_ptr = Wd.data_ptr() + s.ffn * s.hidden * 2
    tp.tp_mlp_forward(plan, dev(inp["X"]), Wd, W3_ptr, dev(inp["W2"]), None, None, P, Z, ws, nws)
    sync_ok(plan)
    ref = oracle.mlp_packed_gate_up(True, s.tp, host64(inp["X"]), host64(Wgu), host64(inp["W2"]))
    assert_close(host64(Z), ref, what="packed gate_up MLP")
    wrong = oracle.mlp_packed_gate_up(False, s.tp, host64(inp["X"]), host64(Wgu), host64(inp["W2"]))
    assert np.abs(host64(Z) - wrong).max() > 0.1 * np.abs(ref).max()
