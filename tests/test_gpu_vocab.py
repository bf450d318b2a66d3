"""GPU parity of the vocab-parallel embedding and the vocab-parallel
cross-entropy (max / sum exchange) against the fp64 oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import megatron_tensor_transformer_colwise_gb300 as tp
import oracle
import synth
from gpu_util import assert_close, bf16_bits, dev, host64, sync_ok

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("M,v,h,t", [(300, 4608, 128, 8), (37, 512, 64, 1), (1000, 2048, 256, 4)])
def test_embedding_bit_exact(M, v, h, t):
    g = torch.Generator().manual_seed(M + v)
    ids = torch.randint(0, v, (M,), generator=g, dtype=torch.int32)
    ids[5] = -3
    ids[6] = v + 7                      # owned by no shard: zero row
    E = synth.normal_bf16((v, h), 1.0, 91)
    out = torch.empty(M, h, dtype=torch.bfloat16, device="cuda")
    tp.tp_vocab_embedding_forward(dev(ids), M, dev(E), v, h, t, out)
    sync_ok()
    ref = oracle.embedding_vocab_parallel(t, ids.numpy(), host64(E))
    assert np.array_equal(bf16_bits(out), oracle.round_bf16_bits(ref).reshape(ref.shape))


@pytest.mark.parametrize("M,v,t", [(300, 4608, 8), (129, 1024, 1), (64, 6144, 3)])
def test_cross_entropy_from_bf16_logits(M, v, t):
    logits = synth.normal_bf16((M, v), 3.0, 92)
    g = torch.Generator().manual_seed(93)
    labels = torch.randint(0, v, (M,), generator=g, dtype=torch.int32)
    labels[0] = -100
    labels[1] = v + 1                   # invalid: NaN
    stats = torch.empty(3 * t * M, dtype=torch.float32, device="cuda")
    loss = torch.empty(M, dtype=torch.float32, device="cuda")
    tp.tp_vocab_parallel_cross_entropy(dev(logits), M, v, t, dev(labels), stats, loss)
    sync_ok()
    ref, st = oracle.cross_entropy_vocab_parallel(t, host64(logits), labels.numpy(), want_stats=True)
    got = loss.cpu().double().numpy()
    assert got[0] == 0.0 and np.isnan(got[1]) and np.isnan(ref[1])
    ok = slice(2, None)
    assert np.abs(got[ok] - ref[ok]).max() <= 1e-3 * np.abs(ref[ok]).max()
    gst = stats.cpu().double().numpy().reshape(3, t, M)
    assert np.abs(gst[0] - st[0]).max() <= 1e-5 * np.abs(st[0]).max()           # shard maxima
    assert np.abs(gst[1] - st[1]).max() <= 1e-4 * np.abs(st[1]).max()           # shard sums
    assert np.array_equal(gst[2][:, 2:], st[2][:, 2:])                          # target logits


@pytest.mark.parametrize("M,v,h,t", [(300, 4608, 128, 8), (130, 2048, 64, 2)])
def test_logits_integer_bit_exact_and_loss_end_to_end(M, v, h, t):
    H = synth.integer_bf16((M, h), -2, 2, 94)
    W = synth.integer_bf16((v, h), -1, 1, 95)
    logits = torch.empty(M, v, dtype=torch.bfloat16, device="cuda")
    tp.tp_vocab_logits_forward(dev(H), M, h, dev(W), v, t, logits)
    sync_ok()
    z = oracle.linear(host64(H), host64(W))
    assert np.array_equal(bf16_bits(logits), oracle.round_bf16_bits(z).reshape(z.shape))
    # End to end from normal inputs: logits GEMM + loss_parallel.
    Hn = synth.normal_bf16((M, h), 1.0, 96)
    Wn = synth.normal_bf16((v, h), 0.1, 97)
    labels = torch.randint(0, v, (M,), generator=torch.Generator().manual_seed(98), dtype=torch.int32)
    tp.tp_vocab_logits_forward(dev(Hn), M, h, dev(Wn), v, t, logits)
    stats = torch.empty(3 * t * M, dtype=torch.float32, device="cuda")
    loss = torch.empty(M, dtype=torch.float32, device="cuda")
    tp.tp_vocab_parallel_cross_entropy(logits, M, v, t, dev(labels), stats, loss)
    sync_ok()
    ref = oracle.cross_entropy(oracle.linear(host64(Hn), host64(Wn)), labels.numpy())
    assert_close(loss.cpu().double().numpy(), ref, what="logits + cross-entropy")


def test_full_vocab_loss_sampled_rows():
    # Llama-3-sized output layer: 8192 tokens, h = 4096, v = 128256, t = 8.
    M, h, v, t = 8192, 4096, 128256, 8
    Hn = synth.normal_bf16((M, h), 1.0, 4100)
    Wn = synth.normal_bf16((v, h), 0.02, 4101)
    labels = torch.randint(0, v, (M,), generator=torch.Generator().manual_seed(4102), dtype=torch.int32)
    logits = torch.empty(M, v, dtype=torch.bfloat16, device="cuda")
    tp.tp_vocab_logits_forward(dev(Hn), M, h, dev(Wn), v, t, logits)
    stats = torch.empty(3 * t * M, dtype=torch.float32, device="cuda")
    loss = torch.empty(M, dtype=torch.float32, device="cuda")
    tp.tp_vocab_parallel_cross_entropy(logits, M, v, t, dev(labels), stats, loss)
    sync_ok()
    rows = [0, 1, 777, 4096, 8191]
    ref = oracle.cross_entropy(oracle.linear(host64(Hn[rows]), host64(Wn)), labels[rows].numpy())
    assert_close(loss.cpu().double().numpy()[rows], ref, what="full-vocab loss rows")
    assert np.isfinite(loss.cpu().numpy()).all()
