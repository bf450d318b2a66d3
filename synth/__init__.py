"""Seeded synthetic inputs shared by the oracle, the tests and the bench.

This module draws random numbers and rounds them; it holds none of the
tensor-parallel block's arithmetic.  Both the CPU oracle and the CUDA path are
fed from the tensors returned here, so the two sides see identical inputs.

Recipe (all draws on the host with a seeded ``torch.Generator``):

* The worked MLP example of the itwiki page "텐서 병렬화" (Tensor parallelism),
  section "MLP": ``torch.manual_seed(0)`` then ``X = randn(4, 16)``,
  ``A = randn(16, 64)``, ``B = randn(64, 16)`` in that order, kept in fp32.
* Every other workload: activations X ~ N(0, 1), weights ~ N(0, 0.02^2)
  (standard deviation 0.02), drawn in fp32 and rounded to bf16 with
  round-to-nearest-even.  Weights use the ``nn.Linear`` layout ``W[out, in]``.
  Tensor number ``j`` of workload number ``c`` uses seed ``1000 * c + j``, in
  the order X, W1, W3, W2, Wq, Wk, Wv, Wo (absent tensors keep their slot).
* Integer-valued tensors (for bit-exact tests) are uniform in [lo, hi], which
  bf16 holds exactly for small magnitudes.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, Optional

import torch

__all__ = [
    "Shape",
    "SHAPES",
    "worked_example",
    "normal_bf16",
    "integer_bf16",
    "workload_inputs",
]

WEIGHT_STD = 0.02
TENSOR_ORDER = ("X", "W1", "W3", "W2", "Wq", "Wk", "Wv", "Wo")


@dataclasses.dataclass(frozen=True)
class Shape:
    """Sizes of one workload (names follow the pages' notation).

    tokens = batch * seq (M); hidden = h; ffn = the MLP inner width (4h in the
    GPT form); heads = a; kv_heads = k; head_dim = d; tp = t.
    """

    name: str
    batch: int
    seq: int
    hidden: int
    ffn: int = 0
    heads: int = 0
    kv_heads: int = 0
    head_dim: int = 0
    tp: int = 1
    act: str = "gelu"  # "gelu", "gelu_tanh", "swiglu", "none"
    index: int = 0  # workload number used for seeds

    @property
    def tokens(self) -> int:
        return self.batch * self.seq


# The five workloads the block is measured and checked on.
SHAPES: Dict[str, Shape] = {
    # Worked example: b=4 rows, h=16, 4h=64, t=4 (fp32, from manual_seed(0)).
    "worked": Shape("worked", 1, 4, 16, ffn=64, tp=4, act="gelu", index=0),
    # GPT-style GeLU MLP: 2048 tokens, h=1024, ffn=4096, t=4.
    "gpt_mlp": Shape("gpt_mlp", 1, 2048, 1024, ffn=4096, tp=4, act="gelu", index=1),
    # Llama-3-8B-shaped SwiGLU MLP: 4096 tokens, h=4096, ffn=14336, t=4.
    "llama_mlp": Shape("llama_mlp", 1, 4096, 4096, ffn=14336, tp=4, act="swiglu", index=2),
    # Head-sharded causal GQA attention: 1 x 2048, h=4096, 32 q / 8 kv heads, d=128, t=8.
    "attn": Shape("attn", 1, 2048, 4096, heads=32, kv_heads=8, head_dim=128, tp=8, act="none", index=3),
    # Full layer: 4 x 2048 tokens, h=4096, 32/8 heads, d=128, SwiGLU ffn=14336, t=8.
    "layer": Shape("layer", 4, 2048, 4096, ffn=14336, heads=32, kv_heads=8, head_dim=128, tp=8,
                   act="swiglu", index=4),
}


def _generator(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def worked_example() -> Dict[str, torch.Tensor]:
    """X[4,16], A[16,64], B[64,16] drawn exactly as the page's listing does."""
    torch.manual_seed(0)
    b, h = 4, 16
    X = torch.randn(b, h)
    A = torch.randn(h, 4 * h)
    B = torch.randn(4 * h, h)
    return {"X": X, "A": A, "B": B}


def normal_bf16(shape, std: float, seed: int) -> torch.Tensor:
    """fp32 N(0, std^2) draw rounded to bf16 (round-to-nearest-even)."""
    x = torch.randn(*shape, generator=_generator(seed), dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(torch.bfloat16)


def integer_bf16(shape, lo: int, hi: int, seed: int) -> torch.Tensor:
    """Integers uniform in [lo, hi] stored as bf16 (exact for |v| <= 256)."""
    x = torch.randint(lo, hi + 1, tuple(shape), generator=_generator(seed), dtype=torch.int32)
    return x.to(torch.bfloat16)


def workload_inputs(shape: Shape, seed_base: Optional[int] = None,
                    integer: Optional[tuple] = None) -> Dict[str, torch.Tensor]:
    """bf16 CPU tensors for one workload, keyed by X, W1, W3, W2, Wq, Wk, Wv, Wo.

    ``integer=(lo, hi)`` draws integer-valued tensors instead of normals.
    Only the tensors the workload uses are returned.
    """
    base = 1000 * shape.index if seed_base is None else seed_base
    M, h = shape.tokens, shape.hidden
    dims = {"X": (M, h)}
    if shape.ffn:
        dims["W1"] = (shape.ffn, h)
        if shape.act == "swiglu":
            dims["W3"] = (shape.ffn, h)
        dims["W2"] = (h, shape.ffn)
    if shape.heads:
        a, k, d = shape.heads, shape.kv_heads, shape.head_dim
        dims["Wq"] = (a * d, h)
        dims["Wk"] = (k * d, h)
        dims["Wv"] = (k * d, h)
        dims["Wo"] = (h, a * d)
    out = {}
    for j, name in enumerate(TENSOR_ORDER):
        if name not in dims:
            continue
        if integer is not None:
            out[name] = integer_bf16(dims[name], integer[0], integer[1], base + j)
        else:
            std = 1.0 if name == "X" else WEIGHT_STD
            out[name] = normal_bf16(dims[name], std, base + j)
    return out


def grad_output(shape: Shape, seed_base: Optional[int] = None) -> torch.Tensor:
    """Upstream gradient dL/dZ for a block's backward: [tokens][hidden] bf16,
    N(0, 1), seeded after the workload's own tensors."""
    base = 1000 * shape.index if seed_base is None else seed_base
    return normal_bf16((shape.tokens, shape.hidden), 1.0, base + len(TENSOR_ORDER))
