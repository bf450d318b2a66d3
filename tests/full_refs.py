"""Oracle results at the workloads' full sizes, computed once per test
session and shared by the tests that compare against them (not a test
module).

They use the oracle's composed forms (numpy matrix products, the C attention
core and norms), which the oracle pins equal to its all-C definitions."""
import functools

import oracle
import synth
from synth import SHAPES

LAYER_WEIGHTS = ("Wq", "Wk", "Wv", "Wo", "W1", "W3", "W2")


def f64(t):
    return t.detach().to("cpu").double().numpy()


@functools.lru_cache(maxsize=None)
def layer_forward():
    """(inputs, y, h1) of the full layer: 4 x 2048 tokens, h 4096, 32 / 8
    heads of 128, SwiGLU ffn 14336."""
    s = SHAPES["layer"]
    inp = synth.workload_inputs(s)
    Y, h1 = oracle.layer_composed(s.batch, s.seq, s.heads, s.kv_heads, s.head_dim, f64(inp["X"]),
                                  *(f64(inp[n]) for n in LAYER_WEIGHTS), want_h1=True)
    return inp, Y, h1


@functools.lru_cache(maxsize=None)
def layer_backward():
    """(inputs, dY, (dX, dWq, dWk, dWv, dWo, dW1, dW3, dW2)) of the full layer."""
    s = SHAPES["layer"]
    inp = synth.workload_inputs(s)
    dY = synth.grad_output(s)
    out = oracle.layer_backward_composed(s.batch, s.seq, s.heads, s.kv_heads, s.head_dim, f64(inp["X"]),
                                         *(f64(inp[n]) for n in LAYER_WEIGHTS), f64(dY))
    return inp, dY, out
