#!/usr/bin/env python
"""Benchmark of the tensor-parallel transformer layer on one GB300 (or N
independent replicas, one per GPU).

A step is one pass of the whole hot path over one batch: tp_layer_forward on
the full-layer workload (8192 tokens = 4 x 2048, h=4096, 32 query / 8 KV
heads, d=128, SwiGLU ffn=14336, t=8, bf16), i.e. RMSNorm, the colwise QKV
GEMM, causal GQA attention, the rowwise o_proj with the g reduction fused in
its accumulator (+ residual), RMSNorm, the colwise W1/W3 GEMM with the
SiLU*gate epilogue, and the rowwise W2 with g fused (+ residual); both
RMSNorms are folded into the GEMMs as per-row scales.

Printed (rank 0, one JSON line): whole-job TFLOP/s over the timed steps
(algorithmic FLOPs: GEMMs 2*M*N*K, causal attention core counted as half of
4*s^2*d*a per sequence), the dominant kernel's roofline measured live with
CUDA events on the launching stream, the g partial-sum reduce in GB/s
(PARTIALS-mode [t][M][h] fp32 partials of the same layer), an end-to-end
figure through the C ABI with host buffers, SM clocks sampled during the
timed region, and the fp64 oracle timed on the host cores on a bounded
sample.  ``--impl reference`` times the oracle itself as the reference arm.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402
from synth import SHAPES, Shape  # noqa: E402

METRIC = ("sharded-MLP/attn TFLOP/s & % BF16 peak; partial-reduce GB/s & % HBM (1×GB300)")
UNIT = "TFLOP/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# Context denominators: the vendor's dense BF16 figure (no 2:4 sparsity) and
# the tensor rate per SM and clock that tcgen05 kind::f16 issues at (a
# 128 x 256 x 16 MMA step every 128 cycles: 8192 FLOP per SM per clock).
SPEC_BF16_TFLOPS = 2250.0
SPEC_BF16_SOURCE = "NVIDIA GB300 dense BF16, 2.25 PFLOP/s per GPU without sparsity (datasheet)"
TENSOR_FLOP_PER_SM_CLK = 8192.0
NOMINAL_HBM_GBS = 8000.0
# A timed region shorter than this runs at the burst clock (the power cap
# needs about a second of full load to pull the clock down).
BURST_REGION_S = 1.0


# ------------------------------------------------------------------ work model

def gemm_flops(M, N, K):
    return 2.0 * M * N * K


def attn_core_flops(s: Shape):
    # QK^T and PV: 2 * 2 * s^2 * d per head and sequence; causal -> half.
    return 0.5 * 4.0 * s.batch * s.seq * s.seq * s.head_dim * s.heads


def layer_kernel_flops(s: Shape):
    """Algorithmic FLOPs of each kernel of the FUSED layer, in launch order
    (the two RMSNorms are folded into the GEMMs as per-row scales; the
    first kernel only computes the row statistics of x)."""
    M, h, f, a, k, d = s.tokens, s.hidden, s.ffn, s.heads, s.kv_heads, s.head_dim
    return [
        ("row_sumsq_x", 0.0),
        ("qkv_colwise_gemm+norm", gemm_flops(M, (a + 2 * k) * d, h)),
        ("attention_core", attn_core_flops(s)),
        ("o_proj_rowwise_gemm+g", gemm_flops(M, h, a * d)),
        ("w1w3_colwise_gemm+norm+swiglu", gemm_flops(M, 2 * f, h)),
        ("w2_rowwise_gemm+g", gemm_flops(M, h, f)),
    ]


def layer_kernel_bytes(s: Shape):
    """Algorithmic HBM bytes of the row-statistics kernel (read x once)."""
    return {"row_sumsq_x": 2.0 * s.tokens * s.hidden}


def mlp_backward_kernel_flops(M, h, f, glu=True):
    """Algorithmic FLOPs of the MLP backward's GEMMs, in launch order: dH =
    dZ W2 (+ activation gradient), dX = [dU | dG] [W1 ; W3] (f's all-reduce
    in the K loop), dW2 = dZ^T H, [dW1 ; dW3] = [dU | dG]^T X."""
    wu = (2 if glu else 1) * f
    return [
        ("bwd_dh_gemm+act_grad", gemm_flops(M, f, h)),
        ("bwd_dx_gemm+f", gemm_flops(M, h, wu)),
        ("bwd_dw2_gemm", gemm_flops(h, f, M)),
        ("bwd_dw13_gemm", gemm_flops(wu, h, M)),
    ]


def attn_backward_kernel_flops(s: Shape):
    """Algorithmic FLOPs of the attention block's backward, in launch order
    (the core backward is five matmuls of the forward's two sizes: S and dP
    recomputed, dV, dK, dQ)."""
    M, h, a, k, d = s.tokens, s.hidden, s.heads, s.kv_heads, s.head_dim
    return [
        ("bwd_do_gemm", gemm_flops(M, a * d, h)),
        ("bwd_dwo_gemm", gemm_flops(h, a * d, M)),
        ("attn_bwd_core", 2.5 * attn_core_flops(s)),
        ("bwd_dx_gemm+f", gemm_flops(M, h, (a + 2 * k) * d)),
        ("bwd_dwqkv_gemm", gemm_flops((a + 2 * k) * d, h, M)),
    ]


def tensor_roofline(achieved, peaks, peak_src, timed_s, sm_mhz, n_sm):
    """Fractions of a contraction's achieved TFLOP/s.  `peak`/`frac` use the
    measured burst peak when the timed region is shorter than BURST_REGION_S
    and the measured sustained one otherwise; the other fractions are
    context: both measured peaks, the vendor's dense figure, and the tensor
    rate at the SM clock sampled during the timed region."""
    burst = timed_s < BURST_REGION_S
    key = "bf16_tflops" if burst else "bf16_tflops_sustained"
    out = {"peak": peaks[key], "frac": achieved / peaks[key],
           "peak_source": f"{peak_src} {key} (timed region {timed_s:.3f} s: "
                          f"{'under' if burst else 'over'} {BURST_REGION_S:.0f} s, "
                          f"{'burst' if burst else 'sustained'} clocks)",
           "frac_of_burst": achieved / peaks["bf16_tflops"],
           "frac_of_sustained": achieved / peaks["bf16_tflops_sustained"],
           "frac_of_spec": achieved / SPEC_BF16_TFLOPS, "spec_peak": SPEC_BF16_TFLOPS,
           "spec_source": SPEC_BF16_SOURCE}
    if sm_mhz:
        at_clock = n_sm * TENSOR_FLOP_PER_SM_CLK * sm_mhz * 1e6 / 1e12
        out["per_clock"] = {"sm_mhz": sm_mhz, "n_sm": n_sm,
                            "tensor_peak_at_clock": at_clock,
                            "frac_at_clock": achieved / at_clock,
                            "flop_per_sm_clk": TENSOR_FLOP_PER_SM_CLK}
    return out


def layer_flops(s: Shape):
    return sum(v for _, v in layer_kernel_flops(s))


def reduce_bytes(t, n, partial_bytes=4, residual=True):
    return t * n * partial_bytes + n * 2 + (n * 2 if residual else 0)


# ------------------------------------------------------------------ environment

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            d = json.load(fh)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons while running."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.lines = []
        self.proc = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50", "-i", self.gpu_id],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.6)  # let the first samples arrive

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark_start(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ts, line in self.lines:
            if self.t0 is None or not (self.t0 - 0.15 <= ts <= self.t1 + 0.15):
                continue
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def gpu_id_for(torch, dev_index: int) -> str:
    try:
        props = torch.cuda.get_device_properties(dev_index)
        bus = getattr(props, "pci_bus_id", None)
        dom = getattr(props, "pci_domain_id", 0)
        devid = getattr(props, "pci_device_id", 0)
        if bus is not None:
            return f"{dom:08x}:{bus:02x}:{devid:02x}.0"
    except Exception:
        pass
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        return vis.split(",")[dev_index]
    return str(dev_index)


def profiled_traffic(kernel_name: str):
    """DRAM bytes per launch of `kernel_name` from the committed ncu summary
    (profiles/dram_traffic.json) with the command that took them and the
    spread over the recorded captures, or None when the GEMM kernel sources
    have changed since those counters were taken."""
    import hashlib
    try:
        with open(os.path.join(ROOT, "profiles", "dram_traffic.json")) as fh:
            entry = json.load(fh)[kernel_name]
        h = hashlib.sha256()
        for f in ("tp_gemm.cu", "tp_device.cuh", "tp_packed.cuh"):
            with open(os.path.join(ROOT, "megatron_tensor_transformer_colwise_gb300", "csrc", f), "rb") as fh:
                h.update(fh.read())
        if h.hexdigest()[:16] != entry["source_sha256_16"]:
            return None
        out = {"bytes_per_launch": entry["bytes_per_launch"], "source": entry.get("command")}
        if "captures" in entry:
            vals = [c["bytes_per_launch"] for c in entry["captures"]]
            out["spread"] = {"captures": len(vals), "min": min(vals), "max": max(vals)}
        return out
    except Exception:
        return None


# ------------------------------------------------------------------ distributed glue

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(value: float, world: int, device=None) -> float:
    """Maximum of a per-rank scalar (the step time) over all ranks."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_value(flops_per_step_per_rank: float, world: int, seconds_per_step: float) -> float:
    """TFLOP/s of all ranks together (each rank runs its own replica)."""
    return flops_per_step_per_rank * world / seconds_per_step / 1e12


# ------------------------------------------------------------------ CPU oracle leg

def oracle_sample(s: Shape, inp, tokens: int):
    """Time the fp64 oracle on the first `tokens` positions of sequence 0 of
    the layer (causal: identical to the full layer's outputs there)."""
    import oracle
    sub = Shape("sample", 1, tokens, s.hidden, ffn=s.ffn, heads=s.heads, kv_heads=s.kv_heads,
                head_dim=s.head_dim, tp=s.tp, act=s.act)
    f64 = {k: v.double().numpy() for k, v in inp.items() if k != "X"}
    X = inp["X"][:tokens].double().numpy()
    t0 = time.perf_counter()
    oracle.layer(1, tokens, s.heads, s.kv_heads, s.head_dim, s.tp, X, f64["Wq"], f64["Wk"], f64["Wv"],
                 f64["Wo"], f64["W1"], f64["W3"], f64["W2"], sharded=True)
    dt = time.perf_counter() - t0
    fl = layer_flops(sub)
    return {"value": fl / dt / 1e12, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
            "seconds": dt,
            "sample": f"layer forward (sharded t={s.tp} form) on the first {tokens} tokens of one "
                      f"sequence, full h={s.hidden}/ffn={s.ffn} weights, fp64 ({fl / 1e9:.1f} GFLOP)"}


def run_reference(args):
    """The reference arm: the fp64 oracle as it stands, timed on the host
    cores.  Each step is a bounded sample (a causal prefix of one sequence of
    the layer workload) sized so that warm-up plus the timed steps take about
    two minutes in total."""
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    s = SHAPES["layer"]
    import oracle
    oracle.lib()
    inp = synth.workload_inputs(s)
    # Calibrate: seconds per token at a small prefix, then size the sample.
    cal = oracle_sample(s, inp, 8)["seconds"] / 8
    budget = 120.0 / max(1, args.steps + args.warmup)
    tokens = int(max(4, min(256, budget / max(cal, 1e-6))))
    if args.ref_tokens:
        tokens = args.ref_tokens
    for _ in range(args.warmup):
        oracle_sample(s, inp, tokens)
    times = []
    r = None
    for _ in range(args.steps):
        r = oracle_sample(s, inp, tokens)
        times.append(r["seconds"])
    sub = Shape("sample", 1, tokens, s.hidden, ffn=s.ffn, heads=s.heads, kv_heads=s.kv_heads,
                head_dim=s.head_dim, tp=s.tp, act=s.act)
    per = sum(times) / len(times)
    value = layer_flops(sub) / per / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": per * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1) activations, N(0,0.02^2) weights, bf16-rounded)",
        "config": {"workload": "tp_layer_forward: 8192 tokens (4 x 2048), h=4096, 32 q / 8 kv "
                               "heads d=128, SwiGLU ffn=14336, t=8 -- each step a %d-token causal "
                               "prefix of one sequence on the fp64 CPU oracle" % tokens},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.num_threads(),
                         "kind": "oracle", "sample": r["sample"] if r else ""},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


def run_blocks(args):
    """The configurations' blocks alone (the ``blocks`` object of the bench
    line), for profiling."""
    import torch
    import megatron_tensor_transformer_colwise_gb300 as tp
    torch.cuda.set_device(0)
    peaks, _ = load_peaks()
    print(json.dumps(time_blocks(tp, torch, torch.device("cuda", 0), torch.cuda.current_stream(), peaks,
                                 reps=args.steps)))
    return 0


def run_case(args):
    """Single-kernel loops on the layer's shapes, for profiling one kernel:
    w13 (colwise W1/W3 + SwiGLU), qkv (colwise QKV), gelu (colwise GeLU, same
    shape as qkv), o_proj / w2 (rowwise, g fused), attn (attention core),
    reduce (g of [8][8192][4096] fp32 partials + residual)."""
    import torch
    import megatron_tensor_transformer_colwise_gb300 as tp
    torch.cuda.set_device(0)
    s = SHAPES["layer"]
    M, h, f, a, k, d, t = s.tokens, s.hidden, s.ffn, s.heads, s.kv_heads, s.head_dim, s.tp
    peaks, _ = load_peaks()
    stream = torch.cuda.current_stream()
    bf = lambda shape, std, seed: synth.normal_bf16(shape, std, seed).cuda()
    mk = lambda **kw: tp.Plan(tp.make_config(tokens=M, hidden=h, tp_degree=t, batch=s.batch,
                                             seq=s.seq, **kw))
    unit, peak = "TFLOP/s", peaks["bf16_tflops"]
    if args.case == "w13":
        X, W1, W3 = bf((M, h), 1.0, 4000), bf((f, h), 0.02, 4001), bf((f, h), 0.02, 4002)
        H = torch.empty(M, f, dtype=torch.bfloat16, device="cuda")
        plan = mk(ffn=f, act="swiglu")
        fn = lambda: tp.tp_colwise_forward(plan, X, W1, W3, H, stream)
        work = gemm_flops(M, 2 * f, h)
    elif args.case in ("qkv", "gelu"):
        n = (a + 2 * k) * d
        X = bf((M, h), 1.0, 4000)
        if args.case == "qkv":
            Wq, Wk, Wv = bf((a * d, h), 0.02, 4003), bf((k * d, h), 0.02, 4004), bf((k * d, h), 0.02, 4005)
            out = torch.empty(M, n, dtype=torch.bfloat16, device="cuda")
            plan = mk(n_heads=a, n_kv_heads=k, head_dim=d, act="none")
            fn = lambda: tp.tp_qkv_forward(plan, X, Wq, Wk, Wv, out, stream)
        else:
            W1 = bf((n, h), 0.02, 4003)
            out = torch.empty(M, n, dtype=torch.bfloat16, device="cuda")
            plan = mk(ffn=n, act="gelu")
            fn = lambda: tp.tp_colwise_forward(plan, X, W1, None, out, stream)
        work = gemm_flops(M, n, h)
    elif args.case in ("o_proj", "w2"):
        K = a * d if args.case == "o_proj" else f
        Y, W = bf((M, K), 1.0, 4006), bf((h, K), 0.02, 4007)
        res = bf((M, h), 1.0, 4008)
        Z = torch.empty(M, h, dtype=torch.bfloat16, device="cuda")
        plan = mk(ffn=K, act="gelu")
        fn = lambda: tp.tp_rowwise_forward(plan, Y, W, None, res, None, Z, stream)
        work = gemm_flops(M, h, K)
    elif args.case == "packed":
        # Fused Q, K, V, gate, up projection of a single-stream block with an
        # MLP ratio of 3 (blocks [1,1,1,3,3] x 3072), 4096 tokens, t = 4.
        hp, Mp, tpk = 3072, 4096, 4
        blocks = [hp, hp, hp, 3 * hp, 3 * hp]
        X = bf((Mp, hp), 1.0, 4010)
        Wp = bf((sum(blocks), hp), 0.02, 4011)
        out = torch.empty(Mp, sum(blocks), dtype=torch.bfloat16, device="cuda")
        fn = lambda: tp.tp_packed_colwise_forward(X, Mp, hp, Wp, blocks, tpk, out, stream)
        work = gemm_flops(Mp, sum(blocks), hp)
    elif args.case in ("vocab_logits", "vocab_ce", "embedding"):
        # Llama-3-sized output layer / embedding: 8192 tokens, h = 4096,
        # v = 128256, vocab split t = 8.
        Mv, hv, vv, tv = 8192, 4096, 128256, 8
        if args.case == "vocab_logits":
            Hn, Wn = bf((Mv, hv), 1.0, 4100), bf((vv, hv), 0.02, 4101)
            logits = torch.empty(Mv, vv, dtype=torch.bfloat16, device="cuda")
            fn = lambda: tp.tp_vocab_logits_forward(Hn, Mv, hv, Wn, vv, tv, logits, stream)
            work = gemm_flops(Mv, vv, hv)
        elif args.case == "vocab_ce":
            logits = bf((Mv, vv), 3.0, 4103)
            labels = torch.randint(0, vv, (Mv,), dtype=torch.int32, device="cuda")
            stats = torch.empty(3 * tv * Mv, dtype=torch.float32, device="cuda")
            loss = torch.empty(Mv, dtype=torch.float32, device="cuda")
            fn = lambda: tp.tp_vocab_parallel_cross_entropy(logits, Mv, vv, tv, labels, stats, loss,
                                                            stream)
            # logits read once; the exchanged statistics and the loss are small
            work, unit, peak = Mv * vv * 2 + 3 * tv * Mv * 4 * 2 + Mv * 8, "GB/s", peaks["hbm_gbs"]
        else:
            E = bf((vv, hv), 1.0, 4104)
            ids = torch.randint(0, vv, (Mv,), dtype=torch.int32, device="cuda")
            out = torch.empty(Mv, hv, dtype=torch.bfloat16, device="cuda")
            fn = lambda: tp.tp_vocab_embedding_forward(ids, Mv, E, vv, hv, tv, out, stream)
            work, unit, peak = 2 * Mv * hv * 2 + Mv * 4, "GB/s", peaks["hbm_gbs"]
    elif args.case in ("sp_layer", "sp_layer_partials", "partials_layer"):
        # The sequence-parallel layer (all-gather entries, reduce-scatter
        # exits, sequence-split residual stream) with g in the accumulator
        # (sp_layer) or through HBM partials (sp_layer_partials), and the
        # replicated layer with HBM partials (partials_layer).
        inp = synth.workload_inputs(s)
        d = {k: v.cuda() for k, v in inp.items()}
        fused = args.case == "sp_layer"
        plan = tp.Plan(tp.make_config(tokens=M, hidden=h, ffn=f, n_heads=a, n_kv_heads=k,
                                      head_dim=s.head_dim, tp_degree=t, act=s.act,
                                      batch=s.batch, seq=s.seq,
                                      reduce_mode=tp.TP_REDUCE_FUSED if fused else tp.TP_REDUCE_PARTIALS,
                                      sequence_parallel=0 if args.case == "partials_layer" else 1))
        nws = tp.tp_plan_workspace_bytes(plan, tp.TP_OP_LAYER)
        wsb = torch.empty(nws, dtype=torch.uint8, device="cuda")
        Yl = torch.empty(M, h, dtype=torch.bfloat16, device="cuda")
        wd = {kk: vv for kk, vv in d.items() if kk != "X"}
        fn = lambda: tp.tp_layer_forward(plan, d["X"], wd, Yl, wsb, nws, stream)
        work = layer_flops(s)
    elif args.case in ("mlp_backward", "mlp_backward_recompute"):
        # Backward of the layer's MLP (8192 tokens, h 4096, f 14336, SwiGLU,
        # t 8): the pre-activations saved by the forward, or recomputed.
        # --tokens shrinks M for a profiler capture.
        if args.tokens:
            M = args.tokens
            mk = lambda **kw: tp.Plan(tp.make_config(tokens=M, hidden=h, tp_degree=t, **kw))
        X, W1, W3 = bf((M, h), 1.0, 4000), bf((f, h), 0.02, 4001), bf((f, h), 0.02, 4002)
        W2, dZ = bf((h, f), 0.02, 4007), bf((M, h), 1.0, 4012)
        plan = mk(ffn=f, act="swiglu")
        nf = tp.tp_plan_workspace_bytes(plan, tp.TP_OP_MLP)
        fws = torch.empty(nf, dtype=torch.uint8, device="cuda")
        Z = torch.empty(M, h, dtype=torch.bfloat16, device="cuda")
        UG = torch.empty(M, 2 * f, dtype=torch.bfloat16, device="cuda")
        tp.tp_mlp_forward_train(plan, X, W1, W3, W2, None, None, None, Z, UG, fws, nf, stream)
        del fws
        if args.case == "mlp_backward_recompute":
            UG = None
        nws = tp.tp_plan_workspace_bytes(plan, tp.TP_OP_MLP_BACKWARD)
        wsb = torch.empty(nws, dtype=torch.uint8, device="cuda")
        dX = torch.empty(M, h, dtype=torch.bfloat16, device="cuda")
        dW1, dW3 = (torch.empty(f, h, dtype=torch.float32, device="cuda") for _ in range(2))
        dW2 = torch.empty(h, f, dtype=torch.float32, device="cuda")
        db2 = torch.empty(h, dtype=torch.float32, device="cuda")
        fn = lambda: tp.tp_mlp_backward(plan, X, W1, W3, W2, dZ, UG, dX, dW1, dW3, dW2, db2, False,
                                        wsb, nws, stream)
        work = sum(v for _, v in mlp_backward_kernel_flops(M, h, f))
    elif args.case in ("attn_backward", "attn_backward_recompute"):
        # Backward of the layer's attention block (4 x 2048 tokens, h 4096,
        # 32 query / 8 KV heads of 128, t 8), with the forward's QKV, O and
        # softmax statistics saved, or recomputed.
        inp = synth.workload_inputs(s)
        dd = {kk: inp[kk].cuda() for kk in ("X", "Wq", "Wk", "Wv", "Wo")}
        dOut = bf((M, h), 1.0, 4013)
        plan = tp.Plan(tp.make_config(tokens=M, hidden=h, n_heads=a, n_kv_heads=k, head_dim=d,
                                      tp_degree=t, act="none", batch=s.batch, seq=s.seq))
        qb_, ob_, lb_ = tp.tp_plan_attn_saved_bytes(plan)
        QKVs = torch.empty(qb_, dtype=torch.uint8, device="cuda")
        Os = torch.empty(ob_, dtype=torch.uint8, device="cuda")
        LSEs = torch.empty(lb_, dtype=torch.uint8, device="cuda")
        outf = torch.empty(M, h, dtype=torch.bfloat16, device="cuda")
        tp.tp_attn_forward_train(plan, dd["X"], dd["Wq"], dd["Wk"], dd["Wv"], dd["Wo"], None, None,
                                 outf, QKVs, Os, LSEs, stream)
        if args.case == "attn_backward_recompute":
            QKVs = Os = LSEs = None
        nws = tp.tp_plan_workspace_bytes(plan, tp.TP_OP_ATTN_BACKWARD)
        wsb = torch.empty(nws, dtype=torch.uint8, device="cuda")
        dX = torch.empty(M, h, dtype=torch.bfloat16, device="cuda")
        f32 = dict(dtype=torch.float32, device="cuda")
        dWq, dWk = torch.empty(a * d, h, **f32), torch.empty(k * d, h, **f32)
        dWv, dWo = torch.empty(k * d, h, **f32), torch.empty(h, a * d, **f32)
        fn = lambda: tp.tp_attn_backward(plan, dd["X"], dd["Wq"], dd["Wk"], dd["Wv"], dd["Wo"], dOut,
                                         QKVs, Os, LSEs, dX, dWq, dWk, dWv, dWo, False, wsb, nws,
                                         stream)
        work = sum(v for _, v in attn_backward_kernel_flops(s))
    elif args.case == "layer_backward":
        # The layer's training step minus its output: tp_layer_backward
        # recomputes the forward (state kept) and runs the whole backward.
        inp = synth.workload_inputs(s)
        wd = {kk: vv.cuda() for kk, vv in inp.items() if kk != "X"}
        Xd, dY = inp["X"].cuda(), bf((M, h), 1.0, 4014)
        plan = tp.Plan(tp.make_config(tokens=M, hidden=h, ffn=f, n_heads=a, n_kv_heads=k, head_dim=d,
                                      tp_degree=t, act=s.act, batch=s.batch, seq=s.seq))
        nws = tp.tp_plan_workspace_bytes(plan, tp.TP_OP_LAYER_BACKWARD)
        wsb = torch.empty(nws, dtype=torch.uint8, device="cuda")
        dX = torch.empty(M, h, dtype=torch.bfloat16, device="cuda")
        grads = {"d" + kk: torch.empty(tuple(vv.shape), dtype=torch.float32, device="cuda")
                 for kk, vv in wd.items()}
        fn = lambda: tp.tp_layer_backward(plan, Xd, wd, dY, dX, grads, False, wsb, nws, stream)
        # forward (recomputed) + both blocks' backward passes
        work = (layer_flops(s) + sum(v for _, v in mlp_backward_kernel_flops(M, h, f))
                + sum(v for _, v in attn_backward_kernel_flops(s)))
    elif args.case == "attn":
        kvn = max(k // t, 1)
        W = (a // t + 2 * kvn) * d
        QKV = bf((M, t * W), 1.0, 4009)
        O = torch.empty(M, a * d, dtype=torch.bfloat16, device="cuda")
        plan = mk(n_heads=a, n_kv_heads=k, head_dim=d, act="none")
        fn = lambda: tp.tp_attn_core_forward(plan, QKV, O, stream)
        work = attn_core_flops(s)
    else:
        n = M * h
        P = torch.randn(t, M, h, device="cuda")
        res = torch.randn(M, h, device="cuda").to(torch.bfloat16)
        Z = torch.empty_like(res)
        fn = lambda: tp.tp_reduce_partials(P, tp.TP_F32, t, n, h, None, res, Z, stream)
        work, unit, peak = reduce_bytes(t, n), "GB/s", peaks["hbm_gbs"]
    for _ in range(args.warmup):
        fn()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        fn()
    e1.record(stream)
    torch.cuda.synchronize()
    sec = e0.elapsed_time(e1) / args.steps / 1e3
    rate = work / sec / (1e12 if unit == "TFLOP/s" else 1e9)
    print(json.dumps({"case": args.case, "us": sec * 1e6, "achieved": rate, "unit": unit,
                      "peak": peak, "frac": rate / peak}))
    return 0


# ------------------------------------------------------------------ GPU arm

def time_blocks(tp, torch, device, stream, peaks, reps=20):
    """The configurations' blocks through the C ABI (FUSED g), each iteration
    timed alone after an L2 flush (two of the three fit in L2): the GPT-style
    GeLU MLP, the Llama-3-8B-shaped SwiGLU MLP and the batch-1 attention block.
    Returns {name: {...}} with TFLOP/s against the measured bf16 burst peak
    (kernels timed alone)."""
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=device)  # > 129 MB L2
    out = {}
    for name in ("gpt_mlp", "llama_mlp", "attn"):
        s = SHAPES[name]
        inp = {k: v.to(device) for k, v in synth.workload_inputs(s).items()}
        M, h = s.tokens, s.hidden
        plan = tp.Plan(tp.make_config(tokens=M, hidden=h, ffn=s.ffn, n_heads=s.heads,
                                      n_kv_heads=s.kv_heads, head_dim=s.head_dim, tp_degree=s.tp,
                                      act=s.act, batch=s.batch, seq=s.seq))
        Z = torch.empty(M, h, dtype=torch.bfloat16, device=device)
        if s.ffn:
            nws = tp.tp_plan_workspace_bytes(plan, tp.TP_OP_MLP)
            ws = torch.empty(max(nws, 16), dtype=torch.uint8, device=device)
            W3 = inp.get("W3")
            fn = lambda: tp.tp_mlp_forward(plan, inp["X"], inp["W1"], W3, inp["W2"], None, None, None,
                                           Z, ws, nws, stream)
            flops = gemm_flops(M, (2 if s.act == "swiglu" else 1) * s.ffn, h) + gemm_flops(M, h, s.ffn)
            desc = f"tp_mlp_forward: {M} tokens, h={h}, ffn={s.ffn}, {s.act}, t={s.tp}, FUSED g"
        else:
            nws = tp.tp_plan_workspace_bytes(plan, tp.TP_OP_ATTN)
            ws = torch.empty(max(nws, 16), dtype=torch.uint8, device=device)
            fn = lambda: tp.tp_attn_forward(plan, inp["X"], inp["Wq"], inp["Wk"], inp["Wv"], inp["Wo"],
                                            None, None, Z, ws, nws, stream)
            a, k, dh = s.heads, s.kv_heads, s.head_dim
            flops = gemm_flops(M, (a + 2 * k) * dh, h) + attn_core_flops(s) + gemm_flops(M, h, a * dh)
            desc = (f"tp_attn_forward: batch {s.batch} x seq {s.seq}, h={h}, {a} q / {k} kv heads "
                    f"d={dh}, t={s.tp}, FUSED g")
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(reps)]
        for e0, e1 in evs:
            flush.zero_()
            e0.record(stream)
            fn()
            e1.record(stream)
        torch.cuda.synchronize()
        assert tp.tp_get_device_status(plan) == tp.TP_OK, tp.tp_last_error()
        us = sum(e0.elapsed_time(e1) for e0, e1 in evs) / reps * 1e3
        tfl = flops / (us / 1e6) / 1e12
        out[name] = {"workload": desc, "us": us, "tflops": tfl, "frac_bf16": tfl / peaks["bf16_tflops"],
                     "frac_of_spec": tfl / SPEC_BF16_TFLOPS,
                     "gflop": flops / 1e9, "l2": "L2 flushed before every timed iteration",
                     "peak_source": "measured bf16_tflops (burst: each block timed alone)"}
        del inp, ws, Z
    del flush
    return out


def run_ours(args):
    import torch
    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    device = torch.device("cuda", torch.cuda.current_device())
    import megatron_tensor_transformer_colwise_gb300 as tp

    peaks, peak_src = load_peaks()
    s = SHAPES["layer"]
    inp = synth.workload_inputs(s)
    d = {k: v.to(device) for k, v in inp.items()}
    plan = tp.Plan(tp.make_config(tokens=s.tokens, hidden=s.hidden, ffn=s.ffn, n_heads=s.heads,
                                  n_kv_heads=s.kv_heads, head_dim=s.head_dim, tp_degree=s.tp,
                                  act=s.act, batch=s.batch, seq=s.seq,
                                  reduce_mode=tp.TP_REDUCE_FUSED))
    nws = tp.tp_plan_workspace_bytes(plan, tp.TP_OP_LAYER)
    ws = torch.empty(nws, dtype=torch.uint8, device=device)
    Y = torch.empty(s.tokens, s.hidden, dtype=torch.bfloat16, device=device)
    wdict = {k: v for k, v in d.items() if k != "X"}
    weights = tp.layer_weights(wdict)
    stream = torch.cuda.current_stream()
    kf = layer_kernel_flops(s)
    nk = len(kf)

    def mk_events(n):
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        for e in evs:
            e.record(stream)  # materialise the cudaEvent_t
        return evs

    warm_events = mk_events(nk + 1)
    for _ in range(args.warmup):
        tp.tp_layer_forward_traced(plan, d["X"], weights, Y, ws, nws,
                                   [e.cuda_event for e in warm_events], stream)
    torch.cuda.synchronize()
    assert tp.tp_get_device_status(plan) == tp.TP_OK, tp.tp_last_error()

    step_events = [mk_events(nk + 1) for _ in range(args.steps)]
    torch.cuda.synchronize()
    sampler = ClockSampler(gpu_id_for(torch, device.index))
    sampler.start()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler.mark_start()
    start.record(stream)
    for k in range(args.steps):
        tp.tp_layer_forward_traced(plan, d["X"], weights, Y, ws, nws,
                                   [e.cuda_event for e in step_events[k]], stream)
    end.record(stream)
    torch.cuda.synchronize()
    sampler.mark_end()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    clocks = sampler.stop()
    assert tp.tp_get_device_status(plan) == tp.TP_OK, tp.tp_last_error()
    ms_local = start.elapsed_time(end) / args.steps
    ms = max_over_ranks(ms_local, world, device)
    flops = layer_flops(s)
    value = whole_job_value(flops, world, ms / 1e3)

    # Per-kernel durations inside the timed region (same stream, live).
    per_kernel = [0.0] * nk
    for evs in step_events:
        for i in range(nk):
            per_kernel[i] += evs[i].elapsed_time(evs[i + 1])
    per_kernel = [v / args.steps for v in per_kernel]
    total_k = sum(per_kernel)
    kbytes = layer_kernel_bytes(s)
    timed_s = ms_local * args.steps / 1e3
    sm_mhz = clocks.get("sm_mhz") if clocks else None
    n_sm = torch.cuda.get_device_properties(device).multi_processor_count
    kernels = []
    for (name, fl), msk in zip(kf, per_kernel):
        row = {"name": name, "us": msk * 1e3, "share": msk / total_k if total_k else None}
        if fl > 0:
            row["tflops"] = fl / (msk / 1e3) / 1e12
            rl = tensor_roofline(row["tflops"], peaks, peak_src, timed_s, sm_mhz, n_sm)
            row["frac_bf16"] = rl["frac"]
            row["frac_of_spec"] = rl["frac_of_spec"]
            if "per_clock" in rl:
                row["frac_at_clock"] = rl["per_clock"]["frac_at_clock"]
        else:
            row["gbs"] = kbytes[name] / (msk / 1e3) / 1e9
            row["frac_hbm"] = row["gbs"] / peaks["hbm_gbs"]
            row["frac_of_8tbs"] = row["gbs"] / NOMINAL_HBM_GBS
        kernels.append(row)
    dom = max(range(nk), key=lambda i: per_kernel[i])
    dom_name, dom_fl = kf[dom]
    achieved = dom_fl / (per_kernel[dom] / 1e3) / 1e12
    roofline = {"bound": "tensor", "kernel": dom_name, "achieved": achieved, "unit": "TFLOP/s",
                "algorithmic_flops_per_launch": dom_fl, "us_per_launch": per_kernel[dom] * 1e3}
    roofline.update(tensor_roofline(achieved, peaks, peak_src, timed_s, sm_mhz, n_sm))
    if sm_mhz:
        roofline["us_x_mhz"] = per_kernel[dom] * 1e3 * sm_mhz
    tr = args.dominant_traffic if args.dominant_traffic is not None else profiled_traffic(dom_name)
    roofline["traffic"] = tr["bytes_per_launch"] if isinstance(tr, dict) else tr
    if isinstance(tr, dict):
        roofline["traffic_source"] = tr.get("source")
        if "spread" in tr:
            roofline["traffic_spread"] = tr["spread"]

    # The g reduction as a PARTIALS-mode kernel over the layer's partials.
    n = s.tokens * s.hidden
    P = torch.randn(s.tp, s.tokens, s.hidden, dtype=torch.float32, device=device)
    res = torch.randn(s.tokens, s.hidden, device=device).to(torch.bfloat16)
    Zr = torch.empty(s.tokens, s.hidden, dtype=torch.bfloat16, device=device)
    for _ in range(5):
        tp.tp_reduce_partials(P, tp.TP_F32, s.tp, n, s.hidden, None, res, Zr, stream)
    torch.cuda.synchronize()
    r0, r1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    reps = 30
    r0.record(stream)
    for _ in range(reps):
        tp.tp_reduce_partials(P, tp.TP_F32, s.tp, n, s.hidden, None, res, Zr, stream)
    r1.record(stream)
    torch.cuda.synchronize()
    red_us = r0.elapsed_time(r1) / reps * 1e3
    rb = reduce_bytes(s.tp, n, 4, residual=True)
    red_gbs = rb / (red_us / 1e6) / 1e9
    reduce_line = {"bound": "hbm", "kernel": "tp_reduce_partials (t=8 fp32 partials + residual)",
                   "achieved": red_gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                   "frac": red_gbs / peaks["hbm_gbs"], "frac_of_8tbs": red_gbs / NOMINAL_HBM_GBS,
                   "us": red_us, "bytes_per_launch": rb,
                   "peak_source": f"{peak_src} hbm_gbs (kernel timed alone)",
                   "l2": "inputs 1.07 GB > 129 MB L2"}
    del P

    # The configurations' blocks on their own (the MLP configurations are
    # what the sharded-MLP share of the tensor-core peak is quoted on).
    blocks = time_blocks(tp, torch, device, stream, peaks)

    # End to end through the C ABI with host buffers (pinned): every step
    # copies its X in and its Y out.  Copies run on their own streams with
    # double-buffered device X / Y, so step k+1's input copy and step k-1's
    # output copy overlap step k's compute, as a serving loop would run.
    Xh = inp["X"].pin_memory()
    Yh = [torch.empty(s.tokens, s.hidden, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    Xd = [torch.empty_like(d["X"]) for _ in range(2)]
    Yd = [torch.empty_like(Y) for _ in range(2)]
    s_in, s_out = torch.cuda.Stream(device), torch.cuda.Stream(device)
    ev = lambda: torch.cuda.Event()
    in_done, comp_done, out_done = [ev(), ev()], [ev(), ev()], [ev(), ev()]

    def e2e_step(k):
        bi = k % 2
        if k >= 2:
            s_in.wait_event(comp_done[bi])      # Xd[bi] no longer read
        with torch.cuda.stream(s_in):
            Xd[bi].copy_(Xh, non_blocking=True)
        in_done[bi].record(s_in)
        stream.wait_event(in_done[bi])
        if k >= 2:
            stream.wait_event(out_done[bi])     # Yd[bi] copied out
        tp.tp_layer_forward(plan, Xd[bi], wdict, Yd[bi], ws, nws, stream)
        comp_done[bi].record(stream)
        s_out.wait_event(comp_done[bi])
        with torch.cuda.stream(s_out):
            Yh[bi].copy_(Yd[bi], non_blocking=True)
        out_done[bi].record(s_out)

    e2e_steps = max(5, args.steps)
    for k in range(3):
        e2e_step(k)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    s_in.wait_event(e0)
    for k in range(e2e_steps):
        e2e_step(k)
    e1.record(s_out)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, world, device)
    e2e = {"value": whole_job_value(flops, world, e2e_ms / 1e3), "unit": UNIT,
           "h2d_bytes_per_step": Xh.numel() * 2, "d2h_bytes_per_step": Yh[0].numel() * 2,
           "ms_per_step": e2e_ms,
           "pipelining": "copy-in of step k+1 and copy-out of step k-1 overlap step k (2 buffers)"}

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) activations, N(0,0.02^2) weights, bf16-rounded)",
        "config": {"workload": "tp_layer_forward: 8192 tokens (4 x 2048), h=4096, 32 q / 8 kv "
                               "heads d=128, SwiGLU ffn=14336, t=8, FUSED g, bf16",
                   "tokens": s.tokens, "tp_degree": s.tp,
                   "parallelism": f"single-GPU t={s.tp} shards" + (f", {world} replicas" if world > 1 else ""),
                   "gflop_per_step": flops / 1e9,
                   "l2": "inputs larger than L2 (436 MB of weights per step)"},
        "roofline": roofline,
        "reduce": reduce_line,
        "blocks": blocks,
        "kernels": kernels,
        "e2e": e2e,
        "clocks": clocks,
        "gpu_launches": nk * args.steps,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = oracle_sample(s, inp, args.cpu_tokens)
        del line["cpu_baseline"]["seconds"]
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-tokens", type=int, default=256,
                    help="tokens of the bounded oracle sample for cpu_baseline")
    ap.add_argument("--ref-tokens", type=int, default=0,
                    help="tokens of the oracle sample per reference step (0 = sized to ~2 min)")
    ap.add_argument("--case", default="layer",
                    choices=["layer", "w13", "qkv", "gelu", "o_proj", "w2", "attn", "reduce",
                             "packed", "vocab_logits", "vocab_ce", "embedding", "sp_layer", "sp_layer_partials",
                             "partials_layer", "mlp_backward", "mlp_backward_recompute",
                             "attn_backward", "attn_backward_recompute", "layer_backward", "blocks"],
                    help="layer = the benchmark step; others = one kernel alone (profiling)")
    ap.add_argument("--tokens", type=int, default=0,
                    help="mlp_backward cases: tokens (0 = the layer's 8192), for small captures")
    ap.add_argument("--dominant-traffic", type=float, default=None,
                    help="DRAM bytes per launch of the dominant kernel from an ncu capture")
    args = ap.parse_args(argv)
    if args.warmup < 3 and args.impl == "ours":
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        return run_reference(args)
    if args.case == "blocks":
        return run_blocks(args)
    if args.case != "layer":
        return run_case(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
