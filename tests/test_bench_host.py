"""Host-side logic of bench.py: the work model and the N-replica timing
aggregation (max over ranks, whole-job value), the latter run as two gloo
ranks on the CPU."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench
from synth import SHAPES


def test_layer_flop_model_matches_the_workload_arithmetic():
    s = SHAPES["layer"]
    parts = dict(bench.layer_kernel_flops(s))
    assert parts["qkv_colwise_gemm+norm"] == pytest.approx(412.3e9, rel=1e-3)
    assert parts["o_proj_rowwise_gemm+g"] == pytest.approx(274.9e9, rel=1e-3)
    assert parts["attention_core"] == pytest.approx(137.4e9, rel=1e-3)
    mlp = parts["w1w3_colwise_gemm+norm+swiglu"] + parts["w2_rowwise_gemm+g"]
    assert mlp == pytest.approx(2886.2e9, rel=1e-3)
    assert bench.layer_flops(s) == pytest.approx(3710.9e9, rel=1e-3)


def test_bench_entry_points_exist():
    for name in ("run_ours", "run_reference", "run_case", "main", "oracle_sample"):
        assert callable(getattr(bench, name)), name


def test_reduce_byte_model():
    # t partials in fp32 read once, residual read once, output written once.
    assert bench.reduce_bytes(8, 8192 * 4096, 4, True) == 8 * 8192 * 4096 * 4 + 2 * 8192 * 4096 * 2
    assert bench.reduce_bytes(4, 100, 2, False) == 4 * 100 * 2 + 100 * 2


def test_whole_job_value_sums_replicas():
    assert bench.whole_job_value(1e12, 1, 1.0) == pytest.approx(1.0)
    assert bench.whole_job_value(1e12, 4, 0.5) == pytest.approx(8.0)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = [3.0, 5.0][rank]                     # per-rank step time
    worst = bench.max_over_ranks(ms, world)
    value = bench.whole_job_value(2e12, world, worst / 1e3)
    dist.barrier()
    q.put((rank, worst, value, bench.dist_env()))
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(2))
    for rank, worst, value, env in got:
        assert worst == 5.0                   # both ranks see the slowest rank's time
        assert value == pytest.approx(2e12 * 2 / 5e-3 / 1e12)
        assert env == (2, rank, rank)
