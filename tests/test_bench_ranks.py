"""The benchmark's multi-rank bookkeeping on CPU: two `gloo` ranks, each with
its own timing, must agree on the slowest rank's time, and the whole-job
throughput must count the work of every rank over that time.  The GEMM has no
exchange step, so N GPUs run N independent replicas and this aggregation is
the only thing the ranks share.
"""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist

    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        my_ms = [12.5, 40.0, 7.0, 33.0][rank]
        ms = bench.max_over_ranks(my_ms, dist, device="cpu")
        value = bench.job_throughput(0.25, 10, world, ms)
        ref = bench.run_reference(type("A", (), {"warmup": 3, "steps": 1})(), rank, world, "c1") if rank else None
        out.put((rank, ms, value, ref))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 4])
def test_max_over_ranks_and_job_throughput(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    slowest = max([12.5, 40.0, 7.0, 33.0][:world])
    for rank, ms, value, ref in got:
        assert ms == slowest, f"rank {rank} saw {ms}"
        # world ranks x 10 steps x 0.25 units in the slowest rank's time
        assert value == pytest.approx(world * 10 * 0.25 / (slowest / 1e3))
        assert ref is None  # only rank 0 runs the reference arm


def test_single_process_needs_no_group():
    import bench

    assert bench.max_over_ranks(3.5, None) == 3.5
    assert bench.job_throughput(2.0, 4, 1, 8.0) == pytest.approx(2.0 * 4 / 8e-3)


def test_custom_dense_shape_uses_the_c2_recipe():
    import bench
    import synth

    cfg = bench.register_shape("96,40,24")
    p = bench.make_problem(cfg)
    ref = synth.config2(M=96, N=40, K=24)
    assert (p.M, p.N, p.K) == (96, 40, 24)
    assert (p.A == ref.A).all() and (p.B == ref.B).all() and (p.C == ref.C).all()
    assert (p.alpha, p.beta) == (1.5, 0.5)
    assert "M=96 N=40 K=24" in bench.WORKLOADS[cfg]["desc"]
