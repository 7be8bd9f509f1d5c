"""The multi-GPU path of bench.py is replicas only: one process per GPU, each running its own
layer on its own tokens, a barrier around every timed region, the maximum of each timing over
the ranks, and the whole-job value = the tokens of all ranks / that time. This checks the
aggregation with real process groups of two ranks on the CPU (gloo), and that the reference
arm prints from rank 0 only."""

import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, local, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        got = bench.max_over_ranks(local[rank], world)
        value = bench.job_throughput(16384, 10, world, got[0])
        q.put((rank, got, value))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_value_with_two_gloo_ranks():
    world = 2
    local = [[4.75, 13.0, 1.5], [5.25, 12.0, 1.75]]  # each rank's timings (ms)
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, local, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    want = [max(a, b) for a, b in zip(*local)]
    for rank, got, value in res:
        assert got == want, (rank, got)
        # 2 ranks x 10 steps x 16384 tokens over the slowest rank's 5.25 ms
        assert value == pytest.approx(2 * 10 * 16384 / 5.25e-3)


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks([3.0, 4.0], 1) == [3.0, 4.0]
    assert bench.job_throughput(100, 5, 1, 10.0) == pytest.approx(100 * 5 / 10e-3)


def test_reference_arm_prints_from_rank_zero_only():
    argv = sys.argv
    try:
        sys.argv = ["bench.py", "--impl", "reference", "--config", "1", "--steps", "1",
                    "--warmup", "1"]
        args = bench.parse()
    finally:
        sys.argv = argv
    assert bench.run_reference(args, rank=1, world=2) is None
    line = bench.run_reference(args, rank=0, world=2)
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    # the line's contract: the oracle on the host, same metric and unit as the GPU arm
    assert line["metric"] == bench.METRIC and line["unit"] == bench.UNIT
    assert line["higher_is_better"] is True and line["dtype"] == "f64"
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == line["value"] and cb["cores"] >= 1
    assert line["e2e"] == {"value": line["value"], "unit": line["unit"],
                           "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
