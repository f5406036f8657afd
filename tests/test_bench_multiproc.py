"""The N > 1 bench path on the host: replicas joined by a gloo process group
(world size 2, CPU), the max-over-ranks time and the whole-job rate, and the
reference arm's rank-0-only output."""
import multiprocessing as mp
import os
import socket

import pytest

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    try:
        dist.init_process_group("gloo", rank=rank, world_size=world)
        ms_local = 10.0 + 5.0 * rank                   # rank 1 is the slow one
        ms = bench.max_over_ranks(ms_local, dist, torch.device("cpu"))
        dist.barrier()
        q.put((rank, bench.dist_setup(None), ms, bench.job_tflops(1e12, 4, world, ms)))
        dist.destroy_process_group()
    except Exception as e:                             # reported to the parent, which fails the test
        q.put((rank, "error", repr(e), None))


def test_two_gloo_ranks_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, setup, ms, value in res:
        assert setup != "error", ms
        assert setup == (2, rank, rank)
        assert ms == 15.0                              # both ranks see the slow rank's time
        # 2 ranks x 4 steps x 1e12 flops in 15 ms
        assert value == pytest.approx(2 * 4 * 1e12 / 15e-3 / 1e12)


def test_single_process_needs_no_group():
    assert bench.max_over_ranks(3.5, None, None) == 3.5


def test_reference_arm_prints_on_rank_0_only(capsys):
    import json

    class A:
        workload = "tiny_f32"
        steps = 1
        warmup = 0
        gpus = 2
    bench.run_reference(A, world=2, rank=1)
    assert capsys.readouterr().out == ""
    bench.run_reference(A, world=2, rank=0)
    lines = capsys.readouterr().out.strip().splitlines()
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["higher_is_better"] is True
