"""The multi-rank path of bench.py on CPU: two gloo ranks on 127.0.0.1.

On the GPU the bench runs one independent replica per GPU (the path needs
no exchange): a barrier around the timed region, the step time taken as the
maximum over ranks, and the whole-job value = ranks x bytes / that time.
These tests run the same aggregation code with world_size 2 over gloo."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        ms = bench._max_over_ranks(times[rank], dist)
        q.put((rank, ms, bench.replica_value(world, 1_000_000_000, ms)))
    finally:
        dist.destroy_process_group()


def test_step_time_is_the_slowest_rank_and_value_counts_every_replica():
    world, times = 2, [0.5, 0.8]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, times, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, value in got:
        assert ms == pytest.approx(0.8)                 # max over ranks, on every rank
        assert value == pytest.approx(2 * 1.0 / 0.8e-3)  # 2 replicas x 1 GB / 0.8 ms, in GB/s


def test_replica_value_single_gpu():
    assert bench.replica_value(1, 1_690_845_184, 0.5) == pytest.approx(3381.690368)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    # Under torchrun the other ranks of the reference arm exit 0 without work.
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    assert bench.main(["--impl", "reference", "--steps", "1", "--warmup", "1"]) == 0
    assert capsys.readouterr().out == ""
