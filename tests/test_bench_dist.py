"""The benchmark's multi-rank plumbing on CPU (gloo, world size 2).

Replicas only: each rank runs the whole step on its own GPU and the job's
time is the slowest rank's.  Here two CPU processes check the barrier, the
max-over-ranks reduction and the whole-job throughput formula.
"""

import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist

    dist.init_process_group("gloo", rank=rank, world_size=world)
    bench.barrier(dist)
    local_ms = 10.0 + 5.0 * rank  # rank 1 is the slow one
    out[rank] = bench.reduce_max(local_ms, dist)
    bench.barrier(dist)
    dist.destroy_process_group()


def test_max_over_ranks_and_barrier_gloo():
    world, port = 2, _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
    assert out[0] == out[1] == 15.0


def test_job_throughput_counts_every_rank():
    # 1 GB per rank per step, 2 ranks, slowest rank 1 ms/step -> 2000 GB/s
    assert bench.job_throughput(10**9, 2, 1.0) == pytest.approx(2000.0)
    assert bench.job_throughput(10**9, 1, 0.5) == pytest.approx(2000.0)


def test_reference_arm_other_ranks_do_nothing(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    assert bench.run_reference(bench.parse_args(["--impl", "reference", "--steps", "1", "--warmup", "0"])) is None
    assert capsys.readouterr().out == ""


def test_stage_inputs_round_trip_on_cpu():
    """One packed buffer carries every input: copying it fills all views."""
    import torch

    host = {"a": torch.arange(7, dtype=torch.int64), "b": torch.randn(3, 5).to(torch.bfloat16),
            "c": torch.tensor([1, -1], dtype=torch.int32)}
    packed, views, dev_buf = bench.stage_inputs(host, torch.device("cpu"), pin=False)
    assert packed.numel() == 256 * 3  # each slice padded to 256 bytes
    for v in views.values():
        assert v.data_ptr() % 256 == 0 or v.data_ptr() % 16 == 0
    dev_buf.copy_(packed)
    for k, t in host.items():
        assert torch.equal(views[k], t)
