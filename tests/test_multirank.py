"""The N > 1 path of bench.py on CPU: two gloo ranks (world_size 2).

Each rank runs its own replica of the workload (weak scaling); the job time is
the maximum over ranks and the throughput counts the work of every rank. Here
each rank reports a different timed total and both must agree on the max and
on the aggregate; the reference arm must do nothing on ranks other than 0.
"""

import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    import sys

    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local_total_ms = [120.0, 150.0][rank]      # rank 1 is the slow one
    mx = bench.reduce_max(local_total_ms, dist, "cpu")
    flops = 2.0 * 4096 ** 3
    gf = bench.whole_job_gflops(mx, world, 100, flops)
    dist.barrier()
    with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
        f.write(f"{mx} {gf}")
    dist.destroy_process_group()


def test_two_rank_max_and_aggregate(tmp_path):
    world, port = 2, _free_port()
    mp.spawn(_worker, args=(world, port, str(tmp_path)), nprocs=world, join=True)
    vals = [tuple(map(float, open(tmp_path / f"rank{r}.txt").read().split())) for r in range(world)]
    assert vals[0] == vals[1]
    mx, gf = vals[0]
    assert mx == 150.0
    expect = world * 100 * 2.0 * 4096 ** 3 / 0.150 / 1e9
    assert abs(gf - expect) <= 1e-9 * expect


def test_single_rank_identity():
    import bench

    assert bench.reduce_max(7.5, None) == 7.5
    assert bench.whole_job_gflops(1000.0, 1, 1, 2e9) == pytest.approx(2.0)


def test_reference_arm_is_rank0_only(monkeypatch, capsys):
    import bench

    class Args:
        gpus, steps, warmup = 2, 1, 0

    monkeypatch.setenv("RANK", "1")
    bench.run_reference(Args(), rank=1)
    assert capsys.readouterr().out == ""

