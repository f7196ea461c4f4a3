"""The multi-rank path of bench.py on CPU (gloo, world size 2).

Each rank runs its own full workload (weak scaling, no data-path
collective); the only collectives are the timing barrier and the maximum of
the elapsed times over ranks.  Here two gloo ranks check that aggregation,
the whole-job throughput formula, and that only rank 0 of the reference arm
prints a line.
"""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank_main(rank, world, port, out_dir):
    import torch
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    # rank r pretends its timed region took (r + 1) * 10 ms, its kernel 2 + r ms
    got = bench._max_over_ranks([10.0 * (rank + 1), 2.0 + rank, 7.0 - rank], torch.device("cpu"))
    dist.barrier()
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as fh:
        json.dump(got, fh)
    dist.destroy_process_group()


def test_max_over_ranks_with_two_gloo_ranks(tmp_path):
    import socket
    import torch.multiprocessing as mp
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    mp.start_processes(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True,
                       start_method="spawn")
    for r in range(2):
        assert json.load(open(tmp_path / f"rank{r}.json")) == [20.0, 3.0, 7.0]


def test_job_throughput_is_weak_scaling():
    sys.path.insert(0, ROOT)
    import bench
    one = bench._job_tflops(1, 1e12, 10, 1000.0)
    assert one == pytest.approx(10.0)
    assert bench._job_tflops(4, 1e12, 10, 1000.0) == pytest.approx(4 * one)


@pytest.mark.parametrize("rank", [0, 1])
def test_reference_arm_prints_only_on_rank0(rank):
    env = dict(os.environ, WORLD_SIZE="2", RANK=str(rank), LOCAL_RANK=str(rank))
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "small", "--steps", "1", "--warmup", "3"],
                       capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    if rank == 0:
        line = json.loads(lines[-1])
        assert line["impl"] == "reference" and line["unit"] == "TFLOP/s"
        assert line["e2e"]["h2d_bytes_per_step"] == 0
    else:
        assert lines == []
