"""The N > 1 path of bench.py on CPU with gloo (world size 2).

With several GPUs every rank runs its own independent simulated ZeRO-2 step
(replicas only: no collective on the data path); the job is timed from a
barrier to a barrier and its time is the slowest rank's.  These tests run that
host logic -- max over ranks, whole-job throughput, rank-0-only output of the
reference arm -- as two real processes over gloo on 127.0.0.1.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    local_ms = [5.0, 7.5][rank]
    ms = bench.max_over_ranks(local_ms, world, "cpu")
    value = bench.job_throughput(1_000_000, world, ms)
    dist.barrier()
    with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
        json.dump({"ms": ms, "value": value}, f)
    dist.destroy_process_group()


def test_max_over_ranks_and_job_throughput(tmp_path):
    port = _free_port()
    mp.spawn(_worker, args=(2, port, str(tmp_path)), nprocs=2, join=True)
    res = [json.load(open(tmp_path / f"r{r}.json")) for r in range(2)]
    for r in res:
        assert r["ms"] == 7.5                       # the slowest rank
        assert r["value"] == pytest.approx(2 * 1_000_000 / 7.5e-3)


def test_single_rank_is_a_no_op():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.25, 1, "cpu") == 3.25
    assert bench.job_throughput(10, 1, 1.0) == pytest.approx(10_000.0)


def test_reference_arm_prints_on_rank_zero_only():
    outs = []
    for rank in (0, 1):
        env = dict(os.environ, RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE="2",
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(_free_port()))
        r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                            "--gpus", "2", "--steps", "1", "--warmup", "3",
                            "--cpu-sample-elems", str(1 << 18)],
                           cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
        assert r.returncode == 0, r.stderr[-2000:]
        outs.append(r.stdout.strip())
    line = json.loads(outs[0].splitlines()[-1])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert outs[1] == ""
