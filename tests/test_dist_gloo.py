"""The multi-process logic of bench.py on CPU with the gloo backend, world size 2: each rank
takes a disjoint shard of the seeded token stream (weak scaling, no data exchange), the job
time is the maximum over the ranks, and the whole-job value counts every rank's tokens.  The
reference arm does its work on rank 0 only."""
import json
import os
import socket
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank: int, ws: int, port: int, out_dir: str) -> None:
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=ws)
    local_ms = [40.0, 55.0][rank]
    ms_max = bench.reduce_max(local_ms, torch.device("cpu"), ws)
    shard = bench.token_shard(rank, 256)
    value = bench.weak_value(ws, 256, 3, ms_max)
    with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
        json.dump({"ms_max": ms_max, "shard": shard, "value": value}, f)
    dist.barrier()
    dist.destroy_process_group()


def test_two_ranks_shard_and_reduce(tmp_path):
    import torch.multiprocessing as mp
    port = _free_port()
    mp.spawn(_worker, args=(2, port, str(tmp_path)), nprocs=2, join=True)
    r = [json.load(open(tmp_path / f"r{i}.json")) for i in range(2)]
    assert r[0]["ms_max"] == r[1]["ms_max"] == 55.0           # the slowest rank's time
    assert r[0]["value"] == r[1]["value"] == pytest.approx(2 * 256 * 3 / 0.055)
    (a0, n0), (a1, n1) = r[0]["shard"], r[1]["shard"]
    assert n0 == n1 == 256 and a1 == a0 + n0                  # disjoint, contiguous shards


def test_reference_arm_other_ranks_exit_without_work(tmp_path):
    """Under torchrun the reference arm runs on rank 0 only: rank 1 prints nothing and exits 0."""
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1", MASTER_ADDR="127.0.0.1",
               MASTER_PORT=str(_free_port()))
    p = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--steps", "1", "--warmup", "3"], env=env, capture_output=True, text=True, timeout=120)
    assert p.returncode == 0, p.stderr
    assert p.stdout.strip() == ""
