"""bench.py's multi-rank path on the CPU, as world_size-2 process groups on
the gloo backend, launched the way the GPU runs are (torch.distributed.run,
rendezvous on 127.0.0.1).  On the GPU the same helper reduces over NCCL:
the job's step time is its slowest rank's, and under torchrun the reference
arm runs on rank 0 alone."""
import json
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

WORKER = r'''
import json, os, sys
sys.path.insert(0, {root!r})
import torch.distributed as dist
dist.init_process_group("gloo")
import bench
rank, world = dist.get_rank(), dist.get_world_size()
# rank r reports a step of 1 + r, an end-to-end time of 10 - r, and r
got = bench.max_over_ranks([1.0 + rank, 10.0 - rank, float(rank)], "cpu")
with open(os.path.join({out!r}, f"rank{{rank}}.json"), "w") as f:
    json.dump({{"rank": rank, "world": world, "got": got}}, f)
dist.barrier()
dist.destroy_process_group()
'''


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_max_over_ranks_world_size_2(tmp_path):
    script = tmp_path / "worker.py"
    script.write_text(WORKER.format(root=ROOT, out=str(tmp_path)))
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes", "1",
           "--nproc-per-node", "2", "--master-addr", "127.0.0.1", "--master-port",
           str(_free_port()), str(script)]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, timeout=300)
    assert r.returncode == 0, r.stderr.decode()[-2000:]
    for rank in range(2):
        d = json.loads((tmp_path / f"rank{rank}.json").read_text())
        assert d["world"] == 2 and d["rank"] == rank
        assert d["got"] == [2.0, 10.0, 1.0]  # every rank sees the maxima


def test_reference_arm_runs_on_rank_0_only():
    """A non-zero rank of the reference arm exits 0 at once and prints
    nothing (rank 0 alone runs the oracle and prints the line)."""
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], cwd=ROOT, env=env, capture_output=True, timeout=300)
    assert r.returncode == 0, r.stderr.decode()[-2000:]
    assert r.stdout.strip() == b""
