"""The N > 1 host logic of bench.py on CPU (gloo, world size 2): process
group setup, the barrier, the max over ranks, and the reference arm under
torchrun (rank 0 alone prints one JSON line; the other rank exits 0 without
work).  The path shards by independent problems (replicas), so there is no
data-path collective to test."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "RANK": str(rank),
                       "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank)})
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist

    w, r, _ = bench.dist_setup()
    assert (w, r) == (world, rank) and dist.get_backend() == "gloo"
    bench.barrier(w)
    got = bench.max_over_ranks(10.0 + rank, w)
    with open(os.path.join(out_dir, f"r{rank}.txt"), "w") as f:
        f.write(repr(got))
    dist.destroy_process_group()


@pytest.mark.skipif(__import__("torch").cuda.is_available(), reason="the CPU (gloo) form of the ranks")
def test_max_over_ranks_gloo(tmp_path):
    mp.start_processes(_rank_main, args=(2, _free_port(), str(tmp_path)), nprocs=2, join=True,
                       start_method="spawn")
    for r in range(2):
        assert float((tmp_path / f"r{r}.txt").read_text()) == 11.0


def test_reference_arm_under_torchrun():
    """`bench.py --impl reference` launched as the driver launches N > 1 runs:
    one JSON line, from rank 0, on the shared workload description."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), "bench.py",
           "--impl", "reference", "--gpus", "2", "--steps", "3", "--warmup", "3",
           "--workload", "tiny_prefill"]
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    p = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600, env=env)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [l for l in p.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, p.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["config"]["workload"].startswith("tiny_prefill: m=64")
