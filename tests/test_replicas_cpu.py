"""The multi-process path of bench.py on the CPU (gloo, world size 2).

The convolution path does not shard (replicas only): every rank runs the whole
chain on its own GPU, the step time is the maximum over ranks, and rank 0 alone
prints.  These tests cover that host logic without a GPU.
"""

import json
import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, port, out):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": "2", "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist

    r, world = bench.dist_init(None)
    bench.barrier(world)
    worst = bench.max_over_ranks(1.5 + rank, world)   # rank 1 is the slower one
    with open(os.path.join(out, f"rank{r}.json"), "w") as f:
        json.dump({"rank": r, "world": world, "backend": dist.get_backend(), "max": worst}, f)
    dist.destroy_process_group()


def test_replica_helpers_gloo(tmp_path):
    mp.start_processes(_rank_main, args=(_free_port(), str(tmp_path)), nprocs=2, join=True,
                       start_method="spawn")
    got = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(2)]
    for r, g in enumerate(got):
        assert g == {"rank": r, "world": 2, "backend": "gloo", "max": 2.5}


def test_reference_arm_two_ranks():
    # torchrun with two ranks: rank 0 times the oracle and prints one line, rank 1
    # exits without work
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
           "--steps", "1", "--warmup", "0"]
    p = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300,
                       env=dict(os.environ, OMP_NUM_THREADS="2"))
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [l for l in p.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"
