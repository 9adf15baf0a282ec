"""The multi-process side of bench.py, on CPU with the gloo backend (world size 2): the job
time is the maximum over ranks, and the reference arm under torch.distributed.run prints
exactly one line (rank 0) while the other rank exits cleanly without work. Each GPU runs its
own replica (requests shard across GPUs, no collective on the data path), so these host-side
steps are all there is to the N > 1 path."""
import json
import os
import socket
import subprocess
import sys

import torch
import torch.multiprocessing as tmp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import bench
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    try:
        got = bench.max_over_ranks(10.0 * (rank + 1) + 0.25, "cpu")
        torch.distributed.barrier()
        with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
            f.write(repr(got))
    finally:
        torch.distributed.destroy_process_group()


def test_max_over_ranks_gloo(tmp_path):
    world = 2
    tmp.spawn(_rank_main, args=(world, free_port(), str(tmp_path)), nprocs=world, join=True)
    for r in range(world):
        assert float((tmp_path / f"rank{r}.txt").read_text()) == 20.25


def test_reference_arm_under_torchrun_prints_one_line():
    env = dict(os.environ, PYTHONPATH=ROOT)
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(free_port()), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3", "--workload", "kivi_b16_4k"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"
