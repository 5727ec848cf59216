"""The multi-process paths of bench.py on CPU: gloo ranks, world size 2."""
import json
import os
import socket
import subprocess
import sys

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_path):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    got = bench.max_over_ranks(10.0 + 5 * rank, dist, "cpu")
    with open(f"{out_path}.{rank}", "w") as f:
        f.write(repr(got))
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_with_gloo(tmp_path):
    port = _free_port()
    out = str(tmp_path / "r")
    mp.start_processes(_rank_main, args=(2, port, out), nprocs=2, start_method="spawn")
    assert [float(open(f"{out}.{r}").read()) for r in range(2)] == [15.0, 15.0]


def test_max_over_ranks_single_process():
    import bench
    assert bench.max_over_ranks(3.5, None) == 3.5


def test_bench_reference_arm_two_ranks():
    """torchrun with 2 ranks: rank 0 alone times the oracle and prints one line."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr=127.0.0.1", f"--master-port={_free_port()}", "bench.py",
           "--impl", "reference", "--config", "tiny", "--steps", "3", "--warmup", "3",
           "--ref-tokens", "2"]
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["steps"] == 3
    assert d["cpu_baseline"]["kind"] == "oracle" and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0
