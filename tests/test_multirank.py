"""The N>1 path of bench.py on CPU: two gloo ranks on 127.0.0.1.

bench.py runs one replica per GPU (the units of work are independent, so there
is no collective on the data path); its only cross-rank steps are the barrier,
the max over ranks of the step time and the sum over ranks of the work.  These
tests run those helpers, and the reference arm under torchrun, as two CPU
processes.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# bench.py picks NCCL (one GPU per rank) when CUDA is visible; these tests are the CPU/gloo form.
pytestmark = pytest.mark.skipif(torch.cuda.is_available(), reason="gloo CPU test (CUDA visible here)")


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out_dir: str):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist

    r, w, local = bench.dist_setup(world)
    bench.barrier(w)
    res = {"rank": r, "world": w, "local": local, "backend": dist.get_backend(),
           "max": bench.max_over_ranks(1.5 + r, w), "sum": bench.sum_over_ranks(1.5 + r, w)}
    bench.barrier(w)
    dist.destroy_process_group()
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump(res, f)


def test_max_and_sum_over_two_gloo_ranks(tmp_path):
    world = 2
    mp.spawn(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    for r, d in enumerate(res):
        assert d["rank"] == r and d["world"] == world and d["local"] == r
        assert d["backend"] == "gloo"
        assert d["max"] == 2.5           # the slowest rank decides the step time
        assert d["sum"] == 1.5 + 2.5     # the work of every rank counts


def test_reference_arm_under_torchrun_prints_one_line_from_rank0():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl", "reference",
           "--gpus", "2", "--steps", "1", "--warmup", "0", "--workload", "tiny_d64_f16"]
    env = dict(os.environ, OMP_NUM_THREADS="2")
    p = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600, env=env)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [l for l in p.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, p.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2
    assert d["metric"].startswith("attention fwd TFLOP/s")
    assert d["value"] > 0 and d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["config"]["workload"] == "tiny_d64_f16"
