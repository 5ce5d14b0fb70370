"""The benchmark's reference arm (the fp64 oracle on the host cores) finishes
within a bounded wall time and times the oracle's arithmetic, not data
preparation.  CPU only."""
import json
import os
import subprocess
import sys
import time

import numpy as np
import attn_inputs
import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_sample_rows_is_linear_and_distinct():
    t0 = time.perf_counter()
    pairs = attn_inputs.sample_rows(8192, 64, 65536, seed=1)
    dt = time.perf_counter() - t0
    assert len(pairs) == 65536 and len(set(pairs)) == 65536
    assert dt < 1.0, f"sampling 65536 rows took {dt:.2f} s"
    for bh in (0, 63):
        for r in (0, 1, 127, 128, 129, 8191):
            assert (bh, r) in set(pairs)


def test_sample_rows_clips_to_the_population():
    pairs = attn_inputs.sample_rows(5, 3, 100, seed=2)
    assert sorted(pairs) == [(b, r) for b in range(3) for r in range(5)]


def test_widened_workload_equals_sampled_rows():
    q, k, v = attn_inputs.make_qkv(2, 3, 200, 260, 32, "bf16", 11, "cpu")
    pairs = attn_inputs.sample_rows(200, 6, 150, seed=3)
    wide = oracle.WidenedWorkload(q, k, v)
    o1, l1 = wide.rows(wide.gather(pairs), True, 0.3)
    o2, l2 = oracle.sampled_rows(q, k, v, pairs, True, 0.3)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
    # grouped K/V heads follow the same head mapping as sampled_rows
    kg, vg = k[:, :1].contiguous(), v[:, :1].contiguous()
    wide_g = oracle.WidenedWorkload(q, kg, vg)
    o1, l1 = wide_g.rows(wide_g.gather(pairs), False, 0.3)
    o2, l2 = oracle.sampled_rows(q, kg, vg, pairs, False, 0.3)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_reference_arm_exact_driver_command():
    """`bench.py --impl reference --gpus 1 --steps 20 --warmup 5` prints its JSON line in bounded time."""
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    t0 = time.perf_counter()
    p = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--gpus", "1", "--steps", "20",
                        "--warmup", "5"], cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    wall = time.perf_counter() - t0
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [ln for ln in p.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["unit"] == "TFLOP/s" and line["value"] > 0
    assert line["steps"] == 20 and line["warmup"] == 5
    assert line["config"]["workload"] == "b2h32_n8192_d128_bf16_causal"
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    # 20 steps of about 2 s plus warm-up and set-up
    assert wall < 300
    assert line["ms_per_step"] < 4000
