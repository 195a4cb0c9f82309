"""The bench's output contract, checked on the CPU through its reference arm
(`bench.py --impl reference`, the oracle on a bounded row sample): one JSON line
with the keys and types the contract names."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
                        "fp32_small", "--steps", "1", "--warmup", "0"], capture_output=True, text=True, timeout=300,
                       cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1, r.stdout
    out = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "higher_is_better", "scaling",
                "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e"):
        assert key in out, key
    assert out["impl"] == "reference"
    assert out["n_gpus"] == 1 and out["steps"] == 1 and out["warmup"] == 0
    assert out["unit"] == "TFLOP/s" and out["higher_is_better"] is True
    assert isinstance(out["value"], (int, float)) and out["value"] > 0
    assert out["config"]["workload"].startswith("fp32_small")
    cb = out["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == out["value"] and cb["sample"]
    e2e = out["e2e"]
    assert e2e["value"] == out["value"] and e2e["unit"] == out["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_cuda_arm_rejects_workloads_it_does_not_time():
    """The CUDA arm times the bf16 pipeline; asking it for the fp32 correctness workload (or an
    unknown name) fails before any device work, with the bf16 choices listed."""
    for name in ("fp32_small", "no_such_workload"):
        r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--workload", name, "--steps", "1"],
                           capture_output=True, text=True, timeout=300, cwd=ROOT)
        assert r.returncode == 2 and r.stdout == ""
        assert "dense_16k" in r.stderr and name in r.stderr


def test_cpu_baseline_credits_the_rows_the_oracle_computes():
    """cpu_baseline credits 10 d FLOPs per kept key of each sampled row: the forward row
    (N d products for the scores and N d for P V, multiply and add counted separately)
    and the dQ row (scores, dP and dS K again).  Counted here from the definition, row by
    row, against the helper the bench uses, with and without a block mask."""
    import numpy as np
    sys.path.insert(0, ROOT)
    import bench
    N, d = 512, 64
    rows = np.array([0, 1, 127, 128, 300, 511])
    assert bench.oracle_sample_flops(rows, N, d) == len(rows) * (4 * N * d + 6 * N * d)
    mask = np.zeros((4, 4), dtype=np.uint8)
    mask[0, 0] = 1
    mask[1, :2] = 1
    mask[2, [0, 3]] = 1
    mask[3, :] = 1
    want = 0
    for i in rows:
        keys = sum(1 for j in range(N) if mask[i // 128, j // 128])
        want += 4 * keys * d + 6 * keys * d
    assert bench.oracle_sample_flops(rows, N, d, mask) == want
