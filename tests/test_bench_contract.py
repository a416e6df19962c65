"""The benchmark's reference arm on the CPU: one JSON line with the keys the bench contract
names, the oracle timed on a bounded sample of the chosen workload (here the tiny fp32
exactness case, so the test runs in seconds)."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_contract_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "tiny",
                          "--steps", "1", "--warmup", "0"], capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    line = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "higher_is_better", "dtype", "data",
                "config", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference"
    assert line["value"] > 0 and line["higher_is_better"] is True
    assert line["config"]["workload"].startswith("Tiny exactness case")
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] == 1
    assert line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"] == {"value": line["value"], "unit": line["unit"], "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}


def test_default_workload_is_the_long_configuration():
    sys.path.insert(0, ROOT)
    import bench

    w = bench.WORKLOADS[bench.DEFAULT_WORKLOAD]
    assert (w["P"], w["b"], w["s"], w["h_q"], w["h_kv"], w["d"], w["dtype"], w["masks"]) == \
        (8, 1, 131072, 64, 64, 128, "bf16", (True,))
    # algorithmic flops count visible (query, key) pairs only: 4 b h d s(s+1)/2 under the mask
    assert bench.attn_flops(1, 131072, 64, 128, True) == 4 * 64 * 128 * 131072 * 131073 // 2
    assert bench.attn_flops(2, 4096, 32, 128, False) == 4 * 2 * 32 * 128 * 4096 * 4096
