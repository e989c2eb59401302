"""The bench's reference arm (the CPU oracle timed on the native arm's workload and
metric) runs without a GPU and prints one JSON line with the keys the bench contract
asks for: impl, metric, value, unit, steps, warmup, a cpu_baseline that describes the
run (kind oracle, the host threads it kept busy, the sample) and an e2e block with no
host-device traffic."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

ATTN_METRIC = "decode-attn KV GB/s (% of HBM peak); frame steps/sec at B streams, 1 GB300"
NATIVE_METRIC = {
    None: ATTN_METRIC,
    "talker": ATTN_METRIC,
    "paged": ATTN_METRIC,
    "layer": "talker frame GB/s (weights + KV, % of HBM peak); frame steps/sec",
    "prefill": "prefill: prompt positions per second (B streams, all 28 layers)",
}


@pytest.mark.parametrize("workload", [None, "talker", "paged", "layer", "prefill"])
def test_reference_arm_prints_one_contract_line(workload):
    """None: the default workload (32 batched streams, bf16 KV), as the driver runs it."""
    cmd = [sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "3"]
    if workload is not None:
        cmd += ["--workload", workload]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["metric"] == NATIVE_METRIC[workload]
    assert d["steps"] == 1 and d["warmup"] == 3
    assert d["value"] > 0 and d["higher_is_better"] is True
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["unit"] == d["unit"]
    assert isinstance(cb["cores"], int) and cb["cores"] >= 1 and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
