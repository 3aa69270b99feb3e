"""bench.py's reference arm (the CPU oracle on a bounded sample of the
decode workload) runs without a GPU: one JSON line with the contract's keys,
and the sample is prepared once, so steps cost only the oracle's step."""
import json
import os
import subprocess
import sys
import time

from conftest import ROOT


def test_reference_arm_prints_one_contract_line():
    t0 = time.time()
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "4",
                        "--warmup", "3"], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["value"] > 0
    assert d["steps"] == 4 and d["warmup"] == 3 and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    # per step only the oracle's decode step on 2048 weight rows (well under
    # a few seconds), not the preparation of the weight sample
    assert d["ms_per_step"] < 5000
    assert time.time() - t0 < 300
