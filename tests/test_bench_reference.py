"""The reference arm of bench.py (the fp64 oracle on the host cores) runs without a GPU and prints
the one JSON line the bench contract asks for, on the workload and metric of the GPU arm."""
import json
import math
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_contract_line():
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1",
                        "--warmup", "0"], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["metric"] == "KDA fwd tokens/s (B=4,H=96,T=8192,d=128,C=64)"
    assert d["unit"] == "tokens/s" and d["higher_is_better"] is True
    assert d["steps"] == 1 and d["warmup"] == 0 and d["value"] > 0
    assert d["config"]["workload"] == "kda_bf16_B4_H96_T8192_d128_C64"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"]
    assert cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0
    # tokens/s from the timed sample: steps * sequences * T / H over the measured time
    n_seq = int(cb["sample"].split()[2])
    assert math.isclose(d["value"] * d["ms_per_step"] * 1e-3, n_seq * 8192 / 96, rel_tol=1e-9)
