"""The reference arm of bench.py (the oracle timed on the host cores) prints the JSON line the
benchmark contract asks for, on CPU: the oracle needs no GPU."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.timeout(600)
def test_reference_arm_prints_one_contract_line():
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "3",
                        "--ref-rows", "1"], cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["steps"] == 1 and d["warmup"] == 3 and d["n_gpus"] == 1
    assert d["value"] > 0 and d["higher_is_better"] is True and d["unit"] == "query-tokens/s"
    assert d["config"]["workload"] == "decode_b32_sq1_h128_topk2048_R352"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_sweep_oracle_rates_on_cpu():
    sys.path.insert(0, ROOT)
    import bench
    import synth
    r = bench.oracle_decode_rate(synth.tiny_decode(seed=0))
    assert r["oracle_query_tokens_per_s"] > 0 and r["oracle_cores"] >= 1
    assert r["oracle_sample"].startswith("1 of 1 query rows")
    a = bench.oracle_append_rate(synth.write_path(seed=0, T=256, num_slots=1024), n_tokens=128)
    assert a["oracle_tokens_per_s"] > 0 and a["oracle_sample"] == "128 of 256 tokens"
