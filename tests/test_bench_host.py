"""Host-side checks of bench.py: the reference arm's JSON line (the oracle on
the host cores, run here on a small workload) and the roofline arithmetic
the GPU arm reports."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from kv_cache_eviction_03_gb300 import accounting as A  # noqa: E402
from kv_cache_eviction_03_gb300 import workload as W  # noqa: E402


def test_reference_arm_prints_one_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--config", "tiny-ref",
                        "--steps", "1", "--warmup", "0"], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == bench.UNIT and d["metric"] == bench.METRIC
    assert d["value"] > 0 and d["higher_is_better"] is True and d["steps"] == 1 and d["warmup"] == 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]
    assert d["config"]["workload"].startswith("tiny-ref")


def test_decode_roofline_arithmetic():
    w = W.WORKLOADS["opt-6.7b"]
    r = bench.decode_roofline(w, 10.0, 6785.9)
    nbytes = A.decode_step_bytes(w.pairs, w.cache_slots, w.head_dim, 2)
    assert r["algorithmic_bytes_per_launch"] == nbytes
    assert r["achieved_gbs"] == pytest.approx(nbytes / 10.0 / 1e3)
    assert r["frac"] == pytest.approx(r["achieved_gbs"] / 6785.9)
    assert r["tokens_per_s_per_layer"] == pytest.approx(w.batch / 10e-6)


def test_traffic_record_is_keyed_to_the_decode_sources():
    rec = json.load(open(os.path.join(ROOT, "profiles", "decode_traffic.json")))
    assert set(rec["workloads"]) == set(W.WORKLOAD_ORDER)
    want = bench.decode_traffic_record("opt-6.7b")
    if rec["decode_sources_sha256"] == bench.decode_source_digest():
        assert want == rec["workloads"]["opt-6.7b"]["dram_bytes_per_launch"]
    else:
        assert want is None  # the kernel changed since the counters were taken
