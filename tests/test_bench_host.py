"""Host-side logic of bench.py, on CPU: the reference arm's JSON line, the
recorded-traffic provenance check, and the clock-sample summary."""
import hashlib
import io
import json
import os
import sys
from contextlib import redirect_stdout

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_reference_arm_prints_one_line_with_the_contract_keys():
    buf = io.StringIO()
    with redirect_stdout(buf):
        rc = bench.main(["--impl", "reference", "--steps", "1", "--warmup", "3",
                         "--workload", "tiny", "--oracle-rows", "32"])
    assert rc == 0
    lines = [l for l in buf.getvalue().splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
              "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC
    assert d["value"] > 0 and d["cpu_baseline"]["kind"] == "oracle"
    assert d["cpu_baseline"]["value"] == d["value"] and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0


def _sha(name):
    with open(os.path.join(ROOT, "bit_w4a4_diffusion_quantize_b300", "csrc", name), "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()


def test_recorded_traffic_is_void_once_a_source_changes(monkeypatch):
    for kernel, rec in bench.MEASURED_TRAFFIC.items():
        current = all(_sha(n) == d for n, d in rec["sources"].items())
        assert bench.measured_traffic(kernel) == (rec["bytes"] if current else None), kernel
        assert os.path.exists(os.path.join(ROOT, rec["profile"])), rec["profile"]
    rec = dict(bench.MEASURED_TRAFFIC["svdq_gemm_w4a4"])
    rec["sources"] = {n: _sha(n) for n in rec["sources"]}
    monkeypatch.setitem(bench.MEASURED_TRAFFIC, "svdq_gemm_w4a4", rec)
    assert bench.measured_traffic("svdq_gemm_w4a4") == rec["bytes"]
    rec["sources"] = dict(rec["sources"], **{"gemm_w4a4.cu": "0" * 64})
    assert bench.measured_traffic("svdq_gemm_w4a4") is None


def test_clock_summary_median_and_reasons():
    c = bench.ClockSampler(0)
    c.t0, c.t1 = 0.0, 1.5
    c.lines = [
        "2032, 2032, 700.5, Not Active, Not Active, Not Active, Not Active",
        "1980, 2032, 1090.0, Not Active, Not Active, Not Active, Active",
        "2032, 2032, 800.0, Not Active, Not Active, Not Active, Not Active",
        "garbage line",
    ]
    s = c.summary()
    assert s["sm_mhz"] == 2032.0 and s["sm_max_mhz"] == 2032.0 and s["samples"] == 3
    assert s["reasons"] == ["sw_power_cap"] and s["power_w_max"] == 1090.0
    c.lines = ["1200, 2032, 900.0, Active, Not Active, Not Active, Not Active"]
    assert c.summary()["reasons"] == ["hw_slowdown"]
    c.lines = []
    assert c.summary()["samples"] == 0
