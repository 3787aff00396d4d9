"""The JSON line contract of bench.py, checked on the CPU: the reference arm (the
float64 oracle on a small row sample) and the traffic lookup that guards against
counters taken on other sources."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_the_contract_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "1",
                        "--cpu-rows", "2"], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["value"] > 0 and d["steps"] == 1 and d["warmup"] == 1
    assert d["unit"] == "TFLOP/s" and d["higher_is_better"] is True
    import bench
    assert d["metric"] == bench.METRIC
    assert d["config"]["workload"] == bench.workload_name()   # the same workload as the measured arm
    assert d["config"]["prefill"] == bench.PREFILL
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_traffic_is_reported_only_for_matching_sources(monkeypatch, tmp_path):
    import bench
    real = bench._source_hash(bench.KERNEL_SOURCES["cp_decode"])
    p = tmp_path / "traffic.json"
    monkeypatch.setattr(bench, "TRAFFIC_JSON", str(p))
    p.write_text(json.dumps({"cp_decode": {"dram_bytes_per_launch": 123, "source_sha256_16": real}}))
    assert bench._traffic("cp_decode") == 123
    p.write_text(json.dumps({"cp_decode": {"dram_bytes_per_launch": 123, "source_sha256_16": "0" * 16}}))
    assert bench._traffic("cp_decode") is None          # counters of other sources are not reported
    assert bench._traffic("ring_attn_bf16") is None     # no entry



def test_headline_line_refuses_workload_overrides():
    # size overrides belong to --parts runs; the headline line always measures the named workload
    for extra in (["--prefill-seq", "32768"], ["--decode-requests", "8"], ["--decode-split", "4"],
                  ["--merge-tokens", "1024"], ["--prefill-shape", "1,8,8,8192,8"]):
        r = subprocess.run([sys.executable, "bench.py", "--steps", "1", "--warmup", "3"] + extra, cwd=ROOT,
                           capture_output=True, text=True, timeout=300)
        assert r.returncode != 0, extra
        assert "--parts" in r.stderr, extra


def test_workload_name_follows_the_sizes(monkeypatch):
    import bench
    assert "S=131072" in bench.workload_name() and "64 req" in bench.workload_name()
    monkeypatch.setitem(bench.PREFILL, "S", 32768)
    assert "S=32768" in bench.workload_name() and "S=131072" not in bench.workload_name()


def test_ring_roofline_reports_burst_and_sustained():
    import bench
    pk = dict(hbm=6000.0, bf16=2000.0, bf16_sus=1600.0, src="measured", sus_mhz=1500.0)
    r = bench.ring_roofline(1500.0, 1.4e14, pk, {"sm_mhz": 2000.0})
    assert r["peak"] == 2000.0 and r["frac"] == 0.75
    assert r["peak_sustained"] == 1600.0 and r["frac_sustained"] == 0.9375
    assert r["sm_mhz_kernel_median"] == 2000.0 and r["sm_mhz_sustained_gemm_median"] == 1500.0
