"""The bench's reference arm (the oracle timed on the host cores) prints one JSON line with the
keys the benchmark contract asks for.  Runs on CPU: the arm never touches a GPU."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1",
                        "--warmup", "0"], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config"):
        assert key in d, key
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert d["steps"] == 1 and d["warmup"] == 0 and d["n_gpus"] == 1
    assert d["unit"] == "tokens/s" and d["higher_is_better"] is True
    assert "workload" in d["config"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"]
    assert cb["value"] == d["value"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_prefill_roofline_counts_the_launches_between_the_stage_events(monkeypatch):
    """With the shared experts on the side stream (a bf16 prefill layer's default) the stage
    events bracket the routed GEMM launches only, so the roofline counts the routed SwiGLU
    FLOPs; MOE_B300_SHARED=serial puts the shared launches inside the events and counts both.
    The launches' measured DRAM traffic is reported only for the set it was captured on."""
    sys.path.insert(0, ROOT)
    import bench
    import moe_inputs
    wl = moe_inputs.workload("dsmoe16b")
    peaks = {"hbm_gbs": 6000.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}
    clocks = {"sm_mhz": 2032, "sm_max_mhz": 2032}
    fb = bench.workload_flops_bytes(wl)
    routed = wl.T * wl.k * 3 * 2 * wl.d * wl.F
    assert fb["routed_flops"] == routed
    assert fb["ffn_flops"] == routed + wl.T * 3 * 2 * wl.d * wl.F_sh
    monkeypatch.delenv("MOE_B300_SHARED", raising=False)
    monkeypatch.delenv("MOE_B300_PATH", raising=False)
    side = bench.prefill_figures(wl, 1.0, [0.5, 0.5], clocks, peaks, "measured")
    assert side["roofline"]["flops_per_step"] == routed
    assert abs(side["roofline"]["achieved"] - routed / 0.5e-3 / 1e12) < 1e-6
    assert side["roofline"]["traffic"] == bench.GEMM_TRAFFIC_BYTES[("dsmoe16b", 8192, 64)]
    monkeypatch.setenv("MOE_B300_SHARED", "serial")
    serial = bench.prefill_figures(wl, 1.0, [0.5, 0.5], clocks, peaks, "measured")
    assert serial["roofline"]["flops_per_step"] == fb["ffn_flops"]
    assert serial["roofline"]["traffic"] is None
    # a decode-sized batch never uses the side stream
    monkeypatch.delenv("MOE_B300_SHARED")
    assert not bench.shared_on_side_stream(wl.replace(T=64))
    assert bench.shared_on_side_stream(wl)
    assert not bench.shared_on_side_stream(moe_inputs.workload("mixtral"))


def test_peak_follows_the_power_cap_of_the_timed_region():
    """Burst peak at full clock; the sustained (power-capped) peak when the median clock sat
    below 95% of the maximum, or the power-cap reason held for at least half of the samples
    while the median clock sat below the maximum."""
    sys.path.insert(0, ROOT)
    import bench
    peaks = {"bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}
    full = {"sm_mhz": 2032, "sm_max_mhz": 2032, "reason_share": {"sw_power_cap": 0.1}}
    assert bench.choose_peak(peaks, "measured", full)[0] == 1800.0
    slow = {"sm_mhz": 1837, "sm_max_mhz": 2032, "reason_share": {}}
    assert bench.choose_peak(peaks, "measured", slow)[0] == 1400.0
    capped = {"sm_mhz": 1935, "sm_max_mhz": 2032, "reason_share": {"sw_power_cap": 0.9}}
    peak, kind = bench.choose_peak(peaks, "measured", capped)
    assert peak == 1400.0 and "90%" in kind
    assert bench.choose_peak(peaks, "measured", {"sm_mhz": None})[0] == 1800.0
    # the cap flag raised while the clock held its maximum does not count
    held = {"sm_mhz": 2032, "sm_max_mhz": 2032, "reason_share": {"sw_power_cap": 1.0}}
    assert bench.choose_peak(peaks, "measured", held)[0] == 1800.0
