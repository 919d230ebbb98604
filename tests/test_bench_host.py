"""Host-side pieces of bench.py on the CPU: the clock record read from
nvidia-smi samples, the committed ncu traffic figures (used only while the
kernel sources are the ones they were taken on), and the peak denominators."""
import bench


def _sampler_with(tmp_path, lines):
    s = bench.ClockSampler(0)
    s.path = str(tmp_path / "clocks.csv")
    with open(s.path, "w") as f:
        f.write("\n".join(lines) + "\n")
    return s


def test_clock_summary_median_under_load_and_reasons(tmp_path):
    idle = "0, 345, 2070, 180.5, 0x0, Not Active, Not Active, Not Active, Not Active"
    load = "0, {}, 2070, {}, 0x4, Not Active, Not Active, Not Active, {}"
    rows = [idle, load.format(2070, 1100.0, "Not Active"), load.format(2040, 1390.0, "Active"),
            load.format(2055, 1200.0, "Not Active"), idle]
    got = _sampler_with(tmp_path, rows).summary()
    # idle samples (below half the top clock) are left out of the median
    assert got["sm_mhz"] == 2055.0
    assert got["sm_max_mhz"] == 2070.0
    assert got["power_w_max"] == 1390.0
    assert got["samples"] == 5
    assert got["reasons"] == ["sw_power_cap"]


def test_clock_summary_reports_throttling_reasons(tmp_path):
    row = "0, 1500, 2070, 900.0, 0x68, Active, Not Active, Active, Not Active"
    got = _sampler_with(tmp_path, [row, row]).summary()
    assert got["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"]
    assert got["sm_mhz"] == 1500.0


def test_clock_summary_without_samples(tmp_path):
    s = _sampler_with(tmp_path, ["garbage line"])
    assert s.summary() == {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}


def test_profiled_traffic_follows_the_source_key(monkeypatch):
    # a summary counts only while the kernel sources hash to its recorded key
    for w in ("prefill_T2048", "prefill_T256", "decode_T1", "moe_T1", "moe_T256"):
        real = bench.kernel_source_hash(w)
        monkeypatch.setattr(bench, "kernel_source_hash", lambda workload=None: "0" * 16)
        assert bench.profiled_traffic(w) is None
        monkeypatch.undo()
        assert bench.kernel_source_hash(w) == real
    assert bench.profiled_traffic("no_such_workload") is None


def test_source_key_covers_each_workloads_kernels():
    # different kernel sources per workload family, one key within a family
    keys = {w: bench.kernel_source_hash(w) for w in
            ("prefill_T2048", "prefill_T256", "decode_T1", "moe_T1", "moe_T256")}
    assert keys["prefill_T2048"] == keys["prefill_T256"]
    assert keys["moe_T1"] == keys["decode_T1"]
    assert len({keys["prefill_T2048"], keys["decode_T1"], keys["moe_T256"]}) == 3


def test_peaks_fall_back_without_the_measured_file(monkeypatch, tmp_path):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    p = bench.load_peaks()
    assert p["source"] == "fallback" and p["hbm"] == 6800.0 and p["bf16"] == 1900.0
    (tmp_path / "MEASURED_PEAKS.json").write_text('{"hbm_gbs": 6692.0, "bf16_tflops": 1941.8}')
    p = bench.load_peaks()
    assert p["source"] == "measured" and p["hbm"] == 6692.0
    assert p["bf16"] == p["bf16_sustained"] == 1941.8


def test_clock_record_rejection_rule():
    ok = {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": []}
    assert bench.clocks_rejected(ok) is None
    # a power cap under load is kept, even with the clock below its maximum
    assert bench.clocks_rejected(dict(ok, sm_mhz=1650.0, reasons=["sw_power_cap"])) is None
    for r in ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"):
        assert r in bench.clocks_rejected(dict(ok, reasons=[r, "sw_power_cap"]))
    # stuck well below the maximum with nothing reported: a leftover clock lock
    assert "no reason" in bench.clocks_rejected(dict(ok, sm_mhz=1400.0))
    assert bench.clocks_rejected(dict(ok, sm_mhz=1900.0)) is None
    # no samples (no nvidia-smi): nothing to reject on
    assert bench.clocks_rejected({"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}) is None
