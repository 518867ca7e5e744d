"""bench.py's host-side bookkeeping on CPU: the clock summary taken from
nvidia-smi samples (window, device filter, throttle reasons), the recorded
DRAM traffic that is used only while the staged-kernel sources are the ones it
was captured on, and the roofline denominator's fallback."""
import os

import bench

BUS = "00000009:01:00.0"
OTHER = "00000019:01:00.0"


def _row(bus, sm, mx, hw="Not Active", thermal="Not Active", sw_thermal="Not Active",
         power="Not Active"):
    return [bus, str(sm), str(mx), "900.0", "0x0", hw, thermal, sw_thermal, power]


def _sampler(samples, bus=BUS):
    s = bench.ClockSampler.__new__(bench.ClockSampler)
    s.samples = samples
    s.proc = None
    s.bus = bus[:-2] if bus else None  # the sampler keeps domain:bus:device
    return s


def test_clock_summary_uses_the_timed_window_and_this_device():
    samples = [(0.0, _row(BUS, 1000, 2070)),            # before the window
               (1.0, _row(BUS, 2070, 2070)),
               (1.1, _row(OTHER, 800, 2070, hw="Active")),  # another GPU of the machine
               (1.2, _row(BUS, 2040, 2070, power="Active")),
               (1.3, _row(BUS, 2070, 2070)),
               (9.0, _row(BUS, 500, 2070, thermal="Active"))]  # after the window
    got = _sampler(samples).summary(1.0, 1.3)
    assert got["sm_mhz"] == 2070.0 and got["sm_max_mhz"] == 2070.0
    assert got["reasons"] == ["sw_power_cap"]  # the other GPU's hw_slowdown is not ours
    assert got["samples"] == 3 and got["in_timed_window"] is True


def test_clock_summary_without_samples_in_the_window_uses_all():
    samples = [(0.0, _row(BUS, 2070, 2070, hw="Active")), (0.05, _row(BUS, 2060, 2070))]
    got = _sampler(samples).summary(5.0, 6.0)
    assert got["in_timed_window"] is False and got["samples"] == 2
    assert got["reasons"] == ["hw_slowdown"]
    assert got["sm_mhz"] == 2065.0


def test_clock_summary_with_nothing_sampled():
    got = _sampler([]).summary(0.0, 1.0)
    assert got == {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}


def test_recorded_traffic_follows_the_source_hash(tmp_path, monkeypatch):
    f = tmp_path / "traffic.md"
    f.write_text("# x\n\nstaged sources: %s\n\nfwd_d4096: 477398784\n`vjp_d8192: 750947840`\n"
                 % bench.source_hash())
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(f))
    assert bench.recorded_traffic("fwd_d4096") == 477398784
    assert bench.recorded_traffic("vjp_d8192") == 750947840
    assert bench.recorded_traffic("fwd_d8192") is None  # not recorded
    f.write_text("staged sources: 0000000000000000\nfwd_d4096: 477398784\n")
    assert bench.recorded_traffic("fwd_d4096") is None  # other sources: not used
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(tmp_path / "missing.md"))
    assert bench.recorded_traffic("fwd_d4096") is None


def test_source_hash_covers_the_staged_plan_and_kernel_files():
    pkg = os.path.join(bench.ROOT, "rmsnorm_fwd_bwd_add_gb300", "csrc")
    for name in ("planner.h", "staged.cuh", "common.cuh"):
        assert name in bench.STAGED_SOURCES and os.path.exists(os.path.join(pkg, name))
    h = bench.source_hash()
    assert len(h) == 16 and h == bench.source_hash()
    assert bench.source_hash(bench.STAGED_SOURCES[:-1]) != h


def test_measured_peak_falls_back_without_the_file(monkeypatch, tmp_path):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    peak, source = bench.measured_peak()
    assert peak == bench.FALLBACK_HBM_GBS and source == "fallback"
    (tmp_path / "MEASURED_PEAKS.json").write_text('{"hbm_gbs": 6702.2}')
    peak, source = bench.measured_peak()
    assert peak == 6702.2 and source.startswith("measured")
