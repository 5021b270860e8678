"""bench.py's reported figures, checked on the host (no GPU): the
algorithmic bytes it charges per GEMV, the roofline fraction it derives from
bytes (or flops) over event time against the measured peak, the bound it
picks for a contraction that has HBM bytes too, and the rule that a DRAM
traffic figure is reported only for the kernel source it was captured on.
"""
import importlib.util
import json
import os

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_gemv_bytes_per_scale_kind(bench):
    n, k, m = 152064, 4096, 1
    # codes + fp32 block scales + bf16 x + bf16 y (the lm_head call at M = 1)
    assert bench.gemv_bytes(m, n, k) == n * k + 4 * 1188 * 32 + 2 * k + 2 * n == 623_318_528
    # MXFP8: one e8m0 byte per 32 K of a row
    assert bench.gemv_bytes(1, 18432, 7168, mx=True) == 18432 * 7168 + 18432 * 224 + 2 * 7168 + 2 * 18432
    assert bench.gemv_bytes(4, 300, 100, scales="row") == 300 * 100 + 4 * 300 + 2 * 4 * 100 + 2 * 4 * 300
    assert bench.gemv_bytes(4, 300, 100, scales="tensor") == 300 * 100 + 4 + 2 * 4 * 100 + 2 * 4 * 300
    # ragged edges round the scale grid up
    assert bench.gemv_bytes(1, 129, 130) == 129 * 130 + 4 * 2 * 2 + 2 * 130 + 2 * 129


def test_rotation_launch_bytes_match_the_profile(bench):
    """One batched launch of the decode rotation is 24 layers of the four
    projection shapes at M = 1: 1,291,562,496 bytes, the algorithmic figure
    that profiles/traffic.json sets beside the measured DRAM traffic."""
    from fp8_block_scaled_02_gb300 import inputs
    per_layer = sum(bench.gemv_bytes(1, n, k) for n, k in inputs.ROTATION_SHAPES)
    want = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))
    assert 24 * per_layer == want["gemv_batch_kernel<1,0,true> rotation"]["algorithmic_bytes_per_launch"]
    assert bench.gemv_bytes(1, 152064, 4096) == want["decode_kernel<1,0,true> lm_head"]["algorithmic_bytes_per_launch"]


def _wl(calls, dominant, **kw):
    return dict(calls=[(name, m, b, None) for name, m, b in calls], dominant=dominant, **kw)


def test_hbm_roofline_is_bytes_over_event_time(bench, monkeypatch):
    monkeypatch.setattr(bench, "measured_peaks", lambda: (6000.0, "test"))
    monkeypatch.setattr(bench, "measured_traffic", lambda kernel, workload: None)
    wl = _wl([("M=1", 1, 600_000_000), ("M=4", 4, 300_000_000)], ("k", [0]))
    value, unit, per_call, roof = bench.summarize(wl, [0.1, 0.1], total_ms=0.2, steps=1, workload="w")
    assert unit == "GB/s"
    assert value == pytest.approx(900e6 / 0.2e-3 / 1e9)                  # all bytes over the whole step
    assert per_call["M=1"]["gb_s"] == pytest.approx(6000.0)
    assert per_call["M=1"]["frac_of_measured"] == pytest.approx(1.0)
    assert per_call["M=4"]["frac_of_8TBps"] == pytest.approx(3000.0 / 8000.0)
    # the dominant kernel: call 0 only
    assert roof["bound"] == "hbm" and roof["achieved"] == pytest.approx(6000.0) and roof["frac"] == 1.0
    assert roof["peak"] == 6000.0


def test_contraction_bound_follows_the_larger_time_at_the_peaks(bench, monkeypatch):
    monkeypatch.setattr(bench, "measured_peaks", lambda: (6000.0, "test"))
    monkeypatch.setattr(bench, "tensor_peak", lambda: (2000.0, "test"))
    monkeypatch.setattr(bench, "measured_traffic", lambda kernel, workload: None)
    # 1 TFLOP and 1 GB per call: 0.5 ms of flops vs 0.167 ms of bytes -> tensor
    wl = _wl([("a", 512, 1e12)], ("g", [0]), flops=True, hbm_bytes=[1e9])
    _, unit, per_call, roof = bench.summarize(wl, [1.0], total_ms=1.0, steps=1, workload="w")
    assert unit == "TFLOP/s" and roof["bound"] == "tensor"
    assert roof["achieved"] == pytest.approx(1000.0) and roof["frac"] == pytest.approx(0.5)
    assert per_call["a"]["bound"] == "tensor"
    # the same flops with 6 GB: 1 ms of bytes vs 0.5 ms of flops -> HBM, fraction of the copy peak
    wl = _wl([("a", 512, 1e12)], ("g", [0]), flops=True, hbm_bytes=[6e9])
    _, _, per_call, roof = bench.summarize(wl, [2.0], total_ms=2.0, steps=1, workload="w")
    assert roof["bound"] == "hbm" and roof["unit"] == "GB/s"
    assert roof["achieved"] == pytest.approx(3000.0) and roof["frac"] == pytest.approx(0.5)
    assert roof["tensor"]["frac"] == pytest.approx(0.25)
    assert per_call["a"]["bound"] == "hbm"


def test_fp8_contraction_takes_twice_the_bf16_peak(bench, monkeypatch):
    monkeypatch.setattr(bench, "measured_peaks", lambda: (6000.0, "test"))
    monkeypatch.setattr(bench, "tensor_peak", lambda: (2000.0, "test"))
    wl = _wl([("a", 4096, 2e12)], ("w8a8", [0]), flops=True, fp8=True)
    _, _, _, roof = bench.summarize(wl, [1.0], total_ms=1.0, steps=1, workload="w")
    assert roof["peak"] == 4000.0 and roof["frac"] == pytest.approx(0.5) and roof["dtype"] == "e4m3"


def test_traffic_is_reported_only_for_the_captured_source(bench, tmp_path, monkeypatch):
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(
        {"decode_kernel<1,0,true> lm_head": {"source_sha256": "abc", "dram_bytes_per_launch": 626_000_000}}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_hash", lambda kernel: "abc")
    assert bench.measured_traffic("decode_kernel<1,0,true>", "lm_head") == 626_000_000
    monkeypatch.setattr(bench, "kernel_source_hash", lambda kernel: "changed")
    assert bench.measured_traffic("decode_kernel<1,0,true>", "lm_head") is None
    assert bench.measured_traffic("decode_kernel<1,0,true>", "rotation") is None

