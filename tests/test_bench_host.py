"""Host logic of bench.py, on CPU: the stack's byte count, the peaks it divides
by, the clock-log summary that decides whether a run is kept, and the rule
that the ncu traffic figure is reported only for the source it was taken on."""

import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_stack_bytes():
    # 64 layers x (qkv, o, gate_up, down): 4-bit codes + fp16 scales + 4-bit
    # zero points per 128-row group
    per_layer = 0
    for K, N in ((5120, 7168), (5120, 5120), (5120, 55296), (27648, 5120)):
        per_layer += K * N // 2 + (K // 128) * N * 2 + (K // 128) * N // 2
    assert per_layer == 253_317_120
    assert bench.STACK_BYTES == 64 * per_layer == 16_212_295_680


def test_peaks_measured_or_fallback(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.load_peaks()[3] == "fallback"
    (tmp_path / "MEASURED_PEAKS.json").write_text(
        json.dumps({"hbm_gbs": 6000.5, "bf16_tflops": 1700.0, "bf16_tflops_sustained": 1300.0}))
    assert bench.load_peaks() == (6000.5, 1700.0, 1300.0, "measured")


class _Running:
    pass


def _summary(tmp_path, lines):
    path = tmp_path / "clocks.csv"
    path.write_text("\n".join(lines) + "\n")
    s = bench.ClockSampler(0, str(path))
    s.proc = _Running()  # as if nvidia-smi had been started
    return s.summary()


def test_clock_summary(tmp_path):
    ok = "Not Active, Not Active, Not Active, Not Active"
    got = _summary(tmp_path, [
        f"2032, 2032, 900.1, {ok}",
        "1995, 2032, 1100.0, Not Active, Not Active, Not Active, Active",
        f"2010, 2032, 1050.0, {ok}",
        "[N/A], 2032, 1000.0, " + ok,  # unreadable sample: skipped
        "garbage",
    ])
    assert got == {"sm_mhz": 2010.0, "sm_max_mhz": 2032.0, "reasons": ["sw_power_cap"], "samples": 3}


def test_clock_summary_reports_thermal_slowdown(tmp_path):
    got = _summary(tmp_path, ["1500, 2032, 1100.0, Not Active, Active, Not Active, Not Active"])
    assert got["reasons"] == ["hw_thermal_slowdown"]


def test_clock_summary_without_samples(tmp_path):
    assert _summary(tmp_path, []) is None
    s = bench.ClockSampler(0, str(tmp_path / "never_written.csv"))
    assert s.summary() is None  # nvidia-smi never started


def test_traffic_only_for_the_captured_source(tmp_path, monkeypatch):
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "traffic.json").write_text(json.dumps({"k": {"source_sha256": "abc", "bytes_per_launch": 123}}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "decode_source_sha256", lambda: "abc")
    assert bench.traffic_from_profiles("k")["bytes_per_launch"] == 123
    assert bench.traffic_from_profiles("other") is None
    monkeypatch.setattr(bench, "decode_source_sha256", lambda: "changed")
    assert bench.traffic_from_profiles("k") is None


def test_decode_source_hash_covers_the_kernel_sources():
    h = bench.decode_source_sha256()
    assert len(h) == 64
    for f in bench.DECODE_SOURCES:
        assert os.path.exists(os.path.join(ROOT, "bit_weight_only_wise_b300", "csrc", f))


def test_sweep_entry_rates():
    # 4096 x 4096 at M = 16: 8,716,288 weight bytes (codes, fp16 scales,
    # 4-bit zeros) in 10 us, plus X (16 x 4096) read and Y (16 x 4096)
    # written once at 2 bytes each
    e = bench.sweep_entry("C1", 4096, 4096, 16, "f16", 10.0, 8_716_288, 8000.0, 2000.0)
    assert e["GBs"] == round(8_716_288 / 10.0 / 1e3, 1) == 871.6
    assert e["GBs_incl_xy"] == round((8_716_288 + 2 * 16 * 8192) / 10.0 / 1e3, 1)
    assert e["TFLOPs"] == round(2 * 16 * 4096 * 4096 / 10.0 / 1e6, 1)
    assert e["hbm_frac"] == round(871.6288 / 8000.0, 4)
    assert e["bound"] == "hbm"
    assert bench.sweep_entry("x", 4096, 4096, 64, "bf16", 1.0, 1, 1.0, 1.0)["bound"] == "both"
    assert bench.sweep_entry("x", 4096, 4096, 4096, "bf16", 1.0, 1, 1.0, 1.0)["bound"] == "tensor"


def test_stack_xy_bytes():
    assert bench.STACK_XY_BYTES == 64 * 2 * ((5120 + 7168) + (5120 + 5120) + (5120 + 55296) + (27648 + 5120))
    assert bench.STACK_XY_BYTES < bench.STACK_BYTES // 1000  # activations are < 0.1% of the stream at M = 1


def test_sweep_digest_is_short_and_keeps_the_fractions():
    # the bench line carries a digest of the sweep, not the entries (those are
    # printed one per line before it): the count, each configuration's M = 1
    # fraction of the HBM peak and its largest-M fraction of the tensor peak
    entries = [bench.sweep_entry(f"C{c} shape", 4096, 4096 * c, M, "bf16", 10.0 * M ** 0.5, 8 << 20, 8000.0, 2000.0)
               for c in (1, 2, 3) for M in (1, 16, 256, 4096)]
    d = bench.sweep_summary(entries)
    assert d["entries"] == len(entries)
    assert set(d["hbm_frac_at_M1"]) == {f"C{c} shape 4096x{4096 * c} bf16" for c in (1, 2, 3)}
    assert d["hbm_frac_at_M1"]["C1 shape 4096x4096 bf16"] == round(entries[0]["hbm_frac"], 3)
    assert d["tc_frac_at_largest_M"]["C3 shape 4096x12288 bf16 M=4096"] == round(entries[-1]["tc_frac"], 3)
    assert len(json.dumps(d)) < 1500
    assert bench.sweep_summary([]) is None
