"""Host-side arithmetic of bench.py (no GPU): the FLOP count the TFLOPS figure
divides, the roofline fractions against the measured peaks, the traffic
record that is only reported on the sources it was taken on, and the clock
record's parsing of nvidia-smi samples."""
import json

import pytest

import bench


def test_attention_flops_counts_two_gemms_and_halves_under_the_mask():
    # S = Q K^T and O = P V: 2 flops per multiply-add, Nq x Nk x d each
    B, H, N, d = 4, 16, 4096, 128
    assert bench.attention_flops(B, H, N, N, d, False) == 2 * 2 * B * H * N * N * d
    assert bench.attention_flops(B, H, N, N, d, True) == 2 * B * H * N * N * d
    assert bench.attention_flops(1, 64, 1, 131072, 128, False) == 4 * 64 * 131072 * 128


def test_tensor_roofline_fraction_and_fp8_peak():
    peaks = {"hbm_gbs": 6000.0, "bf16_tflops": 2000.0}
    meta = {"flops": 5.0e11, "kernel": "attn_fwd_kernel"}
    r = bench.tensor_roofline("bf16_mha_B4_H16_N4096_d128", meta, [0.25, 0.25], peaks, "measured")
    assert r["achieved"] == pytest.approx(2000.0)      # 5e11 flop in 0.25 ms
    assert r["frac"] == pytest.approx(1.0)
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    # an FP8 workload is measured against twice the BF16 peak (the nominal ratio)
    r8 = bench.tensor_roofline("fp8_e4m3_B4_H16_N4096_d128", {"flops": 5.0e11, "kernel": "x"},
                               [0.25], peaks, "measured")
    assert r8["peak"] == pytest.approx(4000.0) and r8["frac"] == pytest.approx(0.5)


def test_prep_roofline_bytes_over_mean_event_time():
    class Ev:
        def __init__(self, ms):
            self.ms = ms

        def elapsed_time(self, other):
            return other.ms - self.ms

    meta = {"prep_events": [(Ev(0.0), Ev(0.05)), (Ev(1.0), Ev(1.07))], "prep_bytes": 3.0e8}
    r = bench.prep_roofline(meta, {"hbm_gbs": 6000.0})
    assert r["ms_per_step"] == pytest.approx(0.06)
    assert r["achieved"] == pytest.approx(3.0e8 / 0.06e-3 / 1e9)
    assert r["frac"] == pytest.approx(r["achieved"] / 6000.0)
    assert bench.prep_roofline({}, {"hbm_gbs": 1.0}) is None


def test_traffic_record_only_on_the_sources_it_was_taken_on(monkeypatch, tmp_path):
    key = "attn_fwd_kernel|bf16_mha_B4_H16_N4096_d128"
    (tmp_path / "profiles").mkdir()
    rec = {key: {"dram_bytes_per_launch": 244636672, "source_hash": bench.kernel_source_hash()}}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(rec))
    # the record is read from profiles/ under the root; the hash stands for the sources
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_hash", lambda names=None: rec[key]["source_hash"])
    assert bench.recorded_traffic("attn_fwd_kernel", "bf16_mha_B4_H16_N4096_d128") == 244636672
    assert bench.recorded_traffic("attn_fwd_kernel", "no_such_workload") is None
    # once a source changes, the record is stale and not reported
    monkeypatch.setattr(bench, "kernel_source_hash", lambda names=None: "0" * 16)
    assert bench.recorded_traffic("attn_fwd_kernel", "bf16_mha_B4_H16_N4096_d128") is None
    # no record at all
    (tmp_path / "profiles" / "traffic.json").unlink()
    assert bench.recorded_traffic("attn_fwd_kernel", "bf16_mha_B4_H16_N4096_d128") is None


def test_clock_summary_median_and_throttle_reasons():
    s = bench.ClockSampler(0)
    line = "{sm}, 2070, 900.0, 0x0, Not Active, Not Active, Not Active, {cap}"
    s.samples = [(1.0, line.format(sm=1900, cap="Active")),
                 (2.0, line.format(sm=2070, cap="Not Active")),
                 (3.0, line.format(sm=1950, cap="Not Active")),
                 (9.0, line.format(sm=100, cap="Not Active"))]   # after the timed region
    r = s.summary(0.5, 3.5)
    assert r["sm_mhz"] == 1950.0 and r["sm_max_mhz"] == 2070.0
    assert r["reasons"] == ["sw_power_cap"] and r["samples"] == 3
    empty = bench.ClockSampler(0).summary(0.0, 1.0)
    assert empty["sm_mhz"] is None and empty["reasons"] == []


def test_every_workload_has_a_config_record():
    for wl, (B, Hq, Hkv, Nq, Nk, d, causal, kind) in bench.WORKLOADS.items():
        c = bench.config_of(wl)
        assert c["workload"] == wl and c["d"] == d and c["causal"] == causal
        assert Hq % Hkv == 0 and d in (64, 128, 256)
        assert kind in ("bf16", "fp8", "fp8h", "fp8hr", "decode")
    assert bench.DEFAULT_WORKLOAD in bench.WORKLOADS
