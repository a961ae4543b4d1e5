"""Host logic of the bench.  The clock record: NVML reason bits and nvidia-smi
lines map to the same slowdown names, and the sampler polls a (fake) NVML
device from a thread so that a timed region of a few milliseconds still gets
samples.  The oracle's timed sample: disjoint row spans, and a run of many
steps that stays within its time budget.  The roofline arithmetic: the
stricter peak, and the operand bytes of the short-head workloads."""
import os
import sys
import time

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_nvml_reason_bits():
    s = bench.summarize_nvml_samples([(2070.0, 0x0), (2000.0, 0x4), (1980.0, 0x1)], 2070.0)
    assert s["sm_mhz"] == 2000.0 and s["sm_max_mhz"] == 2070.0 and s["samples"] == 3
    assert s["reasons"] == ["sw_power_cap"]  # 0x1 (idle) is not a slowdown
    s = bench.summarize_nvml_samples([(1500.0, 0x8 | 0x40), (1400.0, 0x20 | 0x80)], 2070.0)
    assert s["reasons"] == ["hw_power_brake_slowdown", "hw_slowdown", "hw_thermal_slowdown",
                            "sw_thermal_slowdown"]


def test_smi_lines():
    lines = ["0, 2070, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active",
             "0, 1950, 2070, 1390.0, 0x4, Not Active, Not Active, Not Active, Active",
             "garbage"]
    s = bench.summarize_smi_lines(lines)
    assert s["sm_mhz"] == 2010.0 and s["sm_max_mhz"] == 2070.0 and s["samples"] == 2
    assert s["reasons"] == ["sw_power_cap"]
    assert bench.summarize_smi_lines([])["reasons"] == ["unsampled"]


class _FakeNvml:
    max_mhz = 2070.0

    def __init__(self, index):
        self.n = 0
        self.closed = False

    def sample(self):
        self.n += 1
        return (2070.0 if self.n % 2 else 2055.0), 0x0

    def close(self):
        self.closed = True


def test_sampler_polls_during_a_short_region(monkeypatch):
    monkeypatch.setattr(bench, "_NvmlClocks", _FakeNvml)
    with bench.ClockSampler(0) as clk:
        time.sleep(0.02)
    s = clk.summary()
    assert s["samples"] >= 3 and s["reasons"] == [] and s["sm_max_mhz"] == 2070.0
    assert clk.nvml.closed


def test_sampler_falls_back_without_nvml(monkeypatch):
    def _fail(index):
        raise OSError("no NVML here")
    monkeypatch.setattr(bench, "_NvmlClocks", _fail)
    monkeypatch.setattr(bench.subprocess, "Popen", _fail)
    with bench.ClockSampler(0) as clk:
        pass
    assert clk.summary()["reasons"] == ["unsampled"]


def test_reference_sample_spans_are_disjoint_rows():
    from quantized_attention_gb300 import inputs as I
    for name in ("llm8k", "chunk32k", "vit", "swin", "tiny"):
        wl = I.WORKLOADS[name]
        sub = wl.replace(B=1, Hq=wl.Hq // wl.Hkv, Hkv=1)
        for rows, n in ((4096, 32), (64, 16), (20, 16), (1, 8), (10 ** 6, 64)):
            items = bench.oracle_items(sub, rows, n)
            seen = set()
            for h, lo, hi in items:
                assert 0 <= h < sub.Hq and 0 <= lo < hi <= sub.Nq
                span = {(h, r) for r in range(lo, hi)}
                assert not (span & seen)
                seen |= span
            assert len(seen) == min(rows, sub.Hq * sub.Nq) and len(items) <= n


def test_reference_arm_stays_within_its_budget():
    ops, secs, cores, desc = bench.time_cpu_budgeted("tiny", 2, 40, 4.0)
    assert ops > 0 and cores >= 1
    assert secs < 12.0, (secs, desc)  # timed steps within a few times the budget


PEAKS = {"hbm_gbs": 6773.5, "bf16": 1908.3, "bf16_sustained": 1726.8, "source": "measured"}


def test_tensor_roofline_divides_by_the_stricter_peak():
    """The line's fraction uses the higher of the tcgen05-loop peak and the
    cuBLAS-based burst figure (the stricter fraction); both stay in the line."""
    cub = 1.0 / (0.5 / 1908.3 + 0.5 / (2 * 1908.3))  # QK^T at the bf16 rate, PV at twice it
    loops = {"mixed": 3128.0, "f16": 2345.5, "f8": 4692.9}
    r = bench.tensor_roofline(1573.0, PEAKS, loops)
    assert abs(r["peak_cublas_burst"] - cub) < 1e-9
    assert r["peak"] == 3128.0 and abs(r["frac"] - 1573.0 / 3128.0) < 1e-12
    assert abs(r["frac_cublas_burst"] - 1573.0 / cub) < 1e-12
    weak = dict(loops, mixed=2000.0)  # loops below the cuBLAS figure: that one is stricter
    r2 = bench.tensor_roofline(1573.0, PEAKS, weak)
    assert abs(r2["peak"] - cub) < 1e-9 and abs(r2["frac"] - 1573.0 / cub) < 1e-12
    r3 = bench.tensor_roofline(1573.0, PEAKS, None)  # no loops measured
    assert abs(r3["peak"] - cub) < 1e-9 and "peak_tcgen05_loops" not in r3


def test_prefill_roofline_bytes_for_short_heads():
    """ViT and Swin are bound by their operands' bytes: int8 Q and K codes,
    e4m3 V^T at its padded row length, bf16 O and (Swin) one fp32 bias."""
    from quantized_attention_gb300 import inputs as I
    for name, ldv in (("vit", 208), ("swin", 64)):
        wl = I.WORKLOADS[name]
        ms = 0.05
        r = bench.prefill_roofline(wl, ms, 1e9, wl.has_bias, PEAKS, None, ldv)
        want = (wl.B * wl.Hq * wl.Nq * wl.d + wl.B * wl.Hkv * wl.Nk * wl.d + wl.B * wl.Hkv * wl.d * ldv
                + 2 * wl.B * wl.Hq * wl.Nq * wl.d + (4 * wl.Nq * wl.Nk if wl.has_bias else 0))
        assert r["bound"] == "hbm" and r["algorithmic_bytes"] == want
        assert abs(r["frac"] - want / (ms * 1e-3) / 1e9 / PEAKS["hbm_gbs"]) < 1e-12
    r = bench.prefill_roofline(I.WORKLOADS["llm8k"], 0.35, 549.8e9, False, PEAKS, None, 8192)
    assert r["bound"] == "tensor"
