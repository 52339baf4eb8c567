"""Host-side logic of bench.py that decides what its JSON line reports (no GPU needed): the
roofline denominators, the DRAM traffic taken from a committed ncu summary only while the kernel
sources are unchanged, the launch count, the raw parity statistics on the CPU-baseline sample,
the NVML clock summary and the L2-flush decision."""
from __future__ import annotations

import json
import math
import types

import numpy as np
import pytest

import bench
from workloads import WORKLOADS


def test_peaks_measured_and_fallback(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    fb = bench.peaks()
    assert fb["source"] == "fallback" and fb["bf16"] == 1900.0 and fb["hbm_gbs"] == 6800.0
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps(
        {"bf16_tflops": 1892.3, "bf16_tflops_sustained": 1679.0, "hbm_gbs": 6779.4}))
    pk = bench.peaks()
    assert pk == {"bf16": 1892.3, "bf16_sustained": 1679.0, "hbm_gbs": 6779.4,
                  "source": "measured"}


def test_traffic_only_for_the_sources_it_was_taken_on(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.measured_traffic("w", None) is None          # no summary at all
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "fa_fwd_traffic.json").write_text(json.dumps({
        "w": {"dram_bytes_per_launch": 111, "kernel_sources_sha256": "aaa"},
        "w:pv16": {"dram_bytes_per_launch": 222, "kernel_sources_sha256": "aaa"}}))
    monkeypatch.setattr(bench, "kernel_sources_sha256", lambda: "aaa")
    assert bench.measured_traffic("w", None) == 111
    assert bench.measured_traffic("w", None, "pv16") == 222
    assert bench.measured_traffic("other", None) is None
    assert bench.measured_traffic("w", 5.0) == 5.0             # an explicit value wins
    monkeypatch.setattr(bench, "kernel_sources_sha256", lambda: "bbb")
    assert bench.measured_traffic("w", None) is None           # kernel changed since the capture


def test_kernel_sources_hash_covers_the_forward_sources():
    h = bench.kernel_sources_sha256()
    assert len(h) == 64 and int(h, 16) >= 0
    assert all(s.endswith((".cuh", ".cu")) for s in bench.KERNEL_SOURCES)


def test_launches_per_step():
    args = types.SimpleNamespace(splits=1)
    w = WORKLOADS
    assert bench.launches_per_step(w["b2h32n8192d128_bf16"], args, False) == 1
    assert bench.launches_per_step(w["b2h32n16384d128_e4m3"], args, True) == 1
    # causal fp8 with the fp8 P V: the first 256 query rows of every head run a second launch
    assert bench.launches_per_step(w["b2h32n16384d128_e4m3_causal"], args, True) == 2
    assert bench.launches_per_step(w["b2h32n16384d128_e4m3_causal"], args, False) == 1
    assert bench.launches_per_step(w["b1h1n16384d128_bf16"], types.SimpleNamespace(splits=2),
                                   False) == 2


def test_sample_parity_statistics():
    torch = pytest.importorskip("torch")
    B, H, N, d = 1, 2, 8, 4
    rows = [0, 3, 7]
    ref_o = np.zeros((B, H, len(rows), d))
    ref_o[0, 0, 1, 2] = 3.0          # |O_ref| in [2, 4): half a bf16 ulp is 2^-7
    ref_lse = np.full((B, H, len(rows)), 1.5)
    o = torch.zeros(B, H, N, d, dtype=torch.float64)
    lse = torch.full((B, H, N), 1.5, dtype=torch.float64)
    o[0, 0, 3, 2] = 3.015            # 0.015 off: over 1e-2, under 1e-2 + 2^-7
    o[0, 1, 7, 0] = 0.02             # 0.02 off where O_ref = 0: over both
    lse[0, 1, 0] = 1.5 + 4e-4
    ref = {"nb": B, "heads": H, "rows": rows, "o": ref_o, "lse": ref_lse}
    st = bench.sample_parity(o, lse, ref, "bf16")
    assert st["rows"] == 3 and st["heads"] == 2
    assert math.isclose(st["max_err_o"], 0.02, rel_tol=1e-9)
    assert math.isclose(st["max_err_lse"], 4e-4, rel_tol=1e-6)
    assert (st["tol_o"], st["tol_lse"]) == (1e-2, 1e-3)
    assert st["n_over_tol_o"] == 2 and st["n_over_tol_o_plus_half_ulp"] == 1
    assert bench.sample_parity(o, lse, ref, "e4m3")["n_over_tol_o"] == 0   # 5e-2 for fp8


def test_nvml_summary_median_power_and_reasons():
    clk = object.__new__(bench.NvmlClocks)   # no NVML: feed the samples directly
    clk.nvml, clk.max_mhz, clk.period = object(), 2070.0, 0.002
    clk.rows = [(2070.0, 500.0, 0x0), (1800.0, 1300.0, 0x4), (1900.0, 1350.0, 0x4 | 0x8),
                (1850.0, None, None)]
    s = clk.summary()
    assert s["sm_mhz"] == 1875.0 and s["sm_max_mhz"] == 2070.0
    assert s["power_w_max"] == 1350.0 and s["samples"] == 4 and s["period_ms"] == 2.0
    assert s["reasons"] == ["hw_slowdown", "sw_power_cap"]
    clk.rows = []
    assert clk.summary()["reasons"] == ["no samples"]


def test_l2_flush_only_where_inputs_fit():
    fits = {name: bench.inputs_fit_in_l2(w) for name, w in WORKLOADS.items()}
    assert fits["b1h1n256d64_bf16"] and fits["b4h16n2048d128_bf16_causal"]
    assert fits["b1h1n16384d128_bf16"]
    assert not fits["b2h32n8192d128_bf16"] and not fits["b1h16n32768d64_bf16_causal"]
    assert not fits["b2h32n16384d128_e4m3"]
