"""Benchmark bookkeeping on CPU: algorithmic work counts and the roofline
arithmetic, checked against hand-computed values for two workloads."""
import os

import numpy as np
import pytest

import bench
from selective_state_space_fwd_gb300 import workloads as W


def test_counts_fp32_workload():
    w = W.WORKLOADS[2]
    inp = {"valid_len": None}
    c = bench.algorithmic_counts(w, inp)
    e = 8 * 4096 * 1024
    assert c["elements"] == e and c["valid_elements"] == e
    assert c["exps"] == e * 16                       # one exp per (t, d, n)
    assert c["fp32_ops"] == 4 * e * 16 + 2 * e
    # x, delta read + y written (4 B each) + B, C rows + A + D
    assert c["bytes"] == 3 * e * 4 + 2 * 8 * 4096 * 16 * 4 + 1024 * 16 * 4 + 1024 * 4


def test_counts_masked_gated_workload():
    w = W.WORKLOADS[4]
    vl = np.array([64, 2048, 3000, 0] + [100] * 28, np.int32)
    c = bench.algorithmic_counts(w, {"valid_len": vl})
    rows = 64 + 2048 + 2048 + 0 + 100 * 28             # clamped to L
    ev = rows * 1536
    assert c["valid_elements"] == ev
    assert c["exps"] == ev * 16 + ev                   # + one exp per gated element
    nch = 2048 // 256
    assert c["bytes"] == (3 * ev * 2 + 32 * 2048 * 1536 * 2 + 2 * rows * 16 * 2
                          + 1536 * 16 * 4 + 1536 * 4 + 32 * 4 + 32 * nch * 1536 * 16 * 4)


def test_roof_terms():
    c = {"bytes": 6684.5e9, "exps": 32 * 152 * 2070e6, "fp32_ops": 128 * 152 * 2070e6}
    r = bench.roof(c, {"hbm_gbs": 6684.5}, 152, 2070.0)
    assert r["t_hbm"] == pytest.approx(1.0) and r["t_mufu"] == pytest.approx(1.0)
    assert r["t_fp32"] == pytest.approx(1.0) and r["t_roof"] == pytest.approx(1.0)


def test_measured_traffic_requires_matching_sources():
    assert bench.measured_traffic("stream", "no-such-workload") is None
    assert bench.measured_traffic("serial", W.WORKLOADS[2].name) is None


def test_counts_ssd_workloads():
    """The SSD form's bytes and product flops, by hand for both state sizes."""
    for key, N in ((1, 128), (2, 256)):
        w = W.SSD_WORKLOADS[key]
        c = bench.ssd_counts(w)
        Bt, L, H, P, Q = 8, 4096, 32, 64, 128
        e = Bt * L * H * P
        assert c["elements"] == e
        # x, z read and y written (bf16), delta per (t, head), B and C rows, A and D
        assert c["bytes"] == 3 * e * 2 + Bt * L * H * 2 + 2 * Bt * L * N * 2 + 4 * H + 4 * H * P
        nb = L // Q
        # C B^T once per (batch row, block); per head the block matrix times x, C times the
        # state and the state update (2 flops per multiply-add)
        assert c["flops"] == Bt * nb * 2 * Q * Q * N + Bt * H * nb * (2 * Q * Q * P + 4 * Q * N * P)


def test_counts_backward():
    w = W.WORKLOADS[2]
    c = bench.bwd_counts(w, {"valid_len": None}, 256)
    e = 8 * 4096 * 1024
    assert c["exps"] == e * 16 and c["fp32_ops"] == bench.BWD_FP32_PER_NELT * e * 16
    # reads: x, delta, dy, B, C, A, D, chunk states, valid rows; writes: dx, ddelta, dB, dC, dA, dD
    reads = 3 * e * 4 + 2 * 8 * 4096 * 16 * 4 + 1024 * 16 * 4 + 1024 * 4 \
        + 8 * 16 * 1024 * 16 * 4 + 8 * 4
    writes = 2 * e * 4 + 2 * 8 * 4096 * 16 * 4 + 1024 * 16 * 4 + 1024 * 4
    assert c["bytes"] == reads + writes


def test_roofline_takes_the_binding_term():
    """frac is computed against the largest of the three roof terms, and equals
    roof time / measured time."""
    rates = {"ex2_per_clk_sm": 32.0, "fp32_per_clk_sm": 128.0}
    sms, mhz = 152, 2070.0
    unit = 152 * 2070e6
    peaks = {"hbm_gbs": 1000.0}
    # fp32 binds: 2 s of fp32, 1 s of MUFU, 0.5 s of HBM; measured 4 s
    c = {"bytes": 500e9, "exps": 32 * unit, "fp32_ops": 2 * 128 * unit}
    r = bench.roofline(c, 4.0, peaks, rates, sms, mhz)
    assert r["bound"] == "alu" and r["alu_unit"] == "fp32 FMA pipe"
    assert r["frac"] == pytest.approx(0.5) and r["frac_of_roof"] == pytest.approx(0.5)
    # HBM binds
    c = {"bytes": 3000e9, "exps": 32 * unit, "fp32_ops": 128 * unit}
    r = bench.roofline(c, 6.0, peaks, rates, sms, mhz)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["frac"] == pytest.approx(0.5)
    # MUFU binds
    c = {"bytes": 1e9, "exps": 3 * 32 * unit, "fp32_ops": 128 * unit}
    r = bench.roofline(c, 3.0, peaks, rates, sms, mhz)
    assert r["alu_unit"] == "MUFU ex2" and r["frac"] == pytest.approx(1.0)


def test_unit_rates_without_a_gpu_fall_back_to_nominal():
    rates, src = bench.unit_rates()
    if src == "nominal":
        assert rates["ex2_per_clk_sm"] == 32.0 and rates["fp32_per_clk_sm"] == 128.0
    else:
        assert rates["ex2_per_clk_sm"] > 0 and rates["fp32_per_clk_sm"] > 0


def test_slice_rows_is_pure_indexing():
    w = W.WORKLOADS[4].scaled(batch=4, seqlen=64, dim=16)
    inp = W.make_inputs(w)
    s = bench.slice_rows(inp, 1, 3)
    assert np.array_equal(s["x"], inp["x"][1:3]) and np.array_equal(s["B"], inp["B"][1:3])
    assert np.array_equal(s["valid_len"], inp["valid_len"][1:3])
    assert s["A"] is inp["A"] and s["D"] is inp["D"]


def test_smem_port_floor_by_hand(monkeypatch):
    """The shared-memory port floor: the capture's wavefronts of 128 bytes,
    the busiest SM holding ceil(grid / SMs) of the CTAs, at the load rate."""
    entry = {"smem_wavefronts": 152 * 4 * 1000, "grid": 152 * 4 - 1}
    monkeypatch.setattr(bench, "measured_capture", lambda k, w: entry)
    rates = {"lds_bytes_per_clk_sm": 128.0}
    r = bench.smem_port("stream", "any", 1e-3, rates, 152, 1000.0)
    per_cta = entry["smem_wavefronts"] / entry["grid"]
    floor_s = 4 * per_cta / 1e9  # four CTAs on the busiest SM, one wavefront per clock at 1 GHz
    assert r["floor_us"] == pytest.approx(floor_s * 1e6)
    assert r["frac"] == pytest.approx(floor_s / 1e-3)
    assert r["grid"] == entry["grid"] and r["wavefronts"] == entry["smem_wavefronts"]
    # twice the load rate halves the floor
    r2 = bench.smem_port("stream", "any", 1e-3, {"lds_bytes_per_clk_sm": 256.0}, 152, 1000.0)
    assert r2["floor_us"] == pytest.approx(r["floor_us"] / 2)


def test_smem_port_needs_a_capture_with_wavefronts(monkeypatch):
    assert bench.smem_port("stream", "no-such-workload", 1e-3, {}, 152, 2070.0) is None
    monkeypatch.setattr(bench, "measured_capture", lambda k, w: {"dram_read_bytes": 1})
    assert bench.smem_port("stream", "any", 1e-3, {}, 152, 2070.0) is None


def test_committed_captures_are_current():
    """Every capture recorded in profiles/traffic.json was taken on the kernel
    sources as they are (otherwise the bench would report no traffic)."""
    import json
    import os
    entries = json.load(open(os.path.join(bench.ROOT, "profiles", "traffic.json")))
    assert entries
    for e in entries:
        assert bench.measured_capture(e["kernel"], e["workload"]) is not None, e["workload"]


def test_probe_library_exports_its_entry_points():
    """libssmprobe.so (the roofline's unit-rate and shared-load probes) builds
    and exports every entry the bench and the pattern script call."""
    import ctypes
    import shutil
    if shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"):
        pytest.skip("no CUDA compiler")
    from selective_state_space_fwd_gb300 import build as B
    lib = ctypes.CDLL(B.build_probe())
    for name in ("ssmprobe_unit_rates", "ssmprobe_lds_rates", "ssmprobe_lds_patterns"):
        assert hasattr(lib, name), name
