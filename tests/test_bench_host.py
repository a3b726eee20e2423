"""Host-side logic of bench.py (no GPU): the algorithmic bytes and flops the
roofline divides by, the storage sizes per weight format, the expected
touched-expert count, and the DRAM-traffic lookup keyed by kernel source."""

import hashlib
import os

import pytest

import bench
from routed_expert_ffn_gemm_gb300 import inputs


def test_gate_up_algorithmic_bytes_of_the_headline_layer():
    # Mixtral-shaped, T=64, top-2 over 8 experts, all 8 touched: two bf16
    # weight matrices [14336, 4096] per expert, the 128 gathered rows in,
    # h [128, 14336] out
    shape = inputs.WORKLOADS["mixtral_8x7b"].with_T(64)
    work = bench.stage_work(shape, touched=8, splits=7)
    gu_bytes, gu_flops = work["gate_up"]
    assert gu_bytes == 8 * 2 * 14336 * 4096 * 2 + 128 * 4096 * 2 + 128 * 14336 * 2
    assert gu_flops == 4.0 * 128 * 14336 * 4096
    dn_bytes, dn_flops = work["down"]
    # down: one matrix per expert, h in, 7 fp32 split partials out
    assert dn_bytes == 8 * 4096 * 14336 * 2 + 128 * 14336 * 2 + 7 * 128 * 4096 * 4
    assert dn_flops == 2.0 * 128 * 14336 * 4096


@pytest.mark.parametrize("wfmt,bytes_per_weight", [("f32", 4), ("bf16", 2), ("fp8", 1), ("fp8a8", 1),
                                                   ("mxfp4", 17 / 32)])
def test_bytes_per_weight(wfmt, bytes_per_weight):
    shape = inputs.MoEShape("s", T=1, d=128, ffn=128, E=2, k=1, wfmt=wfmt,
                            act="f32" if wfmt == "f32" else "bf16")
    assert bench.wbytes(shape) == bytes_per_weight


def test_fp8_scales_and_fp8_rows_enter_the_bytes():
    base = inputs.MoEShape("s", T=4, d=256, ffn=128, E=4, k=2, wfmt="fp8")
    a8 = inputs.MoEShape("s", T=4, d=256, ffn=128, E=4, k=2, wfmt="fp8a8")
    b_fp8, _ = bench.stage_work(base, touched=4, splits=1)["gate_up"]
    b_a8, _ = bench.stage_work(a8, touched=4, splits=1)["gate_up"]
    # same weights and per-channel scales; the rows are E4M3 codes + one
    # fp32 scale each (FP8 activations) instead of two E4M3 rows + a scale
    # (FP8 weights on bf16 rows)
    R, d = 8, 256
    assert b_fp8 - b_a8 == R * (2 * d + 4) - R * (d + 4)
    # and the down GEMM reads h's E4M3 codes, one row or two, and row scales
    d_fp8, _ = bench.stage_work(base, touched=4, splits=1)["down"]
    d_a8, _ = bench.stage_work(a8, touched=4, splits=1)["down"]
    f = 128
    assert d_fp8 - d_a8 == R * (2 * f + 4) - R * (f + 4)


def test_expected_touched_closed_form():
    shape = inputs.WORKLOADS["deepseek_v3"].with_T(1)
    assert bench.expected_touched(shape) == pytest.approx(8.0)          # k distinct experts
    shape = inputs.WORKLOADS["mixtral_8x7b"].with_T(64)
    assert bench.expected_touched(shape) == pytest.approx(8 * (1 - (6 / 8) ** 64))
    assert bench.expected_touched(shape.with_T(0)) == 0.0


def test_traffic_lookup_follows_the_kernel_source(tmp_path, monkeypatch):
    (tmp_path / "profiles").mkdir()
    src_dir = tmp_path / "routed_expert_ffn_gemm_gb300" / "csrc"
    src_dir.mkdir(parents=True)
    (src_dir / "grouped_tc.cu").write_bytes(b"kernel v1")
    sha = hashlib.sha256(b"kernel v1").hexdigest()[:16]
    (tmp_path / "profiles" / "dram_traffic.txt").write_text(
        "# comment line\nmixtral_8x7b 64 gate_up %s 1884260104\n" % sha)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    shape = inputs.WORKLOADS["mixtral_8x7b"].with_T(64)
    assert bench.measured_traffic(shape, "gate_up") == 1884260104.0
    assert bench.measured_traffic(shape, "down") is None
    assert bench.measured_traffic(shape.with_T(8), "gate_up") is None
    # the source changes: the old counters no longer describe the kernel
    (src_dir / "grouped_tc.cu").write_bytes(b"kernel v2")
    assert bench.measured_traffic(shape, "gate_up") is None


def test_committed_traffic_file_parses():
    path = os.path.join(bench.ROOT, "profiles", "dram_traffic.txt")
    rows = [ln.split() for ln in open(path) if ln.strip() and not ln.startswith("#")]
    assert rows and all(len(r) == 5 and len(r[3]) == 16 and float(r[4]) > 0 for r in rows)


def test_peaks_measured_else_the_recipe_fallback(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    # no measured file: the earlier GB300 measurement (6.8 TB/s, 1.9 / 1.7 PFLOP/s)
    assert bench.load_peaks() == (6800.0, 1900.0, 1700.0, "fallback")
    (tmp_path / "MEASURED_PEAKS.json").write_text(
        '{"hbm_gbs": 6691.5, "bf16_tflops": 1930.8, "bf16_tflops_sustained": 1723.5}')
    assert bench.load_peaks() == (6691.5, 1930.8, 1723.5, "measured")
    # a file without the figures is not a measurement
    (tmp_path / "MEASURED_PEAKS.json").write_text('{"hbm_gbs": 6691.5}')
    assert bench.load_peaks()[3] == "fallback"


def test_clock_summary_reads_nvidia_smi_lines():
    s = bench.ClockSampler(0)
    s.lines = [(0.0, ln) for ln in (
        "0, 2070, 2070, 900.1, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "0, 1995, 2070, 1390.0, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "0, 2070, 2070, 1200.0, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "garbage line",
        "0, [N/A], 2070, 1.0, 0x0, Not Active, Not Active, Not Active, Not Active",
    )]
    out = s.summary()
    assert out == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 3}
    s.lines = [(0.0, "0, 1500, 2070, 1.0, 0x8, Active, Not Active, Not Active, Not Active")]
    assert s.summary()["reasons"] == ["hw_slowdown"]
    s.lines = []
    assert s.summary()["samples"] == 0


def test_default_workload_is_the_largest_configuration():
    # no flags: the DeepSeek-V3-shaped layer (FP8 experts, bf16 activations,
    # shared expert) at its prefill batch of 4096 tokens
    import sys
    argv, sys.argv = sys.argv, ["bench.py"]
    try:
        args = bench.parse_args()
    finally:
        sys.argv = argv
    assert args.workload == "deepseek_v3" and args.T is None
    shape = inputs.WORKLOADS[args.workload].with_T(bench.DEFAULT_T[args.workload])
    assert (shape.T, shape.d, shape.ffn, shape.E, shape.k, shape.ffn_shared, shape.wfmt, shape.act) == \
        (4096, 7168, 2048, 256, 8, 2048, "fp8", "bf16")


def test_oracle_hook_decodes_each_expert_as_the_oracle_does_and_bounds_its_cache():
    import numpy as np
    import oracle
    shape = inputs.MoEShape("s", T=4, d=128, ffn=64, E=5, k=2, wfmt="fp8")
    case = inputs.make_case(shape, 3, "cpu")
    per = 3 * 64 * 128 * 8
    hook = bench._DecodedExperts(case, shape, cap_bytes=2 * per)
    ew = oracle.ExpertWeights("fp8", *(inputs.to_numpy_stored(case[n]) for n in
                                       ("w_gate", "w_up", "w_down", "s_gate", "s_up", "s_down")))
    for e in range(shape.E):
        for a, b in zip(hook(e), ew.get(e)):
            assert np.array_equal(a, b)
    # at most two decoded experts kept, the oldest dropped first
    assert sorted(hook.cache) == [3, 4]
    t = hook.decode_s
    hook(4)
    assert hook.decode_s == t          # a hit decodes nothing
    hook(0)
    assert hook.decode_s > t and sorted(hook.cache) == [0, 4]


def test_layer_roofline_names_the_binding_bound():
    # 10 GB and 1 TFLOP against 5 TB/s and 2 PFLOP/s: bytes take 2 ms, flops
    # 0.5 ms, so HBM binds; at 4 ms the layer reaches half of it
    r = bench.layer_roofline(10e9, 1e12, 4e-3, 5000.0, 2000.0, 8, 1.0)
    assert r["bound"] == "hbm"
    assert r["t_bytes_us"] == pytest.approx(2000.0) and r["t_flops_us"] == pytest.approx(500.0)
    assert r["frac_binding"] == pytest.approx(0.5)
    r = bench.layer_roofline(1e9, 4e12, 4e-3, 5000.0, 2000.0, 8, 1.0)
    assert r["bound"] == "tensor" and r["frac_binding"] == pytest.approx(0.5)


def test_tensor_peak_follows_the_length_of_the_timed_region():
    # burst figure for a short timed region, sustained for one of a second or more
    assert bench.tensor_peak_for(57.0, 1910.7, 1710.9) == (1910.7, "burst")
    assert bench.tensor_peak_for(999.9, 1910.7, 1710.9) == (1910.7, "burst")
    assert bench.tensor_peak_for(1000.0, 1910.7, 1710.9) == (1710.9, "sustained")
    assert bench.tensor_peak_for(3006.0, 1910.7, 1710.9) == (1710.9, "sustained")
