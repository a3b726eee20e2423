"""The library's tiling, launch-count and workspace rules, asked through the
device-free planning entry points (no GPU): the rows per tile, K splits and
CTA pairs the grouped GEMMs take for the layer's workloads, the rules that
bound them, the number of kernels one layer call launches per weight mode,
and the workspace each needs.  The device entry points are the same
functions at the device's SM count (a GPU test checks that)."""

import dataclasses

import pytest

from routed_expert_ffn_gemm_gb300 import api, build, inputs

SMS = 152  # the GB300's multiprocessors
FORMATS = ("bf16", "fp8", "fp8a8", "mxfp4")


@pytest.fixture(scope="module", autouse=True)
def _library():
    build.build()
    api._lib()


def _shape(name, T=None, wfmt=None, ffn_shared=None):
    s = inputs.WORKLOADS[name]
    return dataclasses.replace(s, T=s.T if T is None else T, wfmt=wfmt or s.wfmt,
                               ffn_shared=s.ffn_shared if ffn_shared is None else ffn_shared)


def _plan(shape, sms=SMS):
    return api.moe_plan_info_for(api.problem_of(shape), sms)


CASES = [("mixtral_8x7b", T, "bf16") for T in (1, 8, 32, 64)] + \
        [("qwen3_30b_a3b", T, "bf16") for T in (1, 16, 128)] + \
        [("qwen3_30b_a3b_prefill", None, "bf16")] + \
        [("deepseek_v3", T, w) for T in (1, 64, 4096) for w in FORMATS]


def test_the_headline_layer_runs_the_measured_plan():
    # the Mixtral-shaped T=64 layer whose bench numbers are recorded ran on
    # 32-row tiles, down GEMM on CTA pairs with 7 K splits, gate/up unsplit
    assert _plan(_shape("mixtral_8x7b", 64)) == {
        "bn_gateup": 32, "bn_down": 32, "splits_down": 7, "grid": SMS, "splits_gateup": 1,
        "pair_gateup": 0, "pair_down": 1}


@pytest.mark.parametrize("name,T,wfmt", CASES)
@pytest.mark.parametrize("sms", [SMS, 148, 132, 2, 1])
def test_plan_bounds(name, T, wfmt, sms):
    s = _shape(name, T, wfmt)
    pl = _plan(s, sms)
    assert pl["grid"] == sms
    assert pl["bn_gateup"] in (32, 128, 160, 256) and pl["bn_down"] in (32, 128, 160, 256)
    if wfmt != "fp8":
        assert 160 not in (pl["bn_gateup"], pl["bn_down"])
    assert 1 <= pl["splits_gateup"] <= 8 and 1 <= pl["splits_down"] <= 8
    # each K split keeps at least 4 stages of at most 128 elements
    for K, S in ((s.d, pl["splits_gateup"]), (s.ffn, pl["splits_down"])):
        if S > 1:
            assert K > (4 * S - 1) * 64, (K, S)
    # a pair tile is 256 output channels: ffn for gate/up, d for down
    if pl["pair_gateup"]:
        assert s.ffn % 256 == 0 and sms >= 2
    if pl["pair_down"]:
        assert s.d % 256 == 0 and sms >= 2


@pytest.mark.parametrize("name,T,wfmt", CASES)
def test_tile_rows_follow_the_rows_per_expert(name, T, wfmt):
    s = _shape(name, T, wfmt)
    pl = _plan(s)
    mean = s.T * s.k / s.E
    if mean <= 4:  # decode: a few rows per expert
        assert (pl["bn_gateup"], pl["bn_down"]) == (32, 32)
        # the gate/up decode tiles stay on single CTAs, except two-term
        # rows (FP8 weights, bf16 activations) whose pair units need no K split
        assert pl["pair_gateup"] == (1 if wfmt == "fp8" and pl["splits_gateup"] == 1 and s.ffn % 256 == 0 else 0)
        assert pl["pair_down"] == (1 if wfmt == "bf16" and s.d % 256 == 0 else 0)
    if mean >= 128:  # prefill: whole 256-row tiles, K unsplit, CTA pairs
        # FP8 weights on two-term rows with about 128 rows per group take
        # 160-row tiles (80 rows per CTA of a pair)
        two_term_160 = wfmt == "fp8" and mean + 3 * mean ** 0.5 + 1 <= 192
        assert pl["bn_down"] == (160 if two_term_160 else 256)
        # weights converted to f16 in tensor memory (MXFP4) keep 128-row
        # gate/up tiles
        assert pl["bn_gateup"] == (128 if wfmt == "mxfp4" else 160 if two_term_160 else 256)
        assert pl["splits_gateup"] == pl["splits_down"] == 1
        assert pl["pair_gateup"] == pl["pair_down"] == 1


@pytest.mark.parametrize("name,T,wfmt", CASES)
def test_pair_switch(name, T, wfmt, monkeypatch):
    s = _shape(name, T, wfmt)
    monkeypatch.setenv("MOE_PAIR", "0")
    pl = _plan(s)
    assert pl["pair_gateup"] == pl["pair_down"] == 0
    monkeypatch.setenv("MOE_PAIR", "2")
    pl = _plan(s)
    if pl["bn_down"] == 32:  # every decode tile that splits into pair tiles runs on pairs
        assert pl["pair_down"] == (1 if s.d % 256 == 0 else 0)
    if pl["bn_gateup"] == 32:
        assert pl["pair_gateup"] == (1 if s.ffn % 256 == 0 else 0)


def test_splits_only_when_the_units_leave_the_sms_idle():
    # prefill: hundreds of tiles per GEMM, no K split; one token: a handful
    # of units, split along K
    assert _plan(_shape("qwen3_30b_a3b_prefill"))["splits_down"] == 1
    one = _plan(_shape("deepseek_v3", 1))
    assert one["splits_gateup"] > 1


@pytest.mark.parametrize("T", [1, 64, 4096])
def test_launch_count_per_weight_mode(T):
    n = {w: api.moe_layer_launch_count_for(api.problem_of(_shape("deepseek_v3", T, w)), SMS) for w in FORMATS}
    # MXFP4 weights: one more pass (x to f16 for the converted operands);
    # FP8 weights: two (x's and h's two-term E4M3 rows); FP8 activations:
    # two (x's and h's per-row E4M3 codes)
    assert n["fp8"] == n["bf16"] + 2
    assert n["mxfp4"] == n["bf16"] + 1
    assert n["fp8a8"] == n["bf16"] + 2


@pytest.mark.parametrize("name,T,wfmt", CASES)
def test_launch_count_bounds(name, T, wfmt):
    s = _shape(name, T, wfmt)
    n = api.moe_layer_launch_count_for(api.problem_of(s), SMS)
    # router (+ top-k), permutation, gate/up, down, combine at the least
    assert 5 <= n <= 16
    if s.ffn_shared:
        n0 = api.moe_layer_launch_count_for(api.problem_of(_shape(name, T, wfmt, ffn_shared=0)), SMS)
        assert n >= n0 + 2  # the shared expert's gate/up and down
    assert api.moe_layer_launch_count_for(api.problem_of(s.with_T(0)), SMS) == 0


@pytest.mark.parametrize("name,T,wfmt", CASES)
def test_workspace_holds_the_intermediates(name, T, wfmt):
    s = _shape(name, T, wfmt)
    p = api.problem_of(s)
    ws = api.moe_workspace_size_for(p, SMS)
    pl = _plan(s)
    R = s.T * s.k
    need = R * 4 * 4            # top-k ids and weights, row maps
    need += R * s.ffn * 2       # h (bf16 or f16)
    need += pl["splits_down"] * R * s.d * 4 if pl["splits_down"] > 1 else R * s.d * 2  # y
    if wfmt == "fp8a8":
        need += R * s.ffn + R * 4  # h's E4M3 codes and row scales
    if s.ffn_shared:
        need += s.T * s.ffn_shared * 2 + s.T * s.d * 2
    assert ws >= need


def test_sm_count_is_validated():
    p = api.problem_of(_shape("mixtral_8x7b", 64))
    for bad in (0, -1, 4097):
        with pytest.raises(api.MoEError):
            api.moe_plan_info_for(p, bad)
        with pytest.raises(api.MoEError):
            api.moe_layer_launch_count_for(p, bad)
        with pytest.raises(api.MoEError):
            api.moe_workspace_size_for(p, bad)
    # and rejected problems are rejected here too
    with pytest.raises(api.MoEError):
        api.moe_plan_info_for(api.problem(4, 100, 128, 8, 2), SMS)  # d not a multiple of 8


def test_the_fp32_path_has_no_tiling():
    p = api.problem(64, 128, 256, 8, 2, act="f32", wfmt="f32")
    assert set(api.moe_plan_info_for(p, SMS).values()) == {0}
    assert api.moe_layer_launch_count_for(p, SMS) > 0


def test_two_term_token_rows_are_gathered_per_token_at_prefill(monkeypatch):
    # FP8 weights on bf16 rows at prefill tiles: the token rows are split
    # once per token (two planes of T rows) and gathered by the gate/up
    # GEMM; MOE_X2_SCATTER=1 writes them to their T*k permuted rows instead,
    # which the workspace shows exactly (two planes of codes and one fp32
    # scale per row)
    s = _shape("deepseek_v3", 4096, "fp8")
    p = api.problem_of(s)
    gathered = api.moe_workspace_size_for(p, SMS)
    monkeypatch.setenv("MOE_X2_SCATTER", "1")
    scattered = api.moe_workspace_size_for(p, SMS)
    R, T = s.T * s.k, s.T
    assert scattered - gathered == 2 * (R - T) * s.d + 4 * (R - T)
