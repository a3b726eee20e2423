"""Pins of the CPU reference to facts outside itself: the page's worked
example, the storage-format definitions, closed forms, library routines,
brute force over tiny inputs, and the invariants the page states.

Run on CPU (no GPU marker).
"""

import math

import numpy as np
import pytest
import scipy.special
import torch
import torch.nn.functional as F

import oracle
from oracle import moe_oracle
from routed_expert_ffn_gemm_gb300 import inputs
from tests import helpers


# ---------------------------------------------------------------------------
# storage formats
# ---------------------------------------------------------------------------

def test_decode_bf16_fixed_values():
    cases = {0x3F80: 1.0, 0xBF80: -1.0, 0x4049: 3.140625, 0x0000: 0.0, 0x4000: 2.0,
             0x3F00: 0.5, 0x0080: 2.0 ** -126, 0x0001: 2.0 ** -133,
             0x7F7F: (2 - 2 ** -7) * 2.0 ** 127, 0x7F80: math.inf, 0xFF80: -math.inf}
    got = oracle.decode_bf16(np.array(list(cases), dtype=np.uint16))
    assert np.array_equal(got, np.array(list(cases.values())))
    assert np.isnan(oracle.decode_bf16(np.array([0x7FC0], np.uint16)))[0]
    assert np.signbit(oracle.decode_bf16(np.array([0x8000], np.uint16)))[0]


def test_decode_bf16_all_patterns_match_binary32_upper_half():
    # bf16 is the upper 16 bits of an IEEE binary32: reinterpret via numpy
    bits = np.arange(1 << 16, dtype=np.uint32)
    with np.errstate(invalid="ignore"):
        ref = (bits << 16).view(np.float32).astype(np.float64)
    got = oracle.decode_bf16(bits.astype(np.uint16))
    both_nan = np.isnan(ref) & np.isnan(got)
    assert np.all(both_nan | (ref == got))


def test_decode_e4m3_fixed_values():
    # OCP 8-bit floating point spec, E4M3: bias 7, max normal 448, min
    # subnormal 2^-9, S.1111.111 is NaN, no infinities
    cases = {0x00: 0.0, 0x38: 1.0, 0x40: 2.0, 0x7E: 448.0, 0xFE: -448.0, 0x01: 2.0 ** -9,
             0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x3C: 1.5, 0x77: 240.0, 0x78: 256.0}
    got = oracle.decode_e4m3(np.array(list(cases), dtype=np.uint8))
    assert np.array_equal(got, np.array(list(cases.values())))
    assert np.isnan(oracle.decode_e4m3(np.array([0x7F, 0xFF], np.uint8))).all()


def test_decode_e4m3_all_codes_match_torch():
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = oracle.decode_e4m3(codes.numpy())
    both_nan = np.isnan(ref) & np.isnan(got)
    assert np.all(both_nan | (ref == got))


# ---------------------------------------------------------------------------
# the worked example (page section 二)
# ---------------------------------------------------------------------------

def test_worked_example_groups_and_rows():
    g, idx, w, groups = helpers.worked_example()
    counts, offsets, perm_token, inv_row = oracle.permutation_maps(idx, g["E"])
    assert counts.tolist() == g["rows_per_expert"] == [3, 2, 2, 1]
    assert int(counts.sum()) == g["assignments"] == 8
    assert offsets.tolist() == [0, 3, 5, 7, 8]
    for e in range(g["E"]):
        assert perm_token[offsets[e]:offsets[e + 1]].tolist() == groups[e]
    # the inverse map sends each assignment to a row of its own token and expert
    for t in range(g["T"]):
        for j in range(g["k"]):
            r = inv_row[t, j]
            assert perm_token[r] == t
            assert offsets[idx[t, j]] <= r < offsets[idx[t, j] + 1]
    assert perm_token.tolist() == [0, 1, 2, 2, 3, 0, 1, 3]
    assert inv_row.tolist() == [[0, 5], [6, 1], [2, 3], [4, 7]]


def test_worked_example_router_reproduces_weights():
    g, idx, w, _ = helpers.worked_example()
    logits = helpers.worked_example_logits(idx, w, g["E"])
    got_idx, got_w = oracle.topk_renorm(logits, g["k"])
    assert got_idx.tolist() == idx.tolist()
    np.testing.assert_allclose(got_w, w, rtol=0, atol=1e-12)
    for t in range(g["T"]):
        printed = {int(e[1:]) - 1: v for e, v in g["routing"][f"T{t + 1}"].items()}
        assert {int(e): float(v) for e, v in zip(got_idx[t], got_w[t])} == pytest.approx(printed, abs=1e-12)


def _library_ffn(x, wg, wu, wd):
    x, wg, wu, wd = (torch.from_numpy(np.asarray(a, np.float64)) for a in (x, wg, wu, wd))
    return F.linear(F.silu(F.linear(x, wg)) * F.linear(x, wu), wd).numpy()


def test_worked_example_combine_of_T1():
    # the page: T1's output is 0.7 * E1(T1) + 0.3 * E3(T1)
    g, idx, w, _ = helpers.worked_example()
    rng = np.random.default_rng(7)
    d, f, E = 6, 10, g["E"]
    Wg, Wu, Wd = rng.normal(size=(E, f, d)), rng.normal(size=(E, f, d)), rng.normal(size=(E, d, f))
    x = rng.normal(size=(g["T"], d))
    ew = oracle.ExpertWeights("f64", Wg, Wu, Wd)
    wr = np.zeros((E, d))
    out_i, _, _ = oracle.moe_forward_per_token(x, wr, ew, g["k"], routing=(idx, w))
    out_ii, _, _ = oracle.moe_forward_grouped(x, wr, ew, g["k"], routing=(idx, w))
    c = g["combine"]["T1"]
    t1 = c["E1"] * _library_ffn(x[:1], Wg[0], Wu[0], Wd[0]) + c["E3"] * _library_ffn(x[:1], Wg[2], Wu[2], Wd[2])
    np.testing.assert_allclose(out_i[0], t1[0], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(out_ii[0], t1[0], rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------------------
# router: library matmul, brute force, closed form
# ---------------------------------------------------------------------------

def test_router_logits_match_library_linear():
    rng = np.random.default_rng(1)
    x, w, b = rng.normal(size=(9, 13)), rng.normal(size=(5, 13)), rng.normal(size=5)
    ref = F.linear(torch.from_numpy(x), torch.from_numpy(w), torch.from_numpy(b)).numpy()
    np.testing.assert_allclose(oracle.router_logits(x, w, b), ref, rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("E,k", [(4, 1), (5, 2), (6, 3), (6, 6), (3, 2)])
def test_topk_brute_force_over_subsets(E, k):
    rng = np.random.default_rng(E * 10 + k)
    logits = rng.normal(size=(40, E)) * 2
    idx, w = oracle.topk_renorm(logits, k)
    best = moe_oracle.brute_force_topk_sets(logits, k)
    for t in range(logits.shape[0]):
        assert set(idx[t].tolist()) == best[t]
        # closed form: renormalised weights = softmax over the chosen logits only
        sub = scipy.special.softmax(logits[t, idx[t]])
        np.testing.assert_allclose(w[t], sub, rtol=1e-13, atol=1e-15)
        # slots in descending weight
        assert np.all(np.diff(w[t]) <= 0)


def test_topk_weights_ignore_unchosen_logits():
    rng = np.random.default_rng(3)
    logits = rng.normal(size=(20, 8))
    idx, w = oracle.topk_renorm(logits, 2)
    moved = logits.copy()
    for t in range(20):
        rest = [e for e in range(8) if e not in idx[t]]
        moved[t, rest] -= rng.uniform(0, 5, size=len(rest))  # stay below the k-th
    idx2, w2 = oracle.topk_renorm(moved, 2)
    assert np.array_equal(idx, idx2)
    np.testing.assert_allclose(w, w2, rtol=1e-13)


def test_topk_ties_go_to_lower_index():
    logits = np.array([[1.0, 3.0, 3.0, 0.0, 3.0]])
    idx, w = oracle.topk_renorm(logits, 2)
    assert idx.tolist() == [[1, 2]]
    np.testing.assert_allclose(w, [[0.5, 0.5]])


def test_topk_gap():
    logits = np.array([[0.0, 5.0, 4.0, 1.0]])
    assert oracle.topk_gap(logits, 2)[0] == pytest.approx(3.0)
    assert np.isinf(oracle.topk_gap(logits, 4)[0])


# ---------------------------------------------------------------------------
# expert FFN: closed-form SiLU values and the library FFN
# ---------------------------------------------------------------------------

def test_silu_closed_form_values():
    z = np.array([0.0, 1.0, -1.0, 2.0, -40.0, 40.0, -800.0])
    want = np.array([0.0, 1 / (1 + math.exp(-1)), -1 / (1 + math.e), 2 / (1 + math.exp(-2)),
                     -40 * math.exp(-40) / (1 + math.exp(-40)), 40 / (1 + math.exp(-40)), 0.0])
    np.testing.assert_allclose(oracle.silu(z), want, rtol=1e-15, atol=1e-300)
    np.testing.assert_allclose(oracle.silu(1.0 * np.array([1.0]))[0], 0.7310585786300049, rtol=1e-15)


def test_silu_matches_library():
    z = np.random.default_rng(0).normal(size=1000) * 10
    np.testing.assert_allclose(oracle.silu(z), F.silu(torch.from_numpy(z)).numpy(), rtol=1e-14, atol=1e-300)


def test_swiglu_expert_matches_library_ffn():
    rng = np.random.default_rng(2)
    x, wg, wu, wd = rng.normal(size=(7, 12)), rng.normal(size=(20, 12)), rng.normal(size=(20, 12)), rng.normal(size=(12, 20))
    np.testing.assert_allclose(oracle.swiglu_expert(x, wg, wu, wd), _library_ffn(x, wg, wu, wd), rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------------------
# special cases of the layer
# ---------------------------------------------------------------------------

def _rand_layer(rng, T=12, d=8, f=16, E=5):
    x = rng.normal(size=(T, d))
    wr = rng.normal(size=(E, d)) / np.sqrt(d)
    Wg, Wu = rng.normal(size=(E, f, d)) / np.sqrt(d), rng.normal(size=(E, f, d)) / np.sqrt(d)
    Wd = rng.normal(size=(E, d, f)) / np.sqrt(d)
    return x, wr, Wg, Wu, Wd


def test_single_expert_is_dense_swiglu():
    rng = np.random.default_rng(11)
    x, wr, Wg, Wu, Wd = _rand_layer(rng, E=1)
    ew = oracle.ExpertWeights("f64", Wg, Wu, Wd)
    for fn in (oracle.moe_forward_per_token, oracle.moe_forward_grouped):
        out, idx, w = fn(x, wr, ew, 1)
        np.testing.assert_allclose(out, _library_ffn(x, Wg[0], Wu[0], Wd[0]), rtol=1e-12, atol=1e-12)
        assert np.all(idx == 0) and np.allclose(w, 1.0)


def test_k_equal_E_is_full_softmax_mixture():
    rng = np.random.default_rng(12)
    x, wr, Wg, Wu, Wd = _rand_layer(rng, E=4)
    ew = oracle.ExpertWeights("f64", Wg, Wu, Wd)
    p = scipy.special.softmax(x @ wr.T, axis=1)
    want = sum(p[:, e:e + 1] * _library_ffn(x, Wg[e], Wu[e], Wd[e]) for e in range(4))
    for fn in (oracle.moe_forward_per_token, oracle.moe_forward_grouped):
        out, _, _ = fn(x, wr, ew, 4)
        np.testing.assert_allclose(out, want, rtol=1e-12, atol=1e-12)


def test_identical_experts_give_the_dense_ffn():
    rng = np.random.default_rng(13)
    x, wr, Wg, Wu, Wd = _rand_layer(rng, E=6)
    Wg[:], Wu[:], Wd[:] = Wg[0], Wu[0], Wd[0]
    ew = oracle.ExpertWeights("f64", Wg, Wu, Wd)
    out, _, _ = oracle.moe_forward_grouped(x, wr, ew, 3)
    np.testing.assert_allclose(out, _library_ffn(x, Wg[0], Wu[0], Wd[0]), rtol=1e-12, atol=1e-12)


def test_zero_tokens_give_zero_output():
    rng = np.random.default_rng(14)
    x, wr, Wg, Wu, Wd = _rand_layer(rng)
    ew = oracle.ExpertWeights("f64", Wg, Wu, Wd)
    out, _, _ = oracle.moe_forward_per_token(np.zeros_like(x), wr, ew, 2)
    assert np.all(out == 0)


def test_shared_expert_is_added_with_weight_one():
    rng = np.random.default_rng(15)
    x, wr, Wg, Wu, Wd = _rand_layer(rng)
    sh = (rng.normal(size=(9, 8)), rng.normal(size=(9, 8)), rng.normal(size=(8, 9)))
    ew = oracle.ExpertWeights("f64", Wg, Wu, Wd)
    base, _, _ = oracle.moe_forward_grouped(x, wr, ew, 2)
    withs, _, _ = oracle.moe_forward_grouped(x, wr, ew, 2, shared=sh)
    np.testing.assert_allclose(withs - base, _library_ffn(x, *sh), rtol=1e-11, atol=1e-11)


# ---------------------------------------------------------------------------
# invariants the page states, and the two formulations
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("T,E,k", [(1, 8, 2), (37, 8, 2), (64, 16, 4), (200, 32, 8), (5, 3, 3)])
def test_permutation_invariants(T, E, k):
    rng = np.random.default_rng(T + E + k)
    idx, w = oracle.topk_renorm(rng.normal(size=(T, E)), k)
    counts, offsets, perm_token, inv_row = oracle.permutation_maps(idx, E)
    assert counts.sum() == T * k and offsets[-1] == T * k
    assert np.array_equal(np.bincount(perm_token, minlength=T), np.full(T, k))  # k rows per token
    for t in range(T):
        assert len(set(idx[t].tolist())) == k  # distinct experts per token
    np.testing.assert_allclose(w.sum(axis=1), 1.0, rtol=1e-14)
    assert np.array_equal(perm_token[inv_row], np.repeat(np.arange(T), k).reshape(T, k))
    assert sorted(inv_row.ravel().tolist()) == list(range(T * k))
    for e in range(E):
        rows = perm_token[offsets[e]:offsets[e + 1]]
        assert np.all(np.diff(rows) > 0)  # ascending token order inside an expert
    # permute then unpermute with weights summing to 1 is the identity
    x = rng.normal(size=(T, 3))
    x_perm = x[perm_token]
    back = (w[:, :, None] * x_perm[inv_row]).sum(axis=1)
    np.testing.assert_allclose(back, x, rtol=1e-13, atol=1e-13)


def test_two_formulations_agree_random_layers():
    rng = np.random.default_rng(21)
    for (T, d, f, E, k) in [(30, 8, 16, 6, 2), (17, 16, 8, 9, 4), (3, 4, 4, 3, 3)]:
        x, wr, Wg, Wu, Wd = _rand_layer(rng, T, d, f, E)
        b = rng.normal(size=E)
        sh = (rng.normal(size=(5, d)), rng.normal(size=(5, d)), rng.normal(size=(d, 5)))
        ew = oracle.ExpertWeights("f64", Wg, Wu, Wd)
        a, ia, wa = oracle.moe_forward_per_token(x, wr, ew, k, bias=b, shared=sh)
        c, ic, wc = oracle.moe_forward_grouped(x, wr, ew, k, bias=b, shared=sh)
        assert np.array_equal(ia, ic)
        np.testing.assert_allclose(a, c, rtol=0, atol=1e-12 * np.abs(a).max())


def test_two_formulations_agree_on_generated_fp8_and_bf16_cases():
    for name, T in [("toy_f32", 64)]:
        shape = inputs.WORKLOADS[name].with_T(T)
        case = inputs.make_case(shape, 0)
        x, wr, b, ew, sh = helpers.oracle_inputs(case, shape)
        a, _, _ = oracle.moe_forward_per_token(x, wr, ew, shape.k, bias=b, shared=sh)
        c, _, _ = oracle.moe_forward_grouped(x, wr, ew, shape.k, bias=b, shared=sh)
        np.testing.assert_allclose(a, c, rtol=0, atol=1e-12 * np.abs(a).max())
    # a small fp8 + shared layer built with the same generator
    small = inputs.MoEShape("small_fp8", T=9, d=32, ffn=16, E=6, k=3, ffn_shared=16, wfmt="fp8")
    case = inputs.make_case(small, 3)
    x, wr, b, ew, sh = helpers.oracle_inputs(case, small)
    a, _, _ = oracle.moe_forward_per_token(x, wr, ew, small.k, shared=sh)
    c, _, _ = oracle.moe_forward_grouped(x, wr, ew, small.k, shared=sh)
    np.testing.assert_allclose(a, c, rtol=0, atol=1e-12 * np.abs(a).max())


@pytest.mark.parametrize("wfmt", ["fp8a8", "mxfp4"])
def test_two_formulations_agree_on_quantised_modes(wfmt):
    # per token over its chosen set, and grouped per expert: the same layer
    # with FP8 activations (x and h rows quantised per row) or MXFP4 weights
    small = inputs.MoEShape("small_q", T=11, d=64, ffn=32, E=6, k=3, ffn_shared=32, wfmt=wfmt)
    case = inputs.make_case(small, 5)
    x, wr, b, ew, sh = helpers.oracle_inputs(case, small)
    act8 = wfmt == "fp8a8"
    a, ia, _ = oracle.moe_forward_per_token(x, wr, ew, small.k, shared=sh, act8=act8)
    c, ic, _ = oracle.moe_forward_grouped(x, wr, ew, small.k, shared=sh, act8=act8)
    assert np.array_equal(ia, ic)
    np.testing.assert_allclose(a, c, rtol=0, atol=1e-12 * np.abs(a).max())
    if act8:  # and the quantisation is really applied: unquantised rows give another answer
        u, _, _ = oracle.moe_forward_grouped(x, wr, ew, small.k, shared=sh)
        assert np.abs(u - a).max() > 1e-6 * np.abs(a).max()


def test_fp8_weights_are_code_times_per_channel_scale():
    small = inputs.MoEShape("small_fp8", T=2, d=16, ffn=8, E=2, k=1, wfmt="fp8")
    case = inputs.make_case(small, 5)
    x, wr, b, ew, sh = helpers.oracle_inputs(case, small)
    wg, wu, wd = ew.get(1)
    codes = case["w_gate"][1].view(torch.float8_e4m3fn).to(torch.float64)
    ref = codes * case["s_gate"][1].to(torch.float64)[:, None]
    np.testing.assert_allclose(wg, ref.numpy(), rtol=0, atol=0)
    # per-channel amax of the decoded codes is 448 (scale = amax / 448)
    assert np.allclose(np.abs(codes.numpy()).max(axis=1), 448.0)


# ---------------------------------------------------------------------------
# the skewed prefill recipe
# ---------------------------------------------------------------------------

def test_zipf_bias_scale_matches_calibration():
    cal = helpers.load_golden("zipf_bias_alpha.json")["qwen3_30b_a3b_prefill"]
    assert inputs.ZIPF_ALPHA["qwen3_30b_a3b_prefill"] == cal["alpha"]
    shape = inputs.WORKLOADS["qwen3_30b_a3b_prefill"]
    wr = inputs._normal((shape.E, shape.d), 1.0 / np.sqrt(shape.d), 0, "w_router", "cpu", torch.bfloat16)
    x = inputs.make_tokens(shape, 0)
    lg = oracle.router_logits(helpers.decode_act(x, "bf16"), helpers.decode_act(wr, "bf16"),
                              inputs.zipf_bias(shape, 0).double().numpy())
    idx, _ = oracle.topk_renorm(lg, shape.k)
    counts, _, _, _ = oracle.permutation_maps(idx, shape.E)
    r = counts.max() / counts.mean()
    assert 7.5 <= r <= 8.5


# ---------------------------------------------------------------------------
# FP8 activations (per-row E4M3 quantisation of the gate/up input)
# ---------------------------------------------------------------------------

def _torch_e4m3_codes(v):
    import torch
    return torch.tensor(np.asarray(v, np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_round_to_e4m3_matches_library_cast_in_range():
    # every midpoint between adjacent finite E4M3 magnitudes (the ties), the
    # values just beside them, and a dense sweep, both signs: the library's
    # float8 cast rounds to nearest, ties to even
    mags = oracle.decode_e4m3(np.arange(0x7F))
    mids = (mags[:-1] + mags[1:]) / 2
    v = np.concatenate([mids, np.nextafter(mids.astype(np.float32), np.float32(0)),
                        np.nextafter(mids.astype(np.float32), np.float32(1e9)),
                        np.linspace(0, 448, 20001)]).astype(np.float32)
    v = np.concatenate([v, -v])
    assert np.array_equal(oracle.round_to_e4m3(v), _torch_e4m3_codes(v))


def test_round_to_e4m3_ties_go_to_even_and_saturates():
    assert oracle.round_to_e4m3(np.float32(1.0625)) == 0x38       # between 1 (0x38) and 1.125 (0x39)
    assert oracle.round_to_e4m3(np.float32(1.1875)) == 0x3A       # between 1.125 (0x39) and 1.25 (0x3A)
    assert oracle.round_to_e4m3(np.float32(3 * 2.0 ** -10)) == 0x02  # between subnormals 1 and 2
    assert oracle.round_to_e4m3(np.float32(2.0 ** -10)) == 0x00   # half the smallest subnormal
    for big in (449.0, 464.0, 1000.0, 3.0e38):
        assert oracle.round_to_e4m3(np.float32(big)) == 0x7E      # 448, never NaN
        assert oracle.round_to_e4m3(np.float32(-big)) == 0xFE


def test_quantize_rows_scale_and_extremes():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((6, 300)).astype(np.float32)
    x[3] = 0.0
    codes, s = oracle.quantize_rows_e4m3(x)
    amax = np.abs(x).max(axis=1)
    nz = amax > 0
    assert np.array_equal(s[nz], (amax[nz] / np.float32(448)).astype(np.float32))
    assert s[3] == 1.0 and not codes[3].any()
    # each nonzero row's largest magnitude lands on the largest code
    for t in np.flatnonzero(nz):
        assert (codes[t] & 0x7F).max() == 0x7E
    # the round trip stays within half an E4M3 step (relative 2^-4) of x
    back = oracle.dequantize_rows_e4m3(codes, s)
    tol = np.maximum(np.abs(x) * 2.0 ** -4, s[:, None] * 2.0 ** -10)
    assert np.all(np.abs(back - x) <= tol + 1e-30)


def test_quantize_rows_lossless_on_representable_rows():
    # rows that are E4M3 values times a power-of-two scale, with one element
    # at 448 * scale, come back exactly
    rng = np.random.default_rng(6)
    codes = rng.integers(0, 0x7E, size=(4, 64)).astype(np.uint8) | (rng.integers(0, 2, size=(4, 64)) * 0x80).astype(np.uint8)
    codes[:, 0] = 0x7E
    scale = np.float32(2.0 ** -9)
    x = (oracle.decode_e4m3(codes) * scale).astype(np.float32)
    c2, s2 = oracle.quantize_rows_e4m3(x)
    assert np.all(s2 == scale) and np.array_equal(oracle.decode_e4m3(c2), oracle.decode_e4m3(codes))


def test_act8_expert_quantises_both_activations():
    # On E4M3-representable rows the input quantisation is lossless, so with
    # an identity down projection the FP8-activation expert returns the rows
    # of h as quantised per row: each row divided by (its max / 448) lies on
    # the E4M3 grid, within half a grid step of the plain h, its maximum kept
    rng = np.random.default_rng(6)
    codes = rng.integers(0, 0x7E, size=(5, 64)).astype(np.uint8)
    codes[:, 0] = 0x7E
    x = (oracle.decode_e4m3(codes) * 2.0 ** -9).astype(np.float32)
    wg, wu = rng.standard_normal((2, 48, 64)) / 8.0
    eye = np.eye(48)
    h8 = oracle.swiglu_expert(x, wg, wu, eye, act8=True)
    h = oracle.swiglu_expert(x, wg, wu, eye)
    grid = np.abs(oracle.decode_e4m3(np.arange(0x7F)))
    for t in range(5):
        s = np.abs(h8[t]).max() / 448.0
        assert np.isin(np.abs(h8[t] / s), grid).all()
        assert np.abs(h8[t] - h[t]).max() <= np.abs(h[t]).max() * 2.0 ** -4
        np.testing.assert_allclose(np.abs(h8[t]).max(), np.abs(h[t]).max(), rtol=1e-6)
    # and with a general down projection: the product of those rows
    wd = rng.standard_normal((64, 48)) / 8.0
    np.testing.assert_allclose(oracle.swiglu_expert(x, wg, wu, wd, act8=True), h8 @ wd.T, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------------------
# MXFP4 expert weights (OCP Microscaling: E2M1 elements, UE8M0 block scales)
# ---------------------------------------------------------------------------

def test_decode_e2m1_fixed_values():
    # the OCP MX element format FP4 E2M1: magnitudes 0, 0.5 (the one
    # subnormal), 1, 1.5, 2, 3, 4, 6; the high bit is the sign
    v = oracle.decode_e2m1(np.arange(16))
    assert v[:8].tolist() == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    assert v[8:].tolist() == [-0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0]
    assert np.signbit(v[8]) and not np.signbit(v[0])


def test_decode_e2m1_agrees_with_e4m3_at_the_same_value():
    # every E2M1 value is an E4M3 value: map the fields (exponent e, bias 1
    # -> bias 7; the fraction bit becomes the top of three) and decode with
    # the (separately pinned) E4M3 decoder
    for c in range(16):
        s, e, m = c >> 3, (c >> 1) & 3, c & 1
        if e == 0:
            f8 = 0 if m == 0 else (6 << 3)          # 0.5 = 2^-1
        else:
            f8 = ((e - 1 + 7) << 3) | (m << 2)
        assert oracle.decode_e2m1(c) == oracle.decode_e4m3((s << 7) | f8)


def test_decode_ue8m0_fixed_values():
    v = oracle.decode_ue8m0(np.array([0, 1, 126, 127, 128, 134, 254, 255]))
    assert v[1:7].tolist() == [2.0 ** -126, 0.5, 1.0, 2.0, 128.0, 2.0 ** 127]
    assert v[0] == 2.0 ** -127 and np.isnan(v[7])


def test_unpack_fp4_nibble_order():
    codes = oracle.unpack_fp4(np.array([[0x21, 0xF0, 0x7A]], np.uint8))
    assert codes.tolist() == [[1, 2, 0, 15, 10, 7]]


def test_decode_mxfp4_hand_block():
    # two rows of 64 weights (two 32-element blocks each); scales [K/32, rows]
    codes = np.zeros((2, 64), np.uint8)
    codes[0, 0], codes[0, 1], codes[0, 33] = 0x7, 0x9, 0x3      # 6, -0.5 | 1.5
    codes[1, 2], codes[1, 40], codes[1, 63] = 0x5, 0xC, 0x1     # 3 | -2, 0.5
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    scales = np.array([[127, 126],      # block 0: row 0 x 1, row 1 x 0.5
                       [128, 130]],     # block 1: row 0 x 2, row 1 x 8
                      np.uint8)
    w = oracle.decode_mxfp4(packed, scales)
    expect = np.zeros((2, 64))
    expect[0, 0], expect[0, 1], expect[0, 33] = 6.0, -0.5, 3.0
    expect[1, 2], expect[1, 40], expect[1, 63] = 1.5, -16.0, 4.0
    assert w.shape == (2, 64) and np.array_equal(w, expect)


def test_mxfp4_storage_matches_the_page():
    # "MoE 推理部署", section 专家量化: the OCP MX 4-bit block format puts a
    # 117B-parameter model in about 60 GB, inside one 80 GB GPU.  The format
    # the oracle decodes spends K/2 code bytes and K/32 scale bytes per row of
    # K weights: 4.25 bits per weight.
    K, rows = 4096, 3
    packed = np.zeros((rows, K // 2), np.uint8)
    scales = np.full((K // 32, rows), 127, np.uint8)
    assert oracle.decode_mxfp4(packed, scales).shape == (rows, K)
    bits_per_weight = 8.0 * (packed.size + scales.size) / (rows * K)
    assert bits_per_weight == 4.25
    gb = 117e9 * bits_per_weight / 8 / 1e9
    assert 55.0 <= gb <= 65.0 and gb < 80.0


def test_mxfp4_expert_weights_decode_per_matrix():
    # ExpertWeights("mxfp4") hands each expert's three matrices through
    # decode_mxfp4 with their own scales; the FFN then sees plain values
    rng = np.random.default_rng(8)
    E, d, f = 2, 64, 32
    wg = rng.integers(0, 256, (E, f, d // 2)).astype(np.uint8)
    wu = rng.integers(0, 256, (E, f, d // 2)).astype(np.uint8)
    wd = rng.integers(0, 256, (E, d, f // 2)).astype(np.uint8)
    sg = rng.integers(120, 130, (E, d // 32, f)).astype(np.uint8)
    su = rng.integers(120, 130, (E, d // 32, f)).astype(np.uint8)
    sd = rng.integers(120, 130, (E, f // 32, d)).astype(np.uint8)
    ew = oracle.ExpertWeights("mxfp4", wg, wu, wd, sg, su, sd)
    g1, u1, d1 = ew.get(1)
    assert np.array_equal(g1, oracle.decode_mxfp4(wg[1], sg[1]))
    assert np.array_equal(u1, oracle.decode_mxfp4(wu[1], su[1]))
    assert np.array_equal(d1, oracle.decode_mxfp4(wd[1], sd[1]))
    assert g1.shape == (f, d) and d1.shape == (d, f)
    # each weight divided by its block's scale is an E2M1 value
    blk = np.repeat(oracle.decode_ue8m0(sg[1]), 32, axis=0).T
    assert np.isin(np.abs(g1 / blk), oracle.decode_e2m1(np.arange(8))).all()
