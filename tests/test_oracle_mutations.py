"""Plant plausible mistakes in the CPU reference (on the CPU, one at a time)
and check that at least one pin catches each: the pins must be sharp enough
that a dropped term, a wrong sign or index, or a swapped operand fails."""

import numpy as np
import pytest

import oracle
from oracle import moe_oracle as M
from tests import test_oracle_pins as pins

_orig = {n: getattr(M, n) for n in ("topk_renorm", "permutation_maps", "silu", "swiglu_expert",
                                      "decode_e4m3", "decode_bf16", "moe_forward_grouped",
                                      "moe_forward_per_token", "shared_expert", "router_logits",
                                      "round_to_e4m3", "quantize_rows_e4m3", "decode_e2m1",
                                      "decode_ue8m0", "unpack_fp4", "decode_mxfp4")}


def _no_renorm(logits, k):
    idx, _ = _orig["topk_renorm"](logits, k)
    p = M.softmax(logits)
    return idx, np.take_along_axis(p, idx.astype(np.int64), axis=1)


def _lowest_k(logits, k):
    return _orig["topk_renorm"](-np.asarray(logits), k)


def _ties_high(logits, k):
    logits = np.asarray(logits, float)
    E = logits.shape[1]
    idx, w = _orig["topk_renorm"](logits[:, ::-1], k)
    return (E - 1 - idx).astype(np.int32), w


def _perm_descending(idx, E):
    counts, offsets, perm_token, inv_row = _orig["permutation_maps"](idx, E)
    pt = perm_token.copy()
    inv = inv_row.copy()
    for e in range(E):
        a, b = offsets[e], offsets[e + 1]
        pt[a:b] = perm_token[a:b][::-1]
        for r in range(a, b):
            t = perm_token[r]
            j = list(idx[t]).index(e)
            inv[t, j] = a + b - 1 - r
    return counts, offsets, pt, inv


def _silu_sign(z):
    return _orig["silu"](-np.asarray(z, float))


def _swiglu_swapped(x, wg, wu, wd, act8=False):
    return _orig["swiglu_expert"](x, wu, wg, wd, act8=act8)


def _swiglu_h_unquantised(x, wg, wu, wd, act8=False):
    if not act8:
        return _orig["swiglu_expert"](x, wg, wu, wd)
    xq = M.dequantize_rows_e4m3(*M.quantize_rows_e4m3(np.asarray(x, float)))
    return _orig["swiglu_expert"](xq, wg, wu, wd)


def _swiglu_no_gate(x, wg, wu, wd, act8=False):
    x = np.asarray(x, float)
    return ((x @ np.asarray(wg).T) * (x @ np.asarray(wu).T)) @ np.asarray(wd).T


def _e4m3_bias8(bits):
    return _orig["decode_e4m3"](bits) / 2.0


def _bf16_sub_as_normal(bits):
    b = np.asarray(bits).astype(np.int64)
    out = _orig["decode_bf16"](bits)
    sub = ((b >> 7) & 0xFF) == 0
    out = np.where(sub & ((b & 0x7F) != 0), out * 2.0, out)
    return out


def _router_transposed_bias(x, w, bias=None):
    lg = _orig["router_logits"](x, w, None)
    return lg if bias is None else lg - np.asarray(bias)[None, :]


def _shared_dropped(x, wg, wu, wd):
    return np.zeros((np.asarray(x).shape[0], np.asarray(wd).shape[0]))


def _e4m3_ties_away(v):
    # round half away from zero instead of half to even
    v32 = np.asarray(v, np.float32)
    c = _orig["round_to_e4m3"](v32)
    nudged = _orig["round_to_e4m3"](np.nextafter(v32, np.copysign(np.float32(1e9), v32)))
    mags = M._E4M3_POS
    a = np.abs(v32).astype(float)
    hi = np.clip(np.searchsorted(mags, a), 0, 0x7E)
    tie = (hi > 0) & (mags[hi] - a == a - mags[np.maximum(hi - 1, 0)])
    return np.where(tie, nudged, c).astype(np.uint8)


def _e4m3_no_saturation(v):
    v32 = np.asarray(v, np.float32)
    c = _orig["round_to_e4m3"](v32)
    return np.where(np.abs(v32) > 464.0, c | 0x7F, c).astype(np.uint8)


def _row_scale_480(x):
    x32 = np.asarray(x, np.float32)
    amax = np.max(np.abs(x32), axis=1)
    s = np.where(amax > 0, amax / np.float32(480.0), np.float32(1.0)).astype(np.float32)
    return M.round_to_e4m3((x32 / s[:, None]).astype(np.float32)), s


def _e2m1_subnormal_quarter(codes):
    v = _orig["decode_e2m1"](codes)
    return np.where(np.abs(v) == 0.5, v / 2.0, v)


def _ue8m0_bias_126(s):
    return _orig["decode_ue8m0"](s) * 2.0


def _fp4_nibbles_swapped(packed):
    b = np.asarray(packed).astype(np.uint8)
    return _orig["unpack_fp4"](((b & 0xF) << 4) | (b >> 4))


def _mxfp4_scales_transposed(packed, scales):
    sc = np.asarray(scales)
    return _orig["decode_mxfp4"](packed, sc.T.reshape(sc.shape))


MUTATIONS = {
    "no_renormalisation": ("topk_renorm", _no_renorm),
    "lowest_k_selected": ("topk_renorm", _lowest_k),
    "ties_to_higher_index": ("topk_renorm", _ties_high),
    "rows_descending_token": ("permutation_maps", _perm_descending),
    "silu_sign_flip": ("silu", _silu_sign),
    "gate_up_swapped": ("swiglu_expert", _swiglu_swapped),
    "activation_dropped": ("swiglu_expert", _swiglu_no_gate),
    "act8_h_not_quantised": ("swiglu_expert", _swiglu_h_unquantised),
    "e4m3_wrong_bias": ("decode_e4m3", _e4m3_bias8),
    "bf16_subnormal_as_normal": ("decode_bf16", _bf16_sub_as_normal),
    "router_bias_sign": ("router_logits", _router_transposed_bias),
    "shared_expert_dropped": ("shared_expert", _shared_dropped),
    "e4m3_ties_away_from_zero": ("round_to_e4m3", _e4m3_ties_away),
    "e4m3_overflow_not_saturated": ("round_to_e4m3", _e4m3_no_saturation),
    "activation_scale_off": ("quantize_rows_e4m3", _row_scale_480),
    "e2m1_subnormal_quarter": ("decode_e2m1", _e2m1_subnormal_quarter),
    "ue8m0_bias_126": ("decode_ue8m0", _ue8m0_bias_126),
    "fp4_nibbles_swapped": ("unpack_fp4", _fp4_nibbles_swapped),
    "mxfp4_scales_transposed": ("decode_mxfp4", _mxfp4_scales_transposed),
}

PIN_CHECKS = [
    pins.test_decode_bf16_fixed_values,
    pins.test_decode_bf16_all_patterns_match_binary32_upper_half,
    pins.test_decode_e4m3_fixed_values,
    pins.test_decode_e4m3_all_codes_match_torch,
    pins.test_worked_example_groups_and_rows,
    pins.test_worked_example_router_reproduces_weights,
    pins.test_worked_example_combine_of_T1,
    pins.test_router_logits_match_library_linear,
    lambda: pins.test_topk_brute_force_over_subsets(6, 3),
    pins.test_topk_ties_go_to_lower_index,
    pins.test_silu_closed_form_values,
    pins.test_swiglu_expert_matches_library_ffn,
    pins.test_single_expert_is_dense_swiglu,
    pins.test_shared_expert_is_added_with_weight_one,
    lambda: pins.test_permutation_invariants(37, 8, 2),
    pins.test_round_to_e4m3_matches_library_cast_in_range,
    pins.test_round_to_e4m3_ties_go_to_even_and_saturates,
    pins.test_quantize_rows_scale_and_extremes,
    pins.test_quantize_rows_lossless_on_representable_rows,
    pins.test_act8_expert_quantises_both_activations,
    pins.test_decode_e2m1_fixed_values,
    pins.test_decode_e2m1_agrees_with_e4m3_at_the_same_value,
    pins.test_decode_ue8m0_fixed_values,
    pins.test_unpack_fp4_nibble_order,
    pins.test_decode_mxfp4_hand_block,
    pins.test_mxfp4_storage_matches_the_page,
    pins.test_mxfp4_expert_weights_decode_per_matrix,
]


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_some_pin_catches_the_mutation(name, monkeypatch):
    attr, fn = MUTATIONS[name]
    monkeypatch.setattr(M, attr, fn)
    monkeypatch.setattr(oracle, attr, fn)
    caught = []
    for check in PIN_CHECKS:
        try:
            check()
        except Exception:  # an assertion, or a shape error, both count
            caught.append(getattr(check, "__name__", "lambda"))
    assert caught, f"mutation {name} passed every pin"


def test_unmutated_oracle_passes_every_check():
    for check in PIN_CHECKS:
        check()
