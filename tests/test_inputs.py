"""The seeded input generators (no GPU): reproducible per (seed, tensor
name), shapes and dtypes of every weight format, and quantised weights that
decode (through the oracle's format decoders) to within one quantisation
step of the fp32 draws they were made from."""

import numpy as np
import pytest
import torch

import oracle
from routed_expert_ffn_gemm_gb300 import inputs


def _small(wfmt, **kw):
    base = dict(T=5, d=256, ffn=128, E=4, k=2, wfmt=wfmt, act="f32" if wfmt == "f32" else "bf16")
    base.update(kw)
    return inputs.MoEShape("gen", **base)


@pytest.mark.parametrize("wfmt", ["f32", "bf16", "fp8", "fp8a8", "mxfp4"])
def test_cases_are_reproducible_and_seeded(wfmt):
    a = inputs.make_case(_small(wfmt), 3, "cpu")
    b = inputs.make_case(_small(wfmt), 3, "cpu")
    c = inputs.make_case(_small(wfmt), 4, "cpu")
    for name, t in a.items():
        if t is None:
            assert b[name] is None
            continue
        assert torch.equal(t, b[name]), name
    assert not torch.equal(a["x"], c["x"]) and not torch.equal(a["w_gate"], c["w_gate"])
    # the per-name streams differ: gate and up are not the same draw
    assert not torch.equal(a["w_gate"], a["w_up"])


@pytest.mark.parametrize("wfmt,w_shape,s_shape", [
    ("bf16", (4, 128, 256), None),
    ("fp8", (4, 128, 256), (4, 128)),
    ("fp8a8", (4, 128, 256), (4, 128)),
    ("mxfp4", (4, 128, 128), (4, 8, 128)),
])
def test_weight_layouts(wfmt, w_shape, s_shape):
    case = inputs.make_case(_small(wfmt), 0, "cpu")
    assert tuple(case["w_gate"].shape) == w_shape
    if s_shape is None:
        assert case["s_gate"] is None
    else:
        assert tuple(case["s_gate"].shape) == s_shape
    if wfmt == "mxfp4":  # down: [E, d, ffn/2] codes, [E, ffn/32, d] scales
        assert tuple(case["w_down"].shape) == (4, 256, 64)
        assert tuple(case["s_down"].shape) == (4, 4, 256)


def _draws(shape, rows, cols, name, e):
    std = 1.0 / np.sqrt(shape.d)
    return inputs._normal((rows, cols), std, 0, f"{name}[{e}]", "cpu", torch.float32).double().numpy()


def test_fp8_weights_decode_near_their_draws():
    shape = _small("fp8")
    case = inputs.make_case(shape, 0, "cpu")
    for e in range(shape.E):
        w = _draws(shape, shape.ffn, shape.d, "w_gate", e)
        dec = oracle.decode_e4m3(case["w_gate"][e].numpy()) * case["s_gate"][e].double().numpy()[:, None]
        # half an E4M3 step (relative 2^-4), or the subnormal step, per element
        tol = np.maximum(np.abs(w) * 2.0 ** -4, case["s_gate"][e].double().numpy()[:, None] * 2.0 ** -10)
        assert np.all(np.abs(dec - w) <= tol * 1.0001)


def test_mxfp4_weights_decode_near_their_draws():
    shape = _small("mxfp4")
    case = inputs.make_case(shape, 0, "cpu")
    for e in range(shape.E):
        w = _draws(shape, shape.ffn, shape.d, "w_gate", e)
        scales = case["s_gate"][e].numpy()                        # [d/32, ffn]
        dec = oracle.decode_mxfp4(case["w_gate"][e].numpy(), scales)
        step = np.repeat(oracle.decode_ue8m0(scales), 32, axis=0).T   # [ffn, d] block scale 2^e
        # E2M1 steps are at most 2 * 2^e (between 4 and 6); values past 6 * 2^e saturate
        # (the block max lands in [4, 8) * 2^e)
        assert np.all(np.abs(dec - w) <= 2.0 * step * 1.0001)
        # each block's largest magnitude decodes to 4 or 6 times its scale
        blk_max = np.abs(dec).reshape(shape.ffn, shape.d // 32, 32).max(axis=2)
        ratio = blk_max / oracle.decode_ue8m0(scales).T
        assert np.isin(ratio, [4.0, 6.0]).all()
