"""GPU parity of MXFP4 routed experts ("MoE 推理部署", section 专家量化:
OCP MX block-scaled 4-bit expert weights):

  grouped SwiGLU and the whole layer against the oracle's decode of the
  same codes and UE8M0 block scales: max|err| <= 5e-2 * max|ref| (the bar
  for quantised experts) and, since the in-kernel conversion is exact for
  block scales 2^-23 .. 2^13, a relative rms error of at most 1e-2 (the f16
  roundings of x and h and the bf16 rounding of y remain).
"""

import numpy as np
import pytest
import torch

import oracle
from routed_expert_ffn_gemm_gb300 import api, build, inputs
from tests import helpers
from tests.test_gpu_parity import DEV, FP8_TOL, GROUP_COUNTS, _bf16_rand, _f64, _layer_check

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _library():
    build.build()
    api._lib()
    yield
    assert api.moe_read_device_status() == 0, "a kernel recorded an error"


def _mx_stack(E, rows, cols, gen, scale_range=None):
    """MXFP4 matrices [E, rows, cols]: random N(0, 1/cols) weights through
    the input generator's quantiser, or (scale_range) uniformly random codes
    with UE8M0 scales drawn from [lo, hi]."""
    w = torch.empty((E, rows, cols // 2), dtype=torch.uint8, device=DEV)
    s = torch.empty((E, cols // 32, rows), dtype=torch.uint8, device=DEV)
    for e in range(E):
        if scale_range is None:
            q, sc = inputs._mxfp4_quantise(torch.randn((rows, cols), generator=gen, device=DEV) * cols ** -0.5)
        else:
            q = torch.randint(0, 256, (rows, cols // 2), generator=gen, device=DEV).to(torch.uint8)
            sc = torch.randint(scale_range[0], scale_range[1] + 1, (cols // 32, rows), generator=gen,
                               device=DEV).to(torch.uint8)
        w[e].copy_(q)
        s[e].copy_(sc)
    return w, s


def _grouped_case(kind, d, f, seed, stacks=None):
    counts = np.array(GROUP_COUNTS[kind])
    E = len(counts)
    R = int(counts.sum())
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    g = torch.Generator(device=DEV).manual_seed(seed)
    x = _bf16_rand((R, d), 1.0, g)
    if stacks is None:
        stacks = (_mx_stack(E, f, d, g), _mx_stack(E, f, d, g), _mx_stack(E, d, f, g))
    else:
        stacks = stacks(E, g)
    (wg, sg), (wu, su), (wd, sd) = stacks
    p = api.problem(R, d, f, E, 1, wfmt="mxfp4")
    y = torch.full((R, d), float("nan"), dtype=torch.bfloat16, device=DEV)
    api.moe_grouped_swiglu(p, x, torch.from_numpy(offsets).to(DEV), wg, wu, wd, sg, su, sd, y,
                           api.workspace_for(p))
    torch.cuda.synchronize()
    ew = oracle.ExpertWeights("mxfp4", *(t.cpu().numpy() for t in (wg, wu, wd, sg, su, sd)))
    xf, got = _f64(x), _f64(y)
    ref = np.zeros_like(got)
    for e in range(E):
        a, b = offsets[e], offsets[e + 1]
        if b > a:
            ref[a:b] = oracle.swiglu_expert(xf[a:b], *ew.get(e))
    return p, got, ref


def _check(got, ref):
    assert np.isfinite(got).all()
    assert np.abs(got - ref).max() <= FP8_TOL * np.abs(ref).max()
    rel = np.sqrt(((got - ref) ** 2).mean()) / np.sqrt((ref ** 2).mean())
    assert rel <= 1e-2, f"relative rms error {rel:.3g}"


@pytest.mark.parametrize("bn,pair", [(32, 0), (128, 0), (256, 0), (32, 1), (128, 1), (256, 1)])
@pytest.mark.parametrize("kind", ["prefill_like", "ragged", "decode"])
def test_grouped_swiglu_mxfp4_every_tile(bn, pair, kind, monkeypatch):
    # every tile-row count of both GEMMs, single CTAs and CTA pairs (32-row
    # tiles on pairs: MOE_PAIR=2), the tensor-memory and the shared-memory
    # operand paths of the converters
    monkeypatch.setenv("MOE_BN_GATEUP", str(bn))
    monkeypatch.setenv("MOE_BN_DOWN", str(bn))
    monkeypatch.setenv("MOE_PAIR", str(2 if pair and bn == 32 else pair))
    monkeypatch.setenv("MOE_SPLITS_GATEUP", "1")
    d, f = 512, 256
    p = api.problem(int(np.sum(GROUP_COUNTS[kind])), d, f, len(GROUP_COUNTS[kind]), 1, wfmt="mxfp4")
    info = api.moe_plan_info(p)
    assert (info["bn_gateup"], info["pair_gateup"], info["pair_down"]) == (bn, pair, pair)
    _, got, ref = _grouped_case(kind, d, f, bn + pair)
    _check(got, ref)


def test_grouped_swiglu_mxfp4_extreme_block_scales():
    # the documented exact range of block scales: gate blocks up to 2^13,
    # up blocks down to 2^-23 (so SiLU(g) * u stays inside f16), every code
    def stacks(E, g):
        wg, sg = _mx_stack(E, 256, 512, g, scale_range=(104, 140))
        sg[:, :, :] = torch.where(sg > 120, sg, torch.full_like(sg, 104))
        wu, su = _mx_stack(E, 256, 512, g, scale_range=(104, 108))
        wd, sd = _mx_stack(E, 512, 256, g)
        return (wg, sg), (wu, su), (wd, sd)
    _, got, ref = _grouped_case("ragged", 512, 256, 5, stacks)
    _check(got, ref)


@pytest.mark.parametrize("splits", [1, 3])
def test_layer_mxfp4_decode(splits, monkeypatch):
    monkeypatch.setenv("MOE_SPLITS_GATEUP", str(splits))
    shape = inputs.MoEShape("mx_small", T=5, d=512, ffn=256, E=16, k=4, ffn_shared=256, wfmt="mxfp4")
    assert api.moe_plan_info(api.problem_of(shape))["splits_gateup"] == splits
    _layer_check(shape, 4, FP8_TOL)


@pytest.mark.parametrize("bn,pair", [(128, 0), (128, 1), (256, 1)])
def test_layer_mxfp4_gathered_rows(bn, pair, monkeypatch):
    monkeypatch.setenv("MOE_BN_GATEUP", str(bn))
    monkeypatch.setenv("MOE_BN_DOWN", str(bn))
    monkeypatch.setenv("MOE_PAIR", str(pair))
    monkeypatch.setenv("MOE_SPLITS_GATEUP", "1")
    shape = inputs.MoEShape("mx_gathered", T=300, d=512, ffn=512, E=8, k=2, ffn_shared=256, wfmt="mxfp4")
    _layer_check(shape, 3, FP8_TOL)


def test_layer_mxfp4_deepseek_like():
    for T in (1, 64):
        shape = inputs.MoEShape("ds_like_mx", T=T, d=1024, ffn=512, E=64, k=8, ffn_shared=512, wfmt="mxfp4")
        _layer_check(shape, helpers.seed_without_near_ties(shape, 0, min_gap=1e-3), FP8_TOL)
