"""GPU parity of the FP8-activation mode ("MOE推理流程解析", section 三:
activations quantised before dispatch; "MoE 推理部署", section 专家量化):

  per-row E4M3 quantisation (moe_quantize_rows_e4m3): codes and scales
  bit-exact against the oracle's quantize_rows_e4m3;
  grouped SwiGLU with FP8 x FP8 gate/up products: max|err| <= 5e-2 *
  max|ref| against the oracle's act8 expert (the bar for FP8 experts), and,
  since the device quantises exactly as the oracle does, a relative rms
  error of at most 1e-2 (the f16 rounding of h and the bf16 rounding of y
  remain), several times below the error against the unquantised expert.
"""

import numpy as np
import pytest
import torch

import oracle
from routed_expert_ffn_gemm_gb300 import api, build
from tests import helpers
from tests.test_gpu_parity import DEV, FP8_TOL, GROUP_COUNTS, _bf16_rand, _f64, _fp8_stack

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _library():
    build.build()
    api._lib()
    yield
    assert api.moe_read_device_status() == 0, "a kernel recorded an error"


def _quantise_on_gpu(x):
    codes = torch.empty(x.shape, dtype=torch.uint8, device=DEV)
    scales = torch.empty(x.shape[0], dtype=torch.float32, device=DEV)
    api.moe_quantize_rows_e4m3(x, codes, scales)
    torch.cuda.synchronize()
    return codes.cpu().numpy(), scales.cpu().numpy()


def _special_rows(cols):
    """Rows whose quotients land on E4M3 rounding ties, in the subnormal
    range, below the smallest subnormal (signed zeros), and all-zero rows."""
    rows = np.zeros((4, cols), np.float32)
    # row 0: amax 448 -> scale exactly 1, the row's values are the quotients:
    # ties between neighbours (1.0625: 1 | 1.125; 17: 16 | 18; 3*2^-10:
    # 2^-9 | 2^-8 in the subnormals; 4.5*2^-9 between two subnormals;
    # 7.5*2^-9 between the largest subnormal and the smallest normal),
    # values below half the smallest subnormal (-> signed zero), -0
    vals = [448.0, 1.0625, 17.0, -17.0, 3 * 2.0 ** -10, -3 * 2.0 ** -10, 2.0 ** -11, -(2.0 ** -11),
            -4.5 * 2.0 ** -9, 7.5 * 2.0 ** -9, 1.1875, 248.0, 0.0, -0.0, 13.0, 3.25]
    rows[0, :len(vals)] = vals[:cols]
    rows[0, len(vals):] = np.linspace(-448, 448, cols - len(vals))
    # row 1: all zero (scale 1, codes 0); row 2: all -0 (codes 0x80)
    rows[2, :] = -0.0
    # row 3: a huge and a tiny magnitude in one row
    rows[3, :] = 1e-3
    rows[3, 0] = 3.0e4
    return torch.from_numpy(rows).to(torch.bfloat16)


@pytest.mark.parametrize("rows,cols,std", [(37, 7168, 1.0), (5, 8, 3.0), (300, 2048, 1e-3), (1, 4096, 50.0)])
def test_quantize_rows_bit_exact(rows, cols, std):
    g = torch.Generator(device=DEV).manual_seed(rows * 7 + cols)
    x = _bf16_rand((rows, cols), std, g)
    special = cols >= 16 and rows >= 4
    if special:
        x[:4] = _special_rows(cols).to(DEV)
    codes, scales = _quantise_on_gpu(x)
    q_ref, s_ref = oracle.quantize_rows_e4m3(_f64(x).astype(np.float32))
    assert np.array_equal(scales.view(np.uint32), s_ref.astype(np.float32).view(np.uint32))
    bad = np.argwhere(codes != q_ref)
    assert bad.size == 0, f"{len(bad)} codes differ, first at {bad[:4].tolist()}"
    if special:
        assert codes[0, :10].tolist() == [0x7E, 0x38, 0x58, 0xD8, 0x02, 0x82, 0x00, 0x80, 0x84, 0x08]
        assert (codes[1] == 0).all() and scales[1] == 1.0
        assert (codes[2] == 0x80).all() and scales[2] == 1.0


def test_quantize_rows_empty_and_argument_errors():
    x = torch.zeros((0, 128), dtype=torch.bfloat16, device=DEV)
    api.moe_quantize_rows_e4m3(x, torch.empty((0, 128), dtype=torch.uint8, device=DEV),
                               torch.empty(0, dtype=torch.float32, device=DEV))
    with pytest.raises(api.MoEError) as e:
        x = torch.zeros((2, 12), dtype=torch.bfloat16, device=DEV)
        api.moe_quantize_rows_e4m3(x, torch.empty((2, 12), dtype=torch.uint8, device=DEV),
                                   torch.empty(2, dtype=torch.float32, device=DEV))
    assert e.value.status == api.ERR_UNSUPPORTED


@pytest.mark.parametrize("bn,pair", [(32, 0), (128, 0), (256, 0), (128, 1), (256, 1)])
@pytest.mark.parametrize("kind", ["prefill_like", "ragged", "decode"])
def test_grouped_swiglu_act8_every_tile(bn, pair, kind, monkeypatch):
    # x_perm rows quantised after dispatch (one scale per row), the gate/up
    # GEMM on FP8 x FP8 instructions for every tile-row count, single CTAs
    # and CTA pairs
    monkeypatch.setenv("MOE_BN_GATEUP", str(bn))
    monkeypatch.setenv("MOE_BN_DOWN", str(bn))
    monkeypatch.setenv("MOE_PAIR", str(pair))
    monkeypatch.setenv("MOE_SPLITS_GATEUP", "1")  # (pairs take unsplit gate/up GEMMs)
    counts = np.array(GROUP_COUNTS[kind])
    E, d, f = len(counts), 384, 256
    R = int(counts.sum())
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    g = torch.Generator(device=DEV).manual_seed(bn + 3 * pair)
    x = _bf16_rand((R, d), 1.0, g)
    busy = int(np.argmax(counts))
    wg, sg = _fp8_stack(E, f, d, g, all_codes_expert=busy)
    wu, su = _fp8_stack(E, f, d, g)
    wd, sd = _fp8_stack(E, d, f, g)
    p = api.problem(R, d, f, E, 1, wfmt="fp8a8")
    info = api.moe_plan_info(p)
    assert (info["bn_gateup"], info["pair_gateup"]) == (bn, pair)
    y = torch.full((R, d), float("nan"), dtype=torch.bfloat16, device=DEV)
    api.moe_grouped_swiglu(p, x, torch.from_numpy(offsets).to(DEV), wg, wu, wd, sg, su, sd, y,
                           api.workspace_for(p))
    torch.cuda.synchronize()
    ew = oracle.ExpertWeights("fp8", wg.cpu().numpy(), wu.cpu().numpy(), wd.cpu().numpy(),
                              sg.cpu().numpy(), su.cpu().numpy(), sd.cpu().numpy())
    xf, got = _f64(x), _f64(y)
    ref, ref16 = np.zeros_like(got), np.zeros_like(got)
    for e in range(E):
        a, b = offsets[e], offsets[e + 1]
        if b > a:
            ref[a:b] = oracle.swiglu_expert(xf[a:b], *ew.get(e), act8=True)
            ref16[a:b] = oracle.swiglu_expert(xf[a:b], *ew.get(e))
    assert np.isfinite(got).all()
    assert np.abs(got - ref).max() <= FP8_TOL * np.abs(ref).max()
    rms = lambda v: float(np.sqrt((v ** 2).mean()))  # noqa: E731
    rel = rms(got - ref) / rms(ref)
    assert rel <= 1e-2, f"relative rms error {rel:.3g} against the act8 oracle"
    # the row quantisation is really applied: the unquantised expert is
    # further away than the act8 one
    assert rms(got - ref16) > 2 * rms(got - ref)


def test_layer_act8_quantises_tokens_before_dispatch():
    # the layer quantises x's T rows once and gathers E4M3 rows by token; a
    # DeepSeek-like small layer (FP8 routed experts, bf16 shared expert)
    from routed_expert_ffn_gemm_gb300 import inputs
    from tests.test_gpu_parity import _layer_check
    for T in (1, 7, 64, 300):
        shape = inputs.MoEShape("ds_like_act8", T=T, d=1024, ffn=512, E=64, k=8, ffn_shared=512, wfmt="fp8a8")
        _layer_check(shape, helpers.seed_without_near_ties(shape, 0, min_gap=1e-3), FP8_TOL)
