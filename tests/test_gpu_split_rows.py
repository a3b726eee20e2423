"""GPU: moe_split_rows_e4m3x2, the two-term E4M3 form in which the FP8-weight
mode hands bf16 rows to the FP8 x FP8 tensor-core instructions
("MoE 推理部署", section 专家量化: FP8 expert weights, activations kept at
higher precision).  Checked through the C ABI against the encoding's
definition: s is the power of two that puts the row maximum in (224, 448];
hi is the nearest E4M3 value of x / s and lo the nearest E4M3 value of
x / s - hi (torch's float8 cast, a library rounding, is the pin for both);
s (hi + lo) returns x exactly for every element within 2^9 of its row
maximum, and within s * 2^-10 below that.  Rows span magnitudes from bf16
subnormals to 1e30, with outliers, zeros and signed zeros."""

import numpy as np
import pytest
import torch

import oracle
from routed_expert_ffn_gemm_gb300 import api, build, inputs

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _library():
    build.build()
    api._lib()
    yield
    assert api.moe_read_device_status() == 0


def _rows(rows, cols, seed):
    g = torch.Generator(device="cpu").manual_seed(seed)
    x = torch.randn((rows, cols), generator=g)
    # per-row magnitudes from bf16 subnormal range to 1e30
    mags = torch.logspace(-38, 30, rows, dtype=torch.float64).to(torch.float32)
    x = x * mags[:, None]
    # outliers: a few elements 1e3 .. 1e5 times their row's typical size
    for r in range(0, rows, 3):
        x[r, (r * 7) % cols] *= 10.0 ** (3 + r % 3)
    # elements far below their row maximum (exercise the inexact tail)
    x[1::4, ::5] *= 1e-6
    if rows > 2:
        x[2] = 0.0              # an all-zero row
    if rows > 5:
        x[5, :4] = -0.0         # signed zeros
    if rows > 7:
        x[7] = torch.where(torch.arange(cols) % 2 == 0, x[7], torch.zeros(()))
    return x.to(torch.bfloat16)


def _split(x):
    rows, cols = x.shape
    codes = torch.full((2, rows, cols), 0x7F, dtype=torch.uint8, device=DEV)  # NaN codes until written
    scales = torch.full((rows,), float("nan"), dtype=torch.float32, device=DEV)
    api.moe_split_rows_e4m3x2(x.to(DEV), codes, scales)
    torch.cuda.synchronize()
    return codes.cpu().numpy(), scales.cpu().numpy()


def _e4m3(v):
    """Nearest E4M3 codes of float64 values exact in float32 (torch's cast)."""
    return torch.from_numpy(np.asarray(v, np.float64).astype(np.float32)).to(torch.float8_e4m3fn) \
        .view(torch.uint8).numpy()


@pytest.mark.parametrize("rows,cols", [(64, 7168), (257, 2048), (3, 8), (1, 128), (129, 3072), (5, 4096), (300, 1000)])
def test_split_rows_is_the_definition(rows, cols):
    x = _rows(rows, cols, rows + cols)
    codes, s = _split(x)
    xf = oracle.decode_bf16(inputs.to_numpy_stored(x))
    amax = np.abs(xf).max(axis=1)
    # s: a power of two putting the row maximum in (224, 448]; 1 for zero rows
    m, _ = np.frexp(s.astype(np.float64))
    assert np.all(m == 0.5), "scales are powers of two"
    nz = amax > 0
    assert np.all(s[~nz] == 1.0)
    assert np.all((amax[nz] / s[nz] > 224.0) & (amax[nz] / s[nz] <= 448.0))
    hi, lo = codes[0], codes[1]
    a = xf / s[:, None].astype(np.float64)  # exact: a power-of-two division
    assert np.array_equal(hi, _e4m3(a))
    hv = oracle.decode_e4m3(hi)
    assert np.array_equal(lo, _e4m3(a - hv))
    # reconstruction: exact within 2^9 of the row maximum, else within s 2^-10
    back = s[:, None].astype(np.float64) * (hv + oracle.decode_e4m3(lo))
    big = np.abs(xf) >= amax[:, None] * 2.0 ** -9
    assert np.array_equal(back[big], xf[big])
    assert np.all(np.abs(back - xf) <= s[:, None] * 2.0 ** -10)
    assert not np.any(np.isnan(back))


def test_split_rows_of_outlier_tokens():
    # token rows with a 1e5 outlier beside N(0,1) values: the outlier and
    # every element within 2^9 of it come back bit for bit; the N(0,1)
    # elements, seventeen binades below it, within s * 2^-10 = 2^8 * 2^-10
    x = torch.randn((16, 4096), generator=torch.Generator().manual_seed(3))
    x[:, 17] = 1e5
    x = x.to(torch.bfloat16)
    codes, s = _split(x)
    assert np.all(s == 2.0 ** 8)  # 99840 / 2^8 = 390 in (224, 448]
    xf = oracle.decode_bf16(inputs.to_numpy_stored(x))
    back = s[:, None].astype(np.float64) * (oracle.decode_e4m3(codes[0]) + oracle.decode_e4m3(codes[1]))
    big = np.abs(xf) >= np.abs(xf).max(axis=1, keepdims=True) * 2.0 ** -9
    assert big[:, 17].all()
    assert np.array_equal(back[big], xf[big])
    assert np.abs(back - xf).max() <= 2.0 ** 8 * 2.0 ** -10
