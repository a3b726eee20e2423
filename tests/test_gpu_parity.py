"""GPU parity: every entry point of the C-ABI library against the CPU
reference, element by element, on seeded inputs.

Bars (written in each test):
  routing indices, counts, offsets, permutation maps, row moves: bit-exact;
  routing weights: fp32 rounding (rtol 2e-6 given the same fp32 logits);
  layer / expert outputs: max|err| <= 2e-2 * max|ref| for bf16 storage,
  <= 5e-2 * max|ref| for FP8 (E4M3) expert weights, <= 1e-4 * max|ref| for
  fp32 storage.
"""

import dataclasses

import numpy as np
import pytest
import torch

import oracle
from routed_expert_ffn_gemm_gb300 import api, build, inputs
from tests import helpers

pytestmark = pytest.mark.gpu
DEV = "cuda"
BF16_TOL = 2e-2
FP8_TOL = 5e-2
F32_TOL = 1e-4


@pytest.fixture(scope="module", autouse=True)
def _library():
    build.build()
    api._lib()
    yield
    assert api.moe_read_device_status() == 0, "a kernel recorded an error"


def _bf16_rand(shape, std, gen):
    return (torch.randn(shape, generator=gen, device=DEV) * std).to(torch.bfloat16)


def _f64(t):
    return helpers.decode_act(t, "bf16" if t.dtype == torch.bfloat16 else "f32")


# ---------------------------------------------------------------------------
# router
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("T,E,k", [(64, 8, 2), (300, 128, 8), (257, 256, 8), (33, 4, 4), (5, 1024, 32),
                                   (1, 8, 1), (16, 8, 8)])
def test_router_topk_bit_exact_given_oracle_logits(T, E, k):
    rng = np.random.default_rng(T * 1000 + E + k)
    for _ in range(50):  # reject near-ties below 1e-6 (several answers would be valid)
        lg = rng.normal(size=(T, E)).astype(np.float32).astype(np.float64)
        if helpers.routing_gap_ok(lg, k, 1e-6):
            break
    idx_ref, w_ref = oracle.topk_renorm(lg, k)
    p = api.problem(T, 128, 128, E, k)
    idx = torch.empty((T, k), dtype=torch.int32, device=DEV)
    w = torch.empty((T, k), dtype=torch.float32, device=DEV)
    api.moe_router_topk(p, None, None, None, torch.from_numpy(lg.astype(np.float32)).to(DEV), None, idx, w)
    torch.cuda.synchronize()
    assert np.array_equal(idx.cpu().numpy(), idx_ref)
    np.testing.assert_allclose(w.cpu().numpy(), w_ref, rtol=2e-6, atol=1e-7)


def test_router_exact_ties_go_to_lower_index():
    lg = np.array([[1.0, 3.0, 3.0, 0.0, 3.0, -1.0, 3.0, 2.0]] * 9, dtype=np.float32)
    p = api.problem(9, 128, 128, 8, 3)
    idx = torch.empty((9, 3), dtype=torch.int32, device=DEV)
    w = torch.empty((9, 3), dtype=torch.float32, device=DEV)
    api.moe_router_topk(p, None, None, None, torch.from_numpy(lg).to(DEV), None, idx, w)
    idx_ref, w_ref = oracle.topk_renorm(lg.astype(np.float64), 3)
    assert np.array_equal(idx.cpu().numpy(), idx_ref)
    assert idx_ref[0].tolist() == [1, 2, 4]
    np.testing.assert_allclose(w.cpu().numpy(), w_ref, rtol=2e-6)


def test_router_selection_order_with_signed_zeros_infinities_and_nan():
    # the kernels' documented order beyond the oracle's finite logits:
    # larger first, -0 and +0 tied (lower index first), -inf after every
    # other number, NaN logits last (lower index first)
    rows = [([0.0, -0.0, 1.0, np.nan, -2.0, 3.0, -0.0, np.nan], [5, 2, 0, 1, 6, 4, 3, 7]),
            ([-np.inf, 0.5, np.inf, -1.0, np.nan, 2.0, -np.inf, 1.0], [2, 5, 7, 1, 3, 0, 6, 4])]
    for vals, order in rows:
        lg = np.array([vals] * 9, dtype=np.float32)
        p = api.problem(9, 128, 128, 8, 8)
        idx = torch.empty((9, 8), dtype=torch.int32, device=DEV)
        w = torch.empty((9, 8), dtype=torch.float32, device=DEV)
        api.moe_router_topk(p, None, None, None, torch.from_numpy(lg).to(DEV), None, idx, w)
        torch.cuda.synchronize()
        assert idx.cpu().numpy().tolist() == [order] * 9


@pytest.mark.parametrize("act,T,d,E,k", [("bf16", 40, 512, 16, 4), ("bf16", 3, 2048, 128, 8), ("f32", 64, 128, 8, 2),
                                         ("bf16", 200, 7168, 256, 8), ("bf16", 64, 4096, 8, 2),
                                         # tensor-core logits (bf16, E % 128 == 0, T >= 256), ragged T
                                         ("bf16", 300, 2048, 128, 8), ("bf16", 1000, 7168, 256, 8),
                                         ("bf16", 257, 512, 384, 6)])
def test_router_logits_and_choice(act, T, d, E, k):
    g = torch.Generator(device=DEV).manual_seed(T + d + E)
    dt = torch.bfloat16 if act == "bf16" else torch.float32
    x = torch.randn((T, d), generator=g, device=DEV).to(dt)
    wr = (torch.randn((E, d), generator=g, device=DEV) / d ** 0.5).to(dt)
    bias = torch.randn((E,), generator=g, device=DEV) * 0.1
    p = api.problem(T, d, 128, E, k, act=act, wfmt=act)
    logits = torch.empty((T, E), dtype=torch.float32, device=DEV)
    idx = torch.empty((T, k), dtype=torch.int32, device=DEV)
    w = torch.empty((T, k), dtype=torch.float32, device=DEV)
    api.moe_router_topk(p, x, wr, bias, None, logits, idx, w)
    torch.cuda.synchronize()
    ref = oracle.router_logits(_f64(x), _f64(wr), bias.double().cpu().numpy())
    lg = logits.cpu().numpy().astype(np.float64)
    # fp32 accumulation of d products: |err| <= 1e-5 * max|l|
    assert np.abs(lg - ref).max() <= 1e-5 * np.abs(ref).max()
    # the choice is exactly the oracle's top-k of the GPU's own logits
    idx_g, w_g = oracle.topk_renorm(lg, k)
    assert np.array_equal(idx.cpu().numpy(), idx_g)
    np.testing.assert_allclose(w.cpu().numpy(), w_g, rtol=2e-6, atol=1e-7)
    # and the oracle's choice on its own logits wherever the decision is clear
    idx_r, _ = oracle.topk_renorm(ref, k)
    clear = oracle.topk_gap(ref, k) >= 1e-3
    assert np.array_equal(idx.cpu().numpy()[clear], idx_r[clear])


# ---------------------------------------------------------------------------
# the worked example (page "MOE推理流程解析", section 二)
# ---------------------------------------------------------------------------

def test_worked_example_through_router_and_permute():
    g, idx_ref, w_ref, groups = helpers.worked_example()
    T, E, k = g["T"], g["E"], g["k"]
    lg = helpers.worked_example_logits(idx_ref, w_ref, E).astype(np.float32)
    p = api.problem(T, 128, 128, E, k)
    idx = torch.empty((T, k), dtype=torch.int32, device=DEV)
    w = torch.empty((T, k), dtype=torch.float32, device=DEV)
    api.moe_router_topk(p, None, None, None, torch.from_numpy(lg).to(DEV), None, idx, w)
    counts = torch.empty(E, dtype=torch.int32, device=DEV)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=DEV)
    perm = torch.empty(T * k, dtype=torch.int32, device=DEV)
    inv = torch.empty(T * k, dtype=torch.int32, device=DEV)
    api.moe_permute(p, idx, None, counts, offsets, perm, inv, None, None)
    torch.cuda.synchronize()
    assert idx.cpu().numpy().tolist() == idx_ref.tolist()
    np.testing.assert_allclose(w.cpu().numpy(), w_ref, rtol=1e-6)
    assert counts.cpu().tolist() == g["rows_per_expert"] == [3, 2, 2, 1]
    assert offsets.cpu().tolist() == [0, 3, 5, 7, 8]
    pt = perm.cpu().numpy()
    for e in range(E):
        assert pt[offsets[e]:offsets[e + 1]].tolist() == groups[e]
    assert inv.cpu().numpy().reshape(T, k).tolist() == [[0, 5], [6, 1], [2, 3], [4, 7]]


# ---------------------------------------------------------------------------
# permutation
# ---------------------------------------------------------------------------

def _random_idx(T, E, k, rng, skew=False):
    if skew:
        p = 1.0 / np.arange(1, E + 1) ** 1.2
        p /= p.sum()
        return np.stack([rng.choice(E, k, replace=False, p=p) for _ in range(T)]).astype(np.int32)
    return np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)


@pytest.mark.parametrize("T,E,k,skew", [(1, 8, 2, False), (64, 8, 2, False), (128, 128, 8, False),
                                        (256, 8, 8, False), (257, 8, 8, False), (1000, 64, 6, True),
                                        (8192, 128, 8, True), (4096, 256, 8, False), (3, 1024, 32, False),
                                        # chunked path, experts not a multiple of the scan's 128 per round
                                        (3000, 300, 4, True), (600, 1000, 8, False),
                                        # half a million rows through the chunked path
                                        (65536, 128, 8, False)])
def test_permute_bit_exact(T, E, k, skew):
    rng = np.random.default_rng(T + E + k)
    idx = _random_idx(T, E, k, rng, skew)
    counts_r, offsets_r, perm_r, inv_r = oracle.permutation_maps(idx, E)
    d = 128
    g = torch.Generator(device=DEV).manual_seed(T)
    x = _bf16_rand((T, d), 1.0, g)
    p = api.problem(T, d, 128, E, k)
    ws = api.workspace_for(p)
    counts = torch.empty(E, dtype=torch.int32, device=DEV)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=DEV)
    perm = torch.empty(T * k, dtype=torch.int32, device=DEV)
    inv = torch.empty(T * k, dtype=torch.int32, device=DEV)
    x_perm = torch.empty((T * k, d), dtype=torch.bfloat16, device=DEV)
    api.moe_permute(p, torch.from_numpy(idx).to(DEV), x, counts, offsets, perm, inv, x_perm, ws)
    torch.cuda.synchronize()
    assert np.array_equal(counts.cpu().numpy(), counts_r)
    assert np.array_equal(offsets.cpu().numpy(), offsets_r)
    assert np.array_equal(perm.cpu().numpy(), perm_r)
    assert np.array_equal(inv.cpu().numpy().reshape(T, k), inv_r)
    assert torch.equal(x_perm.cpu(), x.cpu()[torch.from_numpy(perm_r.astype(np.int64))])


def test_permute_flags_out_of_range_expert():
    T, E, k = 16, 8, 2
    idx = _random_idx(T, E, k, np.random.default_rng(0))
    idx[5, 1] = E  # invalid
    p = api.problem(T, 128, 128, E, k)
    counts = torch.empty(E, dtype=torch.int32, device=DEV)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=DEV)
    perm = torch.empty(T * k, dtype=torch.int32, device=DEV)
    inv = torch.empty(T * k, dtype=torch.int32, device=DEV)
    api.moe_permute(p, torch.from_numpy(idx).to(DEV), None, counts, offsets, perm, inv, None, None)
    assert api.moe_read_device_status() == api.ERR_DEVICE_BOUNDS
    assert int(counts.sum()) == T * k - 1
    assert api.moe_read_device_status() == 0  # reading cleared it


# ---------------------------------------------------------------------------
# combine
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("act", ["bf16", "f32"])
def test_combine_matches_definition(act):
    T, k, d = 37, 4, 256
    R = T * k
    rng = np.random.default_rng(5)
    dt = torch.bfloat16 if act == "bf16" else torch.float32
    g = torch.Generator(device=DEV).manual_seed(5)
    y = torch.randn((R, d), generator=g, device=DEV).to(dt)
    sh = torch.randn((T, d), generator=g, device=DEV).to(dt)
    inv = rng.permutation(R).astype(np.int32)
    w = rng.uniform(0.1, 1.0, size=(T, k))
    w = (w / w.sum(1, keepdims=True)).astype(np.float32)
    out = torch.empty((T, d), dtype=dt, device=DEV)
    p = api.problem(T, d, 128, 8, k, act=act, wfmt=act)
    api.moe_combine(p, y, torch.from_numpy(inv).to(DEV), torch.from_numpy(w).to(DEV), sh, out)
    torch.cuda.synchronize()
    yf, sf = _f64(y), _f64(sh)
    ref = (w.astype(np.float64)[:, :, None] * yf[inv.reshape(T, k)]).sum(1) + sf
    got = _f64(out)
    bound = (2.0 ** -8 if act == "bf16" else 1e-6) * np.abs(ref) + 1e-6 * np.abs(ref).max()
    assert np.all(np.abs(got - ref) <= bound)


# ---------------------------------------------------------------------------
# grouped SwiGLU experts
# ---------------------------------------------------------------------------

GROUP_COUNTS = {
    "ragged": [0, 1, 15, 16, 17, 31, 32, 33, 100, 127, 128, 129, 0, 300, 2, 5],
    "decode": [1, 0, 2, 1, 0, 0, 1, 3, 0, 1, 2, 1, 0, 0, 1, 1],
    "one_hot_expert": [0] * 7 + [517] + [0] * 8,
    "prefill_like": [300, 0, 257, 513, 129, 128, 255, 256, 1, 600, 380, 17, 0, 999, 64, 2],
}


@pytest.mark.parametrize("kind", sorted(GROUP_COUNTS))
@pytest.mark.parametrize("d,f", [(256, 384), (128, 256)])
def test_grouped_swiglu_tensor_path(kind, d, f):
    counts = np.array(GROUP_COUNTS[kind])
    E = len(counts)
    R = int(counts.sum())
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    g = torch.Generator(device=DEV).manual_seed(R + d)
    x = _bf16_rand((R, d), 1.0, g)
    wg, wu = _bf16_rand((E, f, d), d ** -0.5, g), _bf16_rand((E, f, d), d ** -0.5, g)
    wd = _bf16_rand((E, d, f), d ** -0.5, g)
    p = api.problem(R, d, f, E, 1)
    y = torch.full((R, d), float("nan"), dtype=torch.bfloat16, device=DEV)
    ws = api.workspace_for(p)
    api.moe_grouped_swiglu(p, x, torch.from_numpy(offsets).to(DEV), wg, wu, wd, None, None, None, y, ws)
    torch.cuda.synchronize()
    got = _f64(y)
    xf = _f64(x)
    ref = np.zeros_like(got)
    for e in range(E):
        a, b = offsets[e], offsets[e + 1]
        if b > a:
            ref[a:b] = oracle.swiglu_expert(xf[a:b], _f64(wg[e]), _f64(wu[e]), _f64(wd[e]))
    assert np.isfinite(got).all()
    assert np.abs(got - ref).max() <= BF16_TOL * np.abs(ref).max()
    # tighter statistical check: bf16 rounding of h and y only
    assert np.sqrt(((got - ref) ** 2).mean()) <= 1e-2 * np.sqrt((ref ** 2).mean())


def _fp8_stack(E, rows, cols, gen, all_codes_expert=None):
    w = torch.empty((E, rows, cols), dtype=torch.uint8, device=DEV)
    s = torch.empty((E, rows), dtype=torch.float32, device=DEV)
    for e in range(E):
        q, sc = inputs._fp8_quantise(torch.randn((rows, cols), generator=gen, device=DEV) * cols ** -0.5)
        w[e].copy_(q)
        s[e].copy_(sc)
    if all_codes_expert is not None:
        # every finite E4M3 code (NaN codes 0x7F / 0xFF excluded), cycling
        codes = torch.tensor([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=torch.uint8, device=DEV)
        n = rows * cols
        w[all_codes_expert].copy_(codes.repeat(n // len(codes) + 1)[:n].view(rows, cols))
        s[all_codes_expert].fill_(1.0 / 448.0)
    return w, s


TILES = [(32, 0), (128, 0), (256, 0), (32, 1), (128, 1), (256, 1)]


@pytest.mark.parametrize("bn,pair,fmt", [(bn, pr, f) for bn, pr in TILES for f in ("bf16", "fp8", "fp8conv")] +
                         [(160, 0, "fp8"), (160, 1, "fp8")])
def test_grouped_swiglu_every_tile_size(bn, pair, fmt, monkeypatch):
    # the same ragged groups through each tile-row count of both GEMMs, on
    # single CTAs and on CTA pairs (256 output channels per tile; 32-row
    # tiles on pairs with MOE_PAIR=2).  FP8 weights: on two-term E4M3 rows,
    # and on the E4M3 -> f16 weight converters (fp8conv)
    fp8 = fmt != "bf16"
    if fmt == "fp8conv":
        monkeypatch.setenv("MOE_FP8_CONVERT", "1")
    monkeypatch.setenv("MOE_BN_GATEUP", str(bn))
    monkeypatch.setenv("MOE_BN_DOWN", str(bn))
    monkeypatch.setenv("MOE_PAIR", str(2 if pair and bn == 32 else pair))  # 2: pairs at decode tiles too
    counts = np.array(GROUP_COUNTS["prefill_like"])
    E, d, f = len(counts), 256, 256
    R = int(counts.sum())
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    g = torch.Generator(device=DEV).manual_seed(bn)
    x = _bf16_rand((R, d), 1.0, g)
    p = api.problem(R, d, f, E, 1, wfmt="fp8" if fp8 else "bf16")
    if fp8:
        wg, sg = _fp8_stack(E, f, d, g)
        wu, su = _fp8_stack(E, f, d, g)
        wd, sd = _fp8_stack(E, d, f, g)
        ew = oracle.ExpertWeights("fp8", wg.cpu().numpy(), wu.cpu().numpy(), wd.cpu().numpy(),
                                  sg.cpu().numpy(), su.cpu().numpy(), sd.cpu().numpy())
    else:
        wg, wu = _bf16_rand((E, f, d), d ** -0.5, g), _bf16_rand((E, f, d), d ** -0.5, g)
        wd = _bf16_rand((E, d, f), d ** -0.5, g)
        sg = su = sd = None
        ew = oracle.ExpertWeights("bf16", inputs.to_numpy_stored(wg), inputs.to_numpy_stored(wu),
                                  inputs.to_numpy_stored(wd))
    info = api.moe_plan_info(p)
    assert info["bn_gateup"] == bn
    assert (info["pair_gateup"], info["pair_down"]) == (pair, pair)
    y = torch.full((R, d), float("nan"), dtype=torch.bfloat16, device=DEV)
    api.moe_grouped_swiglu(p, x, torch.from_numpy(offsets).to(DEV), wg, wu, wd, sg, su, sd, y, api.workspace_for(p))
    torch.cuda.synchronize()
    xf, got = _f64(x), _f64(y)
    ref = np.zeros_like(got)
    for e in range(E):
        a, b = offsets[e], offsets[e + 1]
        if b > a:
            ref[a:b] = oracle.swiglu_expert(xf[a:b], *ew.get(e))
    assert np.isfinite(got).all()
    assert np.abs(got - ref).max() <= (FP8_TOL if fp8 else BF16_TOL) * np.abs(ref).max()
    assert np.sqrt(((got - ref) ** 2).mean()) <= 1e-2 * np.sqrt((ref ** 2).mean())


@pytest.mark.parametrize("kind", ["ragged", "decode"])
@pytest.mark.parametrize("convert", [False, True])
def test_grouped_swiglu_fp8_weights(kind, convert, monkeypatch):
    if convert:
        monkeypatch.setenv("MOE_FP8_CONVERT", "1")
    counts = np.array(GROUP_COUNTS[kind])
    E, d, f = len(counts), 256, 384
    R = int(counts.sum())
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    g = torch.Generator(device=DEV).manual_seed(77)
    x = _bf16_rand((R, d), 1.0, g)
    busy = int(np.argmax(counts))
    wg, sg = _fp8_stack(E, f, d, g, all_codes_expert=busy)
    wu, su = _fp8_stack(E, f, d, g)
    wd, sd = _fp8_stack(E, d, f, g, all_codes_expert=busy)
    p = api.problem(R, d, f, E, 1, wfmt="fp8")
    y = torch.full((R, d), float("nan"), dtype=torch.bfloat16, device=DEV)
    api.moe_grouped_swiglu(p, x, torch.from_numpy(offsets).to(DEV), wg, wu, wd, sg, su, sd, y, api.workspace_for(p))
    torch.cuda.synchronize()
    ew = oracle.ExpertWeights("fp8", wg.cpu().numpy(), wu.cpu().numpy(), wd.cpu().numpy(),
                              sg.cpu().numpy(), su.cpu().numpy(), sd.cpu().numpy())
    xf, got = _f64(x), _f64(y)
    ref = np.zeros_like(got)
    for e in range(E):
        a, b = offsets[e], offsets[e + 1]
        if b > a:
            ref[a:b] = oracle.swiglu_expert(xf[a:b], *ew.get(e))
    assert np.isfinite(got).all()
    assert np.abs(got - ref).max() <= FP8_TOL * np.abs(ref).max()
    # the dequantisation is exact: only the bf16 roundings of h and y remain
    for e in range(E):
        a, b = offsets[e], offsets[e + 1]
        if b > a:
            rel = np.sqrt(((got[a:b] - ref[a:b]) ** 2).mean()) / np.sqrt((ref[a:b] ** 2).mean())
            assert rel <= 1e-2, f"expert {e}: relative rms error {rel:.3g}"


# ---------------------------------------------------------------------------
# whole layer
# ---------------------------------------------------------------------------

# Logit error the layer's router may have against the oracle's float64
# logits (test_router_logits_and_choice: <= 1e-5 * max|l|); the routing of
# every token is checked within twice that band.
LOGIT_ERR = 1e-5


def _layer_check(shape, seed, tol, x=None, per_token=False):
    """The layer through the C ABI against the oracle on EVERY token: the
    routing within the logit-error band (helpers.check_routing_within_tie_band),
    counts, and the output against the oracle's grouped formulation under the
    device's (verified) routing.  ``per_token``: each token's max|err| is held
    to tol times its own max|ref| (rows of very different magnitudes), else
    the whole output's max|err| to tol times its max|ref|."""
    case = inputs.make_case(shape, seed, DEV)
    if x is not None:
        case["x"] = x
    p = api.problem_of(shape)
    out, idx, w, counts = api.layer_forward(p, case, want_routing=True)
    torch.cuda.synchronize()
    x, wr, b, ew, sh = helpers.oracle_inputs(case, shape)
    lg = oracle.router_logits(x, wr, b)
    idx_g = idx.cpu().numpy()
    w_g = w.cpu().numpy().astype(np.float64)
    helpers.check_routing_within_tie_band(lg, shape.k, idx_g, w_g, 2 * LOGIT_ERR * np.abs(lg).max(), LOGIT_ERR)
    cnt_g = counts.cpu().numpy()
    assert cnt_g.sum() == shape.T * shape.k
    assert np.array_equal(cnt_g, np.bincount(idx_g.ravel(), minlength=shape.E))
    # output: the oracle's layer under the device's routing, every token
    # (decoded experts held ahead: at most about 6 GB of float64 weights)
    ahead = int(max(1, min(12, 6e9 // (3 * shape.ffn * shape.d * 8))))
    hook = helpers.PrefetchedExperts(ew, np.unique(idx_g), ahead=ahead)
    try:
        ref, _, _ = oracle.moe_forward_grouped(x, wr, ew, shape.k, bias=b, shared=sh, routing=(idx_g, w_g),
                                               expert_hook=hook, act8=shape.wfmt == "fp8a8")
    finally:
        hook.close()
    got = helpers.decode_act(out, shape.act)
    assert np.isfinite(got).all()
    if per_token:
        err = np.abs(got - ref).max(axis=1)
        lim = tol * np.abs(ref).max(axis=1)
        bad = np.nonzero(err > lim)[0]
        assert bad.size == 0, f"tokens {bad[:8]}: max|err| {err[bad[:8]]} vs limit {lim[bad[:8]]}"
    else:
        err = np.abs(got - ref).max()
        assert err <= tol * np.abs(ref).max(), f"max|err| {err:.3g} vs max|ref| {np.abs(ref).max():.3g}"
    return case


def test_layer_toy_f32():
    shape = inputs.WORKLOADS["toy_f32"]
    _layer_check(shape, 0, F32_TOL)


def test_worked_example_combine_on_gpu():
    # the page: T1 -> 0.7 * E1(T1) + 0.3 * E3(T1); run the layer's grouped
    # expert and combine entry points on the worked example's routing
    g, idx_ref, w_ref, groups = helpers.worked_example()
    T, E, k = g["T"], g["E"], g["k"]
    d, f = 128, 128
    gen = torch.Generator(device=DEV).manual_seed(11)
    x = _bf16_rand((T, d), 1.0, gen)
    wg, wu, wd = (_bf16_rand((E, f, d), d ** -0.5, gen), _bf16_rand((E, f, d), d ** -0.5, gen),
                  _bf16_rand((E, d, f), d ** -0.5, gen))
    p = api.problem(T, d, f, E, k)
    ws = api.workspace_for(p)
    idx_t = torch.from_numpy(idx_ref).to(DEV)
    counts = torch.empty(E, dtype=torch.int32, device=DEV)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=DEV)
    perm = torch.empty(T * k, dtype=torch.int32, device=DEV)
    inv = torch.empty(T * k, dtype=torch.int32, device=DEV)
    x_perm = torch.empty((T * k, d), dtype=torch.bfloat16, device=DEV)
    y = torch.empty((T * k, d), dtype=torch.bfloat16, device=DEV)
    out = torch.empty((T, d), dtype=torch.bfloat16, device=DEV)
    api.moe_permute(p, idx_t, x, counts, offsets, perm, inv, x_perm, ws)
    api.moe_grouped_swiglu(p, x_perm, offsets, wg, wu, wd, None, None, None, y, ws)
    api.moe_combine(p, y, inv, torch.from_numpy(w_ref.astype(np.float32)).to(DEV), None, out)
    torch.cuda.synchronize()
    xf = _f64(x)
    c = g["combine"]["T1"]
    e1 = oracle.swiglu_expert(xf[:1], _f64(wg[0]), _f64(wu[0]), _f64(wd[0]))[0]
    e3 = oracle.swiglu_expert(xf[:1], _f64(wg[2]), _f64(wu[2]), _f64(wd[2]))[0]
    ref = c["E1"] * e1 + c["E3"] * e3
    got = _f64(out)[0]
    assert np.abs(got - ref).max() <= BF16_TOL * np.abs(ref).max()


@pytest.mark.parametrize("T,d,f,E,k", [(300, 256, 384, 16, 4), (7, 128, 256, 8, 2), (1, 256, 128, 4, 4),
                                       (2100, 128, 128, 32, 1),
                                       # the largest expert count and top-k the library takes
                                       (64, 128, 128, 1024, 32), (3, 256, 128, 1024, 32)])
def test_layer_bf16_small_multi_tile(T, d, f, E, k):
    shape = inputs.MoEShape("small", T=T, d=d, ffn=f, E=E, k=k)
    _layer_check(shape, 1, BF16_TOL)


@pytest.mark.parametrize("T", [1, 8, 32, 64])
def test_layer_mixtral_shaped(T):
    _layer_check(inputs.WORKLOADS["mixtral_8x7b"].with_T(T), 0, BF16_TOL)


@pytest.mark.parametrize("T", [1, 16, 128])
def test_layer_qwen3_30b_a3b_shaped_decode(T):
    _layer_check(inputs.WORKLOADS["qwen3_30b_a3b"].with_T(T), 0, BF16_TOL)


def test_layer_qwen3_30b_a3b_shaped_prefill():
    # all 8192 tokens (65 536 routed rows) against the oracle
    shape = inputs.WORKLOADS["qwen3_30b_a3b_prefill"]
    case = _layer_check(shape, 0, BF16_TOL)
    # the skewed load reached the device: hottest expert holds several times the mean
    p = api.problem_of(shape)
    _, _, _, counts = api.layer_forward(p, case, want_routing=True)
    c = counts.cpu().numpy()
    assert c.max() / c.mean() > 4.0


@pytest.mark.parametrize("T", [1, 64, 4096])
def test_layer_deepseek_v3_shaped_fp8_with_shared_expert(T):
    # every token, at full size: d=7168, 256 FP8 experts, top-8, the bf16
    # shared expert
    _layer_check(inputs.WORKLOADS["deepseek_v3"].with_T(T), 0, FP8_TOL)


@pytest.mark.parametrize("wfmt", ["fp8a8", "mxfp4"])
def test_layer_deepseek_v3_shaped_other_weight_modes(wfmt):
    # the benchmarked FP8-activation and MXFP4 modes at the full
    # DeepSeek-V3 shape (d=7168, 256 experts, the shared expert), every token
    shape = dataclasses.replace(inputs.WORKLOADS["deepseek_v3"].with_T(64), name=f"deepseek_v3_{wfmt}",
                                wfmt=wfmt)
    _layer_check(shape, 0, FP8_TOL)


@pytest.mark.parametrize("T", [4, 2048])
def test_layer_fp8_weights_with_outlier_token_rows(T):
    # bf16 token rows far outside f16's range (outlier elements 1e3 .. 1e5,
    # whole rows scaled by up to 1e4, and rows scaled down to 1e-6): the
    # FP8-weight mode carries bf16 rows as exact two-term E4M3 rows, so every
    # token's output matches the oracle to the FP8 tolerance of its own size
    # (T=4: decode tiles; T=2048: 256 rows per expert, CTA-pair prefill tiles)
    shape = inputs.MoEShape("outliers", T=T, d=1024, ffn=512, E=64, k=8, ffn_shared=512, wfmt="fp8")
    g = torch.Generator(device=DEV).manual_seed(T)
    x = torch.randn((T, shape.d), generator=g, device=DEV)
    for t in range(T):
        kind, n = t % 4, t // 4
        if kind == 0:    # one element at 1e5 beside N(0,1) values
            x[t, (t * 37) % shape.d] = (-1) ** n * 1e5
        elif kind == 1:  # one element at 1e3 .. 1e4
            x[t, (t * 37) % shape.d] = 10.0 ** (3 + n % 2)
        elif kind == 2:  # the whole row scaled up, to 1e4
            x[t] *= 10.0 ** (1 + n % 4)
        else:            # the whole row scaled down
            x[t] *= 1e-6
    x = x.to(torch.bfloat16)
    assert x.float().abs().max() >= 9e4  # (1e5 in bf16 is 99840)
    _layer_check(shape, 5, FP8_TOL, x=x, per_token=True)


def test_layer_forward_captured_in_a_cuda_graph_with_stage_timer():
    # the whole layer is enqueued without host synchronisation, so it can be
    # captured; the stage timer's events become timestamp nodes
    shape = inputs.MoEShape("small", T=40, d=256, ffn=384, E=16, k=4)
    case = inputs.make_case(shape, 2, DEV)
    p = api.problem_of(shape)
    ws = api.workspace_for(p)
    direct = api.layer_forward(p, case, workspace=ws)
    out = torch.empty_like(direct)
    timer = api.StageTimer()
    api.layer_forward(p, case, out=out, workspace=ws, timer=timer)  # warm (function attributes)
    torch.cuda.synchronize()
    out.zero_()
    g = torch.cuda.CUDAGraph()
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g, stream=stream):
            api.layer_forward(p, case, out=out, workspace=ws, timer=timer)
    torch.cuda.current_stream().wait_stream(stream)
    g.replay()
    torch.cuda.synchronize()
    ms = timer.read()
    assert set(ms) == set(api.STAGES) and all(v >= 0.0 for v in ms.values())
    assert ms["gate_up"] > 0.0 and ms["down"] > 0.0
    assert torch.equal(out, direct)  # deterministic: same bits as the direct call
    timer.close()


@pytest.mark.parametrize("splits,bn,d,pair", [(1, 0, 512, 0), (3, 0, 512, 0), (8, 0, 512, 0), (3, 256, 512, 0),
                                               (8, 0, 640, 0), (3, 0, 512, 1), (8, 0, 512, 1)])
@pytest.mark.parametrize("wfmt", ["bf16", "fp8", "fp8conv", "fp8a8"])
def test_layer_gateup_split_k(splits, bn, d, pair, wfmt, monkeypatch):
    # the gate/up GEMM split along its reduction: fp32 partials, then an
    # in-order sum and SiLU*mul pass (chosen automatically at tiny batches);
    # bn=256 forces the 256-row tile through the same partials; ceil-sized
    # splits can leave the last ones without k-blocks (d=640 in 64-element
    # blocks over 8 splits, d=512 in the 128-element FP8 decode blocks)
    monkeypatch.setenv("MOE_SPLITS_GATEUP", str(splits))
    monkeypatch.setenv("MOE_PAIR", str(2 * pair))  # 2: FP8 decode tiles on CTA pairs
    if bn:
        monkeypatch.setenv("MOE_BN_GATEUP", str(bn))
    if wfmt == "fp8conv":
        monkeypatch.setenv("MOE_FP8_CONVERT", "1")
    wfmt = "fp8" if wfmt == "fp8conv" else wfmt
    shape = inputs.MoEShape("small", T=5, d=d, ffn=256, E=16, k=4, ffn_shared=256 if wfmt != "bf16" else 0,
                            wfmt=wfmt)
    info = api.moe_plan_info(api.problem_of(shape))
    assert info["splits_gateup"] == splits
    # decode tiles on CTA pairs (MOE_PAIR=2): split-K partials and the fused
    # finalize per CTA of the pair
    assert info["pair_gateup"] == (pair if not bn else 0)
    _layer_check(shape, 4, FP8_TOL if wfmt != "bf16" else BF16_TOL)


@pytest.mark.parametrize("bn,pair,wfmt", [(bn, pr, w) for bn, pr in ((128, 0), (128, 1), (256, 0), (256, 1))
                                           for w in ("bf16", "fp8", "fp8scatter", "fp8conv", "fp8a8")] +
                         [(160, pr, w) for pr in (0, 1) for w in ("fp8", "fp8scatter")] +
                         [(bn, 1, "fp8wide") for bn in (128, 160, 256)] + [(128, 1, "fp8narrow")])
def test_layer_gathered_rows_every_tile(bn, pair, wfmt, monkeypatch):
    # the gate/up GEMM gathers its token rows (cp.async by the producer warp
    # for tiles of >= 128 rows), on single CTAs and on CTA pairs, with groups
    # spanning several tiles and ragged tails.  FP8 weights: the two-term
    # rows gathered per token, or scattered into permuted order (tile loads;
    # fp8scatter), or the weight converters (fp8conv)
    if wfmt == "fp8scatter":
        monkeypatch.setenv("MOE_X2_SCATTER", "1")
        wfmt = "fp8"
    if wfmt in ("fp8wide", "fp8narrow"):  # 256 elements of K per stage in both GEMMs, or in neither
        monkeypatch.setenv("MOE_X2_WIDE", "3" if wfmt == "fp8wide" else "0")
        wfmt = "fp8"
    monkeypatch.setenv("MOE_BN_GATEUP", str(bn))
    monkeypatch.setenv("MOE_BN_DOWN", str(bn))
    monkeypatch.setenv("MOE_PAIR", str(pair))
    monkeypatch.setenv("MOE_SPLITS_GATEUP", "1")  # (pairs take unsplit gate/up GEMMs)
    if wfmt == "fp8conv":
        monkeypatch.setenv("MOE_FP8_CONVERT", "1")
    wfmt = "fp8" if wfmt == "fp8conv" else wfmt
    shape = inputs.MoEShape("gathered", T=300, d=512, ffn=512, E=8, k=2, wfmt=wfmt,
                            ffn_shared=256 if wfmt != "bf16" else 0)
    info = api.moe_plan_info(api.problem_of(shape))
    assert (info["bn_gateup"], info["pair_gateup"]) == (bn, pair)
    _layer_check(shape, 3, FP8_TOL if wfmt != "bf16" else BF16_TOL)


def test_layer_empty_batch():
    shape = inputs.WORKLOADS["qwen3_30b_a3b"].with_T(0)
    case = inputs.make_weights(shape, 0, DEV)
    case["x"] = torch.empty((0, shape.d), dtype=torch.bfloat16, device=DEV)
    out = api.layer_forward(api.problem_of(shape), case, out=torch.empty((0, shape.d), dtype=torch.bfloat16, device=DEV),
                            workspace=torch.empty(16, dtype=torch.uint8, device=DEV))
    assert out.shape == (0, shape.d)


def test_workspace_too_small_is_rejected():
    shape = inputs.MoEShape("small", T=8, d=128, ffn=128, E=4, k=2)
    case = inputs.make_case(shape, 0, DEV)
    p = api.problem_of(shape)
    with pytest.raises(api.MoEError) as e:
        api.layer_forward(p, case, workspace=torch.empty(64, dtype=torch.uint8, device=DEV))
    assert e.value.status == api.ERR_WORKSPACE


# ---------------------------------------------------------------------------
# failure detection: a bounded wait that expires
# ---------------------------------------------------------------------------

def test_bounded_wait_expires_cleanly_and_context_survives():
    api.moe_selftest_bounded_wait(2_000_000)  # 2 ms on a barrier nothing arrives at
    assert api.moe_read_device_status() == api.ERR_DEVICE_TIMEOUT
    assert api.moe_read_device_status() == 0
    # the context is still usable: a normal layer runs and matches
    shape = inputs.MoEShape("small", T=20, d=128, ffn=256, E=8, k=2)
    _layer_check(shape, 3, BF16_TOL)


@pytest.mark.parametrize("shape", [
    inputs.WORKLOADS["toy_f32"],                                    # CUDA-core path
    inputs.WORKLOADS["qwen3_30b_a3b"].with_T(1),                    # fused top-k, split-K gate/up
    inputs.MoEShape("ds_small", T=2, d=1024, ffn=512, E=64, k=8, ffn_shared=512, wfmt="fp8"),
    inputs.MoEShape("ds_small_act8", T=2, d=1024, ffn=512, E=64, k=8, ffn_shared=512, wfmt="fp8a8"),
    inputs.MoEShape("ds_small_mx", T=2, d=1024, ffn=512, E=64, k=8, ffn_shared=512, wfmt="mxfp4"),
    inputs.MoEShape("chunked", T=400, d=256, ffn=256, E=32, k=8),   # chunked permutation
], ids=lambda s: s.name)
def test_layer_launch_count_matches_the_kernels_launched(shape):
    # moe_layer_launch_count (the bench's gpu_launches) against the kernel
    # nodes of one layer call captured into a CUDA graph (driver API)
    import ctypes
    cu = ctypes.CDLL("libcuda.so.1")
    case = inputs.make_case(shape, 0, DEV)
    p = api.problem_of(shape)
    ws = api.workspace_for(p)
    out = api.layer_forward(p, case, workspace=ws)  # warm (function attributes)
    torch.cuda.synchronize()
    stream = torch.cuda.Stream()
    h = ctypes.c_void_p(stream.cuda_stream)
    assert cu.cuStreamBeginCapture_v2(h, ctypes.c_int(2)) == 0  # relaxed capture mode
    try:
        api.layer_forward(p, case, out=out, workspace=ws, stream=stream)
    finally:
        graph = ctypes.c_void_p()
        assert cu.cuStreamEndCapture(h, ctypes.byref(graph)) == 0
    n = ctypes.c_size_t(0)
    assert cu.cuGraphGetNodes(graph, None, ctypes.byref(n)) == 0
    nodes = (ctypes.c_void_p * n.value)()
    assert cu.cuGraphGetNodes(graph, nodes, ctypes.byref(n)) == 0
    kinds = []
    for nd in nodes:
        t = ctypes.c_int(-1)
        assert cu.cuGraphNodeGetType(ctypes.c_void_p(nd), ctypes.byref(t)) == 0
        kinds.append(t.value)
    cu.cuGraphDestroy(graph)
    assert kinds.count(0) == api.moe_layer_launch_count(p), kinds  # 0: kernel node


@pytest.mark.parametrize("shape", [
    inputs.WORKLOADS["mixtral_8x7b"].with_T(64),
    inputs.WORKLOADS["qwen3_30b_a3b"].with_T(1),
    inputs.WORKLOADS["deepseek_v3"].with_T(4096),
    inputs.WORKLOADS["toy_f32"],
], ids=lambda s: f"{s.name}_T{s.T}")
def test_device_planning_is_the_host_planning_at_the_device_sm_count(shape):
    # the device entry points answer what the device-free ones answer for
    # this device's multiprocessor count
    p = api.problem_of(shape)
    sms = torch.cuda.get_device_properties(DEV).multi_processor_count
    assert api.moe_plan_info(p) == api.moe_plan_info_for(p, sms)
    assert api.moe_layer_launch_count(p) == api.moe_layer_launch_count_for(p, sms)
    assert api.moe_workspace_size(p) == api.moe_workspace_size_for(p, sms)
