"""No kernel writes outside its buffers: every output and the workspace sit
inside canary-filled guard regions (tests/guard.py), and after each call the
guards must be intact.  The workspace guard checks that the library stays
within moe_workspace_size; the output guards check every row, tile and
split-K partial store.  Workloads are those the parity tests run (decode,
split-K, CTA pairs, FP8 activations, MXFP4, the chunked permutation, the
skewed prefill), so this adds no new shapes, only the checks."""

import numpy as np
import pytest
import torch

from routed_expert_ffn_gemm_gb300 import api, build, inputs
from tests.guard import Guarded
from tests.test_gpu_parity import DEV, GROUP_COUNTS, _bf16_rand

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _library():
    build.build()
    api._lib()
    yield
    assert api.moe_read_device_status() == 0, "a kernel recorded an error"


def _all_intact(**bufs):
    bad = {n: g.first_overwrite() for n, g in bufs.items() if not g.intact()}
    assert not bad, f"writes outside the buffer (byte offset from its start): {bad}"


LAYERS = [
    inputs.WORKLOADS["toy_f32"],
    inputs.WORKLOADS["qwen3_30b_a3b"].with_T(1),
    inputs.WORKLOADS["mixtral_8x7b"].with_T(64),
    inputs.WORKLOADS["qwen3_30b_a3b_prefill"],
    inputs.MoEShape("chunked", T=400, d=256, ffn=256, E=32, k=8),
    inputs.MoEShape("gathered", T=300, d=512, ffn=512, E=8, k=2, wfmt="fp8", ffn_shared=256),
    inputs.MoEShape("ds_small", T=2, d=1024, ffn=512, E=64, k=8, ffn_shared=512, wfmt="fp8"),
    inputs.MoEShape("ds_like_act8", T=64, d=1024, ffn=512, E=64, k=8, ffn_shared=512, wfmt="fp8a8"),
    inputs.MoEShape("ds_like_mx", T=64, d=1024, ffn=512, E=64, k=8, ffn_shared=512, wfmt="mxfp4"),
]


@pytest.mark.parametrize("shape", LAYERS, ids=lambda s: f"{s.name}_T{s.T}")
def test_layer_writes_stay_inside_outputs_and_workspace(shape):
    case = inputs.make_case(shape, 0, DEV)
    p = api.problem_of(shape)
    T, k, E = shape.T, shape.k, shape.E
    out = Guarded((T, shape.d), case["x"].dtype, DEV)
    idx = Guarded((T, k), torch.int32, DEV)
    w = Guarded((T, k), torch.float32, DEV)
    counts = Guarded((E,), torch.int32, DEV)
    ws = Guarded((api.moe_workspace_size(p),), torch.uint8, DEV)
    api.moe_layer_forward(p, case["x"], case["w_router"], case["router_bias"], case["w_gate"], case["w_up"],
                          case["w_down"], case["s_gate"], case["s_up"], case["s_down"], case["w_shared_gate"],
                          case["w_shared_up"], case["w_shared_down"], out.t, idx.t, w.t, counts.t, ws.t)
    torch.cuda.synchronize()
    assert api.moe_read_device_status() == 0
    _all_intact(out=out, topk_idx=idx, topk_w=w, counts=counts, workspace=ws)
    # the guarded call computed the layer: the same routing and (to rounding)
    # the same output as a call on plain buffers
    ref, ridx, _, rcounts = api.layer_forward(p, case, want_routing=True)
    torch.cuda.synchronize()
    assert torch.equal(idx.t, ridx) and torch.equal(counts.t, rcounts)
    got, want = out.t.double(), ref.double()
    assert torch.isfinite(got).all()
    assert (got - want).abs().max() <= 1e-2 * want.abs().max()


def test_permute_writes_stay_inside():
    T, E, k, d = 400, 32, 8, 128  # chunked path (T*k > 2048)
    rng = np.random.default_rng(1)
    idx = torch.from_numpy(np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)).to(DEV)
    g = torch.Generator(device=DEV).manual_seed(1)
    x = _bf16_rand((T, d), 1.0, g)
    p = api.problem(T, d, 128, E, k)
    R = T * k
    bufs = dict(counts=Guarded((E,), torch.int32, DEV), offsets=Guarded((E + 1,), torch.int32, DEV),
                perm=Guarded((R,), torch.int32, DEV), inv=Guarded((R,), torch.int32, DEV),
                x_perm=Guarded((R, d), torch.bfloat16, DEV),
                workspace=Guarded((api.moe_workspace_size(p),), torch.uint8, DEV))
    api.moe_permute(p, idx, x, bufs["counts"].t, bufs["offsets"].t, bufs["perm"].t, bufs["inv"].t,
                    bufs["x_perm"].t, bufs["workspace"].t)
    torch.cuda.synchronize()
    assert api.moe_read_device_status() == 0
    _all_intact(**bufs)
    assert int(bufs["counts"].t.sum()) == R


@pytest.mark.parametrize("wfmt", ["bf16", "fp8a8", "mxfp4"])
def test_grouped_writes_stay_inside(wfmt):
    counts = np.array(GROUP_COUNTS["ragged"])
    E, d, f = len(counts), 256, 256
    R = int(counts.sum())
    offsets = torch.from_numpy(np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)).to(DEV)
    shape = inputs.MoEShape("grouped", T=R, d=d, ffn=f, E=E, k=1, wfmt=wfmt)
    wts = inputs.make_weights(shape, 0, DEV)
    g = torch.Generator(device=DEV).manual_seed(2)
    x = _bf16_rand((R, d), 1.0, g)
    p = api.problem(R, d, f, E, 1, wfmt=wfmt)
    y = Guarded((R, d), torch.bfloat16, DEV)
    ws = Guarded((api.moe_workspace_size(p),), torch.uint8, DEV)
    api.moe_grouped_swiglu(p, x, offsets, wts["w_gate"], wts["w_up"], wts["w_down"], wts["s_gate"], wts["s_up"],
                           wts["s_down"], y.t, ws.t)
    torch.cuda.synchronize()
    assert api.moe_read_device_status() == 0
    _all_intact(y=y, workspace=ws)
    assert torch.isfinite(y.t.float()).all()


def test_combine_router_and_quantiser_writes_stay_inside():
    T, k, d, E = 37, 4, 256, 128
    R = T * k
    g = torch.Generator(device=DEV).manual_seed(3)
    y = torch.randn((R, d), generator=g, device=DEV).to(torch.bfloat16)
    inv = torch.from_numpy(np.random.default_rng(3).permutation(R).astype(np.int32)).to(DEV)
    tw = torch.full((T, k), 1.0 / k, dtype=torch.float32, device=DEV)
    p = api.problem(T, d, 128, 8, k)
    out = Guarded((T, d), torch.bfloat16, DEV)
    api.moe_combine(p, y, inv, tw, None, out.t)
    # router on the tensor cores (bf16, E % 128 == 0, T >= 256), logits out
    Tr, dr, kr = 300, 2048, 8
    x = torch.randn((Tr, dr), generator=g, device=DEV).to(torch.bfloat16)
    wr = (torch.randn((E, dr), generator=g, device=DEV) / dr ** 0.5).to(torch.bfloat16)
    pr = api.problem(Tr, dr, 128, E, kr)
    logits = Guarded((Tr, E), torch.float32, DEV)
    idx = Guarded((Tr, kr), torch.int32, DEV)
    w = Guarded((Tr, kr), torch.float32, DEV)
    api.moe_router_topk(pr, x, wr, None, None, logits.t, idx.t, w.t)
    # per-row E4M3 codes and scales
    xq = torch.randn((T, 1024), generator=g, device=DEV).to(torch.bfloat16)
    codes = Guarded((T, 1024), torch.uint8, DEV)
    scales = Guarded((T,), torch.float32, DEV)
    api.moe_quantize_rows_e4m3(xq, codes.t, scales.t)
    torch.cuda.synchronize()
    assert api.moe_read_device_status() == 0
    _all_intact(out=out, logits=logits, topk_idx=idx, topk_w=w, codes=codes, scales=scales)
