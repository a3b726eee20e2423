"""The Python binding's size checks (no GPU): every tensor the C entry points
would read or write is checked against the problem's sizes and element size
before any pointer is taken, so a short or mistyped tensor is a ValueError
on the host instead of an out-of-bounds access on the device.  Correctly
sized CPU tensors get past the checks and stop at the device-tensor check,
before anything reaches the library."""

import pytest
import torch

from routed_expert_ffn_gemm_gb300 import api, inputs

SMALL = [
    inputs.WORKLOADS["toy_f32"],
    inputs.MoEShape("b", T=5, d=256, ffn=128, E=4, k=2, ffn_shared=128),
    inputs.MoEShape("z", T=6, d=256, ffn=128, E=8, k=2),  # (with a router bias: _case)
    inputs.MoEShape("f8", T=3, d=256, ffn=128, E=4, k=2, ffn_shared=128, wfmt="fp8"),
    inputs.MoEShape("a8", T=3, d=256, ffn=128, E=4, k=2, ffn_shared=128, wfmt="fp8a8"),
    inputs.MoEShape("mx", T=3, d=256, ffn=128, E=4, k=2, ffn_shared=128, wfmt="mxfp4"),
]


def _case(shape):
    case = inputs.make_case(shape, 0, "cpu")
    if shape.name == "z":
        case["router_bias"] = inputs.zipf_bias(shape, 0, alpha=1.0)
    return case


def _layer_args(shape, case):
    p = api.problem_of(shape)
    out = torch.empty((shape.T, shape.d), dtype=case["x"].dtype)
    idx = torch.empty((shape.T, shape.k), dtype=torch.int32)
    w = torch.empty((shape.T, shape.k), dtype=torch.float32)
    counts = torch.empty(shape.E, dtype=torch.int32)
    ws = torch.empty(16, dtype=torch.uint8)
    return [p, case["x"], case["w_router"], case["router_bias"], case["w_gate"], case["w_up"], case["w_down"],
            case["s_gate"], case["s_up"], case["s_down"], case["w_shared_gate"], case["w_shared_up"],
            case["w_shared_down"], out, idx, w, counts, ws]


NAMES = ["p", "x", "w_router", "router_bias", "w_gate", "w_up", "w_down", "s_gate", "s_up", "s_down",
         "w_shared_gate", "w_shared_up", "w_shared_down", "out", "topk_idx_out", "topk_w_out", "counts_out",
         "workspace"]


@pytest.mark.parametrize("shape", SMALL, ids=lambda s: s.name)
def test_generated_cases_pass_the_checks(shape):
    # the seeded generators' tensors are what the checks expect for every
    # weight mode; the call then stops at the device-tensor check
    case = _case(shape)
    with pytest.raises(ValueError, match="device tensors"):
        api.moe_layer_forward(*_layer_args(shape, case))


@pytest.mark.parametrize("shape", SMALL, ids=lambda s: s.name)
def test_short_or_mistyped_tensors_are_refused(shape):
    case = _case(shape)
    args = _layer_args(shape, case)
    for i, name in enumerate(NAMES):
        t = args[i]
        if name in ("p", "workspace") or t is None:
            continue
        short = args.copy()
        short[i] = t.reshape(-1)[:-1]
        with pytest.raises(ValueError, match=f"^{name}: "):
            api.moe_layer_forward(*short)
        wide = args.copy()
        wide[i] = torch.empty(t.numel(), dtype=torch.float64)
        with pytest.raises(ValueError, match=f"^{name}: "):
            api.moe_layer_forward(*wide)


def test_index_arrays_must_be_int32():
    shape = SMALL[1]
    p = api.problem_of(shape)
    R = shape.T * shape.k
    i32 = lambda n: torch.empty(n, dtype=torch.int32)  # noqa: E731
    with pytest.raises(ValueError, match="topk_idx"):
        api.moe_permute(p, torch.empty(R, dtype=torch.float32), None, i32(shape.E), i32(shape.E + 1),
                        i32(R), i32(R), None, None)
    with pytest.raises(ValueError, match="offsets"):
        api.moe_permute(p, i32(R), None, i32(shape.E), i32(shape.E), i32(R), i32(R), None, None)
    with pytest.raises(ValueError, match="inv_row"):
        api.moe_combine(p, torch.empty((R, shape.d), dtype=torch.bfloat16), torch.empty(R, dtype=torch.int64),
                        torch.empty(R), None, torch.empty((shape.T, shape.d), dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="logits_in"):
        api.moe_router_topk(p, None, None, None, torch.empty((shape.T, shape.E), dtype=torch.float64), None,
                            i32(R), torch.empty(R))


def test_grouped_and_quantiser_sizes():
    shape = SMALL[5]  # MXFP4
    case = inputs.make_case(shape, 0, "cpu")
    p = api.problem(shape.T * shape.k, shape.d, shape.ffn, shape.E, 1, wfmt="mxfp4")
    R = shape.T * shape.k
    x = torch.empty((R, shape.d), dtype=torch.bfloat16)
    off = torch.empty(shape.E + 1, dtype=torch.int32)
    y = torch.empty((R, shape.d), dtype=torch.bfloat16)
    w = [case[n] for n in ("w_gate", "w_up", "w_down", "s_gate", "s_up", "s_down")]
    with pytest.raises(ValueError, match="device tensors"):
        api.moe_grouped_swiglu(p, x, off, *w, y, None)
    # the block scales of the down matrix: [E, ffn/32, d] bytes
    bad = w.copy()
    bad[5] = case["s_down"][:, :-1]
    with pytest.raises(ValueError, match="s_down"):
        api.moe_grouped_swiglu(p, x, off, *bad, y, None)
    with pytest.raises(ValueError, match="y_perm"):
        api.moe_grouped_swiglu(p, x, off, *w, y[:-1], None)
    xq = torch.empty((4, 128), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="codes"):
        api.moe_quantize_rows_e4m3(xq, torch.empty((4, 127), dtype=torch.uint8), torch.empty(4))
    with pytest.raises(ValueError, match="scales"):
        api.moe_quantize_rows_e4m3(xq, torch.empty((4, 128), dtype=torch.uint8), torch.empty(3))
    with pytest.raises(ValueError, match="device tensors"):
        api.moe_quantize_rows_e4m3(xq, torch.empty((4, 128), dtype=torch.uint8), torch.empty(4))
