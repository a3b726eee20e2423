"""The C-ABI library loads and exports every entry point include/moe.h
declares; host-side argument validation answers without a GPU (no compute
call is made here)."""

import ctypes
import os
import re

import pytest

from routed_expert_ffn_gemm_gb300 import api, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return api._lib()


def declared_entry_points():
    with open(os.path.join(ROOT, "include", "moe.h")) as f:
        text = f.read()
    return re.findall(r"MOE_API\s+[\w\s\*]+?\b(moe_\w+)\s*\(", text)


def test_header_declares_the_boundary():
    names = set(declared_entry_points())
    for n in ("moe_router_topk", "moe_permute", "moe_grouped_swiglu", "moe_combine", "moe_layer_forward",
              "moe_workspace_size", "moe_read_device_status", "moe_status_string"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    names = declared_entry_points()
    assert names
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/moe.h but not exported"
    assert set(names) == set(api.EXPORTS), "binding and header disagree"


def _header_arity():
    with open(os.path.join(ROOT, "include", "moe.h")) as f:
        text = f.read()
    out = {}
    for m in re.finditer(r"MOE_API\s+[\w\s\*]+?\b(moe_\w+)\s*\(([^;]*?)\)\s*;", text, re.S):
        params = m.group(2).strip()
        out[m.group(1)] = 0 if params in ("", "void") else params.count(",") + 1
    return out


def test_binding_arity_matches_header():
    arity = _header_arity()
    assert set(arity) == set(api.EXPORTS)
    for name, n in arity.items():
        assert len(api._SIGS[name]) == n, f"{name}: header has {n} parameters, binding {len(api._SIGS[name])}"


def test_abi_version_and_status_strings(lib):
    assert api.moe_abi_version() == 5
    assert api.moe_status_string(0) == "MOE_OK"
    assert api.moe_status_string(api.ERR_DEVICE_TIMEOUT) == "MOE_ERR_DEVICE_TIMEOUT"
    assert api.moe_status_string(-99) == "MOE_ERR_UNKNOWN"


def _ws_status(lib, p):
    n = ctypes.c_size_t(0)
    return lib.moe_workspace_size(ctypes.byref(p), ctypes.byref(n))


@pytest.mark.parametrize("kw,want", [
    (dict(T=4, d=128, ffn=256, E=4, k=5), api.ERR_INVALID_ARG),          # k > E
    (dict(T=-1, d=128, ffn=256, E=4, k=2), api.ERR_INVALID_ARG),         # negative T
    (dict(T=4, d=0, ffn=256, E=4, k=2), api.ERR_INVALID_ARG),            # empty hidden
    (dict(T=4, d=128, ffn=256, E=2048, k=2), api.ERR_UNSUPPORTED),       # E > 1024
    (dict(T=4, d=100, ffn=256, E=8, k=2, act="f32", wfmt="f32"), api.ERR_UNSUPPORTED),   # d % 8
    (dict(T=4, d=192, ffn=256, E=8, k=2), api.ERR_UNSUPPORTED),          # tensor path: d % 128
    (dict(T=4, d=128, ffn=256, E=8, k=2, act="f32", wfmt="bf16"), api.ERR_UNSUPPORTED),  # mixed
    (dict(T=4, d=128, ffn=256, E=40, k=33), api.ERR_UNSUPPORTED),        # k > 32
    # the quantised weight modes take the tensor path only (bf16 activations,
    # d and ffn multiples of 128)
    (dict(T=4, d=128, ffn=256, E=8, k=2, act="f32", wfmt="fp8"), api.ERR_UNSUPPORTED),
    (dict(T=4, d=128, ffn=256, E=8, k=2, act="f32", wfmt="fp8a8"), api.ERR_UNSUPPORTED),
    (dict(T=4, d=128, ffn=256, E=8, k=2, act="f32", wfmt="mxfp4"), api.ERR_UNSUPPORTED),
    (dict(T=4, d=192, ffn=256, E=8, k=2, wfmt="fp8a8"), api.ERR_UNSUPPORTED),
    (dict(T=4, d=128, ffn=320, E=8, k=2, wfmt="mxfp4"), api.ERR_UNSUPPORTED),
])
def test_problem_validation_without_gpu(lib, kw, want):
    assert _ws_status(lib, api.problem(**kw)) == want


def test_null_pointers_rejected_before_any_launch(lib):
    p = api.problem(T=4, d=128, ffn=256, E=8, k=2, act="f32", wfmt="f32")
    # topk outputs missing
    assert lib.moe_router_topk(ctypes.byref(p), None, None, None, None, None, None, None, None) == api.ERR_INVALID_ARG
    # x_perm requested without x
    assert lib.moe_permute(ctypes.byref(p), None, None, None, None, None, None, None, None, 0, None) == api.ERR_INVALID_ARG
    assert lib.moe_combine(ctypes.byref(p), None, None, None, None, None, None) == api.ERR_INVALID_ARG
    assert lib.moe_layer_forward(ctypes.byref(p), *([None] * 17), 0, None) == api.ERR_INVALID_ARG


def test_empty_batch_is_a_no_op(lib):
    p = api.problem(T=0, d=128, ffn=256, E=8, k=2)
    ws = ctypes.c_size_t(0)
    # T == 0 returns OK before any launch, even with null tensors
    assert lib.moe_grouped_swiglu(ctypes.byref(p), *([None] * 10), 0, None) == 0
    assert lib.moe_combine(ctypes.byref(p), None, None, None, None, None, None) == 0
    assert lib.moe_layer_forward(ctypes.byref(p), *([None] * 17), 0, None) == 0
    del ws


def test_misaligned_pointer_rejected(lib):
    p = api.problem(T=4, d=128, ffn=256, E=8, k=2)
    fake = ctypes.c_void_p(0x1000 + 8)  # never dereferenced: rejected on the host
    assert lib.moe_combine(ctypes.byref(p), fake, fake, fake, None, fake, None) == api.ERR_INVALID_ARG


def test_quantize_rows_arguments_checked_before_any_launch(lib):
    fake = ctypes.c_void_p(0x1000)  # never dereferenced: rejected on the host
    q = lib.moe_quantize_rows_e4m3
    assert q(-1, 128, fake, fake, fake, None) == api.ERR_INVALID_ARG        # negative rows
    assert q(4, 12, fake, fake, fake, None) == api.ERR_UNSUPPORTED          # cols % 8
    assert q(4, 0, fake, fake, fake, None) == api.ERR_UNSUPPORTED           # no columns
    assert q(4, 128, None, fake, fake, None) == api.ERR_INVALID_ARG         # null input
    assert q(4, 128, fake, None, fake, None) == api.ERR_INVALID_ARG         # null codes
    assert q(4, 128, fake, fake, None, None) == api.ERR_INVALID_ARG         # null scales
    assert q(4, 128, ctypes.c_void_p(0x1008), fake, fake, None) == api.ERR_INVALID_ARG  # misaligned
    assert q(0, 128, None, None, None, None) == 0                            # empty: no launch


def test_split_rows_arguments_checked_before_any_launch(lib):
    fake = ctypes.c_void_p(0x1000)  # never dereferenced: rejected on the host
    q = lib.moe_split_rows_e4m3x2
    assert q(-1, 128, fake, fake, fake, None) == api.ERR_INVALID_ARG        # negative rows
    assert q(4, 12, fake, fake, fake, None) == api.ERR_UNSUPPORTED          # cols % 8
    assert q(4, 0, fake, fake, fake, None) == api.ERR_UNSUPPORTED           # no columns
    assert q(4, 128, None, fake, fake, None) == api.ERR_INVALID_ARG         # null input
    assert q(4, 128, fake, None, fake, None) == api.ERR_INVALID_ARG         # null codes
    assert q(4, 128, fake, fake, None, None) == api.ERR_INVALID_ARG         # null scales
    assert q(4, 128, fake, ctypes.c_void_p(0x1008), fake, None) == api.ERR_INVALID_ARG  # misaligned codes
    assert q(0, 128, None, None, None, None) == 0                            # empty: no launch


def test_quantised_modes_need_their_scales(lib):
    # FP8 / MXFP4 weights without scale arrays are rejected on the host
    fake = ctypes.c_void_p(0x1000)
    for wfmt in ("fp8", "fp8a8", "mxfp4"):
        p = api.problem(T=4, d=128, ffn=256, E=8, k=2, wfmt=wfmt)
        args = [fake, fake, None, fake, fake, fake, None, None, None, None, None, None, fake,
                None, None, None, fake]
        assert lib.moe_layer_forward(ctypes.byref(p), *args, 1 << 20, None) == api.ERR_INVALID_ARG


def test_shared_expert_pointers_follow_the_problem(lib):
    # the shared expert's three matrices are all given when ffn_shared > 0
    # and all NULL otherwise; bf16 weights take no scale arrays
    fake = ctypes.c_void_p(0x1000)  # never dereferenced: rejected on the host
    base = [fake, fake, None, fake, fake, fake, None, None, None]
    tail = [fake, None, None, None, fake]
    p = api.problem(T=4, d=128, ffn=256, E=8, k=2, ffn_shared=128)
    for shared in ([fake, fake, None], [None, None, None], [fake, None, fake]):
        assert lib.moe_layer_forward(ctypes.byref(p), *base, *shared, *tail, 1 << 20, None) == api.ERR_INVALID_ARG
    p0 = api.problem(T=4, d=128, ffn=256, E=8, k=2)
    assert lib.moe_layer_forward(ctypes.byref(p0), *base, fake, fake, fake, *tail, 1 << 20, None) \
        == api.ERR_INVALID_ARG
    scaled = [fake, fake, None, fake, fake, fake, fake, fake, fake]
    assert lib.moe_layer_forward(ctypes.byref(p0), *scaled, None, None, None, *tail, 1 << 20, None) \
        == api.ERR_INVALID_ARG


def test_assignment_rows_limit(lib):
    # T * k <= 2^24 assignment rows
    assert _ws_status(lib, api.problem(T=(1 << 21) + 1, d=128, ffn=128, E=8, k=8)) == api.ERR_UNSUPPORTED
    assert api.moe_workspace_size_for(api.problem(T=1 << 21, d=128, ffn=128, E=8, k=8), 152) > 0
