"""Thin ctypes binding of libmoe_gb300.so (include/moe.h), same names.

Argument marshalling only: tensors become device pointers, the stream
defaults to torch's current stream, a non-zero status raises ``MoEError``.
Every step of the layer runs in the library's CUDA kernels; there is no
other implementation behind these functions.  The library is loaded on the
first call and a missing library is an error (build it with
``python -m routed_expert_ffn_gemm_gb300.build``).
"""

from __future__ import annotations

import ctypes
import functools
import os
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmoe_gb300.so")

# "fp8a8": FP8 weights with FP8 (per-row E4M3) gate/up activations;
# "mxfp4": OCP MX 4-bit block-scaled weights
DTYPE = {"f32": 0, "bf16": 1, "fp8": 2, "fp8a8": 3, "mxfp4": 4}
OK = 0
ERR_INVALID_ARG = -1
ERR_UNSUPPORTED = -2
ERR_WORKSPACE = -3
ERR_CUDA = -4
ERR_DEVICE_TIMEOUT = -5
ERR_DEVICE_BOUNDS = -6


class moe_problem(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("T", "d", "ffn", "E", "k", "ffn_shared", "act_dtype", "w_dtype")]


class MoEError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        msg = f"{fn} failed: {moe_status_string(status)}"
        if status == ERR_CUDA:
            msg += f" ({_lib().moe_last_cuda_error().decode()})"
        super().__init__(msg)


_LIB = None
_VP = ctypes.c_void_p
_PP = ctypes.POINTER(moe_problem)

_SIGS = {
    "moe_router_topk": [_PP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP],
    "moe_permute": [_PP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, ctypes.c_size_t, _VP],
    "moe_grouped_swiglu": [_PP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, ctypes.c_size_t, _VP],
    "moe_combine": [_PP, _VP, _VP, _VP, _VP, _VP, _VP],
    "moe_layer_forward": [_PP] + [_VP] * 17 + [ctypes.c_size_t, _VP],
    "moe_workspace_size": [_PP, ctypes.POINTER(ctypes.c_size_t)],
    "moe_read_device_status": [_VP, ctypes.POINTER(ctypes.c_int32)],
    "moe_status_string": [ctypes.c_int32],
    "moe_last_cuda_error": [],
    "moe_abi_version": [],
    "moe_selftest_bounded_wait": [ctypes.c_int64, _VP],
    "moe_stage_timer_create": [ctypes.POINTER(_VP)],
    "moe_stage_timer_destroy": [_VP],
    "moe_stage_timer_read": [_VP, ctypes.POINTER(ctypes.c_float)],
    "moe_layer_forward_timed": [_PP] + [_VP] * 17 + [ctypes.c_size_t, _VP, _VP],
    "moe_layer_launch_count": [_PP, ctypes.POINTER(ctypes.c_int32)],
    "moe_plan_info": [_PP, ctypes.POINTER(ctypes.c_int32)],
    "moe_plan_info_for": [_PP, ctypes.c_int32, ctypes.POINTER(ctypes.c_int32)],
    "moe_layer_launch_count_for": [_PP, ctypes.c_int32, ctypes.POINTER(ctypes.c_int32)],
    "moe_workspace_size_for": [_PP, ctypes.c_int32, ctypes.POINTER(ctypes.c_size_t)],
    "moe_permute_static_scratch": [_PP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP],
    "moe_quantize_rows_e4m3": [ctypes.c_int32, ctypes.c_int32, _VP, _VP, _VP, _VP],
    "moe_split_rows_e4m3x2": [ctypes.c_int32, ctypes.c_int32, _VP, _VP, _VP, _VP],
}
STAGES = ("router", "permute", "gate_up", "down", "shared", "combine")
EXPORTS = tuple(_SIGS)


def _lib():
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m routed_expert_ffn_gemm_gb300.build`")
        lib = ctypes.CDLL(LIB_PATH)
        for name, args in _SIGS.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = ctypes.c_int32
        lib.moe_status_string.restype = ctypes.c_char_p
        lib.moe_last_cuda_error.restype = ctypes.c_char_p
        _LIB = lib
    return _LIB


def problem(T, d, ffn, E, k, ffn_shared=0, act="bf16", wfmt="bf16") -> moe_problem:
    return moe_problem(T, d, ffn, E, k, ffn_shared, DTYPE[act], DTYPE[wfmt])


def problem_of(shape) -> moe_problem:
    """moe_problem of an ``inputs.MoEShape``."""
    return problem(shape.T, shape.d, shape.ffn, shape.E, shape.k, shape.ffn_shared, shape.act, shape.wfmt)


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("the library takes device tensors")
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return t.data_ptr()


# Sizes checked before each call.  The C entry points take bare pointers,
# so a tensor smaller than the problem says, or of another element size,
# would be read or written out of bounds on the device; here it is a
# ValueError instead.  Null pointers, alignment and workspace sizes are the
# library's own checks.

def _check(t: Optional[torch.Tensor], name: str, elems: int, esize: int, dtype=None):
    if t is None:
        return
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name}: dtype {t.dtype}, the call takes {dtype}")
    if t.element_size() != esize:
        raise ValueError(f"{name}: {t.element_size()}-byte elements, the problem needs {esize}-byte ones")
    if t.numel() < elems:
        raise ValueError(f"{name}: {t.numel()} elements, the problem needs {elems}")


def _act_size(p) -> int:
    return 4 if p.act_dtype == DTYPE["f32"] else 2


def _key(p) -> tuple:
    return (p.T, p.d, p.ffn, p.E, p.k, p.ffn_shared, p.act_dtype, p.w_dtype)


@functools.lru_cache(maxsize=256)
def _expert_reqs(key) -> tuple:
    """(name, elements, element size, dtype) of the routed expert weights
    and scales, per weight mode: gate/up [E, ffn, d], down [E, d, ffn]; FP8
    codes with fp32 scales [E, ffn] / [E, d]; MXFP4 codes two per byte with
    UE8M0 block scales [E, d/32, ffn] / [E, ffn/32, d]."""
    _, d, f, E, _, _, _, wdt = key
    if wdt == DTYPE["mxfp4"]:
        w, ws, gs, ds, ss = E * f * d // 2, 1, E * (d // 32) * f, E * (f // 32) * d, 1
    elif wdt in (DTYPE["fp8"], DTYPE["fp8a8"]):
        w, ws, gs, ds, ss = E * f * d, 1, E * f, E * d, 4
    else:
        w, ws, gs, ds, ss = E * f * d, 4 if wdt == DTYPE["f32"] else 2, 0, 0, 4
    return (("w_gate", w, ws, None), ("w_up", w, ws, None), ("w_down", w, ws, None),
            ("s_gate", gs, ss, None), ("s_up", gs, ss, None), ("s_down", ds, ss, None))


@functools.lru_cache(maxsize=256)
def _layer_reqs(key) -> tuple:
    T, d, _, E, k, fs, adt, _ = key
    a = 4 if adt == DTYPE["f32"] else 2
    return ((("x", T * d, a, None), ("w_router", E * d, a, None), ("router_bias", E, 4, torch.float32))
            + _expert_reqs(key)
            + (("w_shared_gate", fs * d, a, None), ("w_shared_up", fs * d, a, None),
               ("w_shared_down", fs * d, a, None), ("out", T * d, a, None),
               ("topk_idx_out", T * k, 4, torch.int32), ("topk_w_out", T * k, 4, torch.float32),
               ("counts_out", E, 4, torch.int32)))


def _verify(reqs, tensors):
    for t, (name, elems, esize, dtype) in zip(tensors, reqs):
        if t is not None and (t.numel() < elems or t.element_size() != esize
                              or (dtype is not None and t.dtype != dtype)):
            _check(t, name, elems, esize, dtype)


def _check_experts(p, w_gate, w_up, w_down, s_gate, s_up, s_down):
    _verify(_expert_reqs(_key(p)), (w_gate, w_up, w_down, s_gate, s_up, s_down))


def _check_layer(p, *tensors):
    """The 16 tensors of moe_layer_forward, x .. counts_out, in order."""
    _verify(_layer_reqs(_key(p)), tensors)


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _call(name, *args):
    st = getattr(_lib(), name)(*args)
    if st != OK:
        raise MoEError(name, st)


def moe_router_topk(p, x, w_router, router_bias, logits_in, logits_out, topk_idx, topk_w, stream=None):
    a = _act_size(p)
    _check(x, "x", p.T * p.d, a)
    _check(w_router, "w_router", p.E * p.d, a)
    _check(router_bias, "router_bias", p.E, 4, torch.float32)
    _check(logits_in, "logits_in", p.T * p.E, 4, torch.float32)
    _check(logits_out, "logits_out", p.T * p.E, 4, torch.float32)
    _check(topk_idx, "topk_idx", p.T * p.k, 4, torch.int32)
    _check(topk_w, "topk_w", p.T * p.k, 4, torch.float32)
    _call("moe_router_topk", ctypes.byref(p), _ptr(x), _ptr(w_router), _ptr(router_bias),
          _ptr(logits_in), _ptr(logits_out), _ptr(topk_idx), _ptr(topk_w), _stream(stream))


def _check_permute(p, topk_idx, x, counts, offsets, perm_token, inv_row, x_perm):
    R, a = p.T * p.k, _act_size(p)
    _check(topk_idx, "topk_idx", R, 4, torch.int32)
    _check(x, "x", p.T * p.d, a)
    _check(counts, "counts", p.E, 4, torch.int32)
    _check(offsets, "offsets", p.E + 1, 4, torch.int32)
    _check(perm_token, "perm_token", R, 4, torch.int32)
    _check(inv_row, "inv_row", R, 4, torch.int32)
    _check(x_perm, "x_perm", R * p.d, a)


def moe_permute(p, topk_idx, x, counts, offsets, perm_token, inv_row, x_perm, workspace, stream=None):
    _check_permute(p, topk_idx, x, counts, offsets, perm_token, inv_row, x_perm)
    _call("moe_permute", ctypes.byref(p), _ptr(topk_idx), _ptr(x), _ptr(counts), _ptr(offsets),
          _ptr(perm_token), _ptr(inv_row), _ptr(x_perm), _ptr(workspace),
          0 if workspace is None else workspace.numel() * workspace.element_size(), _stream(stream))


def moe_permute_static_scratch(p, topk_idx, x, counts, offsets, perm_token, inv_row, x_perm, stream=None):
    """moe_permute for callers that cannot allocate device memory: the
    permutation's scratch comes from a fixed 1 MiB array inside the library
    instead of a caller workspace (see include/moe.h for its limits)."""
    _check_permute(p, topk_idx, x, counts, offsets, perm_token, inv_row, x_perm)
    _call("moe_permute_static_scratch", ctypes.byref(p), _ptr(topk_idx), _ptr(x), _ptr(counts),
          _ptr(offsets), _ptr(perm_token), _ptr(inv_row), _ptr(x_perm), _stream(stream))


def moe_grouped_swiglu(p, x_perm, offsets, w_gate, w_up, w_down, s_gate, s_up, s_down, y_perm,
                       workspace, stream=None):
    R, a = p.T * p.k, _act_size(p)
    _check(x_perm, "x_perm", R * p.d, a)
    _check(offsets, "offsets", p.E + 1, 4, torch.int32)
    _check_experts(p, w_gate, w_up, w_down, s_gate, s_up, s_down)
    _check(y_perm, "y_perm", R * p.d, a)
    _call("moe_grouped_swiglu", ctypes.byref(p), _ptr(x_perm), _ptr(offsets), _ptr(w_gate), _ptr(w_up),
          _ptr(w_down), _ptr(s_gate), _ptr(s_up), _ptr(s_down), _ptr(y_perm), _ptr(workspace),
          0 if workspace is None else workspace.numel() * workspace.element_size(), _stream(stream))


def moe_quantize_rows_e4m3(x, codes, scales, stream=None):
    """Per-row E4M3 codes (uint8 [rows, cols]) and fp32 scales ([rows]) of
    bf16 rows x [rows, cols]."""
    rows, cols = (int(v) for v in x.shape)
    _check(x, "x", rows * cols, 2)
    _check(codes, "codes", rows * cols, 1)
    _check(scales, "scales", rows, 4, torch.float32)
    _call("moe_quantize_rows_e4m3", rows, cols, _ptr(x), _ptr(codes), _ptr(scales), _stream(stream))


def moe_split_rows_e4m3x2(x, codes, scales, stream=None):
    """bf16 rows x [rows, cols] as two E4M3 rows each: codes uint8
    [2, rows, cols] (every row's hi codes, then every row's lo codes) and
    power-of-two fp32 scales [rows], with x = s * (hi + lo)."""
    rows, cols = (int(v) for v in x.shape)
    _check(x, "x", rows * cols, 2)
    _check(codes, "codes", 2 * rows * cols, 1)
    _check(scales, "scales", rows, 4, torch.float32)
    _call("moe_split_rows_e4m3x2", rows, cols, _ptr(x), _ptr(codes), _ptr(scales), _stream(stream))


def moe_combine(p, y_perm, inv_row, topk_w, shared_out, out, stream=None):
    R, a = p.T * p.k, _act_size(p)
    _check(y_perm, "y_perm", R * p.d, a)
    _check(inv_row, "inv_row", R, 4, torch.int32)
    _check(topk_w, "topk_w", R, 4, torch.float32)
    _check(shared_out, "shared_out", p.T * p.d, a)
    _check(out, "out", p.T * p.d, a)
    _call("moe_combine", ctypes.byref(p), _ptr(y_perm), _ptr(inv_row), _ptr(topk_w), _ptr(shared_out),
          _ptr(out), _stream(stream))


def moe_layer_forward(p, x, w_router, router_bias, w_gate, w_up, w_down, s_gate, s_up, s_down,
                      w_shared_gate, w_shared_up, w_shared_down, out, topk_idx_out, topk_w_out,
                      counts_out, workspace, stream=None):
    _check_layer(p, x, w_router, router_bias, w_gate, w_up, w_down, s_gate, s_up, s_down, w_shared_gate,
                 w_shared_up, w_shared_down, out, topk_idx_out, topk_w_out, counts_out)
    _call("moe_layer_forward", ctypes.byref(p), _ptr(x), _ptr(w_router), _ptr(router_bias), _ptr(w_gate),
          _ptr(w_up), _ptr(w_down), _ptr(s_gate), _ptr(s_up), _ptr(s_down), _ptr(w_shared_gate),
          _ptr(w_shared_up), _ptr(w_shared_down), _ptr(out), _ptr(topk_idx_out), _ptr(topk_w_out),
          _ptr(counts_out), _ptr(workspace),
          0 if workspace is None else workspace.numel() * workspace.element_size(), _stream(stream))


def moe_layer_forward_timed(p, x, w_router, router_bias, w_gate, w_up, w_down, s_gate, s_up, s_down,
                            w_shared_gate, w_shared_up, w_shared_down, out, topk_idx_out, topk_w_out,
                            counts_out, workspace, timer, stream=None):
    _check_layer(p, x, w_router, router_bias, w_gate, w_up, w_down, s_gate, s_up, s_down, w_shared_gate,
                 w_shared_up, w_shared_down, out, topk_idx_out, topk_w_out, counts_out)
    _call("moe_layer_forward_timed", ctypes.byref(p), _ptr(x), _ptr(w_router), _ptr(router_bias),
          _ptr(w_gate), _ptr(w_up), _ptr(w_down), _ptr(s_gate), _ptr(s_up), _ptr(s_down),
          _ptr(w_shared_gate), _ptr(w_shared_up), _ptr(w_shared_down), _ptr(out), _ptr(topk_idx_out),
          _ptr(topk_w_out), _ptr(counts_out), _ptr(workspace),
          0 if workspace is None else workspace.numel() * workspace.element_size(), _stream(stream),
          timer.handle)


class StageTimer:
    """moe_stage_timer: CUDA events between the stages of one layer call."""

    def __init__(self):
        h = ctypes.c_void_p(None)
        _call("moe_stage_timer_create", ctypes.byref(h))
        self.handle = h

    def read(self):
        """{stage: milliseconds} of the last timed call (waits for it)."""
        ms = (ctypes.c_float * len(STAGES))()
        _call("moe_stage_timer_read", self.handle, ms)
        return dict(zip(STAGES, (float(v) for v in ms)))

    def close(self):
        if self.handle is not None:
            _lib().moe_stage_timer_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def moe_layer_launch_count(p) -> int:
    n = ctypes.c_int32(0)
    _call("moe_layer_launch_count", ctypes.byref(p), ctypes.byref(n))
    return int(n.value)


def _plan_dict(info) -> dict:
    return {"bn_gateup": info[0], "bn_down": info[1], "splits_down": info[2], "grid": info[3],
            "splits_gateup": info[4], "pair_gateup": info[5] & 1, "pair_down": (info[5] >> 1) & 1}


def moe_plan_info(p) -> dict:
    info = (ctypes.c_int32 * 6)()
    _call("moe_plan_info", ctypes.byref(p), info)
    return _plan_dict(info)


def moe_workspace_size(p) -> int:
    n = ctypes.c_size_t(0)
    _call("moe_workspace_size", ctypes.byref(p), ctypes.byref(n))
    return int(n.value)


# The planning answers for a device with `num_sms` SMs, computed on the host
# (no device needed).

def moe_plan_info_for(p, num_sms: int) -> dict:
    info = (ctypes.c_int32 * 6)()
    _call("moe_plan_info_for", ctypes.byref(p), int(num_sms), info)
    return _plan_dict(info)


def moe_layer_launch_count_for(p, num_sms: int) -> int:
    n = ctypes.c_int32(0)
    _call("moe_layer_launch_count_for", ctypes.byref(p), int(num_sms), ctypes.byref(n))
    return int(n.value)


def moe_workspace_size_for(p, num_sms: int) -> int:
    n = ctypes.c_size_t(0)
    _call("moe_workspace_size_for", ctypes.byref(p), int(num_sms), ctypes.byref(n))
    return int(n.value)


def moe_read_device_status(stream=None) -> int:
    v = ctypes.c_int32(0)
    _call("moe_read_device_status", _stream(stream), ctypes.byref(v))
    return int(v.value)


def moe_status_string(status: int) -> str:
    return _lib().moe_status_string(int(status)).decode()


def moe_abi_version() -> int:
    return int(_lib().moe_abi_version())


def moe_selftest_bounded_wait(timeout_ns: int, stream=None):
    _call("moe_selftest_bounded_wait", int(timeout_ns), _stream(stream))


# ---------------------------------------------------------------------------
# conveniences over the C calls (allocation through torch)
# ---------------------------------------------------------------------------

def workspace_for(p, device="cuda") -> torch.Tensor:
    """A device workspace of moe_workspace_size(p) bytes (16-byte aligned)."""
    return torch.empty(max(16, moe_workspace_size(p)), dtype=torch.uint8, device=device)


def layer_forward(p, case, out=None, workspace=None, want_routing=False, stream=None, timer=None):
    """moe_layer_forward (or moe_layer_forward_timed when a StageTimer is
    given) on a case dict (``inputs.make_case`` keys)."""
    x = case["x"]
    if out is None:
        out = torch.empty_like(x)
    if workspace is None:
        workspace = workspace_for(p, x.device)
    idx = w = counts = None
    if want_routing:
        idx = torch.empty((p.T, p.k), dtype=torch.int32, device=x.device)
        w = torch.empty((p.T, p.k), dtype=torch.float32, device=x.device)
        counts = torch.empty((p.E,), dtype=torch.int32, device=x.device)
    args = (p, x, case["w_router"], case["router_bias"], case["w_gate"], case["w_up"],
            case["w_down"], case["s_gate"], case["s_up"], case["s_down"],
            case["w_shared_gate"], case["w_shared_up"], case["w_shared_down"], out,
            idx, w, counts, workspace)
    if timer is None:
        moe_layer_forward(*args, stream=stream)
    else:
        moe_layer_forward_timed(*args, timer, stream=stream)
    return (out, idx, w, counts) if want_routing else out
