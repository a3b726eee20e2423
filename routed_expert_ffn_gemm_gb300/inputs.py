"""Seeded synthetic inputs for the MoE FFN layer.

This module only draws random numbers and stores them in the layer's input
formats; it holds none of the layer's arithmetic (no router, no top-k, no
expert FFN).  Both the CUDA path and the CPU oracle consume what it makes.

Value recipe (shapes are the workloads in ``WORKLOADS``):
  x                ~ N(0, 1), stored in the activation dtype (fp32 or bf16,
                   rounded to nearest even);
  W_r, W_g, W_u, W_d ~ N(0, 1/d) with d the hidden size, for every matrix;
  FP8 experts      drawn as above in fp32, then per output channel
                   scale = amax / 448 and code = E4M3(w / scale) (torch's
                   round-to-nearest cast after clamping to +-448);
  router bias      optional; for the skewed prefill workload
                   b_e = -alpha * s * ln(rank_e) with a seeded permutation
                   of ranks 1..E (Zipf exponent s, alpha calibrated offline).
Random streams: one ``torch.Generator`` per (seed, tensor name), on the
device that holds the tensor, so a case is reproducible on one device.
"""

from __future__ import annotations

import dataclasses
import hashlib
import math
from typing import Dict, Optional

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class MoEShape:
    """One MoE layer workload: T tokens, hidden d, expert ffn, E experts,
    top-k, optional shared expert width, storage formats."""
    name: str
    T: int
    d: int
    ffn: int
    E: int
    k: int
    ffn_shared: int = 0
    act: str = "bf16"          # "f32" | "bf16"
    # "f32" | "bf16" | "fp8" | "fp8a8" (FP8 weights, FP8 gate/up activations)
    # | "mxfp4" (OCP MX 4-bit block-scaled weights)
    wfmt: str = "bf16"
    router_bias: str = "none"  # "none" | "zipf"
    zipf_s: float = 1.2

    def with_T(self, T: int) -> "MoEShape":
        return dataclasses.replace(self, T=T)

    @property
    def R(self) -> int:
        return self.T * self.k


# The workloads.  Names describe the model whose MoE layer shape is used.
WORKLOADS: Dict[str, MoEShape] = {
    # toy fp32 layer: T=64, d=128, ffn=256, E=8, top-2
    "toy_f32": MoEShape("toy_f32", T=64, d=128, ffn=256, E=8, k=2, act="f32", wfmt="f32"),
    # Mixtral-8x7B-shaped layer, bf16, decode batches T in {1, 8, 32, 64}
    "mixtral_8x7b": MoEShape("mixtral_8x7b", T=64, d=4096, ffn=14336, E=8, k=2),
    # Qwen3-30B-A3B-shaped layer, bf16, decode T in {1, 16, 128}
    "qwen3_30b_a3b": MoEShape("qwen3_30b_a3b", T=128, d=2048, ffn=768, E=128, k=8),
    # Qwen3-30B-A3B-shaped prefill, T=8192, Zipf(1.2)-skewed expert load
    "qwen3_30b_a3b_prefill": MoEShape("qwen3_30b_a3b_prefill", T=8192, d=2048, ffn=768,
                                      E=128, k=8, router_bias="zipf"),
    # DeepSeek-V3-shaped layer: FP8 routed experts + one bf16 shared expert
    "deepseek_v3": MoEShape("deepseek_v3", T=64, d=7168, ffn=2048, E=256, k=8,
                            ffn_shared=2048, wfmt="fp8"),
}

DECODE_T = {
    "toy_f32": (64,),
    "mixtral_8x7b": (1, 8, 32, 64),
    "qwen3_30b_a3b": (1, 16, 128),
    "qwen3_30b_a3b_prefill": (8192,),
    "deepseek_v3": (1, 64, 4096),
}

# Scale of the skewing router bias per workload.  Calibrated offline on the
# seeded CPU sample (seed 0) with the CPU reference router so that the
# hottest expert holds about 8x the mean rows; the calibration script and
# its output live in tests/golden/, and a CPU test re-checks the value.
ZIPF_ALPHA = {"qwen3_30b_a3b_prefill": 0.355469}


def zipf_alpha(shape: MoEShape) -> float:
    a = ZIPF_ALPHA.get(shape.name)
    if a is None:
        raise ValueError(f"no calibrated router-bias scale for {shape.name}")
    return float(a)


def zipf_bias(shape: MoEShape, seed: int, alpha: Optional[float] = None, device="cpu") -> torch.Tensor:
    """Per-expert router bias b_e = -alpha * s * ln(rank_e), ranks 1..E in a
    seeded order, fp32.  Skews expert load roughly as a Zipf law."""
    a = zipf_alpha(shape) if alpha is None else float(alpha)
    g = _gen(seed, "zipf_ranks", "cpu")
    ranks = torch.randperm(shape.E, generator=g).to(torch.float64) + 1.0
    return (-a * shape.zipf_s * torch.log(ranks)).to(torch.float32).to(device)


def _gen(seed: int, name: str, device) -> torch.Generator:
    h = hashlib.sha256(f"{seed}:{name}".encode()).digest()
    g = torch.Generator(device=device)
    g.manual_seed(int.from_bytes(h[:8], "little") & ((1 << 63) - 1))
    return g


def _torch_dtype(fmt: str):
    return {"f32": torch.float32, "bf16": torch.bfloat16}[fmt]


def _normal(shape, std, seed, name, device, out_dtype):
    g = _gen(seed, name, device)
    return (torch.randn(shape, generator=g, device=device, dtype=torch.float32) * std).to(out_dtype)


def _fp8_quantise(w: torch.Tensor):
    """Per-output-channel E4M3 codes and fp32 scales of a [rows, cols] block."""
    amax = w.abs().amax(dim=1).clamp_min(1e-30)
    scale = (amax / 448.0).to(torch.float32)
    q = (w / scale[:, None]).clamp(-448.0, 448.0).to(torch.float8_e4m3fn)
    return q.view(torch.uint8), scale


_E2M1_MAGS = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)


def _mxfp4_quantise(w: torch.Tensor):
    """MXFP4 codes of a [rows, cols] fp32 block: per 32 consecutive values of
    a row, the scale 2^e with e = floor(log2(block max)) - 2 (the block's
    largest magnitude lands in [4, 8), saturating at 6), codes the nearest
    E2M1 magnitude (ties up) with the sign bit.  Returns packed codes
    [rows, cols/2] (element 2i in the low nibble) and UE8M0 scales
    [cols/32, rows]."""
    rows, cols = w.shape
    blk = w.reshape(rows, cols // 32, 32)
    amax = blk.abs().amax(dim=2).clamp_min(2.0 ** -100)
    e = (torch.floor(torch.log2(amax)) - 2).clamp(-127, 127)
    q = blk / torch.exp2(e)[..., None]
    mags = torch.tensor(_E2M1_MAGS, device=w.device)
    code = torch.bucketize(q.abs().clamp(max=6.0), (mags[1:] + mags[:-1]) / 2)
    code = (code | ((q < 0).to(code.dtype) << 3)).reshape(rows, cols).to(torch.uint8)
    packed = code[:, 0::2] | (code[:, 1::2] << 4)
    return packed.contiguous(), (e + 127).to(torch.uint8).t().contiguous()


def _expert_stack(shape: MoEShape, rows: int, cols: int, seed: int, name: str, device):
    """[E, rows, cols] expert matrices ~ N(0, 1/d), generated per expert so
    that large layers never hold an fp32 copy of the whole stack."""
    std = 1.0 / math.sqrt(shape.d)
    E = shape.E
    if shape.wfmt == "mxfp4":
        w = torch.empty((E, rows, cols // 2), dtype=torch.uint8, device=device)
        s = torch.empty((E, cols // 32, rows), dtype=torch.uint8, device=device)
        for e in range(E):
            q, sc = _mxfp4_quantise(_normal((rows, cols), std, seed, f"{name}[{e}]", device, torch.float32))
            w[e].copy_(q)
            s[e].copy_(sc)
        return w, s
    if shape.wfmt in ("fp8", "fp8a8"):
        w = torch.empty((E, rows, cols), dtype=torch.uint8, device=device)
        s = torch.empty((E, rows), dtype=torch.float32, device=device)
        for e in range(E):
            q, sc = _fp8_quantise(_normal((rows, cols), std, seed, f"{name}[{e}]", device, torch.float32))
            w[e].copy_(q)
            s[e].copy_(sc)
        return w, s
    dt = _torch_dtype(shape.wfmt)
    w = torch.empty((E, rows, cols), dtype=dt, device=device)
    for e in range(E):
        w[e].copy_(_normal((rows, cols), std, seed, f"{name}[{e}]", device, dt))
    return w, None


def make_weights(shape: MoEShape, seed: int, device="cpu") -> Dict[str, Optional[torch.Tensor]]:
    """Router, routed-expert and shared-expert weights of one layer."""
    act = _torch_dtype(shape.act)
    std = 1.0 / math.sqrt(shape.d)
    out: Dict[str, Optional[torch.Tensor]] = {}
    out["w_router"] = _normal((shape.E, shape.d), std, seed, "w_router", device, act)
    out["router_bias"] = zipf_bias(shape, seed, device=device) if shape.router_bias == "zipf" else None
    out["w_gate"], out["s_gate"] = _expert_stack(shape, shape.ffn, shape.d, seed, "w_gate", device)
    out["w_up"], out["s_up"] = _expert_stack(shape, shape.ffn, shape.d, seed, "w_up", device)
    out["w_down"], out["s_down"] = _expert_stack(shape, shape.d, shape.ffn, seed, "w_down", device)
    if shape.ffn_shared:
        # the shared expert stays in the activation dtype (higher precision
        # than the FP8 routed experts)
        fs = shape.ffn_shared
        out["w_shared_gate"] = _normal((fs, shape.d), std, seed, "w_shared_gate", device, act)
        out["w_shared_up"] = _normal((fs, shape.d), std, seed, "w_shared_up", device, act)
        out["w_shared_down"] = _normal((shape.d, fs), std, seed, "w_shared_down", device, act)
    else:
        out["w_shared_gate"] = out["w_shared_up"] = out["w_shared_down"] = None
    return out


def make_tokens(shape: MoEShape, seed: int, device="cpu", step: int = 0) -> torch.Tensor:
    """Token hidden states x [T, d] ~ N(0, 1) in the activation dtype."""
    return _normal((shape.T, shape.d), 1.0, seed, f"x:{step}", device, _torch_dtype(shape.act))


def make_case(shape: MoEShape, seed: int, device="cpu"):
    case = make_weights(shape, seed, device)
    case["x"] = make_tokens(shape, seed, device)
    return case


# ---------------------------------------------------------------------------
# Host views of stored values (bit patterns), for the oracle
# ---------------------------------------------------------------------------

def to_numpy_stored(t: Optional[torch.Tensor]):
    """A tensor's stored values as numpy: float32 stays float32, bf16 becomes
    its uint16 bit patterns, uint8 (E4M3 codes) stays uint8."""
    if t is None:
        return None
    t = t.detach().to("cpu").contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()
