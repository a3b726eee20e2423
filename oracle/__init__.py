"""Plain fp64 CPU oracle for one Mixture-of-Experts FFN layer forward.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline / reference legs may import this package.  The
product path (the CUDA library and its Python binding) never imports it, and
this package never imports the product path.

Every function states the passage of the source page it follows.  The page
that states the per-layer algorithm is "MOE推理流程解析" (ffner.com); sections
are cited by their numbers there (一 … 十一).  Precision context comes from
"MoE 推理部署" (zzmblog.top), section "专家量化".

Parity status per function (what pins each one is listed in the tests):
  decode_bf16, decode_e4m3          pinned (format definitions, fixed values)
  router_logits                     pinned (brute force, linearity)
  topk_renorm                       pinned (worked example, brute force over
                                    k-subsets, closed form)
  permutation_maps                  pinned (worked example, invariants)
  silu, swiglu_expert               pinned (closed-form values, library FFN)
  moe_forward_per_token             pinned (worked example combine, special
                                    cases, formulation (ii))
  moe_forward_grouped               pinned (formulation (i), special cases)
  shared_expert                     pinned (library FFN)
  round_to_e4m3                     pinned (library float8 cast on every
                                    in-range midpoint and a dense sweep;
                                    saturation; ties to even)
  quantize_rows_e4m3 /              pinned (scale = row max / 448 hits code
  dequantize_rows_e4m3              0x7E; lossless on E4M3-representable
                                    rows; zero rows)
  decode_e2m1, decode_ue8m0,        pinned (the OCP MX element and scale
  unpack_fp4, decode_mxfp4          definitions at fixed codes, the page's
                                    storage figure for a 117B-parameter model,
                                    a hand-decoded block, nibble order and
                                    scale layout by construction)
"""

from .moe_oracle import (  # noqa: F401
    decode_bf16,
    decode_e4m3,
    ExpertWeights,
    router_logits,
    softmax,
    topk_renorm,
    topk_gap,
    permutation_maps,
    silu,
    swiglu_expert,
    moe_forward_per_token,
    moe_forward_grouped,
    shared_expert,
    round_to_e4m3,
    quantize_rows_e4m3,
    dequantize_rows_e4m3,
    decode_e2m1,
    decode_ue8m0,
    unpack_fp4,
    decode_mxfp4,
)
