"""Calibrate the scale of the skewing router bias of the Zipf-skewed
Qwen3-30B-A3B-shaped prefill workload (T=8192, d=2048, E=128, top-8).

Uses only the CPU reference (``oracle``) on the seeded CPU sample (seed 0):
bisects alpha so that the hottest expert receives ~8x the mean number of
rows (max/mean in [7.5, 8.5]) and writes the result to
``zipf_bias_alpha.json`` beside this script.  The value is then copied into
``ZIPF_ALPHA`` of the input generator; a CPU test checks the two agree.

Run from the repository root:  python tests/golden/calibrate_zipf_bias.py
"""

import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from routed_expert_ffn_gemm_gb300 import inputs  # noqa: E402


def max_over_mean(logits0, bias, k, E):
    idx, _ = oracle.topk_renorm(logits0 + bias[None, :], k)
    counts, _, _, _ = oracle.permutation_maps(idx, E)
    return counts.max() / counts.mean()


def main():
    shape = inputs.WORKLOADS["qwen3_30b_a3b_prefill"]
    seed = 0
    w = inputs._normal((shape.E, shape.d), 1.0 / np.sqrt(shape.d), seed, "w_router", "cpu",
                       inputs._torch_dtype(shape.act))
    x = inputs.make_tokens(shape, seed, "cpu")
    xs = oracle.decode_bf16(inputs.to_numpy_stored(x))
    ws = oracle.decode_bf16(inputs.to_numpy_stored(w))
    logits0 = oracle.router_logits(xs, ws)
    lo, hi = 0.0, 4.0
    for _ in range(30):
        mid = 0.5 * (lo + hi)
        b = inputs.zipf_bias(shape, seed, alpha=mid).double().numpy()
        r = max_over_mean(logits0, b, shape.k, shape.E)
        print(f"alpha={mid:.6f} max/mean={r:.4f}", flush=True)
        if 7.95 <= r <= 8.05:
            break
        if r < 8.0:
            lo = mid
        else:
            hi = mid
    alpha = round(mid, 6)
    b = inputs.zipf_bias(shape, seed, alpha=alpha).double().numpy()
    r = float(max_over_mean(logits0, b, shape.k, shape.E))
    out = {f"{shape.name}": {"alpha": alpha, "seed": seed, "T": shape.T,
                             "max_over_mean_rows": round(r, 4),
                             "note": "oracle routing of the seeded CPU sample"}}
    with open(os.path.join(os.path.dirname(os.path.abspath(__file__)), "zipf_bias_alpha.json"), "w") as f:
        json.dump(out, f, indent=1)
        f.write("\n")
    print(json.dumps(out))


if __name__ == "__main__":
    main()
