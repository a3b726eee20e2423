"""Test helpers: turn a generated case into the CPU reference's inputs, and
pick seeds without near-ties in the routing decision."""

import json
import os

import numpy as np

import oracle
from routed_expert_ffn_gemm_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load_golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def worked_example():
    """The page's 4-token / 4-expert top-2 example, 0-based: idx [T, k] with
    slots in descending weight, w [T, k], and the printed groups."""
    g = load_golden("worked_example_4tok_4exp_top2.json")
    T, E, k = g["T"], g["E"], g["k"]
    idx = np.zeros((T, k), dtype=np.int32)
    w = np.zeros((T, k))
    for t in range(T):
        pairs = [(int(e[1:]) - 1, float(v)) for e, v in g["routing"][f"T{t + 1}"].items()]
        pairs.sort(key=lambda p: (-p[1], p[0]))
        idx[t] = [p[0] for p in pairs]
        w[t] = [p[1] for p in pairs]
    groups = [[int(s[1:]) - 1 for s in g["groups"][f"E{e + 1}"]] for e in range(E)]
    return g, idx, w, groups


def worked_example_logits(w_idx, w_val, E):
    """Logits that route the worked example: ln(w) on the chosen experts and
    min(ln w) - 20 elsewhere.  Renormalised softmax over the chosen set then
    returns w exactly (the other logits cancel)."""
    T, k = w_idx.shape
    logits = np.zeros((T, E))
    for t in range(T):
        lw = np.log(w_val[t])
        logits[t, :] = lw.min() - 20.0
        logits[t, w_idx[t]] = lw
    return logits


def decode_act(t, fmt):
    a = inputs.to_numpy_stored(t)
    if a is None:
        return None
    return oracle.decode_bf16(a) if fmt == "bf16" else np.asarray(a, np.float64)


def oracle_inputs(case, shape):
    """(x, w_router, bias, ExpertWeights, shared) for the CPU reference, from
    the stored values of a generated case (tensors may live on any device)."""
    x = decode_act(case["x"], shape.act)
    wr = decode_act(case["w_router"], shape.act)
    bias = None if case["router_bias"] is None else inputs.to_numpy_stored(case["router_bias"]).astype(np.float64)
    if shape.wfmt == "mxfp4":
        ew = oracle.ExpertWeights("mxfp4", _Lazy(case["w_gate"]), _Lazy(case["w_up"]), _Lazy(case["w_down"]),
                                  _Lazy(case["s_gate"]), _Lazy(case["s_up"]), _Lazy(case["s_down"]))
    elif shape.wfmt in ("fp8", "fp8a8"):
        ew = oracle.ExpertWeights("fp8", _Lazy(case["w_gate"]), _Lazy(case["w_up"]), _Lazy(case["w_down"]),
                                  _Lazy(case["s_gate"]), _Lazy(case["s_up"]), _Lazy(case["s_down"]))
    else:
        ew = oracle.ExpertWeights(shape.wfmt, _Lazy(case["w_gate"]), _Lazy(case["w_up"]), _Lazy(case["w_down"]))
    shared = None
    if shape.ffn_shared:
        shared = tuple(decode_act(case[n], shape.act) for n in ("w_shared_gate", "w_shared_up", "w_shared_down"))
    return x, wr, bias, ew, shared


class _Lazy:
    """Indexable view of a [E, ...] tensor that copies one expert to the host
    (as stored values) on access, so huge stacks are never copied whole."""

    def __init__(self, t):
        self.t = t
        self.shape = tuple(t.shape)

    def __getitem__(self, e):
        return inputs.to_numpy_stored(self.t[e])

    def __len__(self):
        return self.shape[0]


def routing_gap_ok(logits, k, min_gap):
    return bool(np.all(oracle.topk_gap(logits, k) >= min_gap))


def seed_without_near_ties(shape, first_seed=0, min_gap=1e-3, tries=50, device="cpu"):
    """First seed >= first_seed whose oracle logits have a k-th/(k+1)-th gap of
    at least min_gap for every token (rejected seeds advance by one)."""
    for s in range(first_seed, first_seed + tries):
        w = inputs.make_weights(shape, s, device)
        x = inputs.make_tokens(shape, s, device)
        lg = oracle.router_logits(decode_act(x, shape.act), decode_act(w["w_router"], shape.act),
                                  None if w["router_bias"] is None else
                                  inputs.to_numpy_stored(w["router_bias"]).astype(np.float64))
        if routing_gap_ok(lg, shape.k, min_gap):
            return s
    raise RuntimeError("no seed without near-ties found")
