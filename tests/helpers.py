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


class PrefetchedExperts:
    """``expert_hook`` for the oracle's grouped formulation: decodes, in worker
    threads and ahead of the grouped loop, the experts that loop will visit
    (``experts``: ascending ids of the experts holding rows), each through the
    oracle's own ``ExpertWeights.get``; at most ``ahead`` decoded experts are
    held at once.  Decoding is most of the oracle's time on the large
    FP8 / MXFP4 layers, and numpy runs it outside the interpreter lock."""

    def __init__(self, ew, experts, workers=8, ahead=12):
        from concurrent.futures import ThreadPoolExecutor
        self.ew = ew
        self.order = [int(e) for e in experts]
        self.pool = ThreadPoolExecutor(max_workers=workers)
        self.futures = {e: self.pool.submit(ew.get, e) for e in self.order[:ahead]}
        self.next = min(ahead, len(self.order))

    def __call__(self, e):
        f = self.futures.pop(int(e), None)
        w = f.result() if f is not None else self.ew.get(int(e))
        if self.next < len(self.order):
            n = self.order[self.next]
            self.next += 1
            self.futures[n] = self.pool.submit(self.ew.get, n)
        return w

    def close(self):
        self.pool.shutdown(wait=True, cancel_futures=True)


def check_routing_within_tie_band(logits, k, idx, w, band, rel_err=1e-5):
    """Routing check for every token, given the oracle's float64 logits and a
    device whose logits may differ from them by up to band / 2 each:
      * the device's k experts are distinct;
      * every expert whose logit exceeds the (k+1)-th largest by more than
        band is among them (no device rounding can drop it);
      * every expert among them is within band of the k-th largest logit
        (no device rounding can raise anything lower into the top k);
      * the weights are the softmax of the oracle's logits over the device's
        set, renormalised, slots in non-increasing weight.  Logits off by up
        to d each move a renormalised weight by a factor within e^(+-2d), so
        the tolerance is 1e-4 plus twice ``rel_err`` times the token's
        largest logit magnitude (the relative logit error the device is
        held to, applied to this token).
    Tokens whose k-th and (k+1)-th logits are further apart than band get
    exactly the oracle's set this way; near-tie tokens get one of the sets
    that are valid under the logit error."""
    logits = np.asarray(logits, np.float64)
    idx = np.asarray(idx)
    w = np.asarray(w, np.float64)
    T, E = logits.shape
    srt = -np.sort(-logits, axis=1)
    kth = srt[:, k - 1]
    k1 = srt[:, k] if k < E else np.full(T, -np.inf)
    for t in range(T):
        chosen = idx[t]
        assert len(set(chosen.tolist())) == k, f"token {t}: repeated experts {chosen}"
        assert np.all((chosen >= 0) & (chosen < E)), f"token {t}: expert out of range"
        must = np.nonzero(logits[t] > k1[t] + band)[0]
        missing = set(must.tolist()) - set(chosen.tolist())
        assert not missing, f"token {t}: experts {sorted(missing)} clearly in the top {k} are missing"
        assert np.all(logits[t, chosen] >= kth[t] - band), f"token {t}: an expert below the top-{k} band"
        z = logits[t, chosen] - logits[t, chosen].max()
        ref = np.exp(z) / np.exp(z).sum()
        rtol = 1e-4 + 2.0 * np.expm1(2.0 * rel_err * np.abs(logits[t]).max())
        np.testing.assert_allclose(w[t], ref, rtol=rtol, atol=1e-6, err_msg=f"token {t}: weights")
        assert np.all(np.diff(w[t]) <= 1e-6), f"token {t}: slots not in descending weight"


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
