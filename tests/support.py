"""Test helpers: routing-margin predicate and oracle marshalling.

The margin rule keeps every routing decision clear of rounding: for each token,
consecutive selection keys that decide a pick (the top k+1 of the eligible
experts, the group-cut boundary, and each group's winner boundary) differ by at
least `margin`.  Softmax layers measure it on the logits (softmax is monotone,
and probabilities of ~1/768 cannot be 1e-3 apart); sigmoid layers on the keys.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import synth

MARGIN = 1e-3


def _gaps_ok(v: np.ndarray, n: int, margin: float) -> bool:
    """Sorted descending, the first n adjacent gaps (positions 0..n) are >= margin."""
    s = np.sort(v)[::-1]
    n = min(n, len(s) - 1)
    return bool(np.all(s[:n] - s[1:n + 1] >= margin)) if n > 0 else True


def margin_rows(spec: dict, x: torch.Tensor, w_r: torch.Tensor, bias, margin: float = MARGIN):
    """Bool array [T]: True where the token's routing has clear margins."""
    b = None if bias is None else bias.numpy()
    logits = oracle.router_logits(spec, synth.bf16_bits(x), w_r.numpy(), b)
    _, _, _, keys = oracle.select(spec, logits, b)
    use_logits = spec["score"] == "softmax" and spec["bias_mode"] != "select"
    space = logits if use_logits else keys
    E, k = synth.n_experts(spec), spec["top_k"]
    ng = spec["n_group"]
    G = E // ng
    ok = np.ones(x.shape[0], dtype=bool)
    for t in range(x.shape[0]):
        v = space[t]
        if ng == 1:
            ok[t] = _gaps_ok(v, k, margin)
        elif spec["per_group_k"] == 0:
            kt = keys[t].reshape(ng, G)
            top2 = np.sort(kt, axis=1)[:, ::-1][:, :min(2, G)].sum(axis=1)
            good = _gaps_ok(top2, spec["topk_group"], margin)
            keep = np.argsort(-top2, kind="stable")[:spec["topk_group"]]
            allowed = np.concatenate([v[g * G:(g + 1) * G] for g in sorted(keep)])
            ok[t] = good and _gaps_ok(allowed, k, margin)
        else:
            pk = spec["per_group_k"]
            vg = v.reshape(ng, G)
            good = all(_gaps_ok(vg[g], pk, margin) for g in range(ng))
            winners = np.concatenate([np.sort(vg[g])[::-1][:pk] for g in range(ng)])
            ok[t] = good and _gaps_ok(winners, len(winners) - 1, margin)
    return ok


def make_inputs(spec: dict, seed: int = 0):
    """(x, w_r, bias, redraws) with margins enforced through the oracle's keys."""
    return synth.make_inputs(spec, seed,
                             accept_rows=lambda x, w, b: margin_rows(spec, x, w, b))


def np_bias(bias):
    return None if bias is None else bias.numpy()


def expert_lists(weights: dict, experts=None):
    """Per-expert numpy lists (gate, up, down) of bf16 bit patterns; experts not in
    `experts` are None (the oracle then refuses to route to them)."""
    E = weights["w_gate"].shape[0]
    want = set(range(E)) if experts is None else set(int(e) for e in experts)
    g, u, d = [], [], []
    for e in range(E):
        if e in want:
            g.append(synth.bf16_bits(weights["w_gate"][e]))
            u.append(synth.bf16_bits(weights["w_up"][e]))
            d.append(synth.bf16_bits(weights["w_down"][e]))
        else:
            g.append(None)
            u.append(None)
            d.append(None)
    return g, u, d


def shared_tuple(weights: dict):
    if "shared_gate" not in weights:
        return None
    return tuple(synth.bf16_bits(weights[k]) for k in ("shared_gate", "shared_up", "shared_down"))


def oracle_layer(spec, x, w_r, bias, weights, experts=None):
    g, u, d = expert_lists(weights, experts)
    return oracle.layer(spec, synth.bf16_bits(x), w_r.numpy(), np_bias(bias), g, u, d,
                        shared_tuple(weights))


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
