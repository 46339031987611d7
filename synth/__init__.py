"""Seeded synthetic inputs for the sparse MoE expert layer.

This module holds the layer descriptions (shapes, routing rule, weight type)
and draws random tensors for them.  It contains none of the layer's arithmetic:
no routing, no matmul, no quantiser.  Both the CUDA path's tests/benchmark and
the CPU oracle read inputs made here.

Recipe (every tensor comes from its own torch.Generator, seeded from
(seed, layer name, tensor name, expert index) through a 64-bit mix):
  * x ~ N(0, 1) drawn fp32 and rounded to bf16 (round to nearest even).
  * router weights W_r ~ N(0, 1/H) fp32, so logits are ~N(0, 1) before bias;
    the skewed prefill layer uses N(0, 1.645/H) and a popularity bias
    b_e = -1.1 * ln(rank_e + 1) (Zipf s = 1.1 over a seeded random ranking).
  * LongCat-shaped layer: one i.i.d. N(0, 0.25^2) logit bias per expert.  The
    768 experts stay exchangeable, so a third of the picks land on the 256
    zero-computation experts in expectation.
  * expert weights ~ N(0, 0.02^2) drawn fp32, rounded to bf16.
  * int8 expert weights: integer codes round(N(0,1) * 31.75) clipped to +-127,
    with per-output-channel fp32 scales 0.02 * 4/127 * U(0.8, 1.2).

Tensors that dominate memory (expert weights) are drawn directly on the device
that will hold them; the small ones (x, router, bias) on the CPU.
"""
from __future__ import annotations

import math

import torch

# Layer descriptions.  Field names follow the library config.
#   hidden H, inter I, n_routed E_r, n_zero E_z, top_k k, n_group, topk_group,
#   per_group_k, score, renormalize, routed_scale, bias_mode, shared_inter, wdtype.
_BASE = dict(n_zero=0, n_group=1, topk_group=1, per_group_k=0, score="softmax",
             renormalize=False, routed_scale=1.0, bias_mode="none", shared_inter=0,
             wdtype="bf16", router_std_scale=1.0, bias_kind="none")

CONFIGS = {
    # T=16, hidden 256, 8 experts, softmax top-2 renormalised, intermediate 128.
    "tiny": dict(_BASE, T=16, hidden=256, inter=128, n_routed=8, top_k=2, renormalize=True),
    # LongCat-Flash-shaped decode: 512 FFN experts + 256 zero-computation experts.
    "longcat": dict(_BASE, T=64, hidden=6144, inter=2048, n_routed=512, n_zero=256, top_k=12,
                    bias_mode="logit", bias_kind="iid"),
    # DeepSeek-V3-shaped decode: 8 groups, top-4 groups then top-8, sigmoid, x2.5, shared.
    "dsv3": dict(_BASE, T=128, hidden=7168, inter=2048, n_routed=256, top_k=8, n_group=8,
                 topk_group=4, score="sigmoid", renormalize=True, routed_scale=2.5,
                 shared_inter=2048),
    # Pangu-MoGE-shaped decode: 8 groups, exactly top-1 per group, shared expert.
    "pangu": dict(_BASE, T=456, hidden=5120, inter=1536, n_routed=64, top_k=8, n_group=8,
                  per_group_k=1, shared_inter=4096),
    # Skewed W8A8 prefill.
    "w8a8_prefill": dict(_BASE, T=8192, hidden=7168, inter=2048, n_routed=256, top_k=8,
                         wdtype="w8a8", bias_mode="logit", bias_kind="zipf",
                         router_std_scale=1.645),
    # Scaled-down relatives used for element-by-element parity.  They keep each
    # layer's routing rule and stress several tiles plus a ragged tail.
    "longcat_s": dict(_BASE, T=48, hidden=1024, inter=384, n_routed=192, n_zero=96, top_k=12,
                      bias_mode="logit", bias_kind="iid"),
    "dsv3_s": dict(_BASE, T=128, hidden=1024, inter=320, n_routed=64, top_k=8, n_group=8,
                   topk_group=4, score="sigmoid", renormalize=True, routed_scale=2.5,
                   shared_inter=384),
    "pangu_s": dict(_BASE, T=456, hidden=640, inter=384, n_routed=64, top_k=8, n_group=8,
                    per_group_k=1, shared_inter=512),
    "ragged_s": dict(_BASE, T=37, hidden=1000, inter=200, n_routed=24, n_zero=8, top_k=5,
                     bias_mode="logit", bias_kind="iid", shared_inter=136),
    "w8a8_s": dict(_BASE, T=512, hidden=1024, inter=512, n_routed=32, top_k=8, wdtype="w8a8",
                   bias_mode="logit", bias_kind="zipf", router_std_scale=1.645),
    # Profiling-sized LongCat relative: full H and I, ~2 rows per expert like the
    # real layer, 4.8 GB of weights (well above the 129 MB L2, a few GB on device).
    "longcat_prof": dict(_BASE, T=16, hidden=6144, inter=2048, n_routed=64, n_zero=32,
                         top_k=12, bias_mode="logit", bias_kind="iid"),
    # LongCat-shaped decode layer with W8A8 weights (int8 halves the bytes each
    # step must stream): the W8A8 decode workload.
    "longcat_w8": dict(_BASE, T=64, hidden=6144, inter=2048, n_routed=512, n_zero=256, top_k=12,
                       bias_mode="logit", bias_kind="iid", wdtype="w8a8"),
    # LongCat's router and gating shape (T=64, H=6144, 768 experts, k=12) with
    # tiny experts (I=16, 0.3 GB): profiles the routing kernels alone.
    "longcat_router": dict(_BASE, T=64, hidden=6144, inter=16, n_routed=512, n_zero=256,
                           top_k=12, bias_mode="logit", bias_kind="iid"),
    # Profiling-sized relative of the W8A8 decode layer (2.4 GB of int8 weights).
    "longcat_w8_prof": dict(_BASE, T=16, hidden=6144, inter=2048, n_routed=64, n_zero=32,
                            top_k=12, bias_mode="logit", bias_kind="iid", wdtype="w8a8"),
    # DeepSeek-V3-shaped decode layer with W8A8 weights, shared expert included
    # (int8 like the routed experts, fed the same quantised token codes), and its
    # scaled-down relative.
    "dsv3_w8": dict(_BASE, T=128, hidden=7168, inter=2048, n_routed=256, top_k=8, n_group=8,
                    topk_group=4, score="sigmoid", renormalize=True, routed_scale=2.5,
                    shared_inter=2048, wdtype="w8a8"),
    "dsv3_w8_s": dict(_BASE, T=128, hidden=1024, inter=320, n_routed=64, top_k=8, n_group=8,
                      topk_group=4, score="sigmoid", renormalize=True, routed_scale=2.5,
                      shared_inter=384, wdtype="w8a8"),
    # Profiling-sized W8A8 prefill relative: full H and I, 64 experts, Zipf load,
    # 2.8 GB of int8 weights and 235 MB of activation codes.
    "w8a8_prof": dict(_BASE, T=2048, hidden=7168, inter=2048, n_routed=64, top_k=8,
                      wdtype="w8a8", bias_mode="logit", bias_kind="zipf", router_std_scale=1.645),
}

# The five headline layers, in order.
HEADLINE = ["tiny", "longcat", "dsv3", "pangu", "w8a8_prefill"]


def spec(base: str, **overrides) -> dict:
    """Copy of a named layer description; overrides may rename it ('name')."""
    d = dict(CONFIGS[base])
    d["name"] = base
    d.update(overrides)
    return d


def n_experts(s: dict) -> int:
    return s["n_routed"] + s["n_zero"]


def _mix(*parts) -> int:
    """Deterministic 63-bit seed from a tuple of ints/strings (splitmix64 chain)."""
    h = 0x9E3779B97F4A7C15
    for p in parts:
        if isinstance(p, str):
            v = 0
            for ch in p.encode():
                v = (v * 131 + ch) & 0xFFFFFFFFFFFFFFFF
        else:
            v = int(p) & 0xFFFFFFFFFFFFFFFF
        h = (h ^ v) & 0xFFFFFFFFFFFFFFFF
        h = (h + 0x9E3779B97F4A7C15) & 0xFFFFFFFFFFFFFFFF
        z = h
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & 0xFFFFFFFFFFFFFFFF
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & 0xFFFFFFFFFFFFFFFF
        h = z ^ (z >> 31)
    return h & 0x7FFFFFFFFFFFFFFF


def _gen(device, *parts) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(_mix(*parts))
    return g


def _normal(shape, std, device, *parts) -> torch.Tensor:
    return torch.randn(shape, generator=_gen(device, *parts), device=device,
                       dtype=torch.float32).mul_(std)


def draw_x(s: dict, seed: int = 0, T: int | None = None) -> torch.Tensor:
    """Token activations [T, H] bf16 on the CPU."""
    T = s["T"] if T is None else T
    return _normal((T, s["hidden"]), 1.0, "cpu", seed, s["name"], "x").to(torch.bfloat16)


def redraw_x_rows(s: dict, x: torch.Tensor, rows, attempt: int, seed: int = 0) -> None:
    """Replace the given rows of x by fresh draws from per-(row, attempt) substreams."""
    for t in rows:
        x[t] = _normal((s["hidden"],), 1.0, "cpu", seed, s["name"], "x-redraw", int(t),
                       attempt).to(torch.bfloat16)


def draw_router(s: dict, seed: int = 0):
    """(W_r [E_tot, H] fp32, bias [E_tot] fp32 or None) on the CPU."""
    E, H = n_experts(s), s["hidden"]
    std = math.sqrt(s["router_std_scale"] / H)
    w_r = _normal((E, H), std, "cpu", seed, s["name"], "w_router")
    bias = None
    if s["bias_kind"] == "iid":
        bias = _normal((E,), 0.25, "cpu", seed, s["name"], "bias")
    elif s["bias_kind"] == "zipf":
        rank = torch.randperm(E, generator=_gen("cpu", seed, s["name"], "popularity"))
        bias = (-1.1 * torch.log(rank.to(torch.float64) + 1.0)).to(torch.float32)
    return w_r, bias


def draw_expert_bf16(s: dict, which: str, e: int, device="cpu", seed: int = 0) -> torch.Tensor:
    """One expert matrix as bf16: 'gate'/'up' [I, H], 'down' [H, I];
    'shared_gate'/'shared_up' [I_s, H], 'shared_down' [H, I_s]."""
    H = s["hidden"]
    I = s["shared_inter"] if which.startswith("shared") else s["inter"]
    shape = (H, I) if which.endswith("down") else (I, H)
    return _normal(shape, 0.02, device, seed, s["name"], which, e).to(torch.bfloat16)


def draw_expert_int8(s: dict, which: str, e: int, device="cpu", seed: int = 0):
    """One int8 expert matrix with per-output-channel fp32 scales: (q, scale).
    which: 'gate'/'up' [I, H], 'down' [H, I], or the shared expert's
    'shared_gate'/'shared_up' [I_s, H], 'shared_down' [H, I_s]."""
    H = s["hidden"]
    I = s["shared_inter"] if which.startswith("shared") else s["inter"]
    shape = (H, I) if which.endswith("down") else (I, H)
    q = _normal(shape, 31.75, device, seed, s["name"], which + "-q", e).round_().clamp_(-127, 127)
    u = torch.rand((shape[0],), generator=_gen(device, seed, s["name"], which + "-s", e),
                   device=device, dtype=torch.float32)
    scale = (0.8 + 0.4 * u) * (0.02 * 4.0 / 127.0)
    return q.to(torch.int8), scale


def draw_weights(s: dict, device="cpu", seed: int = 0, experts=None) -> dict:
    """Stacked expert weights on `device`.

    bf16: {'w_gate': [E_r, I, H], 'w_up': [E_r, I, H], 'w_down': [E_r, H, I]} bf16, plus
    'shared_gate'/'shared_up' [I_s, H] and 'shared_down' [H, I_s] when shared_inter > 0.
    w8a8: int8 'w_gate'/'w_up'/'w_down' with fp32 's_gate'/'s_up' [E_r, I], 's_down' [E_r, H],
    plus int8 'shared_gate'/'shared_up' [I_s, H], 'shared_down' [H, I_s] with fp32
    's_shared_gate'/'s_shared_up' [I_s], 's_shared_down' [H] when shared_inter > 0.
    `experts`: optional iterable of expert indices to draw; the others stay zero.
    """
    E, H, I = s["n_routed"], s["hidden"], s["inter"]
    todo = range(E) if experts is None else sorted(set(int(e) for e in experts))
    out = {}
    if s["wdtype"] == "bf16":
        out["w_gate"] = torch.zeros((E, I, H), dtype=torch.bfloat16, device=device)
        out["w_up"] = torch.zeros((E, I, H), dtype=torch.bfloat16, device=device)
        out["w_down"] = torch.zeros((E, H, I), dtype=torch.bfloat16, device=device)
        for e in todo:
            out["w_gate"][e] = draw_expert_bf16(s, "gate", e, device, seed)
            out["w_up"][e] = draw_expert_bf16(s, "up", e, device, seed)
            out["w_down"][e] = draw_expert_bf16(s, "down", e, device, seed)
        if s["shared_inter"] > 0:
            for which in ("shared_gate", "shared_up", "shared_down"):
                out[which] = draw_expert_bf16(s, which, 0, device, seed)
    else:
        out["w_gate"] = torch.zeros((E, I, H), dtype=torch.int8, device=device)
        out["w_up"] = torch.zeros((E, I, H), dtype=torch.int8, device=device)
        out["w_down"] = torch.zeros((E, H, I), dtype=torch.int8, device=device)
        out["s_gate"] = torch.zeros((E, I), dtype=torch.float32, device=device)
        out["s_up"] = torch.zeros((E, I), dtype=torch.float32, device=device)
        out["s_down"] = torch.zeros((E, H), dtype=torch.float32, device=device)
        for e in todo:
            for which in ("gate", "up", "down"):
                q, sc = draw_expert_int8(s, which, e, device, seed)
                out["w_" + which][e] = q
                out["s_" + which][e] = sc
        if s["shared_inter"] > 0:
            for which in ("shared_gate", "shared_up", "shared_down"):
                q, sc = draw_expert_int8(s, which, 0, device, seed)
                out[which] = q
                out["s_" + which] = sc
    return out


def make_inputs(s: dict, seed: int = 0, accept_rows=None, max_attempts: int = 64):
    """x [T,H] bf16, W_r, bias on the CPU.

    accept_rows(x, w_r, bias) -> bool tensor [T] marks usable token rows (for
    instance rows whose routing has clear margins).  Rejected rows are redrawn
    from their own substreams until accepted.  Returns (x, w_r, bias, redraws).
    """
    x = draw_x(s, seed)
    w_r, bias = draw_router(s, seed)
    redraws = 0
    if accept_rows is not None:
        for attempt in range(max_attempts):
            ok = torch.as_tensor(accept_rows(x, w_r, bias), dtype=torch.bool)
            bad = torch.nonzero(~ok).flatten().tolist()
            if not bad:
                break
            redraws += len(bad)
            redraw_x_rows(s, x, bad, attempt, seed)
        else:
            raise RuntimeError(f"{s['name']}: rows still rejected after {max_attempts} redraws")
    return x, w_r, bias, redraws


def bf16_bits(t: torch.Tensor):
    """bf16 tensor -> numpy uint16 bit patterns (CPU copy)."""
    return t.detach().to("cpu").contiguous().view(torch.int16).numpy().view("uint16")
