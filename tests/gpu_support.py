"""Helpers for the GPU parity tests: device inputs, layer calls through the C ABI,
and the tolerance checks.

Tolerances: routing ids, permutation, counts and offsets are compared exactly;
routing weights within 1e-5 relative (fp32 vs fp64 scoring); layer outputs
within relative L2 <= 5e-3 and max-abs <= 2e-2 in the fp32-output mode, and in
the bf16-output mode within relative L2 <= 5e-3 and
|out - oracle| <= 2e-2 + half a bf16 ulp of the oracle value (bf16 rounding
alone exceeds 2e-2 once |out| >= 8).
"""
from __future__ import annotations

import numpy as np
import torch

import synth
from tests import support

REL_L2 = 5e-3
MAX_ABS = 2e-2

# Layers small enough for the one-CTA router (T * E * H at most 2^20, x and W_r
# within one CTA's shared memory next to the re-sort's bitmap), with the
# routing rules of the larger layers: DSv3-style groups with a sigmoid, a
# select-only bias and a scale; zero-computation experts and a logit bias at a
# single token and an H that is not a multiple of 64; MoGE per-group picks with
# a shared expert; more tokens than warps.
ONE_CTA = {
    "one_cta_groups": dict(T=5, hidden=136, inter=64, n_routed=32, top_k=4, n_group=4,
                           topk_group=2, score="sigmoid", bias_mode="select", bias_kind="iid",
                           routed_scale=2.5, renormalize=True),
    "one_cta_zero": dict(T=1, hidden=200, inter=48, n_routed=32, n_zero=16, top_k=6,
                         bias_mode="logit", bias_kind="iid", renormalize=False),
    "one_cta_per_group": dict(T=33, hidden=512, inter=64, n_routed=16, top_k=4, n_group=4,
                              per_group_k=1, shared_inter=96),
    "one_cta_tokens": dict(T=64, hidden=256, inter=32, n_routed=24, top_k=3),
}


# Layers small enough for the small-layer FFN kernel (at most 16 tokens, H and I
# multiples of 64 up to 256, no shared expert, one expert's weights within one
# CTA's shared memory): every token on every expert (16 rows per expert, both 8-row MMA tiles),
# and a ragged one (3 tokens, most experts empty, zero-computation experts).
SMALL_FFN = {
    "small_ffn_full": dict(T=16, hidden=256, inter=128, n_routed=8, top_k=8, renormalize=True),
    "small_ffn_ragged": dict(T=3, hidden=192, inter=64, n_routed=16, n_zero=4, top_k=2,
                             bias_mode="logit", bias_kind="iid", renormalize=False),
    # the smallest dimensions (one 16-channel tile per CTA in both passes), one token
    "small_ffn_min": dict(T=1, hidden=64, inter=64, n_routed=4, top_k=2, renormalize=True),
}


def layer_spec(name: str) -> dict:
    """A named layer, or one of the one-CTA routing or small-FFN shapes (built on 'tiny')."""
    if name in ONE_CTA:
        return synth.spec("tiny", name=name, **ONE_CTA[name])
    if name in SMALL_FFN:
        return synth.spec("tiny", name=name, **SMALL_FFN[name])
    return synth.spec(name)

_cache = {}


def lib():
    import __graft_entry__

    __graft_entry__._builder().build()
    import sparse_expert_layer_gb300 as m

    return m


def inputs(spec: dict, device="cuda", weights_on="cpu"):
    """(x, w_r, bias) CPU + device copies and weights (on `weights_on`) for a spec."""
    key = (spec["name"], tuple(sorted((k, str(v)) for k, v in spec.items())), weights_on)
    if key in _cache:
        return _cache[key]
    x, w_r, bias, _ = support.make_inputs(spec)
    wts = synth.draw_weights(spec, device=weights_on)
    d = dict(x=x, w_r=w_r, bias=bias, wts=wts,
             x_d=x.to(device), w_r_d=w_r.to(device),
             bias_d=None if bias is None else bias.to(device),
             wts_d={k: v.to(device) for k, v in wts.items()})
    _cache.clear()
    _cache[key] = d
    return d


def run_layer(m, spec, d, out_fp32=True, gemv_max_rows=0, x=None, combine=0, ffn_launch=0):
    cfg = m.config_from_spec(spec, out_fp32=out_fp32, gemv_max_rows=gemv_max_rows,
                             combine=combine, ffn_launch=ffn_launch)
    x = d["x_d"] if x is None else x
    T = x.shape[0]
    out = torch.empty((T, spec["hidden"]), dtype=torch.float32 if out_fp32 else torch.bfloat16,
                      device=x.device)
    ws = m.workspace(cfg, T, x.device)
    w = d["wts_d"]
    m.moe_layer_forward(cfg, T, x, d["w_r_d"], d["bias_d"], w.get("w_gate"), w.get("w_up"),
                        w.get("w_down"), *m.layer_scales(w), w.get("shared_gate"),
                        w.get("shared_up"), w.get("shared_down"), out, ws)
    torch.cuda.synchronize()
    st = m.moe_check_device_status(ws)
    assert st == m.MOE_OK, f"device status {st}"
    return out


def bf16_half_ulp(v: np.ndarray) -> np.ndarray:
    a = np.abs(v)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, 2.0 ** (e - 8), 0.0)


def check_out(got: torch.Tensor, ref: np.ndarray, bf16_out: bool, what=""):
    g = got.float().cpu().double().numpy()
    d = g - ref
    rel = np.linalg.norm(d) / max(np.linalg.norm(ref), 1e-30)
    mx = np.abs(d).max() if d.size else 0.0
    assert rel <= REL_L2, f"{what}: rel-L2 {rel:.3e} > {REL_L2}"
    if bf16_out:
        bound = MAX_ABS + bf16_half_ulp(ref)
        worst = np.max(np.abs(d) - bound) if d.size else -1
        assert worst <= 0, f"{what}: |d| exceeds 2e-2 + ulp/2 by {worst:.3e}"
    else:
        assert mx <= MAX_ABS, f"{what}: max-abs {mx:.3e} > {MAX_ABS}"
    return rel, mx


def expert_lists_from_device(wts_d: dict, experts):
    """Per-expert CPU bit arrays for only the given experts (others None)."""
    E = wts_d["w_gate"].shape[0]
    want = set(int(e) for e in experts)
    g, u, dn = [], [], []
    for e in range(E):
        if e in want:
            g.append(synth.bf16_bits(wts_d["w_gate"][e]))
            u.append(synth.bf16_bits(wts_d["w_up"][e]))
            dn.append(synth.bf16_bits(wts_d["w_down"][e]))
        else:
            g.append(None)
            u.append(None)
            dn.append(None)
    return g, u, dn
