"""Whole-layer pin of the oracle: an independent numpy float64 restatement.

The layer below is written from the method's steps (router matmul, scoring,
group stage, top-k, weights, per-pick SwiGLU expert, weighted combine with
zero-computation experts and the shared expert; the W8A8 variant's per-row
symmetric quantiser, exact integer matmuls and dequantisation acc * s_row *
s_channel), vectorised with numpy and sharing nothing with ``moe_oracle.c``
beyond the inputs.  Sources, cited by page title and section:
  * "LongCat-Flash与GLM-4.6V，昇腾CANN异构计算深水区突围详解", 拆解MoE困局: the
    768-way choice over 512 FFN and 256 zero-computation experts, dispatch and
    combine.
  * "基于Atlas 900 A3 SuperPoD的LongCat-Flash模型推理性能优化实践", 背景介绍 (a
    token routed to a zero-computation expert passes through unchanged) and
    优化措施三 (Router Matmul; QuantBatchMatmul).
  * "华为技术披露集 VOL.12：昇腾×盘古", opening section (MoGE: one winner per
    group) and 分层混合并行（H2P） (grouped routed experts, shared expert).
  * DeepSeek-V3/R1 on Ascend (Huxiu article), deployment paragraph (one shared
    expert beside the routed ones) and "2. 模型侧并发优化" (quantised
    activations travel with their per-row scales).

Shapes are the headline layers scaled down (tiny as is; DSv3-, Pangu- and
LongCat-shaped relatives; a W8A8 layer whose token scales differ from 1 and
whose per-channel weight scales differ across channels), so that the oracle's
dequantisation, routing weights and combine are each exercised by values that
a dropped factor or a wrong index would change.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests import support


# --------------------------------------------------------------- routing ----

def np_route(spec, x, w_r, bias):
    """-> ids [T,k] (slot order), weights [T,k] float64."""
    T = x.shape[0]
    E, k = synth.n_experts(spec), spec["top_k"]
    b = None if bias is None else bias.astype(np.float64)
    logits = x @ w_r.astype(np.float64).T
    if spec["bias_mode"] == "logit":
        logits = logits + b[None, :]
    if spec["score"] == "softmax":
        z = np.exp(logits - logits.max(axis=1, keepdims=True))
        scores = z / z.sum(axis=1, keepdims=True)
    else:
        scores = 1.0 / (1.0 + np.exp(-logits))
    keys = scores + (b[None, :] if spec["bias_mode"] == "select" else 0.0)
    ng = spec["n_group"]
    G = E // ng
    ids = np.empty((T, k), np.int64)
    for t in range(T):
        kt = keys[t]
        # (key descending, index ascending): a stable sort of the negated keys
        order = np.argsort(-kt, kind="stable")
        if ng == 1:
            pick = order[:k]
        elif spec["per_group_k"] > 0:
            pk = spec["per_group_k"]
            winners = []
            for g in range(ng):
                sub = kt[g * G:(g + 1) * G]
                winners.extend(g * G + np.argsort(-sub, kind="stable")[:pk])
            winners = np.array(winners)
            pick = winners[np.lexsort((winners, -kt[winners]))]
        else:
            gscore = np.sort(kt.reshape(ng, G), axis=1)[:, ::-1][:, :2].sum(axis=1)
            keep = np.argsort(-gscore, kind="stable")[:spec["topk_group"]]
            eligible = np.zeros(E, bool)
            for g in keep:
                eligible[g * G:(g + 1) * G] = True
            pick = np.array([e for e in order if eligible[e]][:k])
        ids[t] = pick
    w = np.take_along_axis(scores, ids, axis=1)
    if spec["renormalize"]:
        w = w / w.sum(axis=1, keepdims=True)
    w = w * float(spec["routed_scale"] or 1.0)
    return ids, w


# ----------------------------------------------------------------- bf16 ----

def _silu(g):
    return g / (1.0 + np.exp(-g))


def np_layer_bf16(spec, x, w_r, bias, wts):
    """out [T,H] float64 of the bf16-weight layer."""
    T, H = x.shape
    ids, w = np_route(spec, x, w_r, bias)
    Er = spec["n_routed"]
    out = np.zeros((T, H))
    wg = wts["w_gate"].to(torch.float64).numpy() if Er else None
    wu = wts["w_up"].to(torch.float64).numpy() if Er else None
    wd = wts["w_down"].to(torch.float64).numpy() if Er else None
    for e in range(synth.n_experts(spec)):
        tok, slot = np.nonzero(ids == e)
        if tok.size == 0:
            continue
        if e >= Er:  # zero-computation expert: the token itself
            y = x[tok]
        else:
            xe = x[tok]
            y = (_silu(xe @ wg[e].T) * (xe @ wu[e].T)) @ wd[e].T
        np.add.at(out, tok, w[tok, slot][:, None] * y)
    if spec["shared_inter"] > 0:
        sg, su, sd = (wts[n].to(torch.float64).numpy()
                      for n in ("shared_gate", "shared_up", "shared_down"))
        out += (_silu(x @ sg.T) * (x @ su.T)) @ sd.T
    return out, ids, w


# ----------------------------------------------------------------- W8A8 ----

def np_quantise(v32):
    """Per-row symmetric int8 in IEEE float32: s = amax/127, q = rint(v/s) clipped."""
    v32 = v32.astype(np.float32)
    amax = np.abs(v32).max(axis=1)
    s = (amax / np.float32(127.0)).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        z = np.rint(v32 / s[:, None])
    z = np.where(amax[:, None] > 0, np.clip(z, -127, 127), 0)
    return z.astype(np.int64), s


def _np_w8_expert(q, rs, qg, sg, qu, su, qd, sd):
    """W8A8 SwiGLU expert on code rows q [n,H] with row scales rs [n,1]."""
    g = (q @ qg.T).astype(np.float64) * rs * sg[None, :]
    u = (q @ qu.T).astype(np.float64) * rs * su[None, :]
    h32 = (_silu(g) * u).astype(np.float32)
    qh, sh = np_quantise(h32)
    return (qh @ qd.T).astype(np.float64) * sh.astype(np.float64)[:, None] * sd[None, :]


def np_layer_w8a8(spec, xbits, w_r, bias, wts):
    """out [T,H] float64 of the W8A8 layer (the shared expert, when present, is
    int8 too and takes the same token codes)."""
    x32 = support.bf16_to_f64(xbits).astype(np.float32)
    x = x32.astype(np.float64)
    T, H = x.shape
    ids, w = np_route(spec, x, w_r, bias)
    Er = spec["n_routed"]
    qx, sx = np_quantise(x32)
    out = np.zeros((T, H))
    qg, qu, qd = (wts[n].numpy().astype(np.int64) for n in ("w_gate", "w_up", "w_down"))
    sg, su, sd = (wts[n].numpy().astype(np.float64) for n in ("s_gate", "s_up", "s_down"))
    for e in range(synth.n_experts(spec)):
        tok, slot = np.nonzero(ids == e)
        if tok.size == 0:
            continue
        if e >= Er:
            y = x[tok]
        else:
            rs = sx[tok].astype(np.float64)[:, None]
            y = _np_w8_expert(qx[tok], rs, qg[e], sg[e], qu[e], su[e], qd[e], sd[e])
        np.add.at(out, tok, w[tok, slot][:, None] * y)
    if spec["shared_inter"] > 0:
        m = lambda n: wts[n].numpy().astype(np.int64)
        f = lambda n: wts[n].numpy().astype(np.float64)
        out += _np_w8_expert(qx, sx.astype(np.float64)[:, None], m("shared_gate"),
                             f("s_shared_gate"), m("shared_up"), f("s_shared_up"),
                             m("shared_down"), f("s_shared_down"))
    return out, ids, w, qx, sx


# ---------------------------------------------------------------- tests ----

def _close(a, b, rtol):
    scale = np.abs(b).max()
    assert np.abs(a - b).max() <= rtol * scale, (np.abs(a - b).max(), scale)


@pytest.mark.parametrize("name", ["tiny", "dsv3_s", "pangu_s", "longcat_s", "ragged_s"])
def test_bf16_layer_matches_numpy_restatement(name):
    s = synth.spec(name)
    x, w_r, bias, _ = support.make_inputs(s)
    wts = synth.draw_weights(s)
    out, ids, w = support.oracle_layer(s, x, w_r, bias, wts)
    xf = support.bf16_to_f64(synth.bf16_bits(x))
    ref, ids_ref, w_ref = np_layer_bf16(s, xf, w_r.numpy(), support.np_bias(bias), wts)
    assert np.array_equal(ids, ids_ref)
    assert np.allclose(w, w_ref, rtol=1e-12, atol=0)
    _close(out, ref, 1e-11)


def test_routing_weights_are_not_all_one():
    # The combine pins above only catch a dropped routing weight if the weights
    # differ from 1; check that for the layers they run.
    for name in ("tiny", "dsv3_s", "pangu_s", "longcat_s"):
        s = synth.spec(name)
        x, w_r, bias, _ = support.make_inputs(s)
        xf = support.bf16_to_f64(synth.bf16_bits(x))
        _, w = np_route(s, xf, w_r.numpy(), support.np_bias(bias))
        assert np.abs(w - 1.0).min() > 1e-3


W8_PIN = dict(synth._BASE, name="w8_numpy_pin", T=40, hidden=256, inter=96, n_routed=8, n_zero=2,
              top_k=3, wdtype="w8a8", bias_mode="logit", bias_kind="iid")


def _w8_case():
    s = dict(W8_PIN)
    x, w_r, bias, _ = support.make_inputs(s)
    wts = synth.draw_weights(s)
    return s, x, w_r, bias, wts


def _oracle_w8(s, x, w_r, bias, wts):
    E = s["n_routed"]
    lst = lambda n: [wts[n][e].numpy() for e in range(E)]
    shared = None
    if s["shared_inter"] > 0:
        shared = tuple(wts[n].numpy() for n in ("shared_gate", "s_shared_gate", "shared_up",
                                                "s_shared_up", "shared_down", "s_shared_down"))
    return oracle.layer_w8a8(s, synth.bf16_bits(x), w_r.numpy(), support.np_bias(bias),
                             lst("w_gate"), lst("s_gate"), lst("w_up"), lst("s_up"),
                             lst("w_down"), lst("s_down"), shared)


def test_w8a8_inputs_exercise_every_scale():
    s, x, w_r, bias, wts = _w8_case()
    _, _, _, qx, sx = np_layer_w8a8(s, synth.bf16_bits(x), w_r.numpy(), support.np_bias(bias),
                                    wts)
    # token scales far from 1 (x ~ N(0,1): amax ~ 3, scale ~ 0.025) and varied
    # (bf16 amax values repeat, so not all distinct)
    assert np.all(np.abs(sx - 1.0) > 0.5) and len(np.unique(sx)) > s["T"] // 2
    # per-channel weight scales differ across the channels of one expert
    for n in ("s_gate", "s_up", "s_down"):
        v = wts[n].numpy()
        assert np.all(v.max(axis=1) / v.min(axis=1) > 1.1)
    # the codes are not all at the clip value, so the scale is not trivially amax
    assert np.mean(np.abs(qx) == 127) < 0.05


def test_w8a8_layer_matches_numpy_restatement():
    s, x, w_r, bias, wts = _w8_case()
    out, ids, w, qx, sx = _oracle_w8(s, x, w_r, bias, wts)
    ref, ids_ref, w_ref, qx_ref, sx_ref = np_layer_w8a8(s, synth.bf16_bits(x), w_r.numpy(),
                                                        support.np_bias(bias), wts)
    assert np.array_equal(ids, ids_ref)
    assert np.allclose(w, w_ref, rtol=1e-12, atol=0)
    assert np.array_equal(sx, sx_ref)
    assert np.array_equal(qx.astype(np.int64), qx_ref)
    assert np.any(ids >= s["n_routed"]) and np.any(ids < s["n_routed"])
    # The intermediate h is rounded to fp32 and re-quantised on both sides; a
    # rounding-boundary straddle between two fp64 evaluations of silu would move
    # one code by one step, far below this bound but far above fp64 noise.
    _close(out, ref, 1e-9)


W8_SHARED_PIN = dict(W8_PIN, name="w8_numpy_shared_pin", n_group=2, topk_group=1, n_zero=0,
                     bias_mode="none", bias_kind="none", score="sigmoid", renormalize=True,
                     routed_scale=2.5, shared_inter=72)


def test_w8a8_layer_with_shared_expert_matches_numpy_restatement():
    # DSv3-like routing (sigmoid, groups, renormalised x 2.5) plus an int8 shared
    # expert fed the same token codes; the shared expert's scales vary by channel
    s = dict(W8_SHARED_PIN)
    x, w_r, bias, _ = support.make_inputs(s)
    wts = synth.draw_weights(s)
    v = wts["s_shared_down"].numpy()
    assert v.max() / v.min() > 1.1
    out, ids, w, qx, sx = _oracle_w8(s, x, w_r, bias, wts)
    ref, ids_ref, w_ref, _, _ = np_layer_w8a8(s, synth.bf16_bits(x), w_r.numpy(),
                                              support.np_bias(bias), wts)
    assert np.array_equal(ids, ids_ref)
    assert np.allclose(w, w_ref, rtol=1e-12, atol=0)
    _close(out, ref, 1e-9)
    # the shared expert's part is not negligible
    no_shared = _oracle_w8(dict(s, shared_inter=0), x, w_r, bias, wts)[0]
    assert np.abs(out - no_shared).max() > 0.05 * np.abs(out).max()
