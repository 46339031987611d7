"""Pins of the fp64 CPU oracle against facts fixed outside it.

Each test checks the oracle against something other than itself: brute force on
tiny inputs, closed forms, invariants, special cases that reduce to a textbook
dense computation, and the structural constants the pages print.  The cases are
chosen so that a plausible slip (wrong order, dropped term, swapped gate/up,
transposed operand, wrong tie rule) fails at least one of them.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import synth
from tests import support

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def mk(**kw):
    d = dict(synth._BASE)
    d.update(kw)
    d.setdefault("name", "pin")
    return d


def bf16(a):
    return synth.bf16_bits(torch.as_tensor(np.asarray(a, dtype=np.float32)).to(torch.bfloat16))


# ---------------------------------------------------------------- scores ----

def test_sigmoid_closed_forms():
    s = mk(hidden=8, inter=8, n_routed=4, top_k=4, score="sigmoid")
    logits = np.array([[0.0, math.log(3.0), -math.log(3.0), 2.0]])
    ids, w, sc, key = oracle.select(s, logits)
    assert sc[0, 0] == 0.5
    assert abs(sc[0, 1] - 0.75) < 1e-15
    assert abs(sc[0, 2] - 0.25) < 1e-15
    assert abs(sc[0, 3] + 1.0 / (1.0 + math.e ** 2) - 1.0) < 1e-15
    # no renormalisation: weights are the picked scores, slots in key order
    assert list(ids[0]) == [3, 1, 0, 2]
    assert np.allclose(w[0], sc[0, ids[0]], rtol=0, atol=0)


def test_softmax_closed_form_and_shift_invariance():
    s = mk(hidden=8, inter=8, n_routed=3, top_k=3)
    base = np.array([0.0, math.log(2.0), math.log(3.0)])
    for c in (0.0, 7.25, -40.0):
        _, _, sc, _ = oracle.select(s, (base + c)[None, :])
        assert np.allclose(sc[0], [1 / 6, 2 / 6, 3 / 6], rtol=0, atol=2e-15)


def test_renormalised_top2_weights_closed_form():
    # top-2 of logits (1, 3, 2, 0) renormalised: the softmax denominator cancels,
    # leaving e^3/(e^3+e^2) = 1/(1+e^-1) and e^-1/(1+e^-1).
    s = mk(hidden=8, inter=8, n_routed=4, top_k=2, renormalize=True, routed_scale=2.5)
    ids, w, _, _ = oracle.select(s, np.array([[1.0, 3.0, 2.0, 0.0]]))
    assert list(ids[0]) == [1, 2]
    a = 1.0 / (1.0 + math.exp(-1.0))
    assert abs(w[0, 0] - 2.5 * a) < 1e-15 and abs(w[0, 1] - 2.5 * (1 - a)) < 1e-15


def test_weights_sum_to_scale_when_renormalised():
    rng = np.random.default_rng(1)
    for score in ("softmax", "sigmoid"):
        s = mk(hidden=8, inter=8, n_routed=32, top_k=6, renormalize=True, routed_scale=2.5,
               score=score)
        _, w, _, _ = oracle.select(s, rng.normal(size=(50, 32)))
        assert np.all(np.abs(w.sum(1) - 2.5) < 1e-14)


def test_ties_go_to_lower_index():
    s = mk(hidden=8, inter=8, n_routed=6, top_k=3)
    ids, _, _, _ = oracle.select(s, np.array([[1.0, 3.0, 3.0, 2.0, 3.0, 0.0]]))
    assert list(ids[0]) == [1, 2, 4]
    s2 = mk(hidden=8, inter=8, n_routed=6, top_k=1)
    ids, _, _, _ = oracle.select(s2, np.array([[5.0, 5.0, 5.0, 5.0, 5.0, 5.0]]))
    assert ids[0, 0] == 0


# ----------------------------------------------------- brute-force top-k ----

def _subset_best(cands, key, k):
    return max(itertools.combinations(cands, k), key=lambda S: sum(key[e] for e in S))


@pytest.mark.parametrize("E,k", [(6, 1), (7, 3), (10, 4), (12, 2)])
def test_flat_topk_matches_brute_force(E, k):
    rng = np.random.default_rng(E * 10 + k)
    s = mk(hidden=8, inter=8, n_routed=E, top_k=k)
    logits = rng.normal(size=(40, E))
    ids, _, _, key = oracle.select(s, logits)
    for t in range(40):
        best = _subset_best(range(E), key[t], k)
        assert set(ids[t]) == set(best)
        assert np.all(np.diff(key[t, ids[t]]) < 0)  # slots in descending key order


@pytest.mark.parametrize("E,ng,tg,k", [(12, 4, 2, 3), (16, 4, 1, 2), (16, 8, 3, 4), (9, 3, 2, 5)])
def test_group_limited_topk_matches_brute_force(E, ng, tg, k):
    rng = np.random.default_rng(E + ng * 7 + tg * 13 + k)
    s = mk(hidden=8, inter=8, n_routed=E, top_k=k, n_group=ng, topk_group=tg, score="sigmoid")
    logits = rng.normal(size=(30, E))
    ids, _, _, key = oracle.select(s, logits)
    G = E // ng
    for t in range(30):
        kt = key[t]
        gscore = [sum(sorted(kt[g * G:(g + 1) * G], reverse=True)[:2]) for g in range(ng)]
        gbest = _subset_best(range(ng), gscore, tg)
        cands = [e for e in range(E) if e // G in gbest]
        best = _subset_best(cands, kt, k)
        assert set(ids[t]) == set(best)
        assert np.all(np.diff(kt[ids[t]]) < 0)


@pytest.mark.parametrize("E,ng,pk", [(8, 4, 1), (12, 3, 2), (16, 8, 1)])
def test_per_group_topk_matches_brute_force(E, ng, pk):
    rng = np.random.default_rng(E * 3 + ng + pk)
    s = mk(hidden=8, inter=8, n_routed=E, top_k=ng * pk, n_group=ng, per_group_k=pk)
    logits = rng.normal(size=(30, E))
    ids, _, _, key = oracle.select(s, logits)
    G = E // ng
    for t in range(30):
        want = set()
        for g in range(ng):
            want |= set(_subset_best(range(g * G, (g + 1) * G), key[t], pk))
        assert set(ids[t]) == want
        assert np.all(np.diff(key[t, ids[t]]) < 0)
        per_group = np.bincount(np.asarray(ids[t]) // G, minlength=ng)
        assert np.all(per_group == pk)  # balanced by construction


def test_select_bias_moves_choice_but_not_weights():
    s = mk(hidden=8, inter=8, n_routed=4, top_k=1, score="sigmoid", bias_mode="select")
    logits = np.array([[2.0, 1.0, 0.0, -1.0]])
    bias = np.array([0.0, 0.5, 0.0, 0.0], np.float32)
    ids, w, sc, key = oracle.select(s, logits, bias)
    assert ids[0, 0] == 1  # sigmoid(1)+0.5 > sigmoid(2)
    assert w[0, 0] == sc[0, 1] == 1.0 / (1.0 + math.exp(-1.0))
    assert key[0, 1] == sc[0, 1] + 0.5


# ---------------------------------------------------------------- router ----

def test_router_one_hot_rows_select_columns():
    rng = np.random.default_rng(3)
    H, E = 24, 5
    s = mk(hidden=H, inter=8, n_routed=E, top_k=1)
    w_r = rng.normal(size=(E, H)).astype(np.float32)
    x = np.zeros((H, H), np.float32)
    np.fill_diagonal(x, 1.0)
    logits = oracle.router_logits(s, bf16(x), w_r)
    assert np.array_equal(logits, w_r.T.astype(np.float64))
    x2 = np.zeros((1, H), np.float32)
    x2[0, 3], x2[0, 7] = 2.0, -0.5
    l2 = oracle.router_logits(s, bf16(x2), w_r)
    assert np.allclose(l2[0], 2.0 * w_r[:, 3].astype(np.float64) - 0.5 * w_r[:, 7], rtol=0,
                       atol=1e-12)


def test_router_logit_bias_is_added():
    rng = np.random.default_rng(4)
    H, E = 16, 6
    w_r = rng.normal(size=(E, H)).astype(np.float32)
    x = bf16(rng.normal(size=(3, H)))
    bias = rng.normal(size=E).astype(np.float32)
    l0 = oracle.router_logits(mk(hidden=H, inter=8, n_routed=E, top_k=1), x, w_r)
    l1 = oracle.router_logits(mk(hidden=H, inter=8, n_routed=E, top_k=1, bias_mode="logit"), x,
                              w_r, bias)
    assert np.allclose(l1 - l0, bias[None, :].astype(np.float64), rtol=0, atol=1e-14)


# --------------------------------------------------------------- permute ----

def test_permutation_invariants_and_brute_force():
    rng = np.random.default_rng(5)
    T, k, E = 37, 5, 23
    ids = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)
    counts, offsets, s2e, e2s = oracle.permute(ids, E)
    flat = ids.reshape(-1)
    assert counts.sum() == T * k and offsets[0] == 0 and offsets[-1] == T * k
    assert np.all(np.diff(offsets) == counts)
    assert np.array_equal(counts, np.bincount(flat, minlength=E))
    assert np.array_equal(s2e[e2s], np.arange(T * k))  # bijection
    assert np.array_equal(e2s[s2e], np.arange(T * k))
    brute = sorted(range(T * k), key=lambda r: (flat[r], r // k))
    assert np.array_equal(s2e, np.array(brute))
    assert np.all(np.diff(flat[s2e]) >= 0)


def test_permutation_rejects_out_of_range_ids():
    with pytest.raises(ValueError):
        oracle.permute(np.array([[0, 4]], np.int32), 4)


# ------------------------------------------------------------------- FFN ----

def test_swiglu_odd_part_identity():
    # gate rows (+a, -a), up rows (1, 1), down row (1, -1):
    # y0 = silu(a) - silu(-a) = a for every a; swapping gate and up breaks it.
    H, I = 2, 2
    wg = bf16([[1.0, 0.0], [-1.0, 0.0]])
    wu = bf16([[0.0, 1.0], [0.0, 1.0]])
    wd = bf16([[1.0, -1.0], [0.0, 0.0]])
    for a in (0.0, 0.75, -3.0, 9.5):
        y, h = oracle.swiglu_expert(np.array([a, 1.0]), wg, wu, wd)
        assert abs(y[0] - a) < 1e-13 and y[1] == 0.0
        assert h[0] > h[1] or a <= 0


def _dense_swiglu(x, wg, wu, wd):
    """Textbook dense SwiGLU FFN with numpy float64 matmuls."""
    g = support.bf16_to_f64(wg) @ x
    u = support.bf16_to_f64(wu) @ x
    return support.bf16_to_f64(wd) @ (g / (1.0 + np.exp(-g)) * u)


def test_single_expert_top1_is_dense_swiglu():
    s = mk(T=9, hidden=40, inter=24, n_routed=1, top_k=1, name="dense1")
    x, w_r, bias, _ = synth.make_inputs(s)
    wts = synth.draw_weights(s)
    out, ids, w = support.oracle_layer(s, x, w_r, bias, wts)
    assert np.all(ids == 0) and np.all(w == 1.0)
    xb = support.bf16_to_f64(synth.bf16_bits(x))
    g, u, d = support.expert_lists(wts)
    for t in range(s["T"]):
        ref = _dense_swiglu(xb[t], g[0], u[0], d[0])
        assert np.allclose(out[t], ref, rtol=1e-12, atol=1e-14)


def test_zero_experts_return_weighted_input_exactly():
    s = mk(T=11, hidden=32, inter=16, n_routed=4, n_zero=4, top_k=3, bias_mode="logit",
           name="zeros")
    x, w_r, _, _ = synth.make_inputs(s)
    bias = torch.tensor([-1e3] * 4 + [0.0] * 4)
    wts = synth.draw_weights(s)
    out, ids, w = support.oracle_layer(s, x, w_r, bias, wts)
    assert np.all(ids >= 4)
    xb = support.bf16_to_f64(synth.bf16_bits(x))
    for t in range(s["T"]):
        acc = np.zeros(s["hidden"])
        for j in range(3):
            acc = acc + w[t, j] * xb[t]
        assert np.array_equal(out[t], acc)


def test_shared_expert_adds_dense_ffn():
    s = mk(T=7, hidden=32, inter=16, n_routed=4, n_zero=4, top_k=2, bias_mode="logit",
           shared_inter=24, name="sharedonly")
    x, w_r, _, _ = synth.make_inputs(s)
    bias = torch.tensor([-1e3] * 4 + [0.0] * 4)
    wts = synth.draw_weights(s)
    out, ids, w = support.oracle_layer(s, x, w_r, bias, wts)
    xb = support.bf16_to_f64(synth.bf16_bits(x))
    sg, su, sd = support.shared_tuple(wts)
    for t in range(s["T"]):
        passthrough = w[t, 0] * xb[t] + w[t, 1] * xb[t]
        ref = _dense_swiglu(xb[t], sg, su, sd)
        assert np.allclose(out[t] - passthrough, ref, rtol=1e-11, atol=1e-13)


def test_token_permutation_equivariance():
    s = synth.spec("tiny")
    x, w_r, bias, _ = support.make_inputs(s)
    wts = synth.draw_weights(s)
    out, ids, _ = support.oracle_layer(s, x, w_r, bias, wts)
    perm = torch.randperm(s["T"], generator=torch.Generator().manual_seed(9))
    out_p, ids_p, _ = support.oracle_layer(s, x[perm], w_r, bias, wts)
    assert np.array_equal(out_p, out[perm.numpy()])
    assert np.array_equal(ids_p, ids[perm.numpy()])


def test_linear_in_down_projection():
    s = synth.spec("tiny")
    x, w_r, bias, _ = support.make_inputs(s)
    wts = synth.draw_weights(s)
    out1, _, _ = support.oracle_layer(s, x, w_r, bias, wts)
    wts2 = dict(wts)
    wts2["w_down"] = wts["w_down"] * 2  # exact in bf16
    out2, _, _ = support.oracle_layer(s, x, w_r, bias, wts2)
    assert np.array_equal(out2, 2.0 * out1)


# ---------------------------------------------------------------- W8A8 ----

def test_quantiser_hand_table():
    cases = json.load(open(os.path.join(GOLDEN, "quantiser_cases.json")))["cases"]
    for c in cases:
        q, sc = oracle.quantize_rows(np.array([c["row"]], np.float32))
        assert sc[0] == np.float32(c["scale"])
        assert list(q[0]) == c["codes"]


def test_int8_matmul_is_exact():
    rng = np.random.default_rng(6)
    a = rng.integers(-127, 128, size=(13, 300)).astype(np.int8)
    w = rng.integers(-127, 128, size=(9, 300)).astype(np.int8)
    acc = oracle.int8_matmul(a, w)
    assert np.array_equal(acc, a.astype(np.int64) @ w.astype(np.int64).T)
    ext = np.full((1, 300), -127, np.int8)
    assert oracle.int8_matmul(ext, ext)[0, 0] == 300 * 127 * 127


def test_w8a8_layer_tracks_bf16_layer_on_representable_weights():
    # Integer-valued tokens with amax 127 quantise exactly (scale 1); weights whose
    # scale is a power of two are exact in bf16.  The two layers then differ only
    # by the intermediate's int8 rounding (<= half a step of amax/127 per element).
    s = mk(T=6, hidden=64, inter=32, n_routed=3, top_k=2, name="w8pin")
    rng = np.random.default_rng(7)
    xi = rng.integers(-100, 101, size=(6, 64)).astype(np.float32)
    xi[:, 0] = 127.0
    x = torch.as_tensor(xi).to(torch.bfloat16)
    w_r = torch.as_tensor(rng.normal(size=(3, 64)).astype(np.float32) / 8)
    sc = 2.0 ** -12
    q = {n: [rng.integers(-127, 128, size=shp).astype(np.int8) for _ in range(3)]
         for n, shp in (("g", (32, 64)), ("u", (32, 64)), ("d", (64, 32)))}
    scales = {n: [np.full(q[n][0].shape[0], sc, np.float32) for _ in range(3)] for n in q}
    out8, ids8, _, qx, sx = oracle.layer_w8a8(s, synth.bf16_bits(x), w_r.numpy(), None, q["g"],
                                              scales["g"], q["u"], scales["u"], q["d"],
                                              scales["d"])
    assert np.all(sx == 1.0) and np.array_equal(qx.astype(np.float32), xi)
    to_bits = lambda a: bf16(a.astype(np.float32) * sc)
    outb, idsb, _ = oracle.layer(s, synth.bf16_bits(x), w_r.numpy(), None,
                                 [to_bits(a) for a in q["g"]], [to_bits(a) for a in q["u"]],
                                 [to_bits(a) for a in q["d"]])
    assert np.array_equal(ids8, idsb)
    rel = np.linalg.norm(out8 - outb) / np.linalg.norm(outb)
    assert rel < 1e-2


# -------------------------------------------------------- page constants ----

def test_layer_descriptions_match_page_constants():
    pc = json.load(open(os.path.join(GOLDEN, "page_constants.json")))
    lc = synth.spec("longcat")
    assert lc["n_routed"] + lc["n_zero"] == pc["longcat_experts"]["total"]
    assert lc["n_routed"] == pc["longcat_experts"]["routed"]
    assert lc["n_zero"] == pc["longcat_experts"]["zero_computation"]
    ds = synth.spec("dsv3")
    ep = pc["deepseek_v3_ep"]
    assert ds["n_routed"] == ep["decode_cards"] * ep["decode_routed_per_card"]
    assert ds["n_routed"] == ep["prefill_cards"] * ep["prefill_routed_per_card"]
    assert ep["shared_per_card"] == 1 and ds["shared_inter"] > 0


def test_margin_rule_holds_after_redraws():
    s = synth.spec("dsv3_s")
    x, w_r, bias, redraws = support.make_inputs(s)
    assert support.margin_rows(s, x, w_r, bias).all()


def test_longcat_zero_expert_share_is_about_a_third():
    # The LongCat-shaped layer's router is drawn so that about a third of the
    # picks land on its 256 zero-computation experts (an i.i.d. per-expert bias
    # keeps the 768 experts exchangeable).  Check the realised share on the
    # seeded inputs, routed by the oracle: within [0.30, 0.37] on the full layer
    # and on its scaled-down relative.
    for name in ("longcat", "longcat_s"):
        s = synth.spec(name)
        x, w_r, bias, _ = support.make_inputs(s)
        ids, _, _, _ = oracle.route(s, synth.bf16_bits(x), w_r.numpy(), support.np_bias(bias))
        share = float(np.mean(ids >= s["n_routed"]))
        assert 0.30 <= share <= 0.37, (name, share)
