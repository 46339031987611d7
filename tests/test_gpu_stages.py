"""Stage-by-stage parity of the CUDA path against the fp64 oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests import gpu_support as gs
from tests import support

pytestmark = pytest.mark.gpu

SMALL = ["tiny", "longcat_s", "dsv3_s", "pangu_s", "ragged_s"]


@pytest.fixture(scope="module")
def m():
    return gs.lib()


def route_gpu(m, spec, d, T=None):
    cfg = m.config_from_spec(spec)
    T = d["x_d"].shape[0] if T is None else T
    k = spec["top_k"]
    ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, k), dtype=torch.float32, device="cuda")
    ws = m.workspace(cfg, T)
    m.moe_route(cfg, T, d["x_d"], d["w_r_d"], d["bias_d"], ids, w, ws)
    torch.cuda.synchronize()
    assert m.moe_check_device_status(ws) == m.MOE_OK
    return ids.cpu().numpy(), w.cpu().numpy()


@pytest.mark.parametrize("name", SMALL)
def test_route_matches_oracle(m, name):
    spec = synth.spec(name)
    d = gs.inputs(spec)
    ids, w = route_gpu(m, spec, d)
    ids_o, w_o, _, _ = oracle.route(spec, synth.bf16_bits(d["x"]), d["w_r"].numpy(),
                                    support.np_bias(d["bias"]))
    assert np.array_equal(ids, ids_o)
    assert np.allclose(w, w_o, rtol=1e-5, atol=1e-7)


def test_route_on_tensor_cores_matches_oracle(m):
    # 1024 tokens x 1024 experts: the router runs as the exact three-term bf16
    # split on tensor cores (the path large prefill batches take)
    spec = synth.spec("tiny", T=1024, hidden=1024, n_routed=1024, top_k=4, renormalize=True,
                      name="router_tc")
    d = gs.inputs(spec)
    ids, w = route_gpu(m, spec, d)
    ids_o, w_o, _, _ = oracle.route(spec, synth.bf16_bits(d["x"]), d["w_r"].numpy(),
                                    support.np_bias(d["bias"]))
    assert np.array_equal(ids, ids_o)
    rel = np.abs(w - w_o) / w_o
    assert np.allclose(w, w_o, rtol=1e-5, atol=1e-7), f"max rel {rel.max():.3e}"


@pytest.mark.parametrize("name,over", [
    # H = 2112: 33 chunks of 64 over clusters of 16 CTAs (three chunks each, the last
    # five CTAs none); 200 tokens (a full and a ragged 72-token tile) x 200 experts
    # (a full and a ragged 72-expert tile); the top-k kernel afterwards
    ("wide_ragged", dict(T=200, hidden=2112, n_routed=150, n_zero=50, top_k=6)),
    # all 96 experts in one tile, 300 tokens in three token tiles (the last one 44
    # rows): the router CTAs pick the top-k themselves, one token per warp
    ("wide_fused", dict(T=300, hidden=2048, n_routed=64, n_zero=32, top_k=4,
                        renormalize=True)),
    # the same with per-group (MoGE) selection over 8 groups
    ("wide_fused_groups", dict(T=300, hidden=2048, n_routed=64, n_zero=0, top_k=8, n_group=8,
                               per_group_k=1, bias_mode="none", bias_kind="none")),
])
def test_route_in_clusters_of_16_matches_oracle(m, name, over):
    spec = synth.spec("longcat_s", name=name, **over)
    d = _route_inputs(spec)
    ids, w = route_gpu(m, spec, d)
    ids_o, w_o, _, _ = oracle.route(spec, synth.bf16_bits(d["x"]), d["w_r"].numpy(),
                                    support.np_bias(d["bias"]))
    assert np.array_equal(ids, ids_o)
    assert np.allclose(w, w_o, rtol=1e-5, atol=1e-7)


@pytest.mark.parametrize("name", ["tiny", *gs.ONE_CTA])
def test_route_in_one_cta_matches_oracle(m, name):
    # the router's x and W_r sit in one CTA's shared memory; its 32 warps compute
    # the logits and then the top-k (a token per warp, two for the 64-token case)
    spec = gs.layer_spec(name)
    d = _route_inputs(spec)
    ids, w = route_gpu(m, spec, d)
    ids_o, w_o, _, _ = oracle.route(spec, synth.bf16_bits(d["x"]), d["w_r"].numpy(),
                                    support.np_bias(d["bias"]))
    assert np.array_equal(ids, ids_o)
    assert np.allclose(w, w_o, rtol=1e-5, atol=1e-7)


def _route_inputs(spec):
    x, w_r, bias, _ = support.make_inputs(spec)
    return dict(x=x, w_r=w_r, bias=bias, x_d=x.cuda(), w_r_d=w_r.cuda(),
                bias_d=None if bias is None else bias.cuda())


def test_route_on_cuda_cores_by_default_matches_oracle(m):
    # 128 tokens x 128 experts x H = 6144: one 128 x 128 tile, so 16 CTAs with six
    # K chunks each on tensor cores; the shape class (a single tile, long H) that
    # keeps the CUDA-core router and its split-K reduction
    spec = synth.spec("dsv3_s", hidden=6144, n_routed=128, name="router_cc")
    d = _route_inputs(spec)
    ids, w = route_gpu(m, spec, d)
    ids_o, w_o, _, _ = oracle.route(spec, synth.bf16_bits(d["x"]), d["w_r"].numpy(),
                                    support.np_bias(d["bias"]))
    assert np.array_equal(ids, ids_o)
    assert np.allclose(w, w_o, rtol=1e-5, atol=1e-7)


@pytest.mark.parametrize("score", ["softmax", "sigmoid"])
def test_route_select_bias_and_groups(m, score):
    spec = synth.spec("dsv3_s", score=score, bias_mode="select", bias_kind="iid",
                      name=f"sel_{score}")
    d = gs.inputs(spec)
    ids, w = route_gpu(m, spec, d)
    ids_o, w_o, _, _ = oracle.route(spec, synth.bf16_bits(d["x"]), d["w_r"].numpy(),
                                    support.np_bias(d["bias"]))
    assert np.array_equal(ids, ids_o)
    assert np.allclose(w, w_o, rtol=1e-5, atol=1e-7)


def permute_gpu(m, spec, d, ids_np):
    cfg = m.config_from_spec(spec)
    T, k = ids_np.shape
    E = synth.n_experts(spec)
    ids = torch.as_tensor(ids_np, device="cuda")
    counts = torch.empty(E, dtype=torch.int32, device="cuda")
    offsets = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    s2e = torch.full((T * k,), -7, dtype=torch.int32, device="cuda")
    e2s = torch.full((T * k,), -7, dtype=torch.int32, device="cuda")
    x_perm = torch.zeros((T * k, spec["hidden"]), dtype=torch.bfloat16, device="cuda")
    ws = m.workspace(cfg, T)
    m.moe_permute(cfg, T, ids, d["x_d"][:T], counts, offsets, s2e, e2s, x_perm, None, ws)
    torch.cuda.synchronize()
    return ws, counts.cpu().numpy(), offsets.cpu().numpy(), s2e.cpu().numpy(), \
        e2s.cpu().numpy(), x_perm


@pytest.mark.parametrize("name", ["tiny", "longcat_s", "pangu_s", "ragged_s"])
def test_permute_matches_oracle(m, name):
    spec = synth.spec(name)
    d = gs.inputs(spec)
    ids_o, _, _, _ = oracle.route(spec, synth.bf16_bits(d["x"]), d["w_r"].numpy(),
                                  support.np_bias(d["bias"]))
    ws, counts, offsets, s2e, e2s, x_perm = permute_gpu(m, spec, d, ids_o)
    assert m.moe_check_device_status(ws) == m.MOE_OK
    c_o, o_o, s_o, e_o = oracle.permute(ids_o, synth.n_experts(spec))
    assert np.array_equal(counts, c_o)
    assert np.array_equal(offsets, o_o)
    assert np.array_equal(s2e, s_o)
    assert np.array_equal(e2s, e_o)
    # gathered rows are the token rows, bit for bit; only FFN-expert picks
    r_real = o_o[spec["n_routed"]]
    k = spec["top_k"]
    want = d["x"][torch.as_tensor(s_o[:r_real] // k)]
    assert torch.equal(x_perm[:r_real].cpu(), want)


@pytest.mark.parametrize("T", [1000, 1300])
def test_permute_many_blocks_and_skew(m, T):
    # One expert takes most picks.  1000 tokens: the one-CTA sort (all tokens'
    # bitmap in shared memory); 1300 tokens: six 256-token blocks of the
    # multi-CTA count / scan / scatter.
    spec = synth.spec("tiny", T=T, n_routed=40, top_k=4, name=f"perm_skew_{T}")
    rng = np.random.default_rng(11)
    ids = np.stack([np.concatenate([[0], rng.choice(np.arange(1, 40), 3, replace=False)])
                    if rng.random() < 0.8 else rng.choice(40, 4, replace=False)
                    for _ in range(T)]).astype(np.int32)
    x = torch.randn(T, spec["hidden"]).to(torch.bfloat16)
    d = dict(x_d=x.cuda())
    ws, counts, offsets, s2e, e2s, x_perm = permute_gpu(m, spec, d, ids)
    c_o, o_o, s_o, e_o = oracle.permute(ids, 40)
    assert np.array_equal(counts, c_o) and np.array_equal(offsets, o_o)
    assert np.array_equal(s2e, s_o) and np.array_equal(e2s, e_o)


def test_permute_bad_id_sets_device_status(m):
    spec = synth.spec("tiny")
    d = gs.inputs(spec)
    ids = np.array([[0, 1]] * 16, np.int32)
    ids[5, 1] = 99  # out of range
    ids[9, 0] = -3
    ws, counts, offsets, s2e, e2s, _ = permute_gpu(m, spec, d, ids)
    assert m.moe_check_device_status(ws) == m.MOE_ERR_DEVICE_CHECK
    assert m.moe_check_device_status(ws) == m.MOE_OK  # cleared by the first read
    assert counts.sum() == 30 and offsets[-1] == 30
    assert e2s[5 * 2 + 1] == -1 and e2s[9 * 2 + 0] == -1


@pytest.mark.parametrize("name", ["tiny", "longcat_s", "dsv3_s", "ragged_s"])
def test_grouped_ffn_matches_oracle(m, name):
    spec = synth.spec(name)
    d = gs.inputs(spec)
    ids_o, _, _, _ = oracle.route(spec, synth.bf16_bits(d["x"]), d["w_r"].numpy(),
                                  support.np_bias(d["bias"]))
    ws, counts, offsets, s2e, e2s, x_perm = permute_gpu(m, spec, d, ids_o)
    cfg = m.config_from_spec(spec)
    T, k, H = spec["T"], spec["top_k"], spec["hidden"]
    y = torch.full((T * k, H), float("nan"), dtype=torch.float32, device="cuda")
    w = d["wts_d"]
    m.moe_grouped_ffn(cfg, T, torch.as_tensor(offsets, device="cuda"), x_perm, None,
                      w["w_gate"], w["w_up"], w["w_down"], None, None, None, y, ws)
    torch.cuda.synchronize()
    assert m.moe_check_device_status(ws) == m.MOE_OK
    r_real = offsets[spec["n_routed"]]
    y = y[:r_real].cpu().double().numpy()
    g, u, dn = support.expert_lists(d["wts"])
    xb = support.bf16_to_f64(synth.bf16_bits(d["x"]))
    ref = np.empty_like(y)
    for p in range(r_real):
        r = s2e[p]
        e = ids_o.reshape(-1)[r]
        ref[p], _ = oracle.swiglu_expert(xb[r // k], g[e], u[e], dn[e])
    gs.check_out(torch.as_tensor(y), ref, bf16_out=False, what=name)


def test_combine_weighted_sum(m):
    # combine alone: a plain weighted sum of given rows, checked in fp64
    spec = synth.spec("ragged_s")
    d = gs.inputs(spec)
    T, k, H, E_r = spec["T"], spec["top_k"], spec["hidden"], spec["n_routed"]
    ids_o, w_o, _, _ = oracle.route(spec, synth.bf16_bits(d["x"]), d["w_r"].numpy(),
                                    support.np_bias(d["bias"]))
    _, _, s2e, e2s = oracle.permute(ids_o, synth.n_experts(spec))
    y = torch.randn(T * k, H, dtype=torch.float32)
    sh = torch.randn(T, H, dtype=torch.float32)
    cfg = m.config_from_spec(spec, out_fp32=True)
    out = torch.empty(T, H, dtype=torch.float32, device="cuda")
    m.moe_combine(cfg, T, y.cuda(), torch.as_tensor(e2s, device="cuda"),
                  torch.as_tensor(ids_o, device="cuda"),
                  torch.as_tensor(w_o.astype(np.float32), device="cuda"), d["x_d"], sh.cuda(), out)
    torch.cuda.synchronize()
    xb = support.bf16_to_f64(synth.bf16_bits(d["x"]))
    yd, shd = y.double().numpy(), sh.double().numpy()
    ref = shd.copy()
    for t in range(T):
        for j in range(k):
            e = ids_o[t, j]
            wj = float(np.float32(w_o[t, j]))
            ref[t] += wj * (yd[e2s[t * k + j]] if e < E_r else xb[t])
    assert np.allclose(out.cpu().double().numpy(), ref, rtol=1e-5, atol=1e-5)
