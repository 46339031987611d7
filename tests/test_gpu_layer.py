"""Whole-layer parity of moe_layer_forward against the fp64 oracle, through the C ABI."""
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


def oracle_out(spec, d, x=None):
    x = d["x"] if x is None else x
    out, ids, w = support.oracle_layer(spec, x, d["w_r"], d["bias"], d["wts"])
    return out


@pytest.mark.parametrize("name", SMALL)
@pytest.mark.parametrize("out_fp32", [True, False])
@pytest.mark.parametrize("gemv_max_rows", [0, 8])  # library default / streaming GEMV path
def test_layer_matches_oracle(m, name, out_fp32, gemv_max_rows):
    spec = synth.spec(name)
    d = gs.inputs(spec)
    ref = oracle_out(spec, d)
    got = gs.run_layer(m, spec, d, out_fp32=out_fp32, gemv_max_rows=gemv_max_rows)
    gs.check_out(got, ref, bf16_out=not out_fp32, what=f"{name} gemv<={gemv_max_rows}")


@pytest.mark.parametrize("name", ["tiny", *gs.SMALL_FFN])
@pytest.mark.parametrize("out_fp32", [True, False])
@pytest.mark.parametrize("combine", ["default", "ordered"])
def test_small_layer_ffn_matches_oracle(m, name, out_fp32, combine):
    # at most 16 tokens: one CTA per expert runs gate/up and down as warp-level
    # MMAs out of shared memory (the library default for such layers); an
    # explicit launch form keeps the persistent tensor-core kernel, which must
    # agree with the oracle too
    spec = gs.layer_spec(name)
    d = gs.inputs(spec)
    ref = oracle_out(spec, d)
    mode = m.COMBINE_ORDERED if combine == "ordered" else 0
    got = gs.run_layer(m, spec, d, out_fp32=out_fp32, combine=mode)
    gs.check_out(got, ref, bf16_out=not out_fp32, what=f"{name} {combine}")
    tc = gs.run_layer(m, spec, d, out_fp32=out_fp32, combine=mode, ffn_launch=m.FFN_LAUNCH_ONE)
    gs.check_out(tc, ref, bf16_out=not out_fp32, what=f"{name} {combine} tensor-core kernel")


@pytest.mark.parametrize("name", list(gs.ONE_CTA))
@pytest.mark.parametrize("combine", ["default", "ordered"])
def test_layer_routed_by_the_sort_matches_oracle(m, name, combine):
    # small layers: the one-CTA re-sort routes the tokens itself, then sorts,
    # gathers and starts the accumulators
    spec = gs.layer_spec(name)
    d = gs.inputs(spec)
    ref = oracle_out(spec, d)
    mode = m.COMBINE_ORDERED if combine == "ordered" else 0
    got = gs.run_layer(m, spec, d, out_fp32=False, combine=mode)
    gs.check_out(got, ref, bf16_out=True, what=f"{name} {combine}")


@pytest.mark.parametrize("name", SMALL)
@pytest.mark.parametrize("out_fp32", [True, False])
def test_layer_with_ordered_combine_matches_oracle(m, name, out_fp32):
    # the per-pick rows and the deterministic combine kernel instead of the
    # down epilogue's scatter-add
    spec = synth.spec(name)
    d = gs.inputs(spec)
    ref = oracle_out(spec, d)
    got = gs.run_layer(m, spec, d, out_fp32=out_fp32, combine=m.COMBINE_ORDERED)
    gs.check_out(got, ref, bf16_out=not out_fp32, what=f"{name} ordered")


@pytest.mark.parametrize("name", ["dsv3_s", "pangu_s", "ragged_s"])
@pytest.mark.parametrize("gemv_max_rows", [0, 8])
def test_fused_and_ordered_combine_agree(m, name, gemv_max_rows):
    # The two combines add the same fp32 products, in a different order: they
    # agree to fp32 rounding (and repeated fused calls agree with each other
    # the same way; their atomic adds may land in any order).
    spec = synth.spec(name)
    d = gs.inputs(spec)
    o = gs.run_layer(m, spec, d, gemv_max_rows=gemv_max_rows, combine=m.COMBINE_ORDERED)
    f1 = gs.run_layer(m, spec, d, gemv_max_rows=gemv_max_rows, combine=m.COMBINE_FUSED)
    f2 = gs.run_layer(m, spec, d, gemv_max_rows=gemv_max_rows, combine=m.COMBINE_FUSED)
    scale = o.abs().max().item()
    assert (f1 - o).abs().max().item() <= 1e-5 * scale
    assert (f2 - f1).abs().max().item() <= 1e-5 * scale


@pytest.mark.parametrize("gemv_max_rows", [1, 3, 1000])
def test_layer_path_choice_does_not_change_result(m, gemv_max_rows):
    spec = synth.spec("pangu_s")
    d = gs.inputs(spec)
    ref = oracle_out(spec, d)
    got = gs.run_layer(m, spec, d, gemv_max_rows=gemv_max_rows)
    gs.check_out(got, ref, bf16_out=False, what=f"gemv_max_rows={gemv_max_rows}")


def test_layer_is_deterministic_with_ordered_combine(m):
    spec = synth.spec("dsv3_s")
    d = gs.inputs(spec)
    a = gs.run_layer(m, spec, d, out_fp32=True, combine=m.COMBINE_ORDERED)
    b = gs.run_layer(m, spec, d, out_fp32=True, combine=m.COMBINE_ORDERED)
    assert torch.equal(a, b)


@pytest.mark.parametrize("name", ["dsv3_s", "w8a8_s"])
@pytest.mark.parametrize("combine", [1, 2])  # ordered, fused
def test_layer_replays_from_a_cuda_graph(m, name, combine):
    # The layer is stream-ordered with no host synchronisation, so one capture
    # replays it: the replay on new inputs matches a direct call, bit for bit
    # with the ordered combine, to fp32 rounding with the fused one.
    spec = synth.spec(name)
    d = gs.inputs(spec)
    cfg = m.config_from_spec(spec, out_fp32=True, combine=combine)
    T, H = spec["T"], spec["hidden"]
    w = d["wts_d"]
    x = d["x_d"].clone()
    out = torch.empty((T, H), dtype=torch.float32, device="cuda")
    ws = m.workspace(cfg, T)

    def call(stream):
        m.moe_layer_forward(cfg, T, x, d["w_r_d"], d["bias_d"], w.get("w_gate"), w.get("w_up"),
                            w.get("w_down"), w.get("s_gate"), w.get("s_up"), w.get("s_down"),
                            w.get("shared_gate"), w.get("shared_up"), w.get("shared_down"), out,
                            ws, stream=stream)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        call(s)  # first call outside capture: per-device set-up happens here
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        call(s)
    x.copy_(torch.flip(d["x_d"], [0]))
    g.replay()
    torch.cuda.synchronize()
    assert m.moe_check_device_status(ws) == m.MOE_OK
    replayed = out.clone()
    direct = gs.run_layer(m, spec, d, out_fp32=True, x=x.clone(), combine=combine)
    if combine == m.COMBINE_ORDERED:
        assert torch.equal(replayed, direct)
    else:
        assert (replayed - direct).abs().max().item() <= 1e-5 * direct.abs().max().item()


def test_single_token_and_empty_batch(m):
    spec = synth.spec("ragged_s")
    d = gs.inputs(spec)
    ref = oracle_out(spec, d, x=d["x"][:1])
    got = gs.run_layer(m, spec, d, x=d["x_d"][:1].contiguous())
    gs.check_out(got, ref, bf16_out=False, what="T=1")
    cfg = m.config_from_spec(spec)
    ws = m.workspace(cfg, 0)
    out = torch.empty(0, spec["hidden"], device="cuda", dtype=torch.bfloat16)
    w = d["wts_d"]
    m.moe_layer_forward(cfg, 0, d["x_d"][:0], d["w_r_d"], d["bias_d"], w["w_gate"], w["w_up"],
                        w["w_down"], None, None, None, w["shared_gate"], w["shared_up"],
                        w["shared_down"], out, ws)


def test_zero_experts_pass_input_through(m):
    spec = synth.spec("longcat_s", name="allzero")
    d = dict(gs.inputs(synth.spec("longcat_s")))
    bias = torch.zeros(synth.n_experts(spec))
    bias[:spec["n_routed"]] = -1e3  # every pick lands on a zero-computation expert
    d["bias"], d["bias_d"] = bias, bias.cuda()
    got = gs.run_layer(m, spec, d, out_fp32=True).cpu().double().numpy()
    _, _, w = support.oracle_layer(spec, d["x"], d["w_r"], bias, d["wts"])
    xb = support.bf16_to_f64(synth.bf16_bits(d["x"]))
    ref = w.sum(1, keepdims=True) * xb
    assert np.allclose(got, ref, rtol=2e-6, atol=1e-6)


def test_single_expert_top1_is_dense_ffn(m):
    spec = dict(synth.spec("tiny"), n_routed=1, top_k=1, renormalize=False, T=40,
                name="dense_gpu")
    d = gs.inputs(spec)
    got = gs.run_layer(m, spec, d, out_fp32=True)
    xb = support.bf16_to_f64(synth.bf16_bits(d["x"]))
    g, u, dn = support.expert_lists(d["wts"])
    G = support.bf16_to_f64(g[0]) @ xb.T
    U = support.bf16_to_f64(u[0]) @ xb.T
    ref = (support.bf16_to_f64(dn[0]) @ (G / (1 + np.exp(-G)) * U)).T
    gs.check_out(got, ref, bf16_out=False, what="dense")


# ------------------------------------------------------- full-size layers ---

def full_size_case(m, name, n_sample=4):
    spec = synth.spec(name)
    x, w_r, bias, redraws = support.make_inputs(spec)
    wts_d = synth.draw_weights(spec, device="cuda")
    d = dict(x=x, w_r=w_r, bias=bias, x_d=x.cuda(), w_r_d=w_r.cuda(),
             bias_d=None if bias is None else bias.cuda(), wts_d=wts_d)
    # routing of every token, bit-exact ids
    cfg = m.config_from_spec(spec)
    T, k = spec["T"], spec["top_k"]
    ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
    wgt = torch.empty((T, k), dtype=torch.float32, device="cuda")
    ws = m.workspace(cfg, T)
    m.moe_route(cfg, T, d["x_d"], d["w_r_d"], d["bias_d"], ids, wgt, ws)
    torch.cuda.synchronize()
    ids_o, w_o, _, _ = oracle.route(spec, synth.bf16_bits(x), w_r.numpy(), support.np_bias(bias))
    assert np.array_equal(ids.cpu().numpy(), ids_o)
    assert np.allclose(wgt.cpu().numpy(), w_o, rtol=1e-5, atol=1e-7)
    # the layer at full size, bf16 out (the benchmarked configuration)
    out = gs.run_layer(m, spec, d, out_fp32=False)
    # oracle on sampled tokens with only the experts they pick
    rng = np.random.default_rng(2)
    sample = np.sort(rng.choice(T, n_sample, replace=False))
    need = set(int(e) for e in ids_o[sample].reshape(-1) if e < spec["n_routed"])
    g, u, dn = gs.expert_lists_from_device(wts_d, need)
    shared = None
    if spec["shared_inter"] > 0:
        shared = tuple(synth.bf16_bits(wts_d[kk]) for kk in
                       ("shared_gate", "shared_up", "shared_down"))
    ref, ids_s, _ = oracle.layer(spec, synth.bf16_bits(x[sample]), w_r.numpy(),
                                 support.np_bias(bias), g, u, dn, shared)
    assert np.array_equal(ids_s, ids_o[sample])
    gs.check_out(out[torch.as_tensor(sample, device="cuda")], ref, bf16_out=True, what=name)
    del wts_d, d
    torch.cuda.empty_cache()


@pytest.mark.parametrize("name", ["longcat", "dsv3", "pangu"])
def test_full_size_decode_layers(m, name):
    full_size_case(m, name)


def test_layer_with_more_tasks_than_the_kernel_caches(m):
    # 1536 experts x 2048 tokens x top-2, all on tensor cores: ~1430 tasks, more than
    # the one-launch FFN keeps in shared memory (1024), so its tile decodes read the
    # work list from global memory; the batch also takes the large-batch router, the
    # multi-CTA re-sort and the work-list kernel
    spec = synth.spec("tiny", T=2048, n_routed=1536, top_k=2, name="many_tasks")
    d = gs.inputs(spec)
    ref = oracle_out(spec, d)
    got = gs.run_layer(m, spec, d, out_fp32=True, gemv_max_rows=-1)
    gs.check_out(got, ref, bf16_out=False, what="1536 experts x 2048 tokens")
    cfg = m.config_from_spec(spec, gemv_max_rows=-1)
    assert m.moe_tile_choice(cfg, 2048)[1]  # the one-launch FFN runs this layer


def _bucket(spec, T):
    m = T * spec["top_k"] / synth.n_experts(spec)
    return next((i for i, v in enumerate([2, 8, 32, 128]) if m < v), 4)


@pytest.mark.parametrize("name,T", [("longcat_s", 16), ("longcat_s", 48), ("dsv3_s", 128),
                                    ("pangu_s", 456), ("dsv3_s", 1024)])
def test_layer_in_every_load_bucket(m, name, T):
    # One layer per load bucket of the tile-parameter table (expected picks per
    # expert < 2, < 8, < 32, < 128, >= 128), with the tiling the table picks
    # (moe_tile_choice), against the oracle.
    spec = synth.spec(name, T=T, name=f"{name}_T{T}")
    d = gs.inputs(spec)
    ref = oracle_out(spec, d)
    got = gs.run_layer(m, spec, d, out_fp32=True)
    gs.check_out(got, ref, bf16_out=False, what=f"{name} T={T} bucket {_bucket(spec, T)}")


def test_load_buckets_are_all_covered():
    cases = [("longcat_s", 16), ("longcat_s", 48), ("dsv3_s", 128), ("pangu_s", 456),
             ("dsv3_s", 1024)]
    assert sorted(_bucket(synth.spec(n), T) for n, T in cases) == [0, 1, 2, 3, 4]
