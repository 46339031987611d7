"""W8A8 path: exact int32 accumulators, bit-exact activation codes, and whole-layer
parity against the oracle's W8A8 layer."""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests import gpu_support as gs
from tests import support

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def m():
    return gs.lib()


def qgemm(m, counts, a, w):
    E, N, K = w.shape
    R = a.shape[0]
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    ws = torch.zeros(m.moe_qgemm_s8_workspace_size(E, K, N, R), dtype=torch.uint8, device="cuda")
    acc = torch.full((R, N), -7, dtype=torch.int32, device="cuda")
    m.moe_qgemm_s8(E, K, N, R, torch.as_tensor(offsets, device="cuda"),
                   torch.as_tensor(a, device="cuda"), torch.as_tensor(w, device="cuda"), acc, ws)
    torch.cuda.synchronize()
    assert m.moe_check_device_status(ws) == m.MOE_OK
    return acc.cpu().numpy(), offsets


def qgemm_ref(offsets, a, w):
    out = np.zeros((a.shape[0], w.shape[1]), np.int64)
    for e in range(w.shape[0]):
        r0, r1 = offsets[e], offsets[e + 1]
        out[r0:r1] = a[r0:r1].astype(np.int64) @ w[e].astype(np.int64).T
    return out


def test_qgemm_exact_on_random_codes(m):
    rng = np.random.default_rng(21)
    counts = [0, 1, 37, 128, 200]
    K, N = 1024, 384
    a = rng.integers(-127, 128, size=(sum(counts), K)).astype(np.int8)
    w = rng.integers(-128, 128, size=(len(counts), N, K)).astype(np.int8)
    acc, off = qgemm(m, counts, a, w)
    assert np.array_equal(acc.astype(np.int64), qgemm_ref(off, a, w))


def test_qgemm_exact_past_the_fp32_integer_range(m):
    # all-+-127 codes over K = 7168: partial sums reach 1.2e8 > 2^24, so these
    # tiles fail the tensor-core exactness guard and take the integer path
    rng = np.random.default_rng(22)
    counts = [40, 3, 90]
    K, N = 7168, 256
    a = (127 * rng.choice([-1, 1], size=(sum(counts), K))).astype(np.int8)
    a[:10] = 127
    w = (127 * rng.choice([-1, 1], size=(len(counts), N, K))).astype(np.int8)
    w[0, :5] = 127
    w[2, 7] = -128
    acc, off = qgemm(m, counts, a, w)
    ref = qgemm_ref(off, a, w)
    assert ref.max() == 127 * 127 * K  # the extreme case is present
    assert np.array_equal(acc.astype(np.int64), ref)


def test_qgemm_ragged_k_and_n(m):
    rng = np.random.default_rng(23)
    counts = [17, 0, 130]
    K, N = 1040, 200
    a = rng.integers(-127, 128, size=(sum(counts), K)).astype(np.int8)
    w = rng.integers(-128, 128, size=(len(counts), N, K)).astype(np.int8)
    acc, off = qgemm(m, counts, a, w)
    assert np.array_equal(acc.astype(np.int64), qgemm_ref(off, a, w))


def test_activation_codes_match_oracle_bit_for_bit(m):
    spec = synth.spec("w8a8_s")
    d = gs.inputs(spec)
    T, k, H = spec["T"], spec["top_k"], spec["hidden"]
    E = synth.n_experts(spec)
    ids_o, _, _, _ = oracle.route(spec, synth.bf16_bits(d["x"]), d["w_r"].numpy(),
                                  support.np_bias(d["bias"]))
    cfg = m.config_from_spec(spec)
    ids = torch.as_tensor(ids_o, device="cuda")
    counts = torch.empty(E, dtype=torch.int32, device="cuda")
    offsets = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    s2e = torch.empty(T * k, dtype=torch.int32, device="cuda")
    e2s = torch.empty(T * k, dtype=torch.int32, device="cuda")
    xq = torch.zeros((T * k, H), dtype=torch.int8, device="cuda")
    sx = torch.zeros(T * k, dtype=torch.float32, device="cuda")
    ws = m.workspace(cfg, T)
    m.moe_permute(cfg, T, ids, d["x_d"], counts, offsets, s2e, e2s, xq, sx, ws)
    torch.cuda.synchronize()
    q_o, s_o = oracle.quantize_rows(d["x"].float().numpy())
    s2e = s2e.cpu().numpy()
    rows = s2e[:T * k] // k
    assert np.array_equal(xq.cpu().numpy(), q_o[rows])
    assert np.array_equal(sx.cpu().numpy(), s_o[rows])


@pytest.mark.parametrize("gemv", [-1, 1000])
def test_w8a8_grouped_ffn_stage_matches_oracle(m, gemv):
    # moe_grouped_ffn on the caller's int8 x_perm (from moe_permute), on tensor
    # cores (-1) and on the streaming path (1000); the reference runs each
    # expert through the oracle's quantiser and exact int8 matmuls
    spec = synth.spec("w8a8_s", T=96, name="w8a8_s_T96")
    d = gs.inputs(spec)
    T, k, H = spec["T"], spec["top_k"], spec["hidden"]
    E, E_r = synth.n_experts(spec), spec["n_routed"]
    ids_o, _, _, _ = oracle.route(spec, synth.bf16_bits(d["x"]), d["w_r"].numpy(),
                                  support.np_bias(d["bias"]))
    cfg = m.config_from_spec(spec, gemv_max_rows=gemv)
    ids = torch.as_tensor(ids_o, device="cuda")
    counts = torch.empty(E, dtype=torch.int32, device="cuda")
    offsets = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    s2e = torch.empty(T * k, dtype=torch.int32, device="cuda")
    e2s = torch.empty(T * k, dtype=torch.int32, device="cuda")
    xq = torch.zeros((T * k, H), dtype=torch.int8, device="cuda")
    sx = torch.zeros(T * k, dtype=torch.float32, device="cuda")
    ws = m.workspace(cfg, T)
    m.moe_permute(cfg, T, ids, d["x_d"], counts, offsets, s2e, e2s, xq, sx, ws)
    y = torch.full((T * k, H), float("nan"), dtype=torch.float32, device="cuda")
    w = d["wts_d"]
    m.moe_grouped_ffn(cfg, T, offsets, xq, sx, w["w_gate"], w["w_up"], w["w_down"], w["s_gate"],
                      w["s_up"], w["s_down"], y, ws)
    torch.cuda.synchronize()
    assert m.moe_check_device_status(ws) == m.MOE_OK
    # reference: the oracle's permutation and codes, per expert
    _, off, s2e_o, _ = oracle.permute(ids_o, E)
    q_o, s_o = oracle.quantize_rows(d["x"].float().numpy())
    L = w8_lists(d["wts"])
    r_real = int(off[E_r])
    ref = np.empty((r_real, H))
    for e in range(E_r):
        a, b = int(off[e]), int(off[e + 1])
        if a == b:
            continue
        rows = s2e_o[a:b] // k
        qa, sa = q_o[rows], s_o[rows].astype(np.float64)[:, None]
        g = oracle.int8_matmul(qa, L["qg"][e]) * sa * L["sg"][e].astype(np.float64)[None, :]
        u = oracle.int8_matmul(qa, L["qu"][e]) * sa * L["su"][e].astype(np.float64)[None, :]
        qh, sh = oracle.quantize_rows((g / (1.0 + np.exp(-g)) * u).astype(np.float32))
        ref[a:b] = (oracle.int8_matmul(qh, L["qd"][e]) * sh.astype(np.float64)[:, None]
                    * L["sd"][e].astype(np.float64)[None, :])
    gs.check_out(y[:r_real], ref, bf16_out=False, what=f"w8a8 grouped ffn gemv<={gemv}")


def w8_lists(wts, experts=None):
    E = wts["w_gate"].shape[0]
    want = set(range(E)) if experts is None else set(int(e) for e in experts)
    out = {k: [] for k in ("qg", "sg", "qu", "su", "qd", "sd")}
    for e in range(E):
        ok = e in want
        for key, name in (("qg", "w_gate"), ("qu", "w_up"), ("qd", "w_down")):
            out[key].append(wts[name][e].cpu().numpy() if ok else None)
        for key, name in (("sg", "s_gate"), ("su", "s_up"), ("sd", "s_down")):
            out[key].append(wts[name][e].cpu().numpy() if ok else None)
    return out


def w8_shared(wts):
    if "shared_gate" not in wts:
        return None
    return tuple(wts[n].cpu().numpy() for n in ("shared_gate", "s_shared_gate", "shared_up",
                                                "s_shared_up", "shared_down", "s_shared_down"))


@pytest.mark.parametrize("out_fp32", [True, False])
@pytest.mark.parametrize("combine", [1, 2])  # ordered, fused
def test_w8a8_layer_with_shared_expert_matches_oracle(m, out_fp32, combine):
    # DSv3-shaped routing (sigmoid, groups, x 2.5) with an int8 shared expert fed
    # the same per-token codes; its scales ride after the routed experts'
    spec = synth.spec("dsv3_w8_s")
    d = gs.inputs(spec)
    L = w8_lists(d["wts"])
    ref, _, _, _, _ = oracle.layer_w8a8(spec, synth.bf16_bits(d["x"]), d["w_r"].numpy(),
                                        support.np_bias(d["bias"]), L["qg"], L["sg"], L["qu"],
                                        L["su"], L["qd"], L["sd"], w8_shared(d["wts"]))
    got = gs.run_layer(m, spec, d, out_fp32=out_fp32, combine=combine)
    gs.check_out(got, ref, bf16_out=not out_fp32, what=f"dsv3_w8_s combine={combine}")


@pytest.mark.parametrize("out_fp32", [True, False])
def test_w8a8_layer_matches_oracle(m, out_fp32):
    spec = synth.spec("w8a8_s")
    d = gs.inputs(spec)
    L = w8_lists(d["wts"])
    ref, _, _, _, _ = oracle.layer_w8a8(spec, synth.bf16_bits(d["x"]), d["w_r"].numpy(),
                                        support.np_bias(d["bias"]), L["qg"], L["sg"], L["qu"],
                                        L["su"], L["qd"], L["sd"])
    got = gs.run_layer(m, spec, d, out_fp32=out_fp32)
    gs.check_out(got, ref, bf16_out=not out_fp32, what="w8a8_s")


@pytest.mark.parametrize("T,gemv,H,I", [(512, 8, 1024, 512), (512, 1000, 1024, 512),
                                         (40, 8, 1024, 512), (40, 1000, 1024, 512),
                                         (40, 2, 1024, 512), (40, 8, 2048, 2048),
                                         (40, 1000, 1040, 272), (200, 8, 1040, 272)])
def test_w8a8_streaming_path_matches_oracle_and_tensor_cores(m, T, gemv, H, I):
    # Experts with <= gemv rows take the dp4a GEMV; both paths accumulate the
    # same exact integers and dequantise with the same fp32 formula, so the
    # layer output is bit-identical to the all-tensor-core run.  H = 1040 and
    # I = 272 leave the last 128-channel tile and the last 128-byte K step of
    # each pass partly outside the matrices (filled with zeros by TMA).
    spec = synth.spec("w8a8_s", T=T, hidden=H, inter=I, name=f"w8a8_s_T{T}_{H}_{I}")
    d = gs.inputs(spec)
    L = w8_lists(d["wts"])
    ref, _, _, _, _ = oracle.layer_w8a8(spec, synth.bf16_bits(d["x"]), d["w_r"].numpy(),
                                        support.np_bias(d["bias"]), L["qg"], L["sg"], L["qu"],
                                        L["su"], L["qd"], L["sd"])
    got = gs.run_layer(m, spec, d, out_fp32=True, gemv_max_rows=gemv)
    gs.check_out(got, ref, bf16_out=False, what=f"w8a8 T={T} gemv<={gemv}")
    ordered = m.COMBINE_ORDERED
    got = gs.run_layer(m, spec, d, out_fp32=True, gemv_max_rows=gemv, combine=ordered)
    tc = gs.run_layer(m, spec, d, out_fp32=True, gemv_max_rows=-1, combine=ordered)
    assert torch.equal(got, tc)


def test_w8a8_full_size_prefill(m):
    spec = synth.spec("w8a8_prefill")
    x, w_r, bias, _ = support.make_inputs(spec)
    wts_d = synth.draw_weights(spec, device="cuda")
    d = dict(x=x, w_r=w_r, bias=bias, x_d=x.cuda(), w_r_d=w_r.cuda(), bias_d=bias.cuda(),
             wts_d=wts_d)
    T, k = spec["T"], spec["top_k"]
    cfg = m.config_from_spec(spec)
    ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
    wgt = torch.empty((T, k), dtype=torch.float32, device="cuda")
    ws = m.workspace(cfg, T)
    m.moe_route(cfg, T, d["x_d"], d["w_r_d"], d["bias_d"], ids, wgt, ws)
    torch.cuda.synchronize()
    ids_o, w_o, _, _ = oracle.route(spec, synth.bf16_bits(x), w_r.numpy(), bias.numpy())
    assert np.array_equal(ids.cpu().numpy(), ids_o)
    loads = np.bincount(ids_o.reshape(-1), minlength=spec["n_routed"])
    assert loads.max() >= 10 * loads.mean()  # Zipf skew: hot experts well above the mean
    out = gs.run_layer(m, spec, d, out_fp32=False)
    rng = np.random.default_rng(3)
    sample = np.sort(rng.choice(T, 3, replace=False))
    L = w8_lists(wts_d, set(ids_o[sample].reshape(-1)))
    ref, ids_s, _, _, _ = oracle.layer_w8a8(spec, synth.bf16_bits(x[sample]), w_r.numpy(),
                                            bias.numpy(), L["qg"], L["sg"], L["qu"], L["su"],
                                            L["qd"], L["sd"])
    assert np.array_equal(ids_s, ids_o[sample])
    gs.check_out(out[torch.as_tensor(sample, device="cuda")], ref, bf16_out=True, what="prefill")
    del wts_d, d
    torch.cuda.empty_cache()


def test_w8a8_layer_exact_fallback_on_guard_failures(m):
    # Activations of +-1 and weight codes of +-127: every row norm is 127^2 H and
    # every gate/up channel norm 127^2 H, so at H = 2048 each gate/up pair breaks
    # the tensor-core guard (127^4 H^2 > 2^48) and both halves of every two-SM
    # gate/up tile are recomputed by the exact integer kernel.  The dp4a
    # streaming path sums the same integers exactly and dequantises with the same
    # fp32 formula, so the two runs agree bit for bit.
    H, I, E = 2048, 256, 8
    assert (127 ** 4) * H * H >= 2 ** 48
    spec = synth.spec("w8a8_s", T=64, hidden=H, inter=I, n_routed=E, top_k=2, name="w8_guard")
    base = gs.inputs(spec)
    rng = np.random.default_rng(31)
    x = torch.as_tensor(rng.choice([-1.0, 1.0], size=(spec["T"], H)), dtype=torch.bfloat16)
    codes = lambda *shape: torch.as_tensor(127 * rng.choice([-1, 1], size=shape), dtype=torch.int8)
    wts = {"w_gate": codes(E, I, H), "w_up": codes(E, I, H), "w_down": codes(E, H, I),
           "s_gate": torch.full((E, I), 1e-4), "s_up": torch.full((E, I), 1e-4),
           "s_down": torch.full((E, H), 1e-3)}
    d = dict(base, x=x, x_d=x.cuda(), wts=wts, wts_d={k: v.cuda() for k, v in wts.items()})
    L = w8_lists(wts)
    ref, _, _, _, _ = oracle.layer_w8a8(spec, synth.bf16_bits(x), d["w_r"].numpy(),
                                        support.np_bias(d["bias"]), L["qg"], L["sg"], L["qu"],
                                        L["su"], L["qd"], L["sd"])
    tc = gs.run_layer(m, spec, d, out_fp32=True, gemv_max_rows=-1)
    gs.check_out(tc, ref, bf16_out=False, what="w8a8 guard fallback")
    ordered = m.COMBINE_ORDERED
    tc = gs.run_layer(m, spec, d, out_fp32=True, gemv_max_rows=-1, combine=ordered)
    stream = gs.run_layer(m, spec, d, out_fp32=True, gemv_max_rows=100000, combine=ordered)
    assert torch.equal(tc, stream)


@pytest.mark.parametrize("combine", [1, 2])  # ordered, fused
def test_w8a8_down_pass_exact_fallback(m, combine):
    # Every token is the same row of ones and every gate/up weight code is +127,
    # so h is the same positive value in every channel and quantises to +127
    # everywhere: with I = 2048 each down-pass pair has 127^4 I^2 > 2^48 and
    # fails the tensor-core guard, as does each gate/up pair (H = 2048).  Both
    # passes then run on the exact integer kernel; with the fused combine, the
    # down tiles' halves that fail add nothing in the tensor-core epilogue and
    # the exact kernel adds them.
    H, I, E = 2048, 2048, 8
    assert (127 ** 4) * I * I >= 2 ** 48
    spec = synth.spec("w8a8_s", T=64, hidden=H, inter=I, n_routed=E, top_k=2,
                      name="w8_guard_down")
    base = gs.inputs(spec)
    rng = np.random.default_rng(37)
    x = torch.ones((spec["T"], H), dtype=torch.bfloat16)
    wts = {"w_gate": torch.full((E, I, H), 127, dtype=torch.int8),
           "w_up": torch.full((E, I, H), 127, dtype=torch.int8),
           "w_down": torch.as_tensor(127 * rng.choice([-1, 1], size=(E, H, I)), dtype=torch.int8),
           "s_gate": torch.full((E, I), 1e-5), "s_up": torch.full((E, I), 1e-5),
           "s_down": torch.as_tensor(rng.uniform(0.5e-3, 1.5e-3, size=(E, H)),
                                     dtype=torch.float32)}
    d = dict(base, x=x, x_d=x.cuda(), wts=wts, wts_d={k: v.cuda() for k, v in wts.items()})
    L = w8_lists(wts)
    ref, _, _, _, _ = oracle.layer_w8a8(spec, synth.bf16_bits(x), d["w_r"].numpy(),
                                        support.np_bias(d["bias"]), L["qg"], L["sg"], L["qu"],
                                        L["su"], L["qd"], L["sd"])
    got = gs.run_layer(m, spec, d, out_fp32=True, gemv_max_rows=-1, combine=combine)
    gs.check_out(got, ref, bf16_out=False, what="w8a8 down-pass guard fallback")


@pytest.mark.parametrize("name", ["longcat_w8", "dsv3_w8"])
def test_w8a8_full_size_decode_layers(m, name):
    # The W8A8 decode layers at full size (LongCat-shaped: 512 int8 experts and
    # 256 zero-computation ones; DSv3-shaped: 256 int8 experts in 8 groups plus
    # the int8 shared expert), bf16 out, the default streaming / tensor-core
    # split: every token's routing exactly, sampled tokens' outputs against the
    # oracle run with only the experts they pick.
    spec = synth.spec(name)
    x, w_r, bias, _ = support.make_inputs(spec)
    wts_d = synth.draw_weights(spec, device="cuda")
    d = dict(x=x, w_r=w_r, bias=bias, x_d=x.cuda(), w_r_d=w_r.cuda(),
             bias_d=None if bias is None else bias.cuda(), wts_d=wts_d)
    T, k = spec["T"], spec["top_k"]
    cfg = m.config_from_spec(spec)
    ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
    wgt = torch.empty((T, k), dtype=torch.float32, device="cuda")
    ws = m.workspace(cfg, T)
    m.moe_route(cfg, T, d["x_d"], d["w_r_d"], d["bias_d"], ids, wgt, ws)
    torch.cuda.synchronize()
    ids_o, w_o, _, _ = oracle.route(spec, synth.bf16_bits(x), w_r.numpy(), support.np_bias(bias))
    assert np.array_equal(ids.cpu().numpy(), ids_o)
    out = gs.run_layer(m, spec, d, out_fp32=False)
    rng = np.random.default_rng(5)
    sample = np.sort(rng.choice(T, 3, replace=False))
    L = w8_lists(wts_d, set(int(e) for e in ids_o[sample].reshape(-1) if e < spec["n_routed"]))
    ref, ids_s, _, _, _ = oracle.layer_w8a8(spec, synth.bf16_bits(x[sample]), w_r.numpy(),
                                            support.np_bias(bias), L["qg"], L["sg"], L["qu"],
                                            L["su"], L["qd"], L["sd"], w8_shared(wts_d))
    assert np.array_equal(ids_s, ids_o[sample])
    gs.check_out(out[torch.as_tensor(sample, device="cuda")], ref, bf16_out=True, what=name)
    del wts_d, d
    torch.cuda.empty_cache()
