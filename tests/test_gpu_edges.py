"""Edge cases on the GPU: the largest supported routing shapes, degenerate layers,
the smallest hidden sizes, an all-zero token under W8A8, and the device-side
failure path (a bounded wait that runs out is reported, not trapped)."""
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


def route_check(m, spec):
    d = gs.inputs(spec)
    cfg = m.config_from_spec(spec)
    T, k = spec["T"], spec["top_k"]
    ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, k), dtype=torch.float32, device="cuda")
    ws = m.workspace(cfg, T)
    m.moe_route(cfg, T, d["x_d"], d["w_r_d"], d["bias_d"], ids, w, ws)
    torch.cuda.synchronize()
    assert m.moe_check_device_status(ws) == m.MOE_OK
    ids_o, w_o, _, _ = oracle.route(spec, synth.bf16_bits(d["x"]), d["w_r"].numpy(),
                                    support.np_bias(d["bias"]))
    assert np.array_equal(ids.cpu().numpy(), ids_o)
    assert np.allclose(w.cpu().numpy(), w_o, rtol=1e-5, atol=1e-7)
    return d


def test_most_experts_and_largest_top_k(m):
    # 4096 experts (the limit) and top-32 (the limit), as 32 groups with one winner each
    spec = synth.spec("tiny", T=40, hidden=64, inter=32, n_routed=4096, top_k=32, n_group=32,
                      per_group_k=1, renormalize=True, name="max_experts")
    d = route_check(m, spec)
    ref, _, _ = support.oracle_layer(spec, d["x"], d["w_r"], d["bias"], d["wts"])
    gs.check_out(gs.run_layer(m, spec, d), ref, bf16_out=False, what="max_experts")


def test_most_groups(m):
    # 64 groups (the limit) of 4 experts, top-8 groups by their top-2 sums, sigmoid scores
    spec = synth.spec("tiny", T=64, hidden=128, inter=64, n_routed=256, top_k=8, n_group=64,
                      topk_group=8, score="sigmoid", renormalize=True, name="max_groups")
    d = route_check(m, spec)
    ref, _, _ = support.oracle_layer(spec, d["x"], d["w_r"], d["bias"], d["wts"])
    gs.check_out(gs.run_layer(m, spec, d), ref, bf16_out=False, what="max_groups")


def test_only_zero_computation_experts(m):
    # no FFN expert at all: every pick passes its token through, weighted
    spec = synth.spec("tiny", T=20, n_routed=0, n_zero=8, top_k=3, renormalize=False,
                      name="zeros_only")
    d = gs.inputs(spec)
    got = gs.run_layer(m, spec, d).cpu().double().numpy()
    ref, _, _ = support.oracle_layer(spec, d["x"], d["w_r"], d["bias"], d["wts"])
    assert np.allclose(got, ref, rtol=2e-6, atol=1e-6)


def test_every_expert_picked(m):
    # top_k equal to the number of experts: every expert gets every token
    spec = synth.spec("tiny", T=24, top_k=8, renormalize=True, name="k_equals_e")
    d = gs.inputs(spec)
    ref, _, _ = support.oracle_layer(spec, d["x"], d["w_r"], d["bias"], d["wts"])
    for g in (0, 8):
        gs.check_out(gs.run_layer(m, spec, d, gemv_max_rows=g), ref, bf16_out=False,
                     what=f"k=E gemv<={g}")


@pytest.mark.parametrize("hidden,inter", [(16, 16), (64, 8), (1032, 264)])
def test_smallest_shapes(m, hidden, inter):
    # one K step and one partial tile on either path; 1032 x 264 ends every
    # pass with an 8-element K step and an 8-channel tile
    spec = synth.spec("tiny", T=9, hidden=hidden, inter=inter, name=f"small_{hidden}_{inter}")
    d = gs.inputs(spec)
    ref, _, _ = support.oracle_layer(spec, d["x"], d["w_r"], d["bias"], d["wts"])
    for g in (0, 8):
        gs.check_out(gs.run_layer(m, spec, d, gemv_max_rows=g), ref, bf16_out=False,
                     what=f"H={hidden} I={inter} gemv<={g}")


def test_w8a8_all_zero_token(m):
    # amax 0: the token's scale is 0, every code is 0 and its expert outputs are 0
    spec = synth.spec("w8a8_s", T=64, name="w8_zero_row")
    d = dict(gs.inputs(spec))
    x = d["x"].clone()
    x[5] = 0
    d["x"], d["x_d"] = x, x.cuda()
    got = gs.run_layer(m, spec, d).cpu().double().numpy()
    assert np.all(got[5] == 0.0)
    from tests.test_gpu_w8a8 import w8_lists
    L = w8_lists(d["wts"])
    ref, _, _, _, _ = oracle.layer_w8a8(spec, synth.bf16_bits(x), d["w_r"].numpy(),
                                        support.np_bias(d["bias"]), L["qg"], L["sg"], L["qu"],
                                        L["su"], L["qd"], L["sd"])
    gs.check_out(torch.as_tensor(got), ref, bf16_out=False, what="w8 zero row")


def test_bounded_wait_runs_out_and_is_reported(m):
    # a ~1 ms limit on a barrier that nothing completes: the kernel records a
    # timeout and returns; the host reads it and the context stays usable
    ws = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    m.moe_selftest_wait_timeout(ws, 2_000_000)
    assert m.moe_check_device_status(ws) == m.MOE_ERR_DEVICE_TIMEOUT
    assert m.moe_check_device_status(ws) == m.MOE_OK  # reading cleared it
    spec = synth.spec("tiny")
    d = gs.inputs(spec)
    ref, _, _ = support.oracle_layer(spec, d["x"], d["w_r"], d["bias"], d["wts"])
    gs.check_out(gs.run_layer(m, spec, d), ref, bf16_out=False, what="after timeout")
