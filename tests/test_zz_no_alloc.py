"""moe_route_noalloc: the routing entry point for callers that cannot hand the
library a workspace (a framework that gives an operator only its input and
output buffers, or a decode loop that must not call cudaMalloc).  Its scratch
is a fixed array inside the library; this checks, through the C ABI, that two
calls in a row give the same routing as moe_route, and that a size beyond the
array is refused.  The file name sorts last so a stop-at-first-failure run has
already run every other test."""
import ctypes

import numpy as np
import pytest
import torch

import synth
from tests import gpu_support as gs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def m():
    return gs.lib()


def _route_with_workspace(m, cfg, T, d):
    k = cfg.top_k
    ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, k), dtype=torch.float32, device="cuda")
    ws = m.workspace(cfg, T)
    m.moe_route(cfg, T, d["x_d"], d["w_r_d"], d["bias_d"], ids, w, ws)
    return ids, w


def _noalloc(m, cfg, T, d):
    k = cfg.top_k
    ids = torch.full((T, k), -1, dtype=torch.int32, device="cuda")
    w = torch.full((T, k), -1.0, dtype=torch.float32, device="cuda")
    st = m.lib.moe_route_noalloc(ctypes.byref(cfg), T, d["x_d"].data_ptr(), d["w_r_d"].data_ptr(),
                                 None if d["bias_d"] is None else d["bias_d"].data_ptr(),
                                 ids.data_ptr(), w.data_ptr(),
                                 torch.cuda.current_stream().cuda_stream)
    assert st == m.MOE_OK
    torch.cuda.synchronize()
    return ids, w


@pytest.mark.parametrize("name", ["tiny", "longcat", "dsv3_s", "pangu_s"])
def test_noalloc_route_matches_moe_route_twice(m, name):
    spec = synth.spec(name)
    x, w_r, bias = synth.draw_x(spec), *synth.draw_router(spec)
    d = dict(x_d=x.cuda(), w_r_d=w_r.cuda(), bias_d=None if bias is None else bias.cuda())
    cfg = m.config_from_spec(spec)
    T = spec["T"]
    ref_ids, ref_w = _route_with_workspace(m, cfg, T, d)
    for _ in range(2):
        ids, w = _noalloc(m, cfg, T, d)
        assert torch.equal(ids, ref_ids)
        assert np.allclose(w.cpu().numpy(), ref_w.cpu().numpy(), rtol=1e-5, atol=1e-7)


def test_noalloc_route_at_the_large_batch_switch(m):
    # 1024 tokens x 1024 experts x H = 1024: the logits fill the whole 4 MiB
    # array, and moe_route takes its large-batch router here while the
    # no-allocation entry point keeps the small-batch one.  With routing margins
    # enforced, ids equal the oracle's (and moe_route's) and weights agree to 1e-5.
    import oracle
    from tests import support

    spec = synth.spec("tiny", T=1024, hidden=1024, n_routed=1024, top_k=4, renormalize=True,
                      name="router_tc")
    d = gs.inputs(spec)
    cfg = m.config_from_spec(spec)
    T = spec["T"]
    ids_o, w_o, _, _ = oracle.route(spec, synth.bf16_bits(d["x"]), d["w_r"].numpy(),
                                    support.np_bias(d["bias"]))
    ref_ids, ref_w = _route_with_workspace(m, cfg, T, d)
    for _ in range(2):
        ids, w = _noalloc(m, cfg, T, d)
        assert np.array_equal(ids.cpu().numpy(), ids_o)
        assert torch.equal(ids, ref_ids)
        assert np.allclose(w.cpu().numpy(), w_o, rtol=1e-5, atol=1e-7)
        assert np.allclose(w.cpu().numpy(), ref_w.cpu().numpy(), rtol=1e-5, atol=1e-7)


def test_noalloc_route_refuses_sizes_beyond_its_array(m):
    spec = synth.spec("w8a8_prefill", wdtype="bf16")  # 8192 tokens x 256 experts: 8 MiB
    cfg = m.config_from_spec(spec)
    fake = 1 << 40  # never dereferenced: the size check fails first
    st = m.lib.moe_route_noalloc(ctypes.byref(cfg), spec["T"], fake, fake, fake, fake, fake, None)
    assert st == m.MOE_ERR_WORKSPACE_TOO_SMALL
