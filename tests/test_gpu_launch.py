"""Launch-order checks of moe_layer_forward.

The library's kernels are launched with programmatic dependent launch: each may
be scheduled while its predecessor on the stream is finishing and waits for it
before touching device memory.  A kernel that read or wrote memory too early
would race with the kernel before it, or with the previous call on the same
workspace.  These tests look for such races and compare against plain launches.
"""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import synth
from tests import gpu_support as gs

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def m():
    return gs.lib()


def _forward(m, spec, d, cfg, x, out, ws):
    w = d["wts_d"]
    m.moe_layer_forward(cfg, x.shape[0], x, d["w_r_d"], d["bias_d"], w.get("w_gate"),
                        w.get("w_up"), w.get("w_down"), w.get("s_gate"), w.get("s_up"),
                        w.get("s_down"), w.get("shared_gate"), w.get("shared_up"),
                        w.get("shared_down"), out, ws)


@pytest.mark.parametrize("name", ["longcat_s", "dsv3_s", "ragged_s", "w8a8_s"])
def test_back_to_back_calls_on_one_workspace(m, name):
    # Calls alternate between two inputs on one stream and one workspace with
    # no synchronisation in between; each must equal its input's result from a
    # synchronised call.  A kernel that ran ahead of its predecessor would mix
    # the two inputs' intermediate buffers.
    spec = synth.spec(name)
    d = gs.inputs(spec)
    xa = d["x_d"]
    xb = torch.flip(xa, dims=[0]).contiguous()
    ordered = m.COMBINE_ORDERED  # bit-exact comparisons need the deterministic combine
    ref_a = gs.run_layer(m, spec, d, out_fp32=True, x=xa, combine=ordered)
    ref_b = gs.run_layer(m, spec, d, out_fp32=True, x=xb, combine=ordered)
    cfg = m.config_from_spec(spec, out_fp32=True, combine=ordered)
    T = xa.shape[0]
    ws = m.workspace(cfg, T, xa.device)
    outs = [torch.empty((T, spec["hidden"]), dtype=torch.float32, device=xa.device)
            for _ in range(12)]
    for i, out in enumerate(outs):
        _forward(m, spec, d, cfg, xa if i % 2 == 0 else xb, out, ws)
    torch.cuda.synchronize()
    assert m.moe_check_device_status(ws) == m.MOE_OK
    for i, out in enumerate(outs):
        assert torch.equal(out, ref_a if i % 2 == 0 else ref_b), f"call {i}"


_PLAIN = r"""
import sys, numpy as np, torch
sys.path.insert(0, sys.argv[1])
import synth
from tests import gpu_support as gs
m = gs.lib()
spec = gs.layer_spec(sys.argv[2])
d = gs.inputs(spec)
out = gs.run_layer(m, spec, d, out_fp32=True, combine=m.COMBINE_ORDERED)
np.save(sys.argv[3], out.cpu().numpy())
"""


@pytest.mark.parametrize("name", ["dsv3_s", "w8a8_s"])
def test_plain_launches_give_the_same_bits(m, name, tmp_path):
    # MOE_PDL=0 (read once per process) launches every kernel in plain stream
    # order; the outputs must be identical.
    spec = synth.spec(name)
    d = gs.inputs(spec)
    got = gs.run_layer(m, spec, d, out_fp32=True, combine=m.COMBINE_ORDERED).cpu().numpy()
    path = str(tmp_path / "plain.npy")
    env = dict(os.environ, MOE_PDL="0", PYTHONPATH=ROOT)
    r = subprocess.run([sys.executable, "-c", _PLAIN, ROOT, name, path], env=env, cwd=ROOT,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    plain = np.load(path)
    assert np.array_equal(got, plain)


@pytest.mark.parametrize("name", ["tiny", "pangu_s", "longcat_s", "ragged_s", "one_cta_groups",
                                  "one_cta_per_group"])
def test_unfolded_launches_give_the_same_bits(m, name, tmp_path):
    # MOE_FOLDS=0 (read once per process) runs the small layers' router, the
    # top-k, the re-sort, the gather and the finalize as launches of their own
    # instead of inside another kernel; the outputs must be identical.
    spec = gs.layer_spec(name)
    d = gs.inputs(spec)
    got = gs.run_layer(m, spec, d, out_fp32=True, combine=m.COMBINE_ORDERED).cpu().numpy()
    path = str(tmp_path / "unfolded.npy")
    env = dict(os.environ, MOE_FOLDS="0", PYTHONPATH=ROOT)
    r = subprocess.run([sys.executable, "-c", _PLAIN, ROOT, name, path], env=env, cwd=ROOT,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    assert np.array_equal(got, np.load(path))


@pytest.mark.parametrize("name", ["tiny", "pangu_s", "dsv3_s", "ragged_s"])
def test_wide_down_tiles_give_the_same_bits(m, name):
    # The one-launch FFN's down pass in 256-channel tiles (two weight boxes per
    # activation box) or in 128-channel ones: each output channel is the same
    # sequence of MMAs either way, so with the ordered combine the outputs are
    # identical.  H = 640 and 1000 leave a partial wide tile; pangu_s's shared
    # expert has row chunks of more than 64 rows.
    spec = gs.layer_spec(name)
    d = gs.inputs(spec)
    ordered = m.COMBINE_ORDERED
    wide = gs.run_layer(m, spec, d, combine=ordered, ffn_launch=m.FFN_LAUNCH_ONE_WIDE)
    narrow = gs.run_layer(m, spec, d, combine=ordered, ffn_launch=m.FFN_LAUNCH_ONE)
    assert torch.equal(wide, narrow)


_ROUTE_CC = r"""
import sys, numpy as np, torch
sys.path.insert(0, sys.argv[1])
import oracle, synth
from tests import gpu_support as gs, support
m = gs.lib()
for name in sys.argv[2:]:
    spec = synth.spec(name)
    x, w_r, bias, _ = support.make_inputs(spec)
    cfg = m.config_from_spec(spec)
    T, k = spec["T"], spec["top_k"]
    ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, k), dtype=torch.float32, device="cuda")
    ws = m.workspace(cfg, T)
    m.moe_route(cfg, T, x.cuda(), w_r.cuda(), None if bias is None else bias.cuda(), ids, w, ws)
    torch.cuda.synchronize()
    assert m.moe_check_device_status(ws) == m.MOE_OK
    ids_o, w_o, _, _ = oracle.route(spec, synth.bf16_bits(x), w_r.numpy(), support.np_bias(bias))
    assert np.array_equal(ids.cpu().numpy(), ids_o), name
    assert np.allclose(w.cpu().numpy(), w_o, rtol=1e-5, atol=1e-7), name
    print("ok", name)
"""


def test_route_with_tensor_core_router_off():
    # MOE_ROUTER_TC=0 (read once per process) keeps small-batch routing on the
    # CUDA-core router; the layers whose shapes pick the tensor-core router by
    # default must still route exactly as the oracle does.
    env = dict(os.environ, MOE_ROUTER_TC="0", PYTHONPATH=ROOT)
    r = subprocess.run([sys.executable, "-c", _ROUTE_CC, ROOT, "dsv3_s", "longcat_s", "tiny"],
                       env=env, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.count("ok ") == 3
