"""The tensor-core (tcgen05) path of the grouped FFN alone: every expert forced
onto tensor-core tiles (gemv_max_rows < 0), checked against the fp64 oracle.
Cases grow from one expert with one 16-row tile to ragged shapes."""
import numpy as np
import pytest

import synth
from tests import gpu_support as gs
from tests import support

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def m():
    return gs.lib()


def dense_ref(d):
    xb = support.bf16_to_f64(synth.bf16_bits(d["x"]))
    g, u, dn = support.expert_lists(d["wts"])
    G = support.bf16_to_f64(g[0]) @ xb.T
    U = support.bf16_to_f64(u[0]) @ xb.T
    return (support.bf16_to_f64(dn[0]) @ (G / (1 + np.exp(-G)) * U)).T


@pytest.mark.parametrize("T", [16, 40, 128])
def test_one_expert_one_tile(m, T):
    spec = dict(synth.spec("tiny"), n_routed=1, top_k=1, renormalize=False, T=T,
                name=f"tc_one_{T}")
    d = gs.inputs(spec)
    got = gs.run_layer(m, spec, d, out_fp32=True, gemv_max_rows=-1)
    gs.check_out(got, dense_ref(d), bf16_out=False, what=spec["name"])


@pytest.mark.parametrize("name", ["tiny", "pangu_s", "dsv3_s", "ragged_s", "longcat_s"])
def test_all_tensor_core(m, name):
    spec = synth.spec(name)
    d = gs.inputs(spec)
    ref, _, _ = support.oracle_layer(spec, d["x"], d["w_r"], d["bias"], d["wts"])
    got = gs.run_layer(m, spec, d, out_fp32=True, gemv_max_rows=-1)
    gs.check_out(got, ref, bf16_out=False, what=name)


def test_more_rows_than_one_task(m):
    # 300 rows on one expert: three tensor-core tasks (128 + 128 + 44 rows)
    spec = dict(synth.spec("tiny"), n_routed=1, top_k=1, renormalize=False, T=300,
                hidden=512, inter=256, name="tc_300")
    d = gs.inputs(spec)
    got = gs.run_layer(m, spec, d, out_fp32=True, gemv_max_rows=-1)
    gs.check_out(got, dense_ref(d), bf16_out=False, what="tc_300")
