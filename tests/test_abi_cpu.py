"""The C-ABI library loads, exports what include/moe.h declares, and rejects bad
arguments on the host before touching a GPU.  No compute call is made here."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def moe():
    import __graft_entry__

    __graft_entry__._builder().build()
    import sparse_expert_layer_gb300 as m

    return m


def declared_functions():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+char\s*\*|moe_status)\s+(moe_\w+)\s*\(", src,
                                 flags=re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for f in ("moe_route", "moe_permute", "moe_grouped_ffn", "moe_combine", "moe_layer_forward",
              "moe_workspace_size", "moe_check_device_status", "moe_status_string"):
        assert f in names


def test_library_exports_every_declared_symbol(moe):
    out = subprocess.run(["nm", "-D", "--defined-only", moe._LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\s[TW]\s+(\w+)$", out, flags=re.M))
    missing = [f for f in declared_functions() if f not in exported]
    assert not missing, missing
    for f in declared_functions():
        getattr(moe.lib, f)  # dlsym through ctypes


def test_binding_names_match_header(moe):
    for f in declared_functions():
        if f in ("moe_status_string", "moe_kernel_name", "moe_timing_enable",
                 "moe_timing_collect", "moe_launch_counts"):
            continue
        assert hasattr(moe, f), f


def test_config_struct_layout_matches_header(moe):
    # 17 int32 + 1 float, no padding
    assert ctypes.sizeof(moe.MoeConfig) == 18 * 4


def _ws(moe, cfg, T):
    return moe.moe_workspace_size(cfg, T)


def test_workspace_size_for_the_headline_layers(moe):
    import synth

    for name in synth.HEADLINE:
        s = synth.spec(name)
        cfg = moe.config_from_spec(s)
        n1 = _ws(moe, cfg, s["T"])
        n2 = _ws(moe, cfg, 2 * s["T"])
        assert 0 < n1 < n2


@pytest.mark.parametrize("field,value,status", [
    ("hidden", 7, 1), ("hidden", 0, 1), ("top_k", 0, 1), ("top_k", 9, 1), ("n_group", 3, 1),
    ("score", 5, 1), ("bias_mode", 3, 1), ("shared_inter", 12, 1), ("inter", 4, 1),
    ("renormalize", 2, 1), ("n_routed", -1, 1), ("combine", 3, 1), ("combine", -1, 1),
    ("ffn_launch", 4, 1), ("ffn_launch", -1, 1),
])
def test_invalid_configs_are_rejected(moe, field, value, status):
    import synth

    cfg = moe.config_from_spec(synth.spec("tiny"))
    setattr(cfg, field, value)
    n = ctypes.c_size_t(0)
    assert moe.lib.moe_workspace_size(ctypes.byref(cfg), 16, ctypes.byref(n)) == status


def test_group_rules(moe):
    import synth

    cfg = moe.config_from_spec(synth.spec("dsv3"))
    n = ctypes.c_size_t(0)
    assert moe.lib.moe_workspace_size(ctypes.byref(cfg), 128, ctypes.byref(n)) == 0
    cfg.topk_group = 9
    assert moe.lib.moe_workspace_size(ctypes.byref(cfg), 128, ctypes.byref(n)) == 1
    cfg = moe.config_from_spec(synth.spec("pangu"))
    assert moe.lib.moe_workspace_size(ctypes.byref(cfg), 456, ctypes.byref(n)) == 0
    cfg.top_k = 7  # must equal n_group * per_group_k
    assert moe.lib.moe_workspace_size(ctypes.byref(cfg), 456, ctypes.byref(n)) == 1


def test_unsupported_sizes(moe):
    import synth

    cfg = moe.config_from_spec(synth.spec("tiny"))
    n = ctypes.c_size_t(0)
    cfg.top_k, cfg.n_routed = 33, 64
    assert moe.lib.moe_workspace_size(ctypes.byref(cfg), 16, ctypes.byref(n)) == 2
    cfg.top_k, cfg.n_routed = 2, 5000
    assert moe.lib.moe_workspace_size(ctypes.byref(cfg), 16, ctypes.byref(n)) == 2


def test_w8a8_rules(moe):
    import synth

    n = ctypes.c_size_t(0)
    cfg = moe.config_from_spec(synth.spec("w8a8_s"))
    assert moe.lib.moe_workspace_size(ctypes.byref(cfg), 512, ctypes.byref(n)) == 0
    cfg.hidden = 1000  # int8 rows must be whole 16-byte vectors
    assert moe.lib.moe_workspace_size(ctypes.byref(cfg), 512, ctypes.byref(n)) == 1
    # the shared expert is int8 too: its intermediate size in whole 16-byte rows
    cfg = moe.config_from_spec(synth.spec("w8a8_s", shared_inter=64))
    assert moe.lib.moe_workspace_size(ctypes.byref(cfg), 512, ctypes.byref(n)) == 0
    cfg = moe.config_from_spec(synth.spec("w8a8_s", shared_inter=72))
    assert moe.lib.moe_workspace_size(ctypes.byref(cfg), 512, ctypes.byref(n)) == 1
    # a shared expert with no routed FFN experts is not supported in this mode
    cfg = moe.config_from_spec(synth.spec("w8a8_s", shared_inter=64, n_routed=0, n_zero=8))
    assert moe.lib.moe_workspace_size(ctypes.byref(cfg), 512, ctypes.byref(n)) == 2
    assert moe.lib.moe_qgemm_s8_workspace_size(4, 1024, 256, 100, ctypes.byref(n)) == 0
    assert moe.lib.moe_qgemm_s8_workspace_size(4, 1000, 256, 100, ctypes.byref(n)) == 1


def test_workspace_errors_are_host_side(moe):
    import synth

    cfg = moe.config_from_spec(synth.spec("tiny"))
    need = _ws(moe, cfg, 16)
    fake = 1 << 40  # never dereferenced: every call below fails before any launch
    r = moe.lib.moe_route(ctypes.byref(cfg), 16, fake, fake, None, fake, fake, None, need, None)
    assert r == moe.MOE_ERR_INVALID_ARG
    r = moe.lib.moe_route(ctypes.byref(cfg), 16, fake, fake, None, fake, fake, fake + 8, need, None)
    assert r == moe.MOE_ERR_ALIGNMENT
    r = moe.lib.moe_route(ctypes.byref(cfg), 16, fake, fake, None, fake, fake, fake, need - 1, None)
    assert r == moe.MOE_ERR_WORKSPACE_TOO_SMALL
    r = moe.lib.moe_route(ctypes.byref(cfg), 16, fake + 2, fake, None, fake, fake, fake, need, None)
    assert r == moe.MOE_ERR_ALIGNMENT
    r = moe.lib.moe_route(ctypes.byref(cfg), 16, None, fake, None, fake, fake, fake, need, None)
    assert r == moe.MOE_ERR_INVALID_ARG


def test_bias_is_required_when_configured(moe):
    import synth

    cfg = moe.config_from_spec(synth.spec("longcat_s"))
    need = _ws(moe, cfg, 48)
    fake = 1 << 40
    r = moe.lib.moe_route(ctypes.byref(cfg), 48, fake, fake, None, fake, fake, fake, need, None)
    assert r == moe.MOE_ERR_INVALID_ARG


def test_empty_batch_is_a_no_op(moe):
    import synth

    cfg = moe.config_from_spec(synth.spec("tiny"))
    need = _ws(moe, cfg, 0)
    fake = 1 << 40
    assert moe.lib.moe_route(ctypes.byref(cfg), 0, None, None, None, None, None, fake, need,
                             None) == 0
    assert moe.lib.moe_layer_forward(ctypes.byref(cfg), 0, *([None] * 13), fake, need, None) == 0


def test_status_strings(moe):
    for s in range(8):
        assert moe.lib.moe_status_string(s)
    assert moe.lib.moe_kernel_name(0) == b"router"
    assert moe.lib.moe_kernel_name(99) == b"unknown"


def test_selftest_arguments_are_checked_on_the_host(moe):
    fake = 1 << 40
    assert moe.lib.moe_selftest_wait_timeout(None, 1000, None) == moe.MOE_ERR_INVALID_ARG
    assert moe.lib.moe_selftest_wait_timeout(fake, 0, None) == moe.MOE_ERR_INVALID_ARG
    assert moe.lib.moe_selftest_wait_timeout(fake, 3_000_000_000, None) == moe.MOE_ERR_INVALID_ARG
    assert moe.lib.moe_selftest_wait_timeout(fake + 16, 1000, None) == moe.MOE_ERR_ALIGNMENT


def _table_choice(table, wdtype, H, I, T, k, E):
    """Independent restatement of the tile-table rule: entries of the same weight
    type, nearest in load bucket, then in log2(H * I); first in table order on ties."""
    import math

    m = T * k / E
    b = next((i for i, v in enumerate(table["buckets"]) if m < v), len(table["buckets"]))
    best, best_d = None, None
    for e in table["entries"]:
        if e["wdtype"] != wdtype:
            continue
        d = 1000.0 * abs(e["bucket"] - b) + abs(math.log2(H * max(I, 1) / (e["hidden"] * e["inter"])))
        if best is None or d < best_d:
            best, best_d = e, d
    return best


def test_tile_choice_follows_the_table(moe):
    import json
    import os

    import numpy as np
    import synth

    path = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                        "sparse_expert_layer_gb300", "tuning", "tile_table.json")
    table = json.load(open(path))
    rng = np.random.default_rng(13)
    for wdtype in ("bf16", "w8a8"):
        for _ in range(60):
            H = int(rng.choice([256, 1024, 4096, 5120, 6144, 7168, 8192]))
            I = int(rng.choice([128, 512, 1536, 2048, 4096]))
            E = int(rng.choice([8, 64, 256, 768]))
            k = int(rng.choice([1, 2, 8]))
            T = int(rng.choice([1, 16, 64, 128, 456, 2048, 8192]))
            s = synth.spec("tiny", hidden=H, inter=I, n_routed=E, top_k=k, wdtype=wdtype)
            g, one, wide = moe.moe_tile_choice(moe.config_from_spec(s), T)
            want = _table_choice(table, wdtype, H, I, T, k, E)
            assert g == want["gemv_max"], (wdtype, H, I, E, k, T)
            assert one == (wdtype == "bf16" and bool(want["one_launch"])), (wdtype, H, I, E, k, T)
            assert wide == (one and bool(want.get("dn_wide", 0))), (wdtype, H, I, E, k, T)
    # explicit settings win over the table
    s = synth.spec("longcat")
    assert moe.moe_tile_choice(moe.config_from_spec(s, gemv_max_rows=5), 64)[0] == 5
    assert moe.moe_tile_choice(moe.config_from_spec(s, gemv_max_rows=-1), 64)[0] == 0
    assert moe.moe_tile_choice(moe.config_from_spec(s, ffn_launch=moe.FFN_LAUNCH_TWO), 64)[1] is False
    assert moe.moe_tile_choice(moe.config_from_spec(s, ffn_launch=moe.FFN_LAUNCH_ONE), 64)[1:] \
        == (True, False)
    assert moe.moe_tile_choice(moe.config_from_spec(s, ffn_launch=moe.FFN_LAUNCH_ONE_WIDE),
                               64)[1:] == (True, True)
    # the table's wide down tiles need one launch; W8A8 layers have neither
    sp = synth.spec("pangu")
    assert moe.moe_tile_choice(moe.config_from_spec(sp, ffn_launch=moe.FFN_LAUNCH_TWO),
                               456)[1:] == (False, False)
    sw = synth.spec("pangu", wdtype="w8a8")
    assert moe.moe_tile_choice(moe.config_from_spec(sw, ffn_launch=moe.FFN_LAUNCH_ONE_WIDE),
                               456)[1:] == (False, False)
