"""Offline sweep that writes the grouped FFN's tile-parameter table.

For each layer shape it times moe_layer_forward on a GB300 over the candidate
tilings (GEMV / tensor-core switch point; for bf16 layers two persistent
launches, one, or one with 256-channel down tiles) and records the fastest in
tuning/tile_table.json, together with every candidate's time.  The library compiles that table in (build.py) and
looks it up per call (moe_tile_choice): the tiling choice made from measured
history of the Pangu Pro MoE disclosure, section SwiftGMM.

    python sparse_expert_layer_gb300/tuning/sweep.py [--layers a,b,...] [--out path]

Needs a CUDA device; a few minutes on one GB300.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

LAYERS = ["longcat", "dsv3", "pangu", "tiny", "longcat_w8", "w8a8_prefill"]
GEMV_BF16 = [-1, 1, 2, 4, 8]
GEMV_W8 = [-1, 2, 4, 8, 16]


def load_bucket(spec, buckets):
    m = spec["T"] * spec["top_k"] / (spec["n_routed"] + spec["n_zero"])
    for b, v in enumerate(buckets):
        if m < v:
            return b
    return len(buckets)


def time_layer(moe, torch, spec, d, gemv, launch, steps, warmup):
    cfg = moe.config_from_spec(spec, out_fp32=False, gemv_max_rows=gemv, ffn_launch=launch)
    layer = moe.MoeLayer(cfg, spec["T"], d["w"], d["w_r"], d["bias"], d["dev"])
    out = torch.empty((spec["T"], spec["hidden"]), dtype=torch.bfloat16, device=d["dev"])
    for _ in range(warmup):
        layer.forward(d["x"], out)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(steps):
        layer.forward(d["x"], out)
    b.record()
    torch.cuda.synchronize()
    if moe.moe_check_device_status(layer.ws) != moe.MOE_OK:
        raise RuntimeError(f"{spec['name']}: device status set")
    return a.elapsed_time(b) / steps


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--layers", default=",".join(LAYERS))
    ap.add_argument("--out", default=os.path.join(HERE, "tile_table.json"))
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    args = ap.parse_args()

    import torch

    import __graft_entry__
    __graft_entry__.build()
    import sparse_expert_layer_gb300 as moe
    import synth

    table = json.load(open(os.path.join(HERE, "tile_table.json")))
    buckets = table["buckets"]
    dev = torch.device("cuda:0")
    entries = []
    for name in args.layers.split(","):
        spec = synth.spec(name)
        x, w_r, bias, _ = synth.make_inputs(spec)
        d = dict(x=x.to(dev), w_r=w_r.to(dev), bias=None if bias is None else bias.to(dev),
                 w=synth.draw_weights(spec, device=dev), dev=dev)
        w8 = spec["wdtype"] == "w8a8"
        suffix = {moe.FFN_LAUNCH_TWO: "_two", moe.FFN_LAUNCH_ONE: "_one",
                  moe.FFN_LAUNCH_ONE_WIDE: "_wide"}
        launches = [moe.FFN_LAUNCH_DEFAULT] if w8 else list(suffix)
        ms = {}
        for gemv in (GEMV_W8 if w8 else GEMV_BF16):
            for launch in launches:
                key = f"gemv{max(gemv, 0)}" + ("" if w8 else suffix[launch])
                ms[key] = round(time_layer(moe, torch, spec, d, gemv, launch, args.steps,
                                           args.warmup), 5)
                print(name, key, ms[key], flush=True)
        best = min(ms, key=ms.get)
        gemv_best = int(best.split("_")[0][4:])
        entries.append({"wdtype": spec["wdtype"], "hidden": spec["hidden"],
                        "inter": spec["inter"], "bucket": load_bucket(spec, buckets),
                        "gemv_max": gemv_best,
                        "one_launch": int(best.endswith("_one") or best.endswith("_wide")),
                        "dn_wide": int(best.endswith("_wide")), "layer": name, "ms": ms})
        del d
        torch.cuda.empty_cache()
    table["entries"] = entries
    tmp = args.out + ".tmp"
    with open(tmp, "w") as f:
        json.dump(table, f, indent=1)
    os.replace(tmp, args.out)
    print("wrote", args.out)


if __name__ == "__main__":
    main()
