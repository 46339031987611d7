"""Benchmark of the GB300 sparse MoE expert layer.

One step = one moe_layer_forward over one batch of synthetic tokens (router ->
top-k -> permute -> grouped SwiGLU FFN -> combine), inputs resident in HBM.
Default workload: the LongCat-Flash-shaped decode layer (T=64 tokens, hidden
6144, 512 SwiGLU experts of intermediate 2048 plus 256 zero-computation
experts, softmax top-12), weights bf16 ~N(0, 0.02).

Prints one JSON line (rank 0).  Its headline is the main workload; its
"configs" object holds the same measurements (ms per step with p50/p90,
tokens/s, the layer's fraction of its roofline, the dominant kernel's roofline,
the step replayed from a CUDA graph,
the oracle timed on a sample) for the other headline layers: the tiny layer, the
DSv3- and Pangu-shaped decode layers and the skewed W8A8 prefill layer, each
generated, measured and freed in turn.  --impl reference times the fp64 CPU
oracle instead, on a bounded sample of the main workload.

Multi-GPU: the layer does not shard across GPUs here (no exchange step is
built), so --gpus N under torchrun runs N independent replicas; the timing
barrier and the max-over-ranks reduction are the only cross-rank calls.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import synth  # noqa: E402

FALLBACK_HBM_GBS = 6800.0
PROFILE_TABLE = os.path.join(ROOT, "profiles", "traffic.json")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="longcat")
    ap.add_argument("--gemv-max-rows", type=int, default=0)
    ap.add_argument("--combine", default="default", choices=["default", "ordered", "fused"],
                    help="how the expert outputs return to their tokens (library default: fused)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--cpu-seconds-extra", type=float, default=5.0)
    ap.add_argument("--extra-configs", default=",".join(EXTRA_CONFIGS),
                    help="comma-separated layers measured after the main one ('none': skip)")
    return ap.parse_args()


# ------------------------------------------------------------ distributed --
def dist_setup(n):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        if not dist.is_initialized():
            dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def whole_job_rate(world, units_per_rank_step, steps, ms_max):
    """Units processed by all ranks per second, timed by the slowest rank."""
    return world * units_per_rank_step * steps / (ms_max / 1e3)


def max_over_ranks(v, world, device):
    if world == 1:
        return v
    import torch.distributed as dist

    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------- clocks --
class ClockSampler:
    """nvidia-smi clock/throttle samples while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            # nvidia-smi takes a moment to start: wait (bounded) for its first
            # sample so the timed region is covered from its start
            t0 = time.time()
            while not self.lines and time.time() - t0 < 5.0 and self.proc.poll() is None:
                time.sleep(0.01)
        except (FileNotFoundError, OSError):
            self.proc = None
        self.first = max(0, len(self.lines) - 1)  # the sample current at the start
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or not self.lines:
            return None
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines[self.first:]:
            p = [s.strip() for s in ln.split(",")]
            if len(p) < 9:
                continue
            try:
                sm.append(float(p[1]))
                mx.append(float(p[2]))
            except ValueError:
                continue
            for nm, v in zip(names, p[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ peaks --
def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(path))
        for key in ("hbm_gbs", "hbm_GBs", "hbm_bandwidth_gbs"):
            if key in d:
                return float(d[key]), "measured"
    except (OSError, ValueError):
        pass
    return FALLBACK_HBM_GBS, "fallback"


FALLBACK_BF16_TFLOPS = 1900.0


def tensor_peak():
    """Dense bf16 (= fp16) tensor peak in TFLOP/s: the sustained figure when
    measured (kernels are timed inside a long step), else the burst one."""
    try:
        d = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
        for key in ("bf16_tflops_sustained", "bf16_tflops"):
            if key in d:
                return float(d[key]), "measured:" + key
    except (OSError, ValueError):
        pass
    return FALLBACK_BF16_TFLOPS, "fallback"


def kernel_work(spec, counts, gemv_max, one_launch):
    """{kernel: (algorithmic bytes, flops)} per launch, from the realised loads.
    A unit (routed expert, or the shared expert over all T rows) with n rows goes
    to the GEMV kernels when n <= the switch point (the library's choice, from
    moe_tile_choice), else to the tensor-core ones; bytes = its weights once + its
    activation rows in and results out.  A W8A8 shared expert always runs on the
    tensor-core kernels; a one-launch bf16 FFN is timed as tc_gate_up (both passes)."""
    H, I, Is, T = spec["hidden"], spec["inter"], spec["shared_inter"], spec["T"]
    w8 = spec["wdtype"] == "w8a8"
    wb = 1 if w8 else 2
    units = [(int(n), I, False) for n in counts[:spec["n_routed"]] if n > 0]
    if Is:
        units.append((T, Is, w8))
    out = {k: [0, 0] for k in ("gemv_gate_up", "gemv_down", "tc_gate_up", "tc_down")}
    for n, inter, force_tc in units:
        p = "gemv_" if n <= gemv_max and not force_tc else "tc_"
        d = "gate_up" if (p == "tc_" and one_launch) else "down"
        out[p + "gate_up"][0] += 2 * inter * H * wb + 2 * n * H + 2 * n * inter
        out[p + "gate_up"][1] += 4 * n * inter * H
        out[p + d][0] += inter * H * wb + 2 * n * inter + 4 * n * H
        out[p + d][1] += 2 * n * inter * H
    return {k: tuple(v) for k, v in out.items() if v[0]}


def kernel_source_hash(files):
    h = hashlib.sha256()
    for f in files:
        h.update(open(os.path.join(ROOT, "sparse_expert_layer_gb300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


def traffic_for(kernel, algorithmic_bytes, wdtype, layer):
    """DRAM bytes of one launch: the committed ncu capture's ratio of DRAM bytes to
    algorithmic bytes times this launch's algorithmic bytes.  A capture of this
    layer itself is preferred; else one of a smaller case of the same kernel
    (traffic grows with the weight bytes streamed).  None when there is no capture
    or the kernel source changed since it was taken."""
    try:
        table = json.load(open(PROFILE_TABLE))
    except (OSError, ValueError):
        return None
    rec = table.get(f"{kernel}/{wdtype}@{layer}") or table.get(f"{kernel}/{wdtype}")
    if not rec or rec.get("source_hash") != kernel_source_hash(rec["source_files"]):
        return None
    return rec["dram_bytes"] / rec["algorithmic_bytes"] * algorithmic_bytes


# ------------------------------------------------------------- workloads --
def describe(spec):
    return (f"{spec['name']}: T={spec['T']} H={spec['hidden']} E={spec['n_routed']}"
            f"+{spec['n_zero']}zero k={spec['top_k']} I={spec['inter']}"
            + (f" shared I={spec['shared_inter']}" if spec["shared_inter"] else ""))


def algorithmic_bytes(spec, counts):
    """Bytes the layer must move: unique routed experts touched + shared expert +
    router weights + bias + x in + out."""
    H, I, Is, E = spec["hidden"], spec["inter"], spec["shared_inter"], synth.n_experts(spec)
    U = int((counts[:spec["n_routed"]] > 0).sum())
    if spec["wdtype"] == "w8a8":
        per = 3 * H * I + 4 * (2 * I + H)  # int8 gate + up + down and their scales
        shared = 3 * H * Is + 4 * (2 * Is + H) if Is else 0
    else:
        per = 6 * H * I  # gate + up + down, bf16
        shared = 6 * H * Is
    b = U * per + shared + 4 * E * H + 2 * 2 * spec["T"] * H
    if spec["bias_mode"] != "none":
        b += 4 * E
    return b, U


# ------------------------------------------------------------ CPU oracle --
def oracle_runner(spec, wts, need, w_r, b):
    """Callable running the fp64 oracle layer on token rows (bf16 bits), with host
    copies of just the experts in `need` (bf16 or int8 + scales)."""
    import oracle

    E = spec["n_routed"]
    if spec["wdtype"] == "w8a8":
        L = {k: [None] * E for k in ("w_gate", "s_gate", "w_up", "s_up", "w_down", "s_down")}
        for e in need:
            for k in L:
                L[k][e] = wts[k][e].cpu().numpy()
        sh = None
        if spec["shared_inter"]:
            sh = tuple(wts[k].cpu().numpy() for k in ("shared_gate", "s_shared_gate", "shared_up",
                                                      "s_shared_up", "shared_down",
                                                      "s_shared_down"))
        return lambda xb: oracle.layer_w8a8(spec, xb, w_r.numpy(), b, L["w_gate"], L["s_gate"],
                                            L["w_up"], L["s_up"], L["w_down"], L["s_down"], sh)
    g, u, dn = [None] * E, [None] * E, [None] * E
    for e in need:
        g[e] = synth.bf16_bits(wts["w_gate"][e])
        u[e] = synth.bf16_bits(wts["w_up"][e])
        dn[e] = synth.bf16_bits(wts["w_down"][e])
    shared = None
    if spec["shared_inter"]:
        shared = tuple(synth.bf16_bits(wts[k]) for k in ("shared_gate", "shared_up",
                                                         "shared_down"))
    return lambda xb: oracle.layer(spec, xb, w_r.numpy(), b, g, u, dn, shared)


def cpu_model():
    """The host CPU's model, from /proc/cpuinfo (x86 'model name', or Arm implementer/part)."""
    import platform

    fields = {}
    try:
        for ln in open("/proc/cpuinfo"):
            if ":" in ln:
                k, v = ln.split(":", 1)
                fields.setdefault(k.strip().lower(), v.strip())
    except OSError:
        pass
    name = fields.get("model name")
    if not name and "cpu part" in fields:
        name = f"implementer {fields.get('cpu implementer', '?')} part {fields['cpu part']}"
    return f"{platform.machine()} {name or 'unknown'}"


def oracle_sample(spec, x, w_r, bias, wts_d, n_tok, target_s):
    """Time the fp64 oracle on the first n_tok tokens (experts copied from HBM)."""
    import oracle

    oracle.build()
    xs = x[:n_tok]
    b = None if bias is None else bias.numpy()
    logits = oracle.router_logits(spec, synth.bf16_bits(xs), w_r.numpy(), b)
    ids, _, _, _ = oracle.select(spec, logits, b)
    need = sorted(set(int(e) for e in ids.reshape(-1) if e < spec["n_routed"]))
    run = oracle_runner(spec, wts_d, need, w_r, b)
    xb = synth.bf16_bits(xs)
    reps, t0 = 0, time.perf_counter()
    while True:
        run(xb)
        reps += 1
        if time.perf_counter() - t0 >= target_s:
            break
    dt = time.perf_counter() - t0
    threads = min(n_tok, int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1)))
    return reps * n_tok / dt, threads, reps, dt, len(need)


def run_reference(args, rank, world):
    if rank != 0:
        return
    spec = synth.spec(args.config)
    dev = torch.device("cuda:0")
    x, w_r, bias, _ = synth.make_inputs(spec)
    n_tok = min(spec["T"], os.cpu_count() or 1)
    import oracle

    oracle.build()
    b = None if bias is None else bias.numpy()
    logits = oracle.router_logits(spec, synth.bf16_bits(x[:n_tok]), w_r.numpy(), b)
    ids, _, _, _ = oracle.select(spec, logits, b)
    need = sorted(set(int(e) for e in ids.reshape(-1) if e < spec["n_routed"]))
    wts = synth.draw_weights(spec, device=dev if torch.cuda.is_available() else "cpu",
                             experts=need)
    times = []
    xb = synth.bf16_bits(x[:n_tok])
    run = oracle_runner(spec, wts, need, w_r, b)
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        run(xb)
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
    total = sum(times)
    value = args.steps * n_tok / total
    cores = min(n_tok, int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1)))
    sample = f"{n_tok} of {spec['T']} tokens per step (all their picks, {len(need)} experts)"
    line = {
        "impl": "reference", "metric": "MoE-layer tokens/s", "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": describe(spec), "tokens_per_step": n_tok},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": sample, "nproc": os.cpu_count(), "cpu_model": cpu_model()},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ ours --
# The other headline layers, measured after the main one in the same run (one
# layer's weights on the device at a time): the tiny layer, the DSv3- and
# Pangu-shaped decode layers and the skewed W8A8 prefill layer.
EXTRA_CONFIGS = ["tiny", "dsv3", "pangu", "w8a8_prefill"]
COMBINE_MODES = {"default": 0, "ordered": 1, "fused": 2}


def zero_pick_share(spec, counts_h):
    """Share of the T*k picks that land on zero-computation experts."""
    return float(counts_h[spec["n_routed"]:].sum()) / (spec["T"] * spec["top_k"])


def measure(args, spec, dev, world, full):
    """Times the layer on one workload.  full: also the launch count, CUDA-graph
    replay and the end-to-end run with host buffers (the main workload)."""
    import sparse_expert_layer_gb300 as moe

    T, H = spec["T"], spec["hidden"]
    x, w_r, bias, _ = synth.make_inputs(spec)
    wts = synth.draw_weights(spec, device=dev)
    cfg = moe.config_from_spec(spec, out_fp32=False, gemv_max_rows=args.gemv_max_rows,
                               combine=COMBINE_MODES[args.combine])
    x_d, w_r_d = x.to(dev), w_r.to(dev)
    bias_d = None if bias is None else bias.to(dev)
    layer = moe.MoeLayer(cfg, T, wts, w_r_d, bias_d, dev)
    out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream(dev)

    # routing once to count the unique experts this batch touches
    E, k = synth.n_experts(spec), spec["top_k"]
    ids = torch.empty((T, k), dtype=torch.int32, device=dev)
    wgt = torch.empty((T, k), dtype=torch.float32, device=dev)
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    s2e = torch.empty(T * k, dtype=torch.int32, device=dev)
    e2s = torch.empty(T * k, dtype=torch.int32, device=dev)
    w8 = spec["wdtype"] == "w8a8"
    x_perm = torch.empty((T * k, H), dtype=torch.int8 if w8 else torch.bfloat16, device=dev)
    x_scale = torch.empty(T * k, dtype=torch.float32, device=dev) if w8 else None
    moe.moe_route(cfg, T, x_d, w_r_d, bias_d, ids, wgt, layer.ws)
    moe.moe_permute(cfg, T, ids, x_d, counts, offsets, s2e, e2s, x_perm, x_scale, layer.ws)
    counts_h = counts.cpu().numpy()
    alg_bytes, U = algorithmic_bytes(spec, counts_h)
    del x_perm
    if spec["name"] in ("longcat", "longcat_w8"):
        # the LongCat-shaped router is drawn so that about a third of the picks
        # land on zero-computation experts
        share = zero_pick_share(spec, counts_h)
        if not 0.30 <= share <= 0.37:
            raise RuntimeError(f"{spec['name']}: zero-expert pick share {share:.3f} "
                               "outside [0.30, 0.37]")

    for _ in range(args.warmup):
        layer.forward(x_d, out)
    torch.cuda.synchronize()
    if moe.moe_check_device_status(layer.ws) != moe.MOE_OK:
        raise RuntimeError("device status set during warm-up")

    # timed region: K steps of the layer call, nothing else on the stream
    launches0 = moe.launch_counts()
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(dev.index or 0) as clk:
        start.record(stream)
        for _ in range(args.steps):
            layer.forward(x_d, out)
        stop.record(stream)
        torch.cuda.synchronize()
    barrier(world)
    ms = start.elapsed_time(stop)
    launches1 = moe.launch_counts()
    gpu_launches = sum(launches1.values()) - sum(launches0.values())
    if moe.moe_check_device_status(layer.ws) != moe.MOE_OK:
        raise RuntimeError("device status set during the timed region")
    ms = max_over_ranks(ms, world, dev)
    ms_step = ms / args.steps
    value = whole_job_rate(world, T, args.steps, ms)

    # per-step spread: the same K steps with an event between steps
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    torch.cuda.synchronize()
    evs[0].record(stream)
    for i in range(args.steps):
        layer.forward(x_d, out)
        evs[i + 1].record(stream)
    torch.cuda.synchronize()
    per_step = sorted(evs[i].elapsed_time(evs[i + 1]) for i in range(args.steps))
    p50 = per_step[len(per_step) // 2]
    p90 = per_step[min(len(per_step) - 1, int(0.9 * len(per_step)))]

    # per-kernel breakdown: the same K steps again, each launch bracketed by
    # CUDA events on its stream (recorded by the library)
    moe.timing_enable(True)
    moe.timing_collect()
    torch.cuda.synchronize()
    for _ in range(args.steps):
        layer.forward(x_d, out)
    torch.cuda.synchronize()
    per_kernel = moe.timing_collect()
    moe.timing_enable(False)

    gemv_max, one_launch, dn_wide = moe.moe_tile_choice(cfg, T)
    res = {"spec": spec, "combine": args.combine, "gemv_max": gemv_max,
           "one_launch": one_launch, "dn_wide": dn_wide, "value": value, "ms_step": ms_step,
           "p50": p50, "p90": p90,
           "gpu_launches": gpu_launches, "clocks": clk.summary(), "per_kernel": per_kernel,
           "counts": counts_h, "alg_bytes": alg_bytes, "U": U}
    res["graph"] = graph_replay(args, layer, x_d, out, dev, world, T)
    if full:
        res["e2e"] = end_to_end(args, layer, x, x_d, out, dev, world, T, H)
    res["cpu"] = None
    if world == 1 and not args.no_cpu_baseline:
        n_tok = min(T, os.cpu_count() or 1)
        secs = args.cpu_seconds if full else args.cpu_seconds_extra
        v, cores, reps, dt, n_exp = oracle_sample(spec, x, w_r, bias, wts, n_tok, secs)
        res["cpu"] = {
            "value": v, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"first {n_tok} of {T} tokens, full layer, {n_exp} experts, "
                      f"{reps} repetitions in {dt:.1f} s",
            "nproc": os.cpu_count(), "cpu_model": cpu_model()}
    del layer, wts
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return res


def graph_replay(args, layer, x_d, out, dev, world, T):
    """The same step replayed from a CUDA graph (launch gaps removed)."""
    import sparse_expert_layer_gb300 as moe

    stream = torch.cuda.current_stream(dev)
    try:
        gs = torch.cuda.Stream(dev)
        gs.wait_stream(stream)
        with torch.cuda.stream(gs):
            layer.forward(x_d, out, stream=gs)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=gs):
            layer.forward(x_d, out, stream=gs)
        g.replay()
        torch.cuda.synchronize()
        g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        g0.record(stream)
        for _ in range(args.steps):
            g.replay()
        g1.record(stream)
        torch.cuda.synchronize()
        gms = max_over_ranks(g0.elapsed_time(g1), world, dev)
        if moe.moe_check_device_status(layer.ws) != moe.MOE_OK:
            raise RuntimeError("device status set during graph replay")
        return {"value": whole_job_rate(world, T, args.steps, gms), "unit": "tokens/s",
                "ms_per_step": gms / args.steps}
    except RuntimeError as exc:  # capture unavailable: report why, keep the line
        return {"unavailable": str(exc)[:200]}


def end_to_end(args, layer, x, x_d, out, dev, world, T, H):
    """Host buffers: the H2D copy of x and the D2H copy of out inside the timed region."""
    stream = torch.cuda.current_stream(dev)
    x_h = x.pin_memory()
    out_h = torch.empty((T, H), dtype=torch.bfloat16).pin_memory()
    x_e = torch.empty_like(x_d)
    for _ in range(2):
        x_e.copy_(x_h, non_blocking=True)
        layer.forward(x_e, out)
        out_h.copy_(out, non_blocking=True)
    barrier(world)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        x_e.copy_(x_h, non_blocking=True)
        layer.forward(x_e, out)
        out_h.copy_(out, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    ms_e2e = max_over_ranks(e0.elapsed_time(e1), world, dev)
    return {"value": whole_job_rate(world, T, args.steps, ms_e2e), "unit": "tokens/s",
            "h2d_bytes_per_step": x.numel() * 2, "d2h_bytes_per_step": out.numel() * 2}


def roofline_of(args, res):
    """Roofline of the dominant kernel, the layer's HBM and tensor fractions."""
    spec, per_kernel, counts_h = res["spec"], res["per_kernel"], res["counts"]
    peak, peak_kind = hbm_peak()
    tpeak, tpeak_kind = tensor_peak()
    dom = max(per_kernel, key=lambda kname: per_kernel[kname][0])
    dom_ms, dom_n = per_kernel[dom]
    work = kernel_work(spec, counts_h, res["gemv_max"], res["one_launch"])
    roof = None
    if dom in work and dom_n:
        kb, kf = work[dom]
        sec = dom_ms / dom_n / 1e3
        # the kernel's own bound: arithmetic intensity against the ridge point of
        # the two measured peaks (tensor FLOP/s over HBM bytes/s)
        if kf / kb > tpeak * 1e12 / (peak * 1e9):
            achieved = kf / sec / 1e12
            roof = {"kernel": dom, "bound": "tensor", "achieved": achieved, "peak": tpeak,
                    "unit": "TFLOP/s", "frac": achieved / tpeak, "peak_source": tpeak_kind,
                    "traffic": traffic_for(dom, kb, spec["wdtype"], spec["name"]),
                    "algorithmic_flops_per_launch": kf, "avg_launch_ms": dom_ms / dom_n}
        else:
            achieved = kb / sec / 1e9
            roof = {"kernel": dom, "bound": "hbm", "achieved": achieved, "peak": peak,
                    "unit": "GB/s", "frac": achieved / peak, "peak_source": peak_kind,
                    "traffic": traffic_for(dom, kb, spec["wdtype"], spec["name"]),
                    "algorithmic_bytes_per_launch": kb, "avg_launch_ms": dom_ms / dom_n}
    ms_step = res["ms_step"]
    layer_gbs = res["alg_bytes"] / (ms_step / 1e3) / 1e9
    layer_flops = sum(f for k_, (b_, f) in work.items() if k_.startswith(("tc_", "gemv_")))
    layer_hbm = {"achieved_gbs": layer_gbs, "algorithmic_bytes": res["alg_bytes"],
                 "frac": layer_gbs / peak, "peak": peak, "peak_source": peak_kind}
    layer_tensor = {"achieved_tflops": layer_flops / (ms_step / 1e3) / 1e12,
                    "expert_flops": layer_flops, "peak": tpeak, "peak_source": tpeak_kind,
                    "frac": layer_flops / (ms_step / 1e3) / 1e12 / tpeak}
    return roof, layer_hbm, layer_tensor


def config_block(spec, res):
    counts_h = res["counts"]
    gb = res["alg_bytes"] / 1e9
    l2 = (f"inputs larger than L2: {gb:.1f} GB of weights streamed per step, 129 MB L2"
          if gb > 0.5 else f"L2-resident: {gb * 1e3:.1f} MB per step, not flushed "
          "(latency-bound layer)")
    return {"workload": describe(spec), "tokens": spec["T"], "unique_experts": res["U"],
            "gemv_max_rows": res["gemv_max"], "ffn_one_launch": res["one_launch"],
            "ffn_wide_down_tiles": res["dn_wide"],
            "real_picks": int(counts_h[:spec["n_routed"]].sum()),
            "zero_pick_share": zero_pick_share(spec, counts_h) if spec["n_zero"] else 0.0,
            "l2": l2, "combine": res["combine"]}


def summary_of(args, res):
    """One entry of the per-layer table: every headline layer but the main one."""
    spec = res["spec"]
    roof, layer_hbm, layer_tensor = roofline_of(args, res)
    w8 = spec["wdtype"] == "w8a8"
    bound = "tensor" if w8 else ("latency" if spec["name"] == "tiny" else "hbm")
    return {
        "config": config_block(spec, res), "dtype": "int8" if w8 else "bf16",
        "steps": args.steps, "warmup": args.warmup,
        "value": res["value"], "unit": "tokens/s", "ms_per_step": res["ms_step"],
        "ms_per_step_p50": res["p50"], "ms_per_step_p90": res["p90"],
        "layer_bound": bound,
        "layer_frac": layer_tensor["frac"] if w8 else layer_hbm["frac"],
        "layer_hbm": layer_hbm, "layer_tensor": layer_tensor, "roofline": roof,
        "kernels_ms_per_step": {k: v[0] / args.steps for k, v in res["per_kernel"].items()
                                if v[1]},
        "gpu_launches": res["gpu_launches"], "clocks": res["clocks"],
        "cuda_graph": res["graph"],
        "cpu_baseline": res["cpu"],
    }


def run_ours(args, rank, world, local):
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    spec = synth.spec(args.config)
    res = measure(args, spec, dev, world, full=True)
    T = spec["T"]
    roof, layer_hbm, layer_tensor = roofline_of(args, res)
    w8 = spec["wdtype"] == "w8a8"
    line = {
        "metric": "MoE-layer tokens/s", "value": res["value"], "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": res["ms_step"], "ms_per_step_p50": res["p50"],
        "ms_per_step_p90": res["p90"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "int8" if w8 else "bf16",
        "data": "synthetic",
        "config": dict(config_block(spec, res), parallelism=f"replicas x{world}"),
        "layer_hbm": layer_hbm, "layer_tensor": layer_tensor,
        "roofline": roof,
        "kernels_ms_per_step": {kname: v[0] / args.steps for kname, v in res["per_kernel"].items()
                                if v[1]},
        "e2e": res["e2e"],
        "cuda_graph": res["graph"],
        "gpu_launches": res["gpu_launches"],
        "clocks": res["clocks"],
    }
    if res["cpu"] is not None and rank == 0:
        line["cpu_baseline"] = res["cpu"]
    extras = [c for c in (args.extra_configs.split(",") if args.extra_configs else [])
              if c and c != "none" and c != args.config]
    if extras:
        line["configs"] = {}
        for name in extras:
            line["configs"][name] = summary_of(args, measure(args, synth.spec(name), dev, world,
                                                             full=False))
    if rank == 0:
        print(json.dumps(line), flush=True)


def main():
    args = parse()
    rank, world, local = dist_setup(args.gpus)
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, world, local)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
