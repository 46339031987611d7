"""fp64 CPU oracle of the sparse MoE expert layer -- TEST INFRASTRUCTURE ONLY.

Only the test-suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never does; it fails
loudly when its CUDA build is missing instead of falling back to anything here.

The arithmetic lives in ``moe_oracle.c`` (plain C, fp64, OpenMP over tokens).
This module only compiles it with gcc and marshals numpy arrays.  It shares no
code with ``sparse_expert_layer_gb300``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "liboracle.so")
_lock = threading.Lock()
_lib = None

SOFTMAX, SIGMOID = 0, 1
BIAS_NONE, BIAS_LOGIT, BIAS_SELECT = 0, 1, 2


def build(force: bool = False) -> str:
    """Compile moe_oracle.c into oracle/_build/liboracle.so (gcc, no fast-math)."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    hdr = os.path.join(_HERE, "moe_oracle.h")
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= max(os.path.getmtime(_SRC), os.path.getmtime(hdr))):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-fno-fast-math", "-ffp-contract=off", "-std=c11",
           "-shared", "-fPIC", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class OrcCfg(ctypes.Structure):
    _fields_ = [
        ("hidden", ctypes.c_int), ("inter", ctypes.c_int), ("n_routed", ctypes.c_int),
        ("n_zero", ctypes.c_int), ("top_k", ctypes.c_int), ("n_group", ctypes.c_int),
        ("topk_group", ctypes.c_int), ("per_group_k", ctypes.c_int), ("score", ctypes.c_int),
        ("renormalize", ctypes.c_int), ("routed_scale", ctypes.c_double),
        ("bias_mode", ctypes.c_int), ("shared_inter", ctypes.c_int),
    ]


def make_cfg(spec: dict) -> OrcCfg:
    """Oracle config from a layer description dict (keys as in synth.CONFIGS)."""
    return OrcCfg(
        hidden=spec["hidden"], inter=spec["inter"], n_routed=spec["n_routed"],
        n_zero=spec.get("n_zero", 0), top_k=spec["top_k"], n_group=spec.get("n_group", 1),
        topk_group=spec.get("topk_group", 1), per_group_k=spec.get("per_group_k", 0),
        score=SIGMOID if spec.get("score", "softmax") == "sigmoid" else SOFTMAX,
        renormalize=int(bool(spec.get("renormalize", False))),
        routed_scale=float(spec.get("routed_scale", 1.0)),
        bias_mode={"none": BIAS_NONE, "logit": BIAS_LOGIT, "select": BIAS_SELECT}[
            spec.get("bias_mode", "none")],
        shared_inter=spec.get("shared_inter", 0),
    )


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            I = ctypes.c_int
            C = ctypes.POINTER(OrcCfg)
            lib.orc_router_logits.argtypes = [C, I, P, P, P, P]
            lib.orc_select.argtypes = [C, I, P, P, P, P, P, P]
            lib.orc_permute.argtypes = [I, I, I, P, P, P, P, P]
            lib.orc_swiglu_expert.argtypes = [I, I, P, P, P, P, P, P]
            lib.orc_swiglu_expert.restype = None
            lib.orc_layer.argtypes = [C, I, P, P, P, P, P, P, P, P, P, P, P, P]
            lib.orc_quantize_rows.argtypes = [I, I, P, P, P]
            lib.orc_quantize_rows.restype = None
            lib.orc_int8_matmul.argtypes = [I, I, I, P, P, P]
            lib.orc_int8_matmul.restype = None
            lib.orc_layer_w8a8.argtypes = [C, I, P, P, P, P, P, P, P, P, P, P, P, P, P, P, P,
                                           P, P, P, P, P]
            for f in ("orc_router_logits", "orc_select", "orc_permute", "orc_layer",
                      "orc_layer_w8a8"):
                getattr(lib, f).restype = ctypes.c_int
            _lib = lib
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def _ptr_array(arrs, dtype):
    """(ctypes array of pointers, keep-alive list) for a per-expert list (None allowed)."""
    keep = [None if a is None else _c(a, dtype) for a in arrs]
    ptrs = (ctypes.c_void_p * max(1, len(keep)))()
    for i, a in enumerate(keep):
        ptrs[i] = None if a is None else a.ctypes.data
    return ptrs, keep


def _check(rc, what):
    if rc != 0:
        raise ValueError(f"oracle {what} rejected its arguments (rc={rc})")


def router_logits(spec, x_bits, w_router, bias=None):
    lib, cfg = _load(), make_cfg(spec)
    x_bits, w_router = _c(x_bits, np.uint16), _c(w_router, np.float32)
    bias = _c(bias, np.float32)
    T = x_bits.shape[0]
    E = cfg.n_routed + cfg.n_zero
    out = np.empty((T, E), np.float64)
    _check(lib.orc_router_logits(ctypes.byref(cfg), T, _p(x_bits), _p(w_router), _p(bias),
                                 _p(out)), "router_logits")
    return out


def select(spec, logits, bias=None):
    """-> ids [T,k] int32, weights [T,k] f64, scores [T,E] f64, keys [T,E] f64."""
    lib, cfg = _load(), make_cfg(spec)
    logits = _c(logits, np.float64)
    bias = _c(bias, np.float32)
    T, E = logits.shape
    k = cfg.top_k
    ids = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float64)
    s = np.empty((T, E), np.float64)
    key = np.empty((T, E), np.float64)
    _check(lib.orc_select(ctypes.byref(cfg), T, _p(logits), _p(bias), _p(ids), _p(w), _p(s),
                          _p(key)), "select")
    return ids, w, s, key


def route(spec, x_bits, w_router, bias=None):
    return select(spec, router_logits(spec, x_bits, w_router, bias), bias)


def permute(ids, n_experts):
    """-> counts [E], offsets [E+1], sorted_to_expanded [R], expanded_to_sorted [R]."""
    lib = _load()
    ids = _c(ids, np.int32)
    T, k = ids.shape
    counts = np.empty(n_experts, np.int32)
    offsets = np.empty(n_experts + 1, np.int32)
    s2e = np.empty(T * k, np.int32)
    e2s = np.empty(T * k, np.int32)
    _check(lib.orc_permute(T, k, n_experts, _p(ids), _p(counts), _p(offsets), _p(s2e), _p(e2s)),
           "permute")
    return counts, offsets, s2e, e2s


def swiglu_expert(x_f64, wg_bits, wu_bits, wd_bits):
    """One expert on one token row -> (y [H], h [I]) in fp64."""
    lib = _load()
    x = _c(x_f64, np.float64)
    wg, wu, wd = (_c(a, np.uint16) for a in (wg_bits, wu_bits, wd_bits))
    I, H = wg.shape
    y = np.empty(H, np.float64)
    h = np.empty(I, np.float64)
    lib.orc_swiglu_expert(H, I, _p(x), _p(wg), _p(wu), _p(wd), _p(y), _p(h))
    return y, h


def layer(spec, x_bits, w_router, bias, wg, wu, wd, shared=None):
    """Whole bf16-weight layer.  wg/wu/wd: per-expert lists of bf16-bit arrays
    (entries may be None for experts no token picks).  shared: (sg, su, sd) or None.
    -> out [T,H] f64, ids [T,k], weights [T,k]."""
    lib, cfg = _load(), make_cfg(spec)
    x_bits, w_router = _c(x_bits, np.uint16), _c(w_router, np.float32)
    bias = _c(bias, np.float32)
    T = x_bits.shape[0]
    pg, kg = _ptr_array(wg, np.uint16)
    pu, ku = _ptr_array(wu, np.uint16)
    pd, kd = _ptr_array(wd, np.uint16)
    sg = su = sd = None
    if shared is not None:
        sg, su, sd = (_c(a, np.uint16) for a in shared)
    out = np.empty((T, cfg.hidden), np.float64)
    ids = np.empty((T, cfg.top_k), np.int32)
    w = np.empty((T, cfg.top_k), np.float64)
    _check(lib.orc_layer(ctypes.byref(cfg), T, _p(x_bits), _p(w_router), _p(bias), pg, pu, pd,
                         _p(sg), _p(su), _p(sd), _p(out), _p(ids), _p(w)), "layer")
    del kg, ku, kd
    return out, ids, w


def quantize_rows(v_f32):
    lib = _load()
    v = _c(v_f32, np.float32)
    R, K = v.shape
    q = np.empty((R, K), np.int8)
    s = np.empty(R, np.float32)
    lib.orc_quantize_rows(R, K, _p(v), _p(q), _p(s))
    return q, s


def int8_matmul(a, w):
    lib = _load()
    a, w = _c(a, np.int8), _c(w, np.int8)
    R, K = a.shape
    N = w.shape[0]
    acc = np.empty((R, N), np.int64)
    lib.orc_int8_matmul(R, N, K, _p(a), _p(w), _p(acc))
    return acc


def layer_w8a8(spec, x_bits, w_router, bias, qg, sg, qu, su, qd, sd, shared=None):
    """Whole W8A8 layer -> out [T,H] f64, ids, weights, q_x [T,H] int8, s_x [T] f32.
    shared: (qsg, ssg, qsu, ssu, qsd, ssd) int8 matrices and fp32 scales, or None."""
    lib, cfg = _load(), make_cfg(spec)
    x_bits, w_router = _c(x_bits, np.uint16), _c(w_router, np.float32)
    bias = _c(bias, np.float32)
    T = x_bits.shape[0]
    arrays = [_ptr_array(qg, np.int8), _ptr_array(sg, np.float32), _ptr_array(qu, np.int8),
              _ptr_array(su, np.float32), _ptr_array(qd, np.int8), _ptr_array(sd, np.float32)]
    out = np.empty((T, cfg.hidden), np.float64)
    ids = np.empty((T, cfg.top_k), np.int32)
    w = np.empty((T, cfg.top_k), np.float64)
    qx = np.empty((T, cfg.hidden), np.int8)
    sx = np.empty(T, np.float32)
    sh = [None] * 6
    if shared is not None:
        sh = [_c(a, np.int8 if i % 2 == 0 else np.float32) for i, a in enumerate(shared)]
    _check(lib.orc_layer_w8a8(ctypes.byref(cfg), T, _p(x_bits), _p(w_router), _p(bias),
                              *[a[0] for a in arrays], *[_p(a) for a in sh], _p(out), _p(ids),
                              _p(w), _p(qx), _p(sx)),
           "layer_w8a8")
    del arrays, sh
    return out, ids, w, qx, sx
