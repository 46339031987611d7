"""Python binding of libmoe.so, the GB300 sparse MoE expert layer.

Argument marshalling only: every step of the layer runs in the library's CUDA
kernels.  Functions carry the C names (moe_route, moe_permute, moe_grouped_ffn,
moe_combine, moe_layer_forward, ...).  Tensor arguments may be torch tensors
(their device pointer is passed), raw integer addresses, or None for NULL.
Streams may be a torch.cuda.Stream, a raw handle, or None for torch's current
stream.

There is no fallback: if the shared library has not been built this module
raises on import.
"""
from __future__ import annotations

import ctypes
import os

from . import build as _build_mod

_LIB_PATH = _build_mod.LIB

if not os.path.exists(_LIB_PATH):
    raise ImportError(
        f"{_LIB_PATH} is missing: build it with sparse_expert_layer_gb300.build.build() "
        "(nvcc, sm_103a); this package has no non-CUDA implementation")

lib = ctypes.CDLL(_LIB_PATH)

# moe_status
MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_UNSUPPORTED = 2
MOE_ERR_ALIGNMENT = 3
MOE_ERR_WORKSPACE_TOO_SMALL = 4
MOE_ERR_CUDA = 5
MOE_ERR_DEVICE_CHECK = 6
MOE_ERR_DEVICE_TIMEOUT = 7
SCORE_SOFTMAX, SCORE_SIGMOID = 0, 1
BIAS_NONE, BIAS_LOGIT, BIAS_SELECT = 0, 1, 2
W_BF16, W8A8 = 0, 1
COMBINE_DEFAULT, COMBINE_ORDERED, COMBINE_FUSED = 0, 1, 2
FFN_LAUNCH_DEFAULT, FFN_LAUNCH_TWO, FFN_LAUNCH_ONE, FFN_LAUNCH_ONE_WIDE = 0, 1, 2, 3

KERNELS = ["router", "topk", "perm_count", "perm_scan", "perm_scatter", "perm_gather",
           "worklist", "gemv_gate_up", "gemv_down", "tc_gate_up", "tc_down", "quant_h", "combine",
           "w8_exact", "sort"]
N_KERNELS = len(KERNELS)


class MoeConfig(ctypes.Structure):
    """Mirror of moe_config in include/moe.h."""
    _fields_ = [(n, ctypes.c_int32) for n in (
        "hidden", "inter", "n_routed", "n_zero", "top_k", "n_group", "topk_group", "per_group_k",
        "score", "renormalize")] + [("routed_scale", ctypes.c_float)] + [
        (n, ctypes.c_int32) for n in (
            "bias_mode", "shared_inter", "wdtype", "out_fp32", "gemv_max_rows", "combine",
            "ffn_launch")]


class MoeError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {lib.moe_status_string(status).decode()} (status {status})")


_P = ctypes.c_void_p
_I = ctypes.c_int32
_C = ctypes.POINTER(MoeConfig)
_SZ = ctypes.c_size_t

lib.moe_status_string.restype = ctypes.c_char_p
lib.moe_status_string.argtypes = [ctypes.c_int]
lib.moe_kernel_name.restype = ctypes.c_char_p
lib.moe_kernel_name.argtypes = [_I]
_SIGS = {
    "moe_workspace_size": [_C, _I, ctypes.POINTER(_SZ)],
    "moe_route": [_C, _I, _P, _P, _P, _P, _P, _P, _SZ, _P],
    "moe_permute": [_C, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P],
    "moe_grouped_ffn": [_C, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P],
    "moe_combine": [_C, _I, _P, _P, _P, _P, _P, _P, _P, _P],
    "moe_layer_forward": [_C, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ,
                          _P],
    "moe_check_device_status": [_P, _P],
    "moe_route_noalloc": [_C, _I, _P, _P, _P, _P, _P, _P],
    "moe_tile_choice": [_C, _I, ctypes.POINTER(_I), ctypes.POINTER(_I)],
    "moe_qgemm_s8_workspace_size": [_I, _I, _I, _I, ctypes.POINTER(_SZ)],
    "moe_qgemm_s8": [_I, _I, _I, _I, _P, _P, _P, _P, _P, _SZ, _P],
    "moe_selftest_wait_timeout": [_P, ctypes.c_int64, _P],
    "moe_timing_enable": [_I],
    "moe_timing_collect": [ctypes.POINTER(ctypes.c_float), ctypes.POINTER(_I), _I],
    "moe_launch_counts": [ctypes.POINTER(ctypes.c_int64), _I],
}
for _name, _args in _SIGS.items():
    _f = getattr(lib, _name)
    _f.argtypes = _args
    _f.restype = ctypes.c_int

EXPORTS = sorted(list(_SIGS) + ["moe_status_string", "moe_kernel_name"])


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(status, what):
    if status != MOE_OK:
        raise MoeError(status, what)


def config_from_spec(spec: dict, out_fp32: bool = False, gemv_max_rows: int = 0,
                     combine: int = COMBINE_DEFAULT,
                     ffn_launch: int = FFN_LAUNCH_DEFAULT) -> MoeConfig:
    """MoeConfig from a layer description dict (the keys used by the input generator)."""
    return MoeConfig(
        hidden=spec["hidden"], inter=spec["inter"], n_routed=spec["n_routed"],
        n_zero=spec.get("n_zero", 0), top_k=spec["top_k"], n_group=spec.get("n_group", 1),
        topk_group=spec.get("topk_group", 1), per_group_k=spec.get("per_group_k", 0),
        score=SCORE_SIGMOID if spec.get("score", "softmax") == "sigmoid" else SCORE_SOFTMAX,
        renormalize=int(bool(spec.get("renormalize", False))),
        routed_scale=float(spec.get("routed_scale", 1.0)),
        bias_mode={"none": BIAS_NONE, "logit": BIAS_LOGIT, "select": BIAS_SELECT}[
            spec.get("bias_mode", "none")],
        shared_inter=spec.get("shared_inter", 0),
        wdtype=W8A8 if spec.get("wdtype", "bf16") == "w8a8" else W_BF16,
        out_fp32=int(bool(out_fp32)), gemv_max_rows=int(gemv_max_rows), combine=int(combine),
        ffn_launch=int(ffn_launch))


def moe_tile_choice(cfg: MoeConfig, T: int):
    """(GEMV switch point, one-launch FFN, 256-channel down tiles) the library
    picks for (cfg, T)."""
    g, o = _I(0), _I(0)
    _check(lib.moe_tile_choice(ctypes.byref(cfg), T, ctypes.byref(g), ctypes.byref(o)),
           "moe_tile_choice")
    return g.value, o.value >= 1, o.value == 2


def moe_workspace_size(cfg: MoeConfig, T: int) -> int:
    n = _SZ(0)
    _check(lib.moe_workspace_size(ctypes.byref(cfg), T, ctypes.byref(n)), "moe_workspace_size")
    return n.value


def workspace(cfg: MoeConfig, T: int, device="cuda"):
    """Zeroed uint8 device tensor of moe_workspace_size bytes (status word cleared)."""
    import torch
    return torch.zeros(moe_workspace_size(cfg, T), dtype=torch.uint8, device=device)


def moe_route(cfg, T, x, w_router, bias, topk_ids, topk_w, ws, stream=None):
    _check(lib.moe_route(ctypes.byref(cfg), T, _ptr(x), _ptr(w_router), _ptr(bias),
                         _ptr(topk_ids), _ptr(topk_w), _ptr(ws), _ws_bytes(ws), _stream(stream)),
           "moe_route")


def moe_route_noalloc(cfg, T, x, w_router, bias, topk_ids, topk_w, stream=None):
    """moe_route without a workspace, for callers that cannot give the library
    any memory besides the tensors (see include/moe.h): its scratch is a fixed
    4 MiB array inside the library, shared by every call on the device, so
    calls that overlap on the GPU must not be issued."""
    _check(lib.moe_route_noalloc(ctypes.byref(cfg), T, _ptr(x), _ptr(w_router), _ptr(bias),
                                 _ptr(topk_ids), _ptr(topk_w), _stream(stream)),
           "moe_route_noalloc")


def moe_permute(cfg, T, topk_ids, x, counts, offsets, sorted_to_expanded, expanded_to_sorted,
                x_perm, x_perm_scale, ws, stream=None):
    _check(lib.moe_permute(ctypes.byref(cfg), T, _ptr(topk_ids), _ptr(x), _ptr(counts),
                           _ptr(offsets), _ptr(sorted_to_expanded), _ptr(expanded_to_sorted),
                           _ptr(x_perm), _ptr(x_perm_scale), _ptr(ws), _ws_bytes(ws),
                           _stream(stream)), "moe_permute")


def moe_grouped_ffn(cfg, T, offsets, x_perm, x_perm_scale, w_gate, w_up, w_down, s_gate, s_up,
                    s_down, y_perm, ws, stream=None):
    _check(lib.moe_grouped_ffn(ctypes.byref(cfg), T, _ptr(offsets), _ptr(x_perm),
                               _ptr(x_perm_scale), _ptr(w_gate), _ptr(w_up), _ptr(w_down),
                               _ptr(s_gate), _ptr(s_up), _ptr(s_down), _ptr(y_perm), _ptr(ws),
                               _ws_bytes(ws), _stream(stream)), "moe_grouped_ffn")


def moe_combine(cfg, T, y_perm, expanded_to_sorted, topk_ids, topk_w, x, shared_out, out,
                stream=None):
    _check(lib.moe_combine(ctypes.byref(cfg), T, _ptr(y_perm), _ptr(expanded_to_sorted),
                           _ptr(topk_ids), _ptr(topk_w), _ptr(x), _ptr(shared_out), _ptr(out),
                           _stream(stream)), "moe_combine")


def moe_layer_forward(cfg, T, x, w_router, bias, w_gate, w_up, w_down, s_gate, s_up, s_down,
                      ws_gate, ws_up, ws_down, out, ws, stream=None):
    _check(lib.moe_layer_forward(ctypes.byref(cfg), T, _ptr(x), _ptr(w_router), _ptr(bias),
                                 _ptr(w_gate), _ptr(w_up), _ptr(w_down), _ptr(s_gate),
                                 _ptr(s_up), _ptr(s_down), _ptr(ws_gate), _ptr(ws_up),
                                 _ptr(ws_down), _ptr(out), _ptr(ws), _ws_bytes(ws),
                                 _stream(stream)), "moe_layer_forward")


def moe_qgemm_s8_workspace_size(n_experts, K, N, R) -> int:
    n = _SZ(0)
    _check(lib.moe_qgemm_s8_workspace_size(n_experts, K, N, R, ctypes.byref(n)),
           "moe_qgemm_s8_workspace_size")
    return n.value


def moe_qgemm_s8(n_experts, K, N, R, offsets, a, w, acc, ws, stream=None):
    """Grouped int8 x int8 -> exact int32 (see include/moe.h)."""
    _check(lib.moe_qgemm_s8(n_experts, K, N, R, _ptr(offsets), _ptr(a), _ptr(w), _ptr(acc),
                            _ptr(ws), _ws_bytes(ws), _stream(stream)), "moe_qgemm_s8")


def moe_check_device_status(ws, stream=None) -> int:
    """Status code (MOE_OK / MOE_ERR_DEVICE_CHECK / MOE_ERR_DEVICE_TIMEOUT); clears it."""
    return lib.moe_check_device_status(_ptr(ws), _stream(stream))


def moe_selftest_wait_timeout(ws, limit_cycles: int, stream=None):
    """Launch a wait that runs out after `limit_cycles` and records a timeout in `ws`."""
    _check(lib.moe_selftest_wait_timeout(_ptr(ws), int(limit_cycles), _stream(stream)),
           "moe_selftest_wait_timeout")


def timing_enable(on: bool = True):
    _check(lib.moe_timing_enable(1 if on else 0), "moe_timing_enable")


def timing_collect() -> dict:
    """{kernel name: (total ms, launches)} since the previous collect (synchronises)."""
    ms = (ctypes.c_float * N_KERNELS)()
    n = (_I * N_KERNELS)()
    _check(lib.moe_timing_collect(ms, n, N_KERNELS), "moe_timing_collect")
    return {KERNELS[i]: (ms[i], n[i]) for i in range(N_KERNELS)}


def launch_counts() -> dict:
    n = (ctypes.c_int64 * N_KERNELS)()
    _check(lib.moe_launch_counts(n, N_KERNELS), "moe_launch_counts")
    return {KERNELS[i]: n[i] for i in range(N_KERNELS)}


def _ws_bytes(ws):
    if ws is None or isinstance(ws, int):
        raise TypeError("pass the workspace as a torch uint8 tensor")
    return ws.numel() * ws.element_size()


def layer_scales(weights: dict):
    """(s_gate, s_up, s_down) as moe_layer_forward takes them: the routed
    experts' per-channel scales, followed (W8A8 with a shared expert) by the
    shared expert's ('s_shared_gate' / '_up' / '_down')."""
    out = []
    for n in ("gate", "up", "down"):
        s = weights.get("s_" + n)
        sh = weights.get("s_shared_" + n)
        if s is not None and sh is not None:
            import torch
            s = torch.cat([s.reshape(-1), sh.reshape(-1)])
        out.append(s)
    return tuple(out)


class MoeLayer:
    """Convenience holder: config + device weights + workspace for a fixed T."""

    def __init__(self, cfg: MoeConfig, T: int, weights: dict, w_router, bias=None,
                 device="cuda"):
        self.cfg, self.T = cfg, T
        self.w = weights
        self.scales = layer_scales(weights)
        self.w_router, self.bias = w_router, bias
        self.ws = workspace(cfg, T, device)

    def forward(self, x, out, stream=None):
        w = self.w
        moe_layer_forward(self.cfg, x.shape[0], x, self.w_router, self.bias, w.get("w_gate"),
                          w.get("w_up"), w.get("w_down"), *self.scales, w.get("shared_gate"),
                          w.get("shared_up"), w.get("shared_down"), out, self.ws, stream)
        return out
