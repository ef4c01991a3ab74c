"""ctypes binding of the C ABI in include/moe_gb300.h (argument marshalling only).

Every function keeps the C name and argument order.  Array arguments accept a
torch tensor (its data_ptr() is passed), a raw integer device address, or
None for a nullable pointer; `stream` defaults to torch's current CUDA stream.
A non-MOE_OK status raises MoeError with the library's own message.  Nothing
here computes any part of the layer: if the CUDA library cannot be loaded,
every call fails loudly.
"""
from __future__ import annotations

import ctypes
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
HEADER = os.path.join(os.path.dirname(HERE), "include", "moe_gb300.h")

(MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_WORKSPACE, MOE_ERR_CUDA, MOE_ERR_DEVICE_CHECK,
 MOE_ERR_TIMEOUT) = range(7)
MOE_F32, MOE_BF16, MOE_Q8_0, MOE_Q4_K, MOE_Q8_0_R, MOE_Q5_K, MOE_Q6_K, MOE_Q3_K, MOE_MXFP4 = range(9)
MOE_ROUTE_SOFTMAX, MOE_ROUTE_SIGMOID_GROUP = range(2)

STATUS_NAMES = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED", 3: "MOE_ERR_WORKSPACE",
                4: "MOE_ERR_CUDA", 5: "MOE_ERR_DEVICE_CHECK", 6: "MOE_ERR_TIMEOUT"}


class MoeError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


class moe_route_cfg(ctypes.Structure):
    _fields_ = [("mode", ctypes.c_int), ("n_experts", ctypes.c_int), ("top_k", ctypes.c_int),
                ("n_groups", ctypes.c_int), ("topk_groups", ctypes.c_int), ("routed_scale", ctypes.c_float),
                ("renormalize", ctypes.c_int)]


class moe_qmat(ctypes.Structure):
    _fields_ = [("qtype", ctypes.c_int), ("data", ctypes.c_void_p), ("rows", ctypes.c_int64),
                ("cols", ctypes.c_int64), ("expert_stride_bytes", ctypes.c_int64)]


class moe_layer_desc(ctypes.Structure):
    _fields_ = [("route", moe_route_cfg), ("hidden", ctypes.c_int), ("intermediate", ctypes.c_int),
                ("x_type", ctypes.c_int), ("W_router", ctypes.c_void_p), ("bias", ctypes.c_void_p),
                ("gate", moe_qmat), ("up", moe_qmat), ("down", moe_qmat),
                ("shared_intermediate", ctypes.c_int), ("s_gate", moe_qmat), ("s_up", moe_qmat),
                ("s_down", moe_qmat), ("accumulate", ctypes.c_int), ("tc_min_tokens", ctypes.c_int),
                ("decode_chain_off", ctypes.c_int), ("norm_gamma", ctypes.c_void_p), ("norm_eps", ctypes.c_float),
                ("expert_counts", ctypes.c_void_p)]


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return os.path.join(HERE, "_build", "libmoe_gb300.so")


def load(build_if_missing: bool = True):
    """The loaded CUDA library (built in-tree on first use when missing)."""
    global _lib
    with _lock:
        if _lib is None:
            path = library_path()
            if build_if_missing:
                from . import build as _build
                path = _build.build()
            if not os.path.exists(path):
                raise OSError(f"the CUDA library {path} is missing; run __graft_entry__.build()")
            _lib = _declare(ctypes.CDLL(path))
    return _lib


def _declare(lib):
    P, I, I64, S, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float
    PS = ctypes.POINTER(ctypes.c_size_t)
    sig = {
        "moe_route": [ctypes.POINTER(moe_route_cfg), P, I, I, I, P, P, P, P, P, P, P],
        "moe_permute_workspace_size": [I, I, I, PS],
        "moe_permute": [P, I, I, I, P, P, P, P, S, P],
        "moe_permute_noalloc": [P, I, I, I, P, P, P, P],
        "moe_expert_counts_add": [P, I, P, P],
        "moe_expert_ffn_workspace_size": [I, I, I, I, I, PS],
        "moe_expert_ffn": [ctypes.POINTER(moe_qmat)] * 3 + [I, P, I, I, I, I, P, P, I, P, P, S, P],
        "moe_expert_gateup": [ctypes.POINTER(moe_qmat)] * 2 + [I, P, I, I, I, I, P, P, I, P, P],
        "moe_expert_down": [ctypes.POINTER(moe_qmat), I, P, I, I, I, P, P, I, P, P],
        "moe_combine": [P, P, P, I, I, I, P, I, P, P],
        "moe_rmsnorm_bf16": [P, P, I, I, F, P, P],
        "moe_layer_plan_create": [ctypes.POINTER(moe_layer_desc), ctypes.POINTER(P)],
        "moe_layer_plan_destroy": [P],
        "moe_layer_workspace_size": [P, I, PS],
        "moe_layer_path": [P, I, ctypes.POINTER(ctypes.c_int)],
        "moe_layer": [P, P, I, P, P, S, P],
        "moe_layer_timed": [P, P, I, P, P, S, P, P, P],
        "moe_layer_debug_views": [P, I, P, ctypes.POINTER(P), ctypes.POINTER(P), ctypes.POINTER(P)],
        "moe_read_device_status": [P, I, P, ctypes.POINTER(ctypes.c_int32), P],
        "moe_permute_read_device_status": [I, I, I, P, ctypes.POINTER(ctypes.c_int32), P],
        "moe_debug_set_waits": [ctypes.c_uint64, I],
        "moe_debug_set_stamps": [P, S],
        "moe_weights_prepare_size": [ctypes.POINTER(moe_qmat), I, PS],
        "moe_weights_prepare": [ctypes.POINTER(moe_qmat), I, P, S, P],
    }
    for name, args in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = ctypes.c_int
    lib.moe_last_error.argtypes = []
    lib.moe_last_error.restype = ctypes.c_char_p
    lib.moe_version.argtypes = []
    lib.moe_version.restype = ctypes.c_char_p
    del I64
    return lib


def _p(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int):
    if status != MOE_OK:
        msg = load().moe_last_error().decode(errors="replace")
        raise MoeError(status, msg)


def qmat(qtype: int, data, rows: int, cols: int, expert_stride_bytes: int = 0) -> moe_qmat:
    return moe_qmat(qtype, _p(data), rows, cols, expert_stride_bytes)


def route_cfg(mode: int, n_experts: int, top_k: int, n_groups: int = 1, topk_groups: int = 1,
              routed_scale: float = 1.0, renormalize: bool = True) -> moe_route_cfg:
    return moe_route_cfg(mode, n_experts, top_k, n_groups, topk_groups, routed_scale, int(renormalize))


# ------------------------------------------------------------------ calls (C names)

def moe_route(cfg, x, x_type, T, H, W_router, bias, logits_in, logits_out, topk_ids, topk_w, stream=None):
    _check(load().moe_route(ctypes.byref(cfg), _p(x), x_type, T, H, _p(W_router), _p(bias), _p(logits_in),
                            _p(logits_out), _p(topk_ids), _p(topk_w), _stream(stream)))


def moe_permute_workspace_size(T, k, E) -> int:
    n = ctypes.c_size_t(0)
    _check(load().moe_permute_workspace_size(T, k, E, ctypes.byref(n)))
    return n.value


def moe_permute(topk_ids, T, k, E, sorted_pairs, offsets, pair_pos, workspace, ws_bytes, stream=None):
    _check(load().moe_permute(_p(topk_ids), T, k, E, _p(sorted_pairs), _p(offsets), _p(pair_pos),
                              _p(workspace), ws_bytes, _stream(stream)))


def moe_expert_counts_add(offsets, E, counts, stream=None):
    """counts[e] += offsets[e+1] - offsets[e] (counts: int64 [E] on the device, a running histogram)."""
    _check(load().moe_expert_counts_add(_p(offsets), E, _p(counts), _stream(stream)))


def moe_permute_noalloc(topk_ids, T, k, E, sorted_pairs, offsets, pair_pos, stream=None):
    """moe_permute without a workspace (fixed library scratch; T*k <= 65536)."""
    _check(load().moe_permute_noalloc(_p(topk_ids), T, k, E, _p(sorted_pairs), _p(offsets), _p(pair_pos),
                                      _stream(stream)))


def moe_expert_ffn_workspace_size(T, k, E, H, I) -> int:
    n = ctypes.c_size_t(0)
    _check(load().moe_expert_ffn_workspace_size(T, k, E, H, I, ctypes.byref(n)))
    return n.value


def moe_expert_ffn(gate, up, down, E, x, x_type, T, H, I, sorted_pairs, offsets, k, y_pairs, workspace,
                   ws_bytes, stream=None):
    _check(load().moe_expert_ffn(ctypes.byref(gate), ctypes.byref(up), ctypes.byref(down), E, _p(x), x_type,
                                 T, H, I, _p(sorted_pairs), _p(offsets), k, _p(y_pairs), _p(workspace),
                                 ws_bytes, _stream(stream)))


def moe_expert_gateup(gate, up, E, x, x_type, T, H, I, sorted_pairs, offsets, k, h, stream=None):
    _check(load().moe_expert_gateup(ctypes.byref(gate), ctypes.byref(up), E, _p(x), x_type, T, H, I,
                                    _p(sorted_pairs), _p(offsets), k, _p(h), _stream(stream)))


def moe_expert_down(down, E, h, T, H, I, sorted_pairs, offsets, k, y_pairs, stream=None):
    _check(load().moe_expert_down(ctypes.byref(down), E, _p(h), T, H, I, _p(sorted_pairs), _p(offsets), k,
                                  _p(y_pairs), _stream(stream)))


def moe_combine(y_pairs, topk_w, pair_pos, T, k, H, shared_out, accumulate, out, stream=None):
    _check(load().moe_combine(_p(y_pairs), _p(topk_w), _p(pair_pos), T, k, H, _p(shared_out),
                              int(accumulate), _p(out), _stream(stream)))


def moe_rmsnorm_bf16(x, gamma, T, H, eps, u, stream=None):
    _check(load().moe_rmsnorm_bf16(_p(x), _p(gamma), T, H, float(eps), _p(u), _stream(stream)))


def moe_layer_plan_create(desc: moe_layer_desc) -> int:
    h = ctypes.c_void_p(0)
    _check(load().moe_layer_plan_create(ctypes.byref(desc), ctypes.byref(h)))
    return h.value


def moe_layer_plan_destroy(plan: int):
    _check(load().moe_layer_plan_destroy(plan))


def moe_layer_workspace_size(plan: int, T: int) -> int:
    n = ctypes.c_size_t(0)
    _check(load().moe_layer_workspace_size(plan, T, ctypes.byref(n)))
    return n.value


MOE_PATH_GEMV, MOE_PATH_DECODE_CHAIN, MOE_PATH_TENSOR = 0, 1, 2
PATH_NAMES = {MOE_PATH_GEMV: "gemv", MOE_PATH_DECODE_CHAIN: "decode_chain", MOE_PATH_TENSOR: "tensor"}


def moe_layer_path(plan, T):
    """Which kernels moe_layer runs for T tokens: one of the MOE_PATH_* values."""
    v = ctypes.c_int(-1)
    _check(load().moe_layer_path(plan, T, ctypes.byref(v)))
    return v.value


def moe_layer(plan, x, T, out, workspace, ws_bytes, stream=None):
    _check(load().moe_layer(plan, _p(x), T, _p(out), _p(workspace), ws_bytes, _stream(stream)))


def moe_layer_timed(plan, x, T, out, workspace, ws_bytes, stream=None, ev_before=None, ev_after=None):
    """moe_layer recording torch.cuda.Event objects around the routed gate/up kernel."""
    eb = ev_before.cuda_event if ev_before is not None else None
    ea = ev_after.cuda_event if ev_after is not None else None
    _check(load().moe_layer_timed(plan, _p(x), T, _p(out), _p(workspace), ws_bytes, _stream(stream), eb, ea))


def moe_layer_debug_views(plan, T, workspace):
    a, b, c = ctypes.c_void_p(0), ctypes.c_void_p(0), ctypes.c_void_p(0)
    _check(load().moe_layer_debug_views(plan, T, _p(workspace), ctypes.byref(a), ctypes.byref(b),
                                        ctypes.byref(c)))
    return a.value, b.value, c.value


def moe_read_device_status(plan, T, workspace, stream=None) -> int:
    code = ctypes.c_int32(0)
    _check(load().moe_read_device_status(plan, T, _p(workspace), ctypes.byref(code), _stream(stream)))
    return code.value


def moe_permute_read_device_status(T, k, E, workspace, stream=None) -> int:
    code = ctypes.c_int32(0)
    _check(load().moe_permute_read_device_status(T, k, E, _p(workspace), ctypes.byref(code), _stream(stream)))
    return code.value


def moe_weights_prepare_size(m: moe_qmat, n_experts: int) -> int:
    n = ctypes.c_size_t(0)
    _check(load().moe_weights_prepare_size(ctypes.byref(m), n_experts, ctypes.byref(n)))
    return n.value


def moe_weights_prepare(m: moe_qmat, n_experts: int, dst, dst_bytes: int, stream=None) -> moe_qmat:
    """Repacks m (Q8_0) into dst; returns the moe_qmat that describes the prepared tensor."""
    out = moe_qmat(m.qtype, m.data, m.rows, m.cols, m.expert_stride_bytes)
    _check(load().moe_weights_prepare(ctypes.byref(out), n_experts, _p(dst), dst_bytes, _stream(stream)))
    return out


def moe_debug_set_stamps(buf, nbytes: int):
    _check(load().moe_debug_set_stamps(_p(buf), int(nbytes)))


def moe_debug_set_waits(limit_ns: int, stall: int):
    _check(load().moe_debug_set_waits(int(limit_ns), int(stall)))


def moe_last_error() -> str:
    return load().moe_last_error().decode(errors="replace")


def moe_version() -> str:
    return load().moe_version().decode()
