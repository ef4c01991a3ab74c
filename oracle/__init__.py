"""fp64 CPU oracle for the routed-expert MoE layer -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product (the CUDA library and its
binding) never does, and the two share no code.

The arithmetic lives in ``oracle.c`` (plain C, fp64, one obvious loop per
definition); this module compiles it with gcc and wraps it with ctypes and
numpy.  Parity status of every function is listed in the header of
``oracle.c``; nothing here is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

Q8_0 = 2
Q4_K = 3
Q5_K = 4
Q6_K = 5
Q3_K = 6
MXFP4 = 7
ROUTE_SOFTMAX = 0
ROUTE_SIGMOID_GROUP = 1


def build(force: bool = False, src: str | None = None, out: str | None = None) -> str:
    """Compile oracle.c (or `src`) into a shared library; returns its path."""
    src = src or _SRC
    out = out or _LIB_PATH
    os.makedirs(os.path.dirname(out), exist_ok=True)
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-fno-fast-math",
           "-ffp-contract=off", src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


class _Layer(ctypes.Structure):
    _fields_ = [
        ("mode", ctypes.c_int), ("E", ctypes.c_int), ("k", ctypes.c_int),
        ("n_groups", ctypes.c_int), ("topk_groups", ctypes.c_int), ("renormalize", ctypes.c_int),
        ("scale", ctypes.c_double), ("H", ctypes.c_int), ("I", ctypes.c_int),
        ("qtype", ctypes.c_int),
        ("gate", ctypes.c_void_p), ("up", ctypes.c_void_p), ("down", ctypes.c_void_p),
        ("expert_stride_gu", ctypes.c_int64), ("expert_stride_d", ctypes.c_int64),
        ("Wr", ctypes.c_void_p), ("bias", ctypes.c_void_p),
        ("shared_qtype", ctypes.c_int), ("I_s", ctypes.c_int),
        ("s_gate", ctypes.c_void_p), ("s_up", ctypes.c_void_p), ("s_down", ctypes.c_void_p),
        ("qtype_down", ctypes.c_int),
    ]


def load(path: str | None = None):
    """Load (building if needed) the oracle library.  `path` loads a variant."""
    global _lib
    if path is not None:
        return _declare(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            _lib = _declare(ctypes.CDLL(build()))
    return _lib


def _declare(lib):
    P, I64, I32, D = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_double
    lib.oracle_half_to_double.argtypes = [ctypes.c_uint16]
    lib.oracle_half_to_double.restype = D
    lib.oracle_e2m1_to_double.argtypes = [I32]
    lib.oracle_e2m1_to_double.restype = D
    lib.oracle_dequant_matrix.argtypes = [I32, P, I64, I64, P]
    lib.oracle_dequant_matrix.restype = I32
    lib.oracle_router_logits.argtypes = [P, I32, I32, P, I32, P]
    lib.oracle_router_logits.restype = None
    lib.oracle_route.argtypes = [I32, P, P, I32, I32, I32, I32, I32, I32, D, P, P, P]
    lib.oracle_route.restype = I32
    lib.oracle_permute.argtypes = [P, I32, I32, I32, P, P, P]
    lib.oracle_permute.restype = I32
    lib.oracle_expert_counts.argtypes = [P, I64, I32, P]
    lib.oracle_expert_counts.restype = I32
    lib.oracle_expert_ffn.argtypes = [I32, P, P, P, I32, I32, P, P, P]
    lib.oracle_expert_ffn.restype = I32
    lib.oracle_expert_ffn_mixed.argtypes = [I32, I32, P, P, P, I32, I32, P, P, P]
    lib.oracle_expert_ffn_mixed.restype = I32
    lib.oracle_moe_layer.argtypes = [ctypes.POINTER(_Layer), P, I32, P, P, P, P, P, P, I32]
    lib.oracle_moe_layer.restype = I32
    lib.oracle_rmsnorm.argtypes = [P, I32, I32, P, D, P]
    lib.oracle_rmsnorm.restype = None
    lib.oracle_round_bf16.argtypes = [D]
    lib.oracle_round_bf16.restype = D
    lib.oracle_moe_stack.argtypes = [ctypes.POINTER(_Layer), P, I32, D, P, I32, P, P, I32]
    lib.oracle_moe_stack.restype = I32
    lib.oracle_max_threads.argtypes = []
    lib.oracle_max_threads.restype = I32
    return lib


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _u8(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.uint8))


_BLOCK = {Q8_0: (32, 34), Q4_K: (256, 144), Q5_K: (256, 176), Q6_K: (256, 210), Q3_K: (256, 110),
          MXFP4: (32, 17)}


def row_bytes(qtype: int, K: int) -> int:
    weights, nbytes = _BLOCK[qtype]
    return K // weights * nbytes


# --------------------------------------------------------------------------- wrappers

def half_to_double(bits: int, lib=None) -> float:
    return (lib or load()).oracle_half_to_double(int(bits))


def e2m1_to_double(nibble: int, lib=None) -> float:
    return (lib or load()).oracle_e2m1_to_double(int(nibble))


def dequant(qtype: int, data, rows: int, K: int, lib=None) -> np.ndarray:
    data = _u8(data)
    assert data.size >= rows * row_bytes(qtype, K)
    out = np.empty((rows, K), dtype=np.float64)
    rc = (lib or load()).oracle_dequant_matrix(qtype, _ptr(data), rows, K, _ptr(out))
    assert rc == 0
    return out


def router_logits(x, Wr, lib=None) -> np.ndarray:
    x = _f64(x)
    Wr = np.ascontiguousarray(Wr, dtype=np.float32)
    T, H = x.shape
    E = Wr.shape[0]
    out = np.empty((T, E), dtype=np.float64)
    (lib or load()).oracle_router_logits(_ptr(x), T, H, _ptr(Wr), E, _ptr(out))
    return out


def route(mode: int, logits, k: int, bias=None, n_groups: int = 1, topk_groups: int = 1,
          renormalize: bool = True, scale: float = 1.0, lib=None):
    """Returns (ids [T,k] int32 ascending, w [T,k] f64, gaps [T,2] f64)."""
    logits = _f64(logits)
    T, E = logits.shape
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    ids = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float64)
    gaps = np.empty((T, 2), dtype=np.float64)
    rc = (lib or load()).oracle_route(mode, _ptr(logits), _ptr(b), T, E, k, n_groups, topk_groups,
                                      int(renormalize), float(scale), _ptr(ids), _ptr(w), _ptr(gaps))
    if rc != 0:
        raise ValueError("oracle_route rejected the arguments")
    return ids, w, gaps


def permute(ids, E: int, lib=None):
    """Returns (sorted_pairs [P], offsets [E+1], pair_pos [P]) as int32."""
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    T, k = ids.shape
    P = T * k
    sp = np.empty(P, dtype=np.int32)
    off = np.empty(E + 1, dtype=np.int32)
    pp = np.empty(P, dtype=np.int32)
    rc = (lib or load()).oracle_permute(_ptr(ids), T, k, E, _ptr(sp), _ptr(off), _ptr(pp))
    if rc != 0:
        raise ValueError("oracle_permute: expert id out of range")
    return sp, off, pp


def expert_counts(ids, E: int, counts=None, lib=None) -> np.ndarray:
    """The running routing histogram: counts (uint64 [E], zeros when None) plus, for each
    expert, the number of pairs of ids routed to it.  Returns the updated counts."""
    ids = np.ascontiguousarray(ids, dtype=np.int32).reshape(-1)
    out = np.zeros(E, dtype=np.uint64) if counts is None else np.array(counts, dtype=np.uint64, copy=True)
    if out.shape != (E,):
        raise ValueError("counts must have E entries")
    rc = (lib or load()).oracle_expert_counts(_ptr(ids), ids.size, E, _ptr(out))
    if rc != 0:
        raise ValueError("oracle_expert_counts: expert id out of range")
    return out


def expert_ffn(qtype: int, gate, up, down, H: int, I: int, x, lib=None, qtype_down: int | None = None):
    """One SwiGLU expert on one token; returns (y [H], h [I]).  qtype_down (default: qtype)
    is the type of the down matrix when it differs from gate and up."""
    gate, up, down = _u8(gate), _u8(up), _u8(down)
    x = _f64(x)
    y = np.empty(H, dtype=np.float64)
    h = np.empty(I, dtype=np.float64)
    lib = lib or load()
    if qtype_down is None:
        rc = lib.oracle_expert_ffn(qtype, _ptr(gate), _ptr(up), _ptr(down), H, I, _ptr(x), _ptr(y), _ptr(h))
    else:
        rc = lib.oracle_expert_ffn_mixed(qtype, qtype_down, _ptr(gate), _ptr(up), _ptr(down), H, I,
                                         _ptr(x), _ptr(y), _ptr(h))
    assert rc == 0
    return y, h


class LayerSpec:
    """Host-side description of one MoE layer's stored tensors (numpy arrays).

    gate/up: uint8 [E, I, row_bytes(H)] in qtype; down: uint8 [E, H, row_bytes(I)] in
    qtype_down (default: qtype); Wr fp32 [E, H]; bias fp32 [E] or None; shared_* uint8 or None.
    """

    def __init__(self, *, mode, E, k, H, I, qtype, gate, up, down, Wr, bias=None,
                 n_groups=1, topk_groups=1, renormalize=True, scale=1.0,
                 shared_qtype=Q8_0, I_s=0, s_gate=None, s_up=None, s_down=None, qtype_down=None):
        self.mode, self.E, self.k, self.H, self.I, self.qtype = mode, E, k, H, I, qtype
        self.qtype_down = qtype if qtype_down is None else qtype_down
        self.gate, self.up, self.down = _u8(gate), _u8(up), _u8(down)
        self.Wr = np.ascontiguousarray(Wr, dtype=np.float32)
        self.bias = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
        self.n_groups, self.topk_groups = n_groups, topk_groups
        self.renormalize, self.scale = renormalize, scale
        self.shared_qtype, self.I_s = shared_qtype, I_s
        self.s_gate = None if s_gate is None else _u8(s_gate)
        self.s_up = None if s_up is None else _u8(s_up)
        self.s_down = None if s_down is None else _u8(s_down)

    def c_struct(self) -> _Layer:
        return _Layer(
            mode=self.mode, E=self.E, k=self.k, n_groups=self.n_groups,
            topk_groups=self.topk_groups, renormalize=int(self.renormalize),
            scale=float(self.scale), H=self.H, I=self.I, qtype=self.qtype,
            gate=_ptr(self.gate), up=_ptr(self.up), down=_ptr(self.down),
            expert_stride_gu=self.I * row_bytes(self.qtype, self.H),
            expert_stride_d=self.H * row_bytes(self.qtype_down, self.I),
            Wr=_ptr(self.Wr), bias=_ptr(self.bias),
            shared_qtype=self.shared_qtype, I_s=self.I_s,
            s_gate=_ptr(self.s_gate), s_up=_ptr(self.s_up), s_down=_ptr(self.s_down),
            qtype_down=self.qtype_down,
        )


def moe_layer(spec: LayerSpec, x, logits=None, n_threads: int = 1, want_y: bool = False, lib=None):
    """Returns dict(out [T,H], ids [T,k], w [T,k], logits [T,E], y [T*k,H] if want_y)."""
    x = _f64(x)
    T, H = x.shape
    assert H == spec.H
    E, k = spec.E, spec.k
    out = np.empty((T, H), dtype=np.float64)
    ids = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float64)
    lg = np.empty((T, E), dtype=np.float64)
    y = np.empty((T * k, H), dtype=np.float64) if want_y else None
    lin = None if logits is None else _f64(logits)
    st = spec.c_struct()
    rc = (lib or load()).oracle_moe_layer(ctypes.byref(st), _ptr(x), T, _ptr(lin), _ptr(out),
                                          _ptr(ids), _ptr(w), _ptr(lg), _ptr(y), int(n_threads))
    if rc != 0:
        raise ValueError("oracle_moe_layer rejected the arguments")
    res = dict(out=out, ids=ids, w=w, logits=lg)
    if want_y:
        res["y"] = y
    return res


def rmsnorm(x, gamma, eps: float = 1e-6, lib=None) -> np.ndarray:
    x = _f64(x)
    T, H = x.shape
    g = np.ascontiguousarray(gamma, dtype=np.float32)
    u = np.empty_like(x)
    (lib or load()).oracle_rmsnorm(_ptr(x), T, H, _ptr(g), float(eps), _ptr(u))
    return u


def round_bf16(v: float, lib=None) -> float:
    return (lib or load()).oracle_round_bf16(float(v))


def moe_stack(specs, gammas, x, eps: float = 1e-6, n_threads: int = 1, lib=None):
    """x_{l+1} = x_l + MoE_l(bf16(RMSNorm_l(x_l))).  Returns (x_out, ids [L,T,k], gaps [L,T,2])."""
    x = _f64(x).copy()
    T, H = x.shape
    n = len(specs)
    structs = (_Layer * n)(*[s.c_struct() for s in specs])
    g_arrays = [np.ascontiguousarray(g, dtype=np.float32) for g in gammas]
    g_ptrs = (ctypes.c_void_p * n)(*[a.ctypes.data for a in g_arrays])
    k = specs[0].k
    ids = np.empty((n, T, k), dtype=np.int32)
    gaps = np.empty((n, T, 2), dtype=np.float64)
    rc = (lib or load()).oracle_moe_stack(structs, ctypes.cast(g_ptrs, ctypes.c_void_p), n, float(eps),
                                          _ptr(x), T, _ptr(ids), _ptr(gaps), int(n_threads))
    if rc != 0:
        raise ValueError("oracle_moe_stack failed")
    return x, ids, gaps


def max_threads(lib=None) -> int:
    return (lib or load()).oracle_max_threads()
