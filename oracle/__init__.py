"""CPU oracle for one MoE FFN layer forward -- TEST INFRASTRUCTURE ONLY.

Only the tests, the package's smoke entry and the benchmark's CPU-baseline leg
may import this package.  The product path (the CUDA library and its binding)
never touches it; the two share no code.  The arithmetic lives in
``moe_oracle.c`` (plain loops, float accumulation, or double in the
``fp64=True`` build); this file only compiles it and marshals numpy arrays.

Parity pins: every function here is pinned by the ``-m "not gpu"`` tests in
``tests/test_oracle_pins.py`` against library routines, closed forms,
invariants and brute force (see that file's docstring for the list).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIBS = {}
_LOCK = threading.Lock()

_C = ctypes
_i64, _i32, _vp = _C.c_int64, _C.c_int32, _C.c_void_p


class _Layer(ctypes.Structure):
    _fields_ = [
        ("hidden", _i32), ("num_experts", _i32), ("top_k", _i32), ("inter", _i32),
        ("shared_inter", _i32), ("wfmt", _i32),
        ("w1", _vp), ("w3", _vp), ("w2", _vp),
        ("s1", _vp), ("s3", _vp), ("s2", _vp),
        ("ws1", _vp), ("ws3", _vp), ("ws2", _vp),
        ("ss1", _vp), ("ss3", _vp), ("ss2", _vp),
        ("shared_gate", _vp),
        ("sb1", _vp), ("sb3", _vp), ("sb2", _vp),
        ("ssb1", _vp), ("ssb3", _vp), ("ssb2", _vp),
    ]

# weight formats of the oracle layer struct
FMT_BF16, FMT_FP8, FMT_NVFP4 = 0, 1, 2


def lib_path(fp64: bool = False) -> str:
    return os.path.join(_BUILD, "libmoe_oracle_f64.so" if fp64 else "libmoe_oracle_f32.so")


def build(force: bool = False) -> None:
    """Compile both oracle builds (float and double accumulation) with gcc."""
    os.makedirs(_BUILD, exist_ok=True)
    for fp64 in (False, True):
        out = lib_path(fp64)
        if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(_SRC):
            continue
        tmp = out + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared", "-std=c11",
               "-fvisibility=hidden", _SRC, "-o", tmp, "-lm"]
        if fp64:
            cmd.insert(1, "-DORACLE_FP64")
        subprocess.run(cmd, check=True)
        os.replace(tmp, out)


def _lib(fp64: bool = False):
    with _LOCK:
        if fp64 not in _LIBS:
            build()
            lib = ctypes.CDLL(lib_path(fp64))
            lib.oracle_e4m3_decode.argtypes = [_vp, _vp, _i64]
            lib.oracle_e4m3_encode.argtypes = [_vp, _vp, _i64]
            lib.oracle_act_quant.argtypes = [_vp, _i64, _vp, _vp, _vp]
            lib.oracle_e2m1_decode.argtypes = [_vp, _vp, _i64]
            lib.oracle_e2m1_encode.argtypes = [_vp, _vp, _i64]
            lib.oracle_nvfp4_quant.argtypes = [_vp, _i64, _vp, _vp, _vp, _vp]
            lib.oracle_router_logits.argtypes = [_vp, _i64, _C.c_int, _vp, _vp, _C.c_int, _vp]
            lib.oracle_topk_softmax.argtypes = [_vp, _i64, _C.c_int, _C.c_int, _vp, _vp, _vp]
            lib.oracle_topk_sigmoid.argtypes = [_vp, _i64, _C.c_int, _C.c_int, _vp, _C.c_int, _C.c_float,
                                                _vp, _vp, _vp]
            lib.oracle_permute.argtypes = [_vp, _i64, _C.c_int, _C.c_int, _vp, _vp, _vp]
            lib.oracle_route_weights.argtypes = [_vp, _i64, _C.c_int, _C.c_int, _vp, _C.c_int, _C.c_int,
                                                 _C.c_float, _vp]
            lib.oracle_residual_rmsnorm.argtypes = [_vp, _i64, _C.c_int, _vp, _vp, _C.c_float, _vp]
            lib.oracle_moe_forward.argtypes = [ctypes.POINTER(_Layer), _vp, _i64, _vp, _i64, _vp, _vp, _vp]
            lib.oracle_moe_forward.restype = _C.c_int
            lib.oracle_set_threads.argtypes = [_C.c_int]
            lib.oracle_set_threads.restype = _C.c_int
            lib.oracle_acc_bits.restype = _C.c_int
            _LIBS[fp64] = lib
        return _LIBS[fp64]


def _np(a, dtype=None):
    """torch tensor (any device) or array -> contiguous numpy array on the host."""
    try:
        import torch
        if isinstance(a, torch.Tensor):
            t = a.detach().cpu().contiguous()
            if t.dtype == torch.bfloat16:
                t = t.view(torch.int16)
                return t.numpy().view(np.uint16)
            a = t.numpy()
    except ImportError:  # pragma: no cover
        pass
    a = np.ascontiguousarray(a)
    if dtype is not None and a.dtype != dtype:
        a = a.astype(dtype)
    return a


def _ptr(a):
    return None if a is None else a.ctypes.data


def set_threads(n: int = 0, fp64: bool = False) -> int:
    """Set the OpenMP thread count (0 keeps the default); returns the count in use."""
    return _lib(fp64).oracle_set_threads(int(n))


def acc_bits(fp64: bool = False) -> int:
    return _lib(fp64).oracle_acc_bits()


def e4m3_decode(codes) -> np.ndarray:
    c = _np(codes, np.uint8)
    out = np.empty(c.shape, np.float32)
    _lib().oracle_e4m3_decode(_ptr(c), _ptr(out), c.size)
    return out


def e4m3_encode(values) -> np.ndarray:
    v = _np(values, np.float32)
    out = np.empty(v.shape, np.uint8)
    _lib().oracle_e4m3_encode(_ptr(v), _ptr(out), v.size)
    return out


def act_quant(values):
    """1x128 block quantisation of a 1-D vector -> (codes, scales, dequantised)."""
    v = _np(values, np.float32).reshape(-1)
    n = v.size
    q = np.empty(n, np.uint8)
    s = np.empty((n + 127) // 128, np.float32)
    d = np.empty(n, np.float32)
    _lib().oracle_act_quant(_ptr(v), n, _ptr(q), _ptr(s), _ptr(d))
    return q, s, d


def e2m1_decode(codes) -> np.ndarray:
    """Values of e2m1 codes (the low 4 bits of each byte)."""
    c = _np(codes, np.uint8)
    out = np.empty(c.shape, np.float32)
    _lib().oracle_e2m1_decode(_ptr(c), _ptr(out), c.size)
    return out


def e2m1_encode(values) -> np.ndarray:
    """e2m1 codes (one per byte) of float values: nearest, ties to even, saturating."""
    v = _np(values, np.float32)
    out = np.empty(v.shape, np.uint8)
    _lib().oracle_e2m1_encode(_ptr(v), _ptr(out), v.size)
    return out


def nvfp4_quant(values):
    """NVFP4 quantisation of each row of a [rows, n] array (n a multiple of 16)
    -> (packed codes uint8 [rows, n/2], e4m3 block-scale codes uint8
    [rows, n/16], row scales float32 [rows], dequantised float32 [rows, n])."""
    v = _np(values, np.float32)
    if v.ndim == 1:
        v = v.reshape(1, -1)
    rows, n = v.shape
    assert n % 16 == 0
    q = np.empty((rows, n // 2), np.uint8)
    sb = np.empty((rows, n // 16), np.uint8)
    g = np.empty(rows, np.float32)
    d = np.empty((rows, n), np.float32)
    lib = _lib()
    for r in range(rows):
        lib.oracle_nvfp4_quant(_ptr(v[r]), n, _ptr(q[r]), _ptr(sb[r]), g[r:].ctypes.data, _ptr(d[r]))
    return q, sb, g, d


def router_logits(x, router_w, router_bias=None, fp64: bool = False) -> np.ndarray:
    xb = _np(x)
    assert xb.dtype == np.uint16, "x must be bf16"
    m, H = xb.shape
    wr = _np(router_w, np.float32)
    E = wr.shape[0]
    b = None if router_bias is None else _np(router_bias, np.float32)
    L = np.empty((m, E), np.float32)
    _lib(fp64).oracle_router_logits(_ptr(xb), m, H, _ptr(wr), _ptr(b), E, _ptr(L))
    return L


def topk_softmax(logits, k: int):
    """-> ids int32 [m,k], weights float32 [m,k], margin float32 [m]."""
    L = _np(logits, np.float32)
    m, E = L.shape
    ids = np.empty((m, k), np.int32)
    w = np.empty((m, k), np.float32)
    margin = np.empty(m, np.float32)
    _lib().oracle_topk_softmax(_ptr(L), m, E, k, _ptr(ids), _ptr(w), _ptr(margin))
    return ids, w, margin


def topk_sigmoid(logits, k: int, bias=None, norm: bool = True, scale: float = 1.0):
    """Sigmoid scores, selection by score + bias -> ids int32 [m,k], weights
    float32 [m,k], margin float32 [m] (in selection-key units)."""
    L = _np(logits, np.float32)
    m, E = L.shape
    b = None if bias is None else _np(bias, np.float32)
    ids = np.empty((m, k), np.int32)
    w = np.empty((m, k), np.float32)
    margin = np.empty(m, np.float32)
    _lib().oracle_topk_sigmoid(_ptr(L), m, E, k, _ptr(b), int(bool(norm)), float(scale), _ptr(ids), _ptr(w),
                               _ptr(margin))
    return ids, w, margin


def route_weights(shape, logits, ids):
    """Routing weights float32 [m,k] for a given selection ids [m,k] (the
    forced-ids mode): the layer's scoring applied to those ids' logits."""
    L = _np(logits, np.float32)
    m, E = L.shape
    a = _np(ids, np.int32)
    k = a.shape[1]
    assert a.shape[0] == m and a.min() >= 0 and a.max() < E
    w = np.empty((m, k), np.float32)
    sigmoid = getattr(shape, "scoring", "softmax") == "sigmoid"
    _lib().oracle_route_weights(_ptr(L), m, E, k, _ptr(a), int(sigmoid),
                                int(bool(getattr(shape, "norm_topk_prob", True))),
                                float(getattr(shape, "routed_scaling", 1.0)), _ptr(w))
    return w


def permute(ids, num_experts: int):
    """-> expert_offsets int32 [E+1], sorted_pair int32 [P], slot_of_pair int32 [P]."""
    a = _np(ids, np.int32)
    m, k = a.shape
    P = m * k
    off = np.empty(num_experts + 1, np.int32)
    sp = np.empty(P, np.int32)
    sl = np.empty(P, np.int32)
    _lib().oracle_permute(_ptr(a), m, k, num_experts, _ptr(off), _ptr(sp), _ptr(sl))
    return off, sp, sl


def _layer_struct(shape, layer, keep):
    def arr(name, dtype):
        t = layer.get(name)
        if t is None:
            return None
        a = _np(t, dtype) if dtype is not None else _np(t)
        keep.append(a)
        return a

    nvfp4 = bool(getattr(shape, "nvfp4", False))
    wdt = np.uint8 if (shape.fp8 or nvfp4) else None
    s = _Layer()
    s.hidden, s.num_experts, s.top_k = shape.hidden, shape.num_experts, shape.top_k
    s.inter, s.shared_inter = shape.inter, shape.shared_inter
    s.wfmt = FMT_NVFP4 if nvfp4 else (FMT_FP8 if shape.fp8 else FMT_BF16)
    for name in ("w1", "w3", "w2", "ws1", "ws3", "ws2"):
        a = arr(name, wdt)
        setattr(s, name, _ptr(a))
    for name in ("s1", "s3", "s2", "ss1", "ss3", "ss2"):
        a = arr(name, np.float32)
        setattr(s, name, _ptr(a))
    for name in ("sb1", "sb3", "sb2", "ssb1", "ssb3", "ssb2"):
        a = arr(name, np.uint8) if nvfp4 else None
        setattr(s, name, _ptr(a))
    s.shared_gate = _ptr(arr("shared_gate", np.float32)) if getattr(shape, "shared_gate", False) else None
    return s


def moe_forward(shape, layer, x, ids, w, rows=None, fp64: bool = False) -> np.ndarray:
    """Layer output (float32 [len(rows) or m, H]) for a given routing (ids, w)."""
    keep = []
    st = _layer_struct(shape, layer, keep)
    xb = _np(x)
    assert xb.dtype == np.uint16, "x must be bf16"
    m = xb.shape[0]
    ids_a = _np(ids, np.int32)
    w_a = _np(w, np.float32)
    assert ids_a.shape == (m, shape.top_k) and w_a.shape == (m, shape.top_k)
    r = None if rows is None else _np(rows, np.int64).reshape(-1)
    n = m if r is None else r.size
    out = np.empty((n, shape.hidden), np.float32)
    rc = _lib(fp64).oracle_moe_forward(ctypes.byref(st), _ptr(xb), m, _ptr(r), n,
                                       _ptr(ids_a), _ptr(w_a), _ptr(out))
    if rc != 0:
        raise ValueError("oracle_moe_forward: token row or expert id out of range")
    return out


def residual_rmsnorm(moe_out, residual, weight, eps: float, fp64: bool = False):
    """Layer tail: -> (new residual bf16 as uint16 [m,H], norm_out uint16 [m,H])."""
    o = _np(moe_out, np.float32)
    r = _np(residual).copy()
    assert r.dtype == np.uint16, "residual must be bf16"
    wv = _np(weight, np.float32)
    m, H = o.shape
    out = np.empty((m, H), np.uint16)
    _lib(fp64).oracle_residual_rmsnorm(_ptr(o), m, H, _ptr(r), _ptr(wv), float(eps), _ptr(out))
    return r, out


def route(shape, layer, x, fp64: bool = False):
    """Router logits + top-k for all tokens -> (logits, ids, w, margin).

    softmax scoring: the bias (if any) is part of the logits.  sigmoid scoring:
    the logits carry no bias; it only selects (oracle_topk_sigmoid)."""
    if getattr(shape, "scoring", "softmax") == "sigmoid":
        L = router_logits(x, layer["router_w"], None, fp64=fp64)
        ids, w, margin = topk_sigmoid(L, shape.top_k, layer.get("router_bias"), shape.norm_topk_prob,
                                      shape.routed_scaling)
        return L, ids, w, margin
    L = router_logits(x, layer["router_w"], layer.get("router_bias"), fp64=fp64)
    ids, w, margin = topk_softmax(L, shape.top_k)
    return L, ids, w, margin


def reference(shape, layer, x, rows=None, fp64: bool = False):
    """The whole layer: route every token, then the expert sum for `rows`."""
    L, ids, w, margin = route(shape, layer, x, fp64=fp64)
    out = moe_forward(shape, layer, x, ids, w, rows=rows, fp64=fp64)
    return {"logits": L, "ids": ids, "w": w, "margin": margin, "out": out}
