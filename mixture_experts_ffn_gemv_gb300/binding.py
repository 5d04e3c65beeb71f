"""ctypes binding of libmoe_ffn_gb300.so (argument marshalling only).

Every entry point keeps the C-ABI's name (moe_route, moe_permute,
moe_experts, moe_forward); the tensors' data pointers and the current torch
CUDA stream are passed straight through.  No computation happens here, and a
missing library is an error: there is no CPU or torch fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from .build import LIB, build_library, up_to_date

MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_WORKSPACE, MOE_ERR_CUDA, MOE_ERR_DEVICE = range(6)
MOE_WEIGHTS_BF16, MOE_WEIGHTS_FP8_E4M3_B128, MOE_WEIGHTS_NVFP4 = 0, 1, 2
MOE_SCORING_SOFTMAX, MOE_SCORING_SIGMOID = 0, 1
MOE_ARM_AUTO, MOE_ARM_GEMV, MOE_ARM_GEMM = 0, 1, 2
ARMS = {"auto": MOE_ARM_AUTO, "gemv": MOE_ARM_GEMV, "gemm": MOE_ARM_GEMM}

EXPORTED = (
    "moe_layer_create", "moe_layer_destroy", "moe_workspace_size", "moe_select_arm", "moe_route",
    "moe_permute", "moe_permute_noalloc", "moe_experts", "moe_shared_expert_add", "moe_forward",
    "moe_forward_residual_rmsnorm",
    "moe_act_quant_fp8", "moe_act_quant_nvfp4", "moe_act_quant_nvfp4_f32", "moe_device_status", "moe_router_planes_size",
    "moe_router_prepare", "moe_layer_set_wait_limit",
    "moe_layer_stall_test",
    "moe_last_launch_count", "moe_kernel_timing_enable", "moe_kernel_timing_read", "moe_kernel_count",
    "moe_kernel_name", "moe_status_string",
)

_vp, _i64, _i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32


class MoeConfig(ctypes.Structure):
    _fields_ = [("hidden", _i32), ("num_experts", _i32), ("top_k", _i32), ("inter", _i32),
                ("shared_inter", _i32), ("weights", _i32), ("scoring", _i32), ("norm_topk_prob", _i32),
                ("routed_scaling_factor", ctypes.c_float), ("expert_begin", _i32), ("expert_end", _i32)]


class MoeExpertWeights(ctypes.Structure):
    _fields_ = [("w1", _vp), ("w3", _vp), ("w2", _vp), ("s1", _vp), ("s3", _vp), ("s2", _vp), ("gate", _vp),
                ("sb1", _vp), ("sb3", _vp), ("sb2", _vp)]


class MoeError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


_lib = None
_lock = threading.Lock()


def load_library(path: str | None = None, build: bool = True):
    """Load (building first if stale) the CUDA library; raises if unavailable."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or LIB
        if build and path is None and not up_to_date():
            build_library()
        if not os.path.exists(p):
            raise RuntimeError(f"CUDA library {p} is missing; build it with build_library()")
        lib = ctypes.CDLL(p)
        lib.moe_layer_create.argtypes = [ctypes.POINTER(MoeConfig), ctypes.POINTER(MoeExpertWeights),
                                         ctypes.POINTER(MoeExpertWeights), ctypes.POINTER(_vp)]
        lib.moe_layer_destroy.argtypes = [_vp]
        lib.moe_workspace_size.argtypes = [_vp, _i64, ctypes.POINTER(ctypes.c_size_t)]
        lib.moe_select_arm.argtypes = [_vp, _i64]
        lib.moe_route.argtypes = [_vp, _vp, _i64, _vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_size_t, _vp]
        lib.moe_permute.argtypes = [_vp, _vp, _i64, _vp, _vp, _vp, _vp, ctypes.c_size_t, _vp]
        lib.moe_permute_noalloc.argtypes = [_vp, _i64, _i32, _i32, _vp, _vp, _vp, _vp]
        lib.moe_experts.argtypes = [_vp, _vp, _i64, _vp, _vp, _vp, ctypes.c_int, _vp, ctypes.c_size_t, _vp]
        lib.moe_shared_expert_add.argtypes = [_vp, _vp, _i64, _vp, ctypes.c_int, _vp, ctypes.c_size_t, _vp]
        lib.moe_forward.argtypes = [_vp, _vp, _i64, _vp, _vp, _vp, _vp, _vp, ctypes.c_int, _vp, ctypes.c_size_t, _vp]
        lib.moe_forward_residual_rmsnorm.argtypes = [_vp, _vp, _i64, _vp, _vp, _vp, _vp, ctypes.c_float, _vp, _vp,
                                                     _vp, ctypes.c_int, _vp, ctypes.c_size_t, _vp]
        lib.moe_act_quant_fp8.argtypes = [_vp, _i64, _i64, _vp, _vp, _vp]
        lib.moe_act_quant_nvfp4.argtypes = [_vp, _i64, _i64, _vp, _vp, _vp, _vp]
        lib.moe_act_quant_nvfp4_f32.argtypes = [_vp, _i64, _i64, _vp, _vp, _vp, _vp]
        lib.moe_device_status.argtypes = [_vp, _vp, ctypes.POINTER(_i32)]
        lib.moe_last_launch_count.argtypes = [_vp]
        lib.moe_router_planes_size.argtypes = [_vp, ctypes.POINTER(ctypes.c_size_t)]
        lib.moe_router_prepare.argtypes = [_vp, _vp, _vp, ctypes.c_size_t, _vp]
        lib.moe_layer_set_wait_limit.argtypes = [_vp, ctypes.c_uint64]
        lib.moe_layer_stall_test.argtypes = [_vp, ctypes.c_int]
        lib.moe_kernel_timing_enable.argtypes = [_vp, ctypes.c_int]
        lib.moe_kernel_timing_read.argtypes = [_vp, ctypes.c_int, ctypes.POINTER(ctypes.c_double),
                                               ctypes.POINTER(_i64)]
        lib.moe_kernel_count.argtypes = []
        lib.moe_kernel_name.argtypes = [ctypes.c_int]
        lib.moe_kernel_name.restype = ctypes.c_char_p
        lib.moe_status_string.argtypes = [ctypes.c_int]
        lib.moe_status_string.restype = ctypes.c_char_p
        _lib = lib
        return lib


def status_string(status: int) -> str:
    try:
        return load_library(build=False).moe_status_string(int(status)).decode()
    except Exception:  # pragma: no cover - library absent
        return "status"


def _check(rc: int, what: str):
    if rc != MOE_OK:
        raise MoeError(rc, what)


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def moe_act_quant_fp8(x, stream=None):
    """x bf16 [rows, n] (device) -> (codes uint8 [rows, n], scales fp32 [rows, n/128])."""
    lib = load_library()
    rows, n = x.shape
    codes = torch.empty(rows, n, dtype=torch.uint8, device=x.device)
    scales = torch.empty(rows, n // 128, dtype=torch.float32, device=x.device)
    _check(lib.moe_act_quant_fp8(_p(x), rows, n, _p(codes), _p(scales), _stream(stream)), "moe_act_quant_fp8")
    return codes, scales


def moe_act_quant_nvfp4(x, stream=None):
    """x bf16 or fp32 [rows, n] (device) -> (packed codes uint8 [rows, n/2],
    e4m3 block-scale codes uint8 [rows, n/16], row scales fp32 [rows])."""
    lib = load_library()
    rows, n = x.shape
    codes = torch.empty(rows, n // 2, dtype=torch.uint8, device=x.device)
    sb = torch.empty(rows, n // 16, dtype=torch.uint8, device=x.device)
    g = torch.empty(rows, dtype=torch.float32, device=x.device)
    if x.dtype == torch.float32:
        fn, name = lib.moe_act_quant_nvfp4_f32, "moe_act_quant_nvfp4_f32"
    else:
        assert x.dtype == torch.bfloat16, x.dtype
        fn, name = lib.moe_act_quant_nvfp4, "moe_act_quant_nvfp4"
    _check(fn(_p(x), rows, n, _p(codes), _p(sb), _p(g), _stream(stream)), name)
    return codes, sb, g


class MoeLayer:
    """A layer handle over caller-owned device weights (see include/moe_ffn.h).

    tensors: dict with w1, w3, w2 (and s1, s3, s2 for fp8; s1, s3, s2 and
    sb1, sb3, sb2 for NVFP4), optionally ws1, ws3, ws2 (+ ss1, ss3, ss2, and
    ssb1, ssb3, ssb2) for the shared expert, as produced by
    ``inputs.make_experts`` and moved to the device.
    """

    def __init__(self, shape, tensors: dict, expert_range=None):
        """expert_range: (begin, end) makes this handle one expert-parallel
        shard holding experts [begin, end) of shape.num_experts; its tensors
        w1, w3, w2 (and s*, sb*) are then stacked over those experts only."""
        self.lib = load_library()
        self.shape = shape
        self._keep = dict(tensors)
        sigmoid = getattr(shape, "scoring", "softmax") == "sigmoid"
        nvfp4 = bool(getattr(shape, "nvfp4", False))
        wfmt = MOE_WEIGHTS_NVFP4 if nvfp4 else (MOE_WEIGHTS_FP8_E4M3_B128 if shape.fp8 else MOE_WEIGHTS_BF16)
        cfg = MoeConfig(shape.hidden, shape.num_experts, shape.top_k, shape.inter, shape.shared_inter, wfmt,
                        MOE_SCORING_SIGMOID if sigmoid else MOE_SCORING_SOFTMAX,
                        int(bool(getattr(shape, "norm_topk_prob", True))),
                        float(getattr(shape, "routed_scaling", 1.0)),
                        *(expert_range if expert_range is not None else (0, 0)))
        sbn = ("sb1", "sb3", "sb2") if nvfp4 else ()
        routed = MoeExpertWeights(*[_p(tensors.get(n)) for n in ("w1", "w3", "w2", "s1", "s3", "s2")], None,
                                  *[_p(tensors.get(n)) for n in sbn])
        shared = None
        if shape.shared_inter:
            gate = _p(tensors.get("shared_gate")) if getattr(shape, "shared_gate", False) else None
            shared = MoeExpertWeights(*[_p(tensors.get(n)) for n in ("ws1", "ws3", "ws2", "ss1", "ss3", "ss2")],
                                      gate, *[_p(tensors.get("s" + n)) for n in sbn])
        self.expert_range = tuple(expert_range) if expert_range is not None else (0, shape.num_experts)
        handle = _vp()
        _check(self.lib.moe_layer_create(ctypes.byref(cfg), ctypes.byref(routed),
                                         ctypes.byref(shared) if shared is not None else None,
                                         ctypes.byref(handle)), "moe_layer_create")
        self.handle = handle
        self._ws = None

    def close(self):
        if getattr(self, "handle", None):
            self.lib.moe_layer_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # ---- workspace
    def workspace_size(self, m: int) -> int:
        n = ctypes.c_size_t()
        _check(self.lib.moe_workspace_size(self.handle, int(m), ctypes.byref(n)), "moe_workspace_size")
        return n.value

    def workspace(self, m: int, device=None) -> torch.Tensor:
        need = self.workspace_size(m)
        if self._ws is None or self._ws.numel() < need:
            dev = device if device is not None else torch.device("cuda", torch.cuda.current_device())
            self._ws = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
        return self._ws

    def select_arm(self, m: int) -> int:
        return self.lib.moe_select_arm(self.handle, int(m))

    def prepare_router(self, router_w, stream=None):
        """Split router_w once into planes this handle keeps (moe_router_prepare);
        router_w=None forgets them."""
        if router_w is None:
            _check(self.lib.moe_router_prepare(self.handle, None, None, 0, _stream(stream)), "moe_router_prepare")
            self._planes = None
            return
        n = ctypes.c_size_t()
        _check(self.lib.moe_router_planes_size(self.handle, ctypes.byref(n)), "moe_router_planes_size")
        self._planes = torch.empty(max(n.value, 256), dtype=torch.uint8, device=router_w.device)
        _check(self.lib.moe_router_prepare(self.handle, _p(router_w), _p(self._planes), self._planes.numel(),
                                           _stream(stream)), "moe_router_prepare")

    def set_wait_limit(self, ns: int):
        """Limit (ns) of the grouped GEMMs' bounded waits; 0 restores 2 s."""
        _check(self.lib.moe_layer_set_wait_limit(self.handle, int(ns)), "moe_layer_set_wait_limit")

    def stall_test(self, enable: bool):
        """Make the bf16 grouped GEMMs wait on a barrier nothing completes."""
        _check(self.lib.moe_layer_stall_test(self.handle, int(bool(enable))), "moe_layer_stall_test")

    def last_launch_count(self) -> int:
        return self.lib.moe_last_launch_count(self.handle)

    def kernel_timing(self, enable: bool):
        """Turn per-kernel event timing on or off (resets the totals)."""
        _check(self.lib.moe_kernel_timing_enable(self.handle, int(bool(enable))), "moe_kernel_timing_enable")

    def kernel_times(self) -> dict:
        """{kernel name: (total ms, launches)} for kernels launched while timing was on."""
        out = {}
        for k in range(self.lib.moe_kernel_count()):
            ms = ctypes.c_double()
            n = _i64()
            _check(self.lib.moe_kernel_timing_read(self.handle, k, ctypes.byref(ms), ctypes.byref(n)),
                   "moe_kernel_timing_read")
            if n.value:
                out[self.lib.moe_kernel_name(k).decode()] = (ms.value, n.value)
        return out

    def device_status(self, stream=None) -> int:
        code = _i32()
        ws = self._ws
        if ws is None:
            return 0
        rc = self.lib.moe_device_status(_p(ws), _stream(stream), ctypes.byref(code))
        if rc not in (MOE_OK, MOE_ERR_DEVICE):
            raise MoeError(rc, "moe_device_status")
        return code.value

    # ---- entry points
    def moe_route(self, x, router_w, router_bias=None, logits=False, stream=None):
        m = x.shape[0]
        dev = x.device
        ids = torch.empty(m, self.shape.top_k, dtype=torch.int32, device=dev)
        w = torch.empty(m, self.shape.top_k, dtype=torch.float32, device=dev)
        lg = torch.empty(m, self.shape.num_experts, dtype=torch.float32, device=dev) if logits else None
        ws = self.workspace(m)
        _check(self.lib.moe_route(self.handle, _p(x), m, _p(router_w), _p(router_bias), _p(lg), _p(ids), _p(w),
                                  _p(ws), ws.numel(), _stream(stream)), "moe_route")
        return (ids, w, lg) if logits else (ids, w)

    def moe_permute(self, topk_ids, stream=None):
        m = topk_ids.shape[0]
        dev = topk_ids.device
        P = m * self.shape.top_k
        n_local = self.expert_range[1] - self.expert_range[0]  # this handle's experts
        off = torch.empty(n_local + 1, dtype=torch.int32, device=dev)
        sp = torch.empty(P, dtype=torch.int32, device=dev)
        sl = torch.empty(P, dtype=torch.int32, device=dev)
        ws = self.workspace(m)
        _check(self.lib.moe_permute(self.handle, _p(topk_ids), m, _p(off), _p(sp), _p(sl), _p(ws), ws.numel(),
                                    _stream(stream)), "moe_permute")
        return off, sp, sl

    def moe_experts(self, x, topk_ids, topk_w, arm="auto", out=None, stream=None):
        m = x.shape[0]
        if out is None:
            out = torch.empty(m, self.shape.hidden, dtype=torch.bfloat16, device=x.device)
        ws = self.workspace(m)
        _check(self.lib.moe_experts(self.handle, _p(x), m, _p(topk_ids), _p(topk_w), _p(out), ARMS[arm], _p(ws),
                                    ws.numel(), _stream(stream)), "moe_experts")
        return out

    def moe_shared_expert_add(self, x, out, arm="auto", stream=None):
        """out (bf16 [m, H], in place) += the shared expert of x."""
        m = x.shape[0]
        ws = self.workspace(m)
        _check(self.lib.moe_shared_expert_add(self.handle, _p(x), m, _p(out), ARMS[arm], _p(ws), ws.numel(),
                                              _stream(stream)), "moe_shared_expert_add")
        return out

    def moe_forward(self, x, router_w, router_bias=None, arm="auto", out=None, return_routing=False, stream=None):
        m = x.shape[0]
        dev = x.device
        if out is None:
            out = torch.empty(m, self.shape.hidden, dtype=torch.bfloat16, device=dev)
        ids = w = None
        if return_routing:
            ids = torch.empty(m, self.shape.top_k, dtype=torch.int32, device=dev)
            w = torch.empty(m, self.shape.top_k, dtype=torch.float32, device=dev)
        ws = self.workspace(m)
        _check(self.lib.moe_forward(self.handle, _p(x), m, _p(router_w), _p(router_bias), _p(out), _p(ids), _p(w),
                                    ARMS[arm], _p(ws), ws.numel(), _stream(stream)), "moe_forward")
        return (out, ids, w) if return_routing else out

    def moe_forward_residual_rmsnorm(self, x, router_w, residual, norm_w, eps=1e-6, router_bias=None, arm="auto",
                                     norm_out=None, return_routing=False, stream=None):
        """The layer with its tail: residual (bf16 [m, H], updated in place) +=
        the layer output, and norm_out = RMSNorm(residual) * norm_w (fp32 [H])."""
        m = x.shape[0]
        dev = x.device
        if norm_out is None:
            norm_out = torch.empty(m, self.shape.hidden, dtype=torch.bfloat16, device=dev)
        ids = w = None
        if return_routing:
            ids = torch.empty(m, self.shape.top_k, dtype=torch.int32, device=dev)
            w = torch.empty(m, self.shape.top_k, dtype=torch.float32, device=dev)
        ws = self.workspace(m)
        _check(self.lib.moe_forward_residual_rmsnorm(self.handle, _p(x), m, _p(router_w), _p(router_bias),
                                                     _p(residual), _p(norm_w), float(eps), _p(norm_out), _p(ids),
                                                     _p(w), ARMS[arm], _p(ws), ws.numel(), _stream(stream)),
               "moe_forward_residual_rmsnorm")
        return (norm_out, ids, w) if return_routing else norm_out
