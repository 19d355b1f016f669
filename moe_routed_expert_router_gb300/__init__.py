"""Python binding of libmoe_nvfp4.so, the C-ABI library of the routed MoE FFN
over NVFP4 weights on GB300 (sm_103a).

Argument marshalling only: every step of the path runs in the library's CUDA
kernels.  torch provides device memory and streams.  There is no fallback: if
the library cannot be loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = _build.LIB

ROUTER_SOFTMAX, ROUTER_SIGMOID = 0, 1
ROUTER_F32, ROUTER_BF16 = 0, 1
WEIGHTS_NVFP4, WEIGHTS_MXFP4 = 0, 1
W4A16, W4A4 = 0, 1

STATUS = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED_SHAPE", 3: "MOE_ERR_MISALIGNED",
          4: "MOE_ERR_NONFINITE", 5: "MOE_ERR_TIMEOUT", 6: "MOE_ERR_CUDA", 7: "MOE_ERR_OOM", 8: "MOE_ERR_DEVICE"}
OK, ERR_INVALID_ARG, ERR_UNSUPPORTED_SHAPE, ERR_MISALIGNED, ERR_NONFINITE, ERR_TIMEOUT, ERR_CUDA, ERR_OOM, \
    ERR_DEVICE = range(9)

EXPORTS = ["moe_plan_create", "moe_plan_destroy", "moe_route", "moe_forward", "moe_forward_host",
           "moe_quantize_act", "moe_quantize_nvfp4", "moe_plan_sync_status", "moe_plan_debug_buffer",
           "moe_plan_set_profiling", "moe_plan_read_profile", "moe_plan_set_path", "moe_plan_check_timeout",
           "moe_route_static", "moe_convert_f32", "moe_quantize_mxfp4", "moe_plan_keep_h", "moe_status_string",
           "moe_version"]
FMT_E4M3, FMT_E2M1 = 0, 1
PATH_AUTO, PATH_CUDA_CORE, PATH_TENSOR_CORE, PATH_WARP_MMA = 0, 1, 2, 3
STAGES = ["route", "group", "quant_x", "permute", "gate_up", "quant_h", "down", "finalize"]


class MoeError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)}")


class Config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "hidden", "inter", "num_experts", "top_k", "max_tokens", "router", "renormalize", "mode",
        "has_shared", "shared_inter", "router_dtype", "weight_format")]


class Nvfp4(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p), ("tensor_scale", ctypes.c_void_p)]


class ExpertSetC(ctypes.Structure):
    _fields_ = [("gate", Nvfp4), ("up", Nvfp4), ("down", Nvfp4)]


_lib = None


def lib():
    """Load the library (building it first if the sources are newer)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH) or not _build.up_to_date():
            _build.build()
        L = ctypes.CDLL(LIB_PATH)
        P, I32 = ctypes.c_void_p, ctypes.c_int32
        L.moe_plan_create.argtypes = [ctypes.POINTER(Config), ctypes.POINTER(P)]
        L.moe_plan_destroy.argtypes = [P]
        L.moe_route.argtypes = [P, P, I32, P, P, P, P, P, P, P]
        L.moe_forward.argtypes = [P, P, I32, P, P, ctypes.POINTER(ExpertSetC), ctypes.POINTER(ExpertSetC), P, P]
        L.moe_forward_host.argtypes = L.moe_forward.argtypes
        L.moe_quantize_act.argtypes = [P, P, I32, P, P, P, P]
        L.moe_quantize_nvfp4.argtypes = [P, I32, I32, I32, P, P, P, P]
        L.moe_plan_sync_status.argtypes = [P, P]
        L.moe_plan_debug_buffer.argtypes = [P, ctypes.c_char_p, ctypes.POINTER(P), ctypes.POINTER(ctypes.c_size_t)]
        L.moe_plan_set_profiling.argtypes = [P, I32]
        L.moe_plan_keep_h.argtypes = [P, I32]
        L.moe_plan_set_path.argtypes = [P, I32]
        L.moe_plan_check_timeout.argtypes = [P, ctypes.c_int64, P]
        L.moe_route_static.argtypes = [P, I32, I32, P, P, I32, I32, I32, I32, P, P, P, P, P]
        L.moe_plan_read_profile.argtypes = [P, P, P, P]
        L.moe_convert_f32.argtypes = [P, ctypes.c_int64, I32, P, P]
        L.moe_quantize_mxfp4.argtypes = [P, ctypes.c_int64, I32, P, P, P]
        L.moe_status_string.argtypes = [I32]
        L.moe_status_string.restype = ctypes.c_char_p
        L.moe_version.restype = ctypes.c_char_p
        for n in EXPORTS:
            if n not in ("moe_status_string", "moe_version"):
                getattr(L, n).restype = I32
        _lib = L
    return _lib


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream=None):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(status: int, where: str):
    if status != OK:
        raise MoeError(status, where)


class NvfpTensor:
    """One NVFP4 weight stacked over experts: codes [n][N][K/2] u8, scales [n][N][K/16] u8, ts [n] f32."""

    def __init__(self, codes: torch.Tensor, scales: torch.Tensor, ts: torch.Tensor):
        self.codes, self.scales, self.ts = codes, scales, ts

    def c(self) -> Nvfp4:
        return Nvfp4(_ptr(self.codes), _ptr(self.scales), _ptr(self.ts))


class ExpertSet:
    def __init__(self, gate: NvfpTensor, up: NvfpTensor, down: NvfpTensor):
        self.gate, self.up, self.down = gate, up, down

    def c(self) -> ExpertSetC:
        return ExpertSetC(self.gate.c(), self.up.c(), self.down.c())


def quantize_nvfp4(w: torch.Tensor, out: NvfpTensor | None = None, stream=None) -> NvfpTensor:
    """NVFP4-quantise fp32 weights [batch][rows][cols] on the device (one tensor scale per item)."""
    assert w.is_cuda and w.dtype == torch.float32 and w.is_contiguous()
    if w.dim() == 2:
        w = w.unsqueeze(0)
    b, r, c = w.shape
    if out is None:
        out = NvfpTensor(torch.empty(b, r, c // 2, dtype=torch.uint8, device=w.device),
                         torch.empty(b, r, c // 16, dtype=torch.uint8, device=w.device),
                         torch.empty(b, dtype=torch.float32, device=w.device))
    _check(lib().moe_quantize_nvfp4(_ptr(w), b, r, c, _ptr(out.codes), _ptr(out.scales), _ptr(out.ts),
                                    _stream(stream)), "moe_quantize_nvfp4")
    return out


def quantize_mxfp4(w: torch.Tensor, out: NvfpTensor | None = None, stream=None) -> NvfpTensor:
    """MXFP4-quantise fp32 weights [batch][rows][cols] (or [rows][cols]) on the
    device: E2M1 codes and E8M0 block-of-32 scales (no tensor scale: ts is None)."""
    assert w.is_cuda and w.dtype == torch.float32 and w.is_contiguous()
    if w.dim() == 2:
        w = w.unsqueeze(0)
    b, r, c = w.shape
    if out is None:
        out = NvfpTensor(torch.empty(b, r, c // 2, dtype=torch.uint8, device=w.device),
                         torch.empty(b, r, c // 32, dtype=torch.uint8, device=w.device), None)
    _check(lib().moe_quantize_mxfp4(_ptr(w), b * r, c, _ptr(out.codes), _ptr(out.scales), _stream(stream)),
           "moe_quantize_mxfp4")
    return out


def convert_f32(src: torch.Tensor, fmt: int, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """The device's fp32 -> E4M3 byte (FMT_E4M3) or E2M1 code (FMT_E2M1) conversion, element-wise."""
    assert src.is_cuda and src.dtype == torch.float32 and src.is_contiguous()
    if out is None:
        out = torch.empty(src.shape, dtype=torch.uint8, device=src.device)
    _check(lib().moe_convert_f32(_ptr(src), src.numel(), fmt, _ptr(out), _stream(stream)), "moe_convert_f32")
    return out


class Plan:
    """A moe_plan: configuration plus device workspace for up to max_tokens tokens."""

    def __init__(self, hidden, inter, num_experts, top_k, max_tokens, router=ROUTER_SOFTMAX, renormalize=True,
                 mode=W4A16, has_shared=False, shared_inter=0, router_dtype=ROUTER_F32, weight_format=WEIGHTS_NVFP4):
        self.cfg = Config(hidden, inter, num_experts, top_k, max_tokens, router, int(bool(renormalize)), mode,
                          int(bool(has_shared)), shared_inter if has_shared else 0, router_dtype, weight_format)
        h = ctypes.c_void_p()
        _check(lib().moe_plan_create(ctypes.byref(self.cfg), ctypes.byref(h)), "moe_plan_create")
        self.handle = h

    def close(self):
        if getattr(self, "handle", None) and self.handle.value:
            lib().moe_plan_destroy(self.handle)
            self.handle = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *a):
        self.close()

    def route(self, x, router_w, router_bias=None, out=None, stream=None):
        T = x.shape[0]
        k, E = self.cfg.top_k, self.cfg.num_experts
        dev = x.device
        if out is None:
            out = dict(topk_ids=torch.empty(T, k, dtype=torch.int32, device=dev),
                       topk_w=torch.empty(T, k, dtype=torch.float32, device=dev),
                       expert_offsets=torch.empty(E + 1, dtype=torch.int32, device=dev),
                       sorted_rows=torch.empty(max(T * k, 1), dtype=torch.int32, device=dev))
        _check(lib().moe_route(self.handle, _ptr(x), T, _ptr(router_w), _ptr(router_bias), _ptr(out["topk_ids"]),
                               _ptr(out["topk_w"]), _ptr(out["expert_offsets"]), _ptr(out["sorted_rows"]),
                               _stream(stream)), "moe_route")
        return out

    def forward(self, x, router_w, router_bias, routed: ExpertSet, shared: ExpertSet | None = None, out=None,
                stream=None):
        T = x.shape[0]
        if out is None:
            out = torch.empty(T, self.cfg.hidden, dtype=torch.bfloat16, device=x.device)
        rs = routed.c()
        ss = shared.c() if shared is not None else None
        _check(lib().moe_forward(self.handle, _ptr(x), T, _ptr(router_w), _ptr(router_bias), ctypes.byref(rs),
                                 ctypes.byref(ss) if ss is not None else None, _ptr(out), _stream(stream)),
               "moe_forward")
        return out

    def forward_host(self, x_host, router_w, router_bias, routed: ExpertSet, shared: ExpertSet | None, out_host,
                     stream=None):
        T = x_host.shape[0]
        rs = routed.c()
        ss = shared.c() if shared is not None else None
        _check(lib().moe_forward_host(self.handle, _ptr(x_host), T, _ptr(router_w), _ptr(router_bias),
                                      ctypes.byref(rs), ctypes.byref(ss) if ss is not None else None,
                                      _ptr(out_host), _stream(stream)), "moe_forward_host")
        return out_host

    def quantize_act(self, x, stream=None):
        T, H = x.shape
        codes = torch.empty(T, H // 2, dtype=torch.uint8, device=x.device)
        scales = torch.empty(T, H // (32 if self.cfg.weight_format == WEIGHTS_MXFP4 else 16), dtype=torch.uint8,
                             device=x.device)
        ts = torch.empty(1, dtype=torch.float32, device=x.device)
        _check(lib().moe_quantize_act(self.handle, _ptr(x), T, _ptr(codes), _ptr(scales), _ptr(ts), _stream(stream)),
               "moe_quantize_act")
        return codes, scales, ts

    def sync_status(self, stream=None) -> int:
        return lib().moe_plan_sync_status(self.handle, _stream(stream))

    def check_timeout(self, wait_ns: int, stream=None):
        _check(lib().moe_plan_check_timeout(self.handle, wait_ns, _stream(stream)), "moe_plan_check_timeout")

    def set_path(self, path: int):
        _check(lib().moe_plan_set_path(self.handle, path), "moe_plan_set_path")

    def keep_h(self, on: bool):
        """Store the fp32 SwiGLU output also where gate/up quantises it itself (MXFP4 W4A4, tensor cores)."""
        _check(lib().moe_plan_keep_h(self.handle, int(bool(on))), "moe_plan_keep_h")

    def set_profiling(self, on: bool):
        _check(lib().moe_plan_set_profiling(self.handle, int(bool(on))), "moe_plan_set_profiling")

    def read_profile(self):
        """Per-stage summed event ms, kernel launches and executions since the last read."""
        import numpy as np
        ms = np.zeros(len(STAGES), np.float32)
        la = np.zeros(len(STAGES), np.int64)
        ca = np.zeros(len(STAGES), np.int64)
        _check(lib().moe_plan_read_profile(self.handle, ms.ctypes.data, la.ctypes.data, ca.ctypes.data),
               "moe_plan_read_profile")
        return {s: (float(ms[i]), int(la[i]), int(ca[i])) for i, s in enumerate(STAGES)}

    def debug_buffer(self, name: str):
        p = ctypes.c_void_p()
        n = ctypes.c_size_t()
        _check(lib().moe_plan_debug_buffer(self.handle, name.encode(), ctypes.byref(p), ctypes.byref(n)),
               "moe_plan_debug_buffer")
        return p.value, n.value


def device_view(ptr: int, nbytes: int, dtype=torch.uint8, device="cuda"):
    """A torch view of plan-owned device memory (for tests)."""
    class _A:
        __cuda_array_interface__ = {"shape": (nbytes,), "typestr": "|u1", "data": (ptr, False), "version": 3}
    t = torch.as_tensor(_A(), device=device)
    return t.view(dtype)
