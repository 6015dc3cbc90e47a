"""Thin ctypes binding of libnvfp4.so (argument marshalling only).

Every function here takes CUDA tensors, checks dtypes and shapes, and passes
raw device pointers, sizes and the current CUDA stream to the C ABI declared
in include/nvfp4.h.  All arithmetic happens in the library's CUDA kernels;
if the library is missing, loading fails loudly: there is no CPU fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

_lib = None
_lock = threading.Lock()

OK, ERR_INVALID_ARG, ERR_SHAPE, ERR_ALIGNMENT, ERR_WORKSPACE, ERR_UNSUPPORTED_DEVICE, ERR_CUDA, \
    ERR_NONFINITE, ERR_TIMEOUT = range(9)
OUT_BF16, OUT_FP32 = 0, 1

EXPORTS = [
    "nvfp4_workspace_bytes", "nvfp4_quantize", "nvfp4_dequantize", "nvfp4_w4a16_lora_gemm",
    "nvfp4_round_scales", "nvfp4_get_device_status", "nvfp4_status_string", "nvfp4_encode_debug",
    "nvfp4_quotient_check", "nvfp4_w4a16_lora_gemm_static", "nvfp4_wait_selftest", "nvfp4_gemm_kernel",
    "nvfp4_scale_qlora_gemm", "nvfp4_w4a16_lora_gemm_dgrad", "nvfp4_dgrad_workspace_bytes",
    "nvfp4_lora_grads", "nvfp4_lora_grads_workspace_bytes", "nvfp4_gemm_list_workspace_bytes",
    "nvfp4_w4a16_lora_gemm_list",
]


class Projection(ctypes.Structure):
    """struct nvfp4_projection (one entry of nvfp4_w4a16_lora_gemm_list)."""
    _fields_ = [("x_bf16", ctypes.c_void_p), ("codes", ctypes.c_void_p), ("scales_e4m3", ctypes.c_void_p),
                ("tensor_scale", ctypes.c_void_p), ("lora_a_bf16", ctypes.c_void_p),
                ("lora_b_bf16", ctypes.c_void_p), ("noise_fp32", ctypes.c_void_p), ("y", ctypes.c_void_p),
                ("N", ctypes.c_int64), ("K", ctypes.c_int64), ("lora_scale", ctypes.c_float)]


class NVFP4Error(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True):
    """Load libnvfp4.so (building it with nvcc when it is missing or stale)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB
        if build_if_missing and _build.is_stale():
            _build.build()
        if not os.path.exists(path):
            raise RuntimeError(f"libnvfp4.so not found at {path}; run nvfp4_weight_only_02_gb300/build.py")
        lib = ctypes.CDLL(path)
        P, i64, u32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint32
        st = ctypes.c_int
        sig = {
            "nvfp4_workspace_bytes": (ctypes.c_size_t, [i64, i64, i64, i64]),
            "nvfp4_quantize": (st, [P, i64, i64, P, P, P, ctypes.c_int, P, ctypes.c_size_t, P]),
            "nvfp4_dequantize": (st, [P, P, P, i64, i64, P, ctypes.c_int, P]),
            "nvfp4_w4a16_lora_gemm": (st, [P, i64, i64, i64, P, P, P, P, P, i64, ctypes.c_float, P, P,
                                           ctypes.c_int, P, ctypes.c_size_t, P]),
            "nvfp4_round_scales": (st, [P, P, i64, i64, P, P, ctypes.c_size_t, P]),
            "nvfp4_get_device_status": (st, [P, P]),
            "nvfp4_status_string": (ctypes.c_char_p, [st]),
            "nvfp4_encode_debug": (st, [P, i64, ctypes.c_int, P, P]),
            "nvfp4_quotient_check": (st, [u32, u32, P, P]),
            "nvfp4_w4a16_lora_gemm_static": (st, [P, i64, i64, i64, P, P, P, P, P, i64, ctypes.c_float,
                                                  P, P, ctypes.c_int, P]),
            "nvfp4_wait_selftest": (st, [P, ctypes.c_int, P]),
            "nvfp4_gemm_kernel": (ctypes.c_char_p, [i64, i64, i64, i64]),
            "nvfp4_scale_qlora_gemm": (st, [P, i64, i64, i64, P, P, P, P, P, P, i64, ctypes.c_float, P, P,
                                            ctypes.c_int, P, ctypes.c_size_t, P]),
            "nvfp4_w4a16_lora_gemm_dgrad": (st, [P, i64, i64, i64, P, P, P, P, P, i64, ctypes.c_float, P, P,
                                                 ctypes.c_int, P, ctypes.c_size_t, P]),
            "nvfp4_dgrad_workspace_bytes": (ctypes.c_size_t, [i64, i64, i64, i64]),
            "nvfp4_lora_grads": (st, [P, P, P, i64, i64, i64, P, P, i64, ctypes.c_float, P, P, P, ctypes.c_size_t,
                                      P]),
            "nvfp4_lora_grads_workspace_bytes": (ctypes.c_size_t, [i64, i64, i64, i64]),
            "nvfp4_gemm_list_workspace_bytes": (ctypes.c_size_t, [P, ctypes.c_int, i64, i64]),
            "nvfp4_w4a16_lora_gemm_list": (st, [P, ctypes.c_int, i64, i64, ctypes.c_int, P, ctypes.c_size_t, P]),
        }
        for name, (res, args) in sig.items():
            f = getattr(lib, name)
            f.restype = res
            f.argtypes = args
        _lib = lib
        return lib


def gemm_kernel(M: int, N: int, K: int, r: int = 0):
    """Kernel family nvfp4_w4a16_lora_gemm runs for these sizes (None if unsupported)."""
    name = load().nvfp4_gemm_kernel(M, N, K, r)
    return None if name is None else name.decode()


def status_string(status: int) -> str:
    return load().nvfp4_status_string(int(status)).decode()


def _check(status: int, where: str):
    if status != OK:
        raise NVFP4Error(status, where)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _need(t, dtype, shape, name):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


# ------------------------------------------------------------------ workspace
def nvfp4_workspace_bytes(M: int, N: int, K: int, r: int) -> int:
    return int(load().nvfp4_workspace_bytes(M, N, K, r))


def new_workspace(nbytes: int, device=None) -> torch.Tensor:
    """A zero-filled workspace (the library keeps it zeroed between calls)."""
    n = max(256, (int(nbytes) + 255) // 256 * 256)
    return torch.zeros(n, dtype=torch.uint8, device=device or "cuda")


def nvfp4_get_device_status(workspace: torch.Tensor) -> int:
    return int(load().nvfp4_get_device_status(_ptr(workspace), _stream()))


# ------------------------------------------------------------------ entry points
def nvfp4_quantize(w: torch.Tensor, codes: torch.Tensor, scales: torch.Tensor,
                   tensor_scale: torch.Tensor, use_given_tensor_scale: bool,
                   workspace: torch.Tensor):
    N, K = w.shape
    _need(w, torch.bfloat16, (N, K), "w")
    _need(codes, torch.uint8, (N, K // 2), "codes")
    _need(scales, torch.uint8, (N, K // 16), "scales")
    _need(tensor_scale, torch.float32, (1,), "tensor_scale")
    st = load().nvfp4_quantize(_ptr(w), N, K, _ptr(codes), _ptr(scales), _ptr(tensor_scale),
                               int(bool(use_given_tensor_scale)), _ptr(workspace),
                               workspace.numel(), _stream())
    _check(st, "nvfp4_quantize")


def nvfp4_dequantize(codes: torch.Tensor, scales: torch.Tensor, tensor_scale: torch.Tensor,
                     out: torch.Tensor):
    N, K2 = codes.shape
    K = K2 * 2
    _need(scales, torch.uint8, (N, K // 16), "scales")
    _need(tensor_scale, torch.float32, (1,), "tensor_scale")
    if out.dtype not in (torch.float32, torch.bfloat16):
        raise ValueError("out must be float32 or bfloat16")
    _need(out, out.dtype, (N, K), "out")
    st = load().nvfp4_dequantize(_ptr(codes), _ptr(scales), _ptr(tensor_scale), N, K, _ptr(out),
                                 OUT_FP32 if out.dtype == torch.float32 else OUT_BF16, _stream())
    _check(st, "nvfp4_dequantize")


def nvfp4_w4a16_lora_gemm(x: torch.Tensor, codes: torch.Tensor, scales: torch.Tensor,
                          tensor_scale: torch.Tensor, lora_a, lora_b, lora_scale: float,
                          noise, y: torch.Tensor, workspace: torch.Tensor):
    M, K = x.shape
    N = codes.shape[0]
    _need(x, torch.bfloat16, (M, K), "x")
    _need(codes, torch.uint8, (N, K // 2), "codes")
    _need(scales, torch.uint8, (N, K // 16), "scales")
    _need(tensor_scale, torch.float32, (1,), "tensor_scale")
    r = 0
    if lora_a is not None:
        r = lora_a.shape[0]
        _need(lora_a, torch.bfloat16, (r, K), "lora_a")
        _need(lora_b, torch.bfloat16, (N, r), "lora_b")
    if noise is not None:
        _need(noise, torch.float32, (K,), "noise")
    if y.dtype not in (torch.float32, torch.bfloat16):
        raise ValueError("y must be float32 or bfloat16")
    _need(y, y.dtype, (M, N), "y")
    st = load().nvfp4_w4a16_lora_gemm(
        _ptr(x), M, N, K, _ptr(codes), _ptr(scales), _ptr(tensor_scale), _ptr(lora_a),
        _ptr(lora_b), r, float(lora_scale), _ptr(noise), _ptr(y),
        OUT_FP32 if y.dtype == torch.float32 else OUT_BF16, _ptr(workspace), workspace.numel(),
        _stream())
    _check(st, "nvfp4_w4a16_lora_gemm")


def _projection_array(entries):
    """entries: (x, codes, scales, tensor_scale, lora_a, lora_b, lora_scale, noise, y) tuples of CUDA
    tensors (lora_a, lora_b, noise may be None).  Returns (ctypes array, M, r, y dtype code)."""
    if len(entries) == 0:
        raise ValueError("empty projection list")
    M = entries[0][0].shape[0]
    r = 0 if entries[0][4] is None else entries[0][4].shape[0]
    ydt = entries[0][8].dtype
    if ydt not in (torch.float32, torch.bfloat16):
        raise ValueError("y must be float32 or bfloat16")
    arr = (Projection * len(entries))()
    for i, (x, codes, scales, ts, a, b, s, z, y) in enumerate(entries):
        K = x.shape[1]
        N = codes.shape[0]
        _need(x, torch.bfloat16, (M, K), f"x[{i}]")
        _need(codes, torch.uint8, (N, K // 2), f"codes[{i}]")
        _need(scales, torch.uint8, (N, K // 16), f"scales[{i}]")
        _need(ts, torch.float32, (1,), f"tensor_scale[{i}]")
        if (a is None) != (r == 0):
            raise ValueError("every entry of a list has the same LoRA rank")
        if a is not None:
            _need(a, torch.bfloat16, (r, K), f"lora_a[{i}]")
            _need(b, torch.bfloat16, (N, r), f"lora_b[{i}]")
        if z is not None:
            _need(z, torch.float32, (K,), f"noise[{i}]")
        _need(y, ydt, (M, N), f"y[{i}]")
        arr[i] = Projection(_ptr(x), _ptr(codes), _ptr(scales), _ptr(ts), _ptr(a), _ptr(b), _ptr(z), _ptr(y),
                            N, K, float(s))
    return arr, M, r, OUT_FP32 if ydt == torch.float32 else OUT_BF16


def nvfp4_gemm_list_workspace_bytes(entries) -> int:
    arr, M, r, _ = _projection_array(entries)
    return int(load().nvfp4_gemm_list_workspace_bytes(arr, len(entries), M, r))


def nvfp4_w4a16_lora_gemm_list(entries, workspace: torch.Tensor):
    """Independent projections of one token count in one call (see _projection_array for an entry)."""
    arr, M, r, ydt = _projection_array(entries)
    st = load().nvfp4_w4a16_lora_gemm_list(arr, len(entries), M, r, ydt, _ptr(workspace), workspace.numel(),
                                           _stream())
    _check(st, "nvfp4_w4a16_lora_gemm_list")


def nvfp4_round_scales(scale_param: torch.Tensor, tensor_scale: torch.Tensor,
                       scales: torch.Tensor, workspace: torch.Tensor):
    N, KB = scale_param.shape
    _need(scale_param, torch.float32, (N, KB), "scale_param")
    _need(scales, torch.uint8, (N, KB), "scales")
    _need(tensor_scale, torch.float32, (1,), "tensor_scale")
    st = load().nvfp4_round_scales(_ptr(scale_param), _ptr(tensor_scale), N, KB * 16,
                                   _ptr(scales), _ptr(workspace), workspace.numel(), _stream())
    _check(st, "nvfp4_round_scales")


def nvfp4_scale_qlora_gemm(x: torch.Tensor, codes: torch.Tensor, scale_param: torch.Tensor,
                           tensor_scale: torch.Tensor, scales: torch.Tensor, lora_a, lora_b,
                           lora_scale: float, noise, y: torch.Tensor, workspace: torch.Tensor):
    M, K = x.shape
    N = codes.shape[0]
    _need(x, torch.bfloat16, (M, K), "x")
    _need(codes, torch.uint8, (N, K // 2), "codes")
    _need(scale_param, torch.float32, (N, K // 16), "scale_param")
    _need(scales, torch.uint8, (N, K // 16), "scales")
    _need(tensor_scale, torch.float32, (1,), "tensor_scale")
    r = 0
    if lora_a is not None:
        r = lora_a.shape[0]
        _need(lora_a, torch.bfloat16, (r, K), "lora_a")
        _need(lora_b, torch.bfloat16, (N, r), "lora_b")
    if noise is not None:
        _need(noise, torch.float32, (K,), "noise")
    if y.dtype not in (torch.float32, torch.bfloat16):
        raise ValueError("y must be float32 or bfloat16")
    _need(y, y.dtype, (M, N), "y")
    st = load().nvfp4_scale_qlora_gemm(
        _ptr(x), M, N, K, _ptr(codes), _ptr(scale_param), _ptr(tensor_scale), _ptr(scales),
        _ptr(lora_a), _ptr(lora_b), r, float(lora_scale), _ptr(noise), _ptr(y),
        OUT_FP32 if y.dtype == torch.float32 else OUT_BF16, _ptr(workspace), workspace.numel(),
        _stream())
    _check(st, "nvfp4_scale_qlora_gemm")


def nvfp4_encode_debug(x: torch.Tensor, which: int) -> torch.Tensor:
    out = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    st = load().nvfp4_encode_debug(_ptr(x), x.numel(), int(which), _ptr(out), _stream())
    _check(st, "nvfp4_encode_debug")
    return out


def nvfp4_wait_selftest(workspace: torch.Tensor, which: int):
    _check(load().nvfp4_wait_selftest(_ptr(workspace), int(which), _stream()), "nvfp4_wait_selftest")


def nvfp4_quotient_check(sig_lo: int, sig_hi: int) -> int:
    cnt = torch.zeros(1, dtype=torch.int64, device="cuda")
    st = load().nvfp4_quotient_check(sig_lo, sig_hi, _ptr(cnt), _stream())
    _check(st, "nvfp4_quotient_check")
    return int(cnt.item())


# ------------------------------------------------------------------ conveniences
class QuantizedWeight:
    """Device buffers of one NVFP4 weight: codes, scales and tensor scale."""

    def __init__(self, codes, scales, tensor_scale):
        self.codes, self.scales, self.tensor_scale = codes, scales, tensor_scale

    @property
    def shape(self):
        return self.codes.shape[0], self.codes.shape[1] * 2


def quantize(w: torch.Tensor, tensor_scale=None, workspace=None) -> QuantizedWeight:
    N, K = w.shape
    dev = w.device
    codes = torch.empty((N, K // 2), dtype=torch.uint8, device=dev)
    scales = torch.empty((N, K // 16), dtype=torch.uint8, device=dev)
    ts = torch.zeros(1, dtype=torch.float32, device=dev)
    if tensor_scale is not None:
        ts.fill_(float(tensor_scale))
    ws = workspace if workspace is not None else new_workspace(256, dev)
    nvfp4_quantize(w, codes, scales, ts, tensor_scale is not None, ws)
    return QuantizedWeight(codes, scales, ts)


def dequantize(q: QuantizedWeight, dtype=torch.float32) -> torch.Tensor:
    out = torch.empty(q.shape, dtype=dtype, device=q.codes.device)
    nvfp4_dequantize(q.codes, q.scales, q.tensor_scale, out)
    return out


def nvfp4_dgrad_workspace_bytes(M: int, N: int, K: int, r: int) -> int:
    return int(load().nvfp4_dgrad_workspace_bytes(M, N, K, r))


def nvfp4_w4a16_lora_gemm_dgrad(dy: torch.Tensor, codes: torch.Tensor, scales: torch.Tensor,
                                tensor_scale: torch.Tensor, lora_a, lora_b, lora_scale: float,
                                noise, dx: torch.Tensor, workspace: torch.Tensor):
    M, N = dy.shape
    K = codes.shape[1] * 2
    _need(dy, torch.bfloat16, (M, N), "dy")
    _need(codes, torch.uint8, (N, K // 2), "codes")
    _need(scales, torch.uint8, (N, K // 16), "scales")
    _need(tensor_scale, torch.float32, (1,), "tensor_scale")
    r = 0
    if lora_a is not None:
        r = lora_a.shape[0]
        _need(lora_a, torch.bfloat16, (r, K), "lora_a")
        _need(lora_b, torch.bfloat16, (N, r), "lora_b")
    if noise is not None:
        _need(noise, torch.float32, (K,), "noise")
    if dx.dtype not in (torch.float32, torch.bfloat16):
        raise ValueError("dx must be float32 or bfloat16")
    _need(dx, dx.dtype, (M, K), "dx")
    st = load().nvfp4_w4a16_lora_gemm_dgrad(
        _ptr(dy), M, N, K, _ptr(codes), _ptr(scales), _ptr(tensor_scale), _ptr(lora_a),
        _ptr(lora_b), r, float(lora_scale), _ptr(noise), _ptr(dx),
        OUT_FP32 if dx.dtype == torch.float32 else OUT_BF16, _ptr(workspace), workspace.numel(),
        _stream())
    _check(st, "nvfp4_w4a16_lora_gemm_dgrad")


def gemm_dgrad(dy, q: "QuantizedWeight", lora_a=None, lora_b=None, lora_scale=0.0, noise=None,
               out_dtype=torch.float32, workspace=None) -> torch.Tensor:
    """dX = (dY deq(W) + s (dY B) A) diag(z), the input gradient of gemm()."""
    M, N = dy.shape
    K = q.shape[1]
    r = 0 if lora_a is None else lora_a.shape[0]
    dx = torch.empty((M, K), dtype=out_dtype, device=dy.device)
    ws = workspace if workspace is not None else new_workspace(nvfp4_dgrad_workspace_bytes(M, N, K, r),
                                                              dy.device)
    nvfp4_w4a16_lora_gemm_dgrad(dy, q.codes, q.scales, q.tensor_scale, lora_a, lora_b, lora_scale, noise,
                                dx, ws)
    return dx


def nvfp4_lora_grads_workspace_bytes(M: int, N: int, K: int, r: int) -> int:
    return int(load().nvfp4_lora_grads_workspace_bytes(M, N, K, r))


def nvfp4_lora_grads(x: torch.Tensor, noise, dy: torch.Tensor, lora_a: torch.Tensor, lora_b: torch.Tensor,
                     lora_scale: float, grad_a: torch.Tensor, grad_b: torch.Tensor, workspace: torch.Tensor):
    M, K = x.shape
    N = dy.shape[1]
    r = lora_a.shape[0]
    _need(x, torch.bfloat16, (M, K), "x")
    _need(dy, torch.bfloat16, (M, N), "dy")
    _need(lora_a, torch.bfloat16, (r, K), "lora_a")
    _need(lora_b, torch.bfloat16, (N, r), "lora_b")
    _need(grad_a, torch.float32, (r, K), "grad_a")
    _need(grad_b, torch.float32, (N, r), "grad_b")
    if noise is not None:
        _need(noise, torch.float32, (K,), "noise")
    st = load().nvfp4_lora_grads(_ptr(x), _ptr(noise), _ptr(dy), M, N, K, _ptr(lora_a), _ptr(lora_b), r,
                                 float(lora_scale), _ptr(grad_a), _ptr(grad_b), _ptr(workspace),
                                 workspace.numel(), _stream())
    _check(st, "nvfp4_lora_grads")


def lora_grads(x, dy, lora_a, lora_b, lora_scale, noise=None, workspace=None):
    """(dA (r, K), dB (N, r)) float32: dA = s (dY B)^T X', dB = s dY^T (X' A^T)."""
    M, K = x.shape
    N = dy.shape[1]
    r = lora_a.shape[0]
    ga = torch.empty((r, K), dtype=torch.float32, device=x.device)
    gb = torch.empty((N, r), dtype=torch.float32, device=x.device)
    ws = workspace if workspace is not None else new_workspace(nvfp4_lora_grads_workspace_bytes(M, N, K, r),
                                                              x.device)
    nvfp4_lora_grads(x, noise, dy, lora_a, lora_b, lora_scale, ga, gb, ws)
    return ga, gb


def gemm_list(items, out_dtype=torch.float32, workspace=None):
    """items: (x, q, lora_a, lora_b, lora_scale, noise) tuples (q a QuantizedWeight; lora_a, lora_b,
    noise may be None).  Returns the list of outputs, each M x N."""
    entries = []
    for x, q, a, b, s, z in items:
        y = torch.empty((x.shape[0], q.shape[0]), dtype=out_dtype, device=x.device)
        entries.append((x, q.codes, q.scales, q.tensor_scale, a, b, s, z, y))
    ws = workspace if workspace is not None else new_workspace(nvfp4_gemm_list_workspace_bytes(entries),
                                                              entries[0][0].device)
    nvfp4_w4a16_lora_gemm_list(entries, ws)
    return [e[8] for e in entries]


def gemm(x, q: QuantizedWeight, lora_a=None, lora_b=None, lora_scale=0.0, noise=None,
         out_dtype=torch.float32, workspace=None) -> torch.Tensor:
    M, K = x.shape
    N = q.shape[0]
    r = 0 if lora_a is None else lora_a.shape[0]
    y = torch.empty((M, N), dtype=out_dtype, device=x.device)
    ws = workspace if workspace is not None else new_workspace(nvfp4_workspace_bytes(M, N, K, r),
                                                              x.device)
    nvfp4_w4a16_lora_gemm(x, q.codes, q.scales, q.tensor_scale, lora_a, lora_b, lora_scale, noise,
                          y, ws)
    return y
