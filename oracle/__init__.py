"""CPU oracle for the NVFP4 weight path (TEST INFRASTRUCTURE ONLY).

The arithmetic lives in ``nvfp4_oracle.c`` (plain C, brute-force encoders,
double-precision triple-loop GEMM).  This module only compiles it with gcc and
marshals numpy arrays through ctypes.  Only the tests, the smoke check and the
benchmark's CPU-baseline leg may import it; the product library never does,
and the two share no code.

Sources of each definition are cited in the C file's header.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "nvfp4_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

OK, NONFINITE, BAD_SHAPE = 0, 1, 2


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (-O2, no FP contraction) if it is stale."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".{os.getpid()}.tmp"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
             "-shared", "-pthread", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def _configure(lib):
    P = ctypes.c_void_p
    i64 = ctypes.c_int64
    lib.orc_bf16_to_f32.restype = ctypes.c_float
    lib.orc_bf16_to_f32.argtypes = [ctypes.c_uint16]
    lib.orc_f32_to_bf16.restype = ctypes.c_uint16
    lib.orc_f32_to_bf16.argtypes = [ctypes.c_float]
    lib.orc_e2m1_value.restype = ctypes.c_double
    lib.orc_e2m1_value.argtypes = [ctypes.c_int]
    lib.orc_e4m3_value.restype = ctypes.c_double
    lib.orc_e4m3_value.argtypes = [ctypes.c_int]
    lib.orc_e2m1_encode.restype = ctypes.c_int
    lib.orc_e2m1_encode.argtypes = [ctypes.c_float]
    lib.orc_e4m3_encode_nonneg.restype = ctypes.c_int
    lib.orc_e4m3_encode_nonneg.argtypes = [ctypes.c_float]
    lib.orc_quantize.restype = ctypes.c_int
    lib.orc_quantize.argtypes = [P, i64, i64, P, ctypes.c_int, P, P, ctypes.c_int]
    lib.orc_dequantize.restype = None
    lib.orc_dequantize.argtypes = [P, P, ctypes.c_float, i64, i64, P, P]
    lib.orc_round_scales.restype = ctypes.c_int
    lib.orc_round_scales.argtypes = [P, ctypes.c_float, i64, P]
    lib.orc_noisy_input.restype = None
    lib.orc_noisy_input.argtypes = [P, P, i64, i64, P]
    lib.orc_encode_array.restype = None
    lib.orc_encode_array.argtypes = [P, i64, ctypes.c_int, P, ctypes.c_int]
    lib.orc_gemm.restype = ctypes.c_int
    lib.orc_gemm.argtypes = [P, i64, i64, i64, P, P, ctypes.c_float, P, P, i64,
                             ctypes.c_float, P, P, ctypes.c_int]
    lib.orc_gemm_dgrad.restype = ctypes.c_int
    lib.orc_gemm_dgrad.argtypes = [P, i64, i64, i64, P, P, ctypes.c_float, P, P, i64,
                                   ctypes.c_float, P, P, ctypes.c_int]
    lib.orc_lora_grads.restype = ctypes.c_int
    lib.orc_lora_grads.argtypes = [P, P, P, i64, i64, i64, P, P, i64, ctypes.c_float, P, P, ctypes.c_int]
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _configure(ctypes.CDLL(build()))
        return _lib


def use_library(path):
    """Point this module at another build of the oracle source (the mutation
    tests load deliberately broken copies); ``None`` restores the default.
    Returns the previous handle."""
    global _lib
    with _lock:
        prev = _lib
        _lib = None if path is None else _configure(ctypes.CDLL(path))
        return prev


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def default_threads() -> int:
    return os.cpu_count() or 1


# ---------------------------------------------------------------- scalars
def bf16_to_f32(bits):
    bits = np.asarray(bits, dtype=np.uint16)
    lib = _load()
    return np.array([lib.orc_bf16_to_f32(int(b)) for b in bits.ravel()],
                    dtype=np.float32).reshape(bits.shape)


def f32_to_bf16(x):
    x = np.asarray(x, dtype=np.float32)
    lib = _load()
    return np.array([lib.orc_f32_to_bf16(float(v)) for v in x.ravel()],
                    dtype=np.uint16).reshape(x.shape)


def e2m1_value(code: int) -> float:
    return _load().orc_e2m1_value(int(code))


def e4m3_value(byte: int) -> float:
    return _load().orc_e4m3_value(int(byte))


def e2m1_encode(x: float) -> int:
    return _load().orc_e2m1_encode(float(np.float32(x)))


def e4m3_encode(x: float) -> int:
    return _load().orc_e4m3_encode_nonneg(float(np.float32(x)))


def encode_array(x, which, nthreads=None):
    """which 0: E2M1 codes (sign in bit 3); which 1: E4M3 bytes of x >= 0."""
    x = _c(x, np.float32).ravel()
    out = np.zeros(x.size, np.uint8)
    _load().orc_encode_array(_ptr(x), x.size, int(which), _ptr(out), nthreads or default_threads())
    return out


# ---------------------------------------------------------------- tensors
def quantize(w_bits, tensor_scale=None, nthreads=None):
    """w_bits: (N, K) uint16 bf16 patterns.  Returns (status, codes (N, K/2)
    uint8, scales (N, K/16) uint8, s_t float32)."""
    w = _c(w_bits, np.uint16)
    N, K = w.shape
    codes = np.zeros((N, K // 2), np.uint8)
    scales = np.zeros((N, max(K // 16, 0)), np.uint8)
    st = np.array([0.0 if tensor_scale is None else tensor_scale], np.float32)
    rc = _load().orc_quantize(_ptr(w), N, K, _ptr(st), int(tensor_scale is not None),
                              _ptr(codes), _ptr(scales), nthreads or default_threads())
    return rc, codes, scales, np.float32(st[0])


def dequantize(codes, scales, s_t):
    """Returns (fp32 (N, K), bf16 bits (N, K))."""
    codes = _c(codes, np.uint8)
    scales = _c(scales, np.uint8)
    N = codes.shape[0]
    K = codes.shape[1] * 2
    f = np.zeros((N, K), np.float32)
    b = np.zeros((N, K), np.uint16)
    _load().orc_dequantize(_ptr(codes), _ptr(scales), float(np.float32(s_t)), N, K,
                           _ptr(f), _ptr(b))
    return f, b


def round_scales(param, s_t):
    """Scale-only update: E4M3 bytes of param / s_t (same shape as param)."""
    p = _c(param, np.float32)
    out = np.zeros(p.shape, np.uint8)
    rc = _load().orc_round_scales(_ptr(p), float(np.float32(s_t)), p.size, _ptr(out))
    return rc, out


def noisy_input(x_bits, z):
    x = _c(x_bits, np.uint16)
    M, K = x.shape
    out = np.zeros((M, K), np.uint16)
    _load().orc_noisy_input(_ptr(x), _ptr(_c(z, np.float32)), M, K, _ptr(out))
    return out


def gemm(x_bits, codes, scales, s_t, a_bits=None, b_bits=None, lora_scale=0.0, z=None,
         nthreads=None):
    """Y (M, N) float64 = X' deq(W)^T + s (X' A^T) B^T."""
    x = _c(x_bits, np.uint16)
    codes = _c(codes, np.uint8)
    scales = _c(scales, np.uint8)
    M, K = x.shape
    N = codes.shape[0]
    A = _c(a_bits, np.uint16)
    B = _c(b_bits, np.uint16)
    r = 0 if A is None or B is None else A.shape[0]
    y = np.zeros((M, N), np.float64)
    rc = _load().orc_gemm(_ptr(x), M, N, K, _ptr(codes), _ptr(scales),
                          float(np.float32(s_t)), _ptr(A), _ptr(B), r, float(lora_scale),
                          _ptr(_c(z, np.float32)), _ptr(y), nthreads or default_threads())
    if rc != OK:
        raise ValueError(f"oracle gemm status {rc}")
    return y


def gemm_dgrad(dy_bits, codes, scales, s_t, a_bits=None, b_bits=None, lora_scale=0.0, z=None,
               nthreads=None):
    """dX (M, K) float64 = (dY deq(W) + s (dY B) A) diag(z): the gradient of
    gemm() with respect to its input, the bf16 rounding of X' taken as the
    identity."""
    dy = _c(dy_bits, np.uint16)
    codes = _c(codes, np.uint8)
    scales = _c(scales, np.uint8)
    M, N = dy.shape
    K = codes.shape[1] * 2
    if codes.shape[0] != N:
        raise ValueError("dY columns must match the weight rows")
    A = _c(a_bits, np.uint16)
    B = _c(b_bits, np.uint16)
    r = 0 if A is None or B is None else A.shape[0]
    dx = np.zeros((M, K), np.float64)
    rc = _load().orc_gemm_dgrad(_ptr(dy), M, N, K, _ptr(codes), _ptr(scales),
                                float(np.float32(s_t)), _ptr(A), _ptr(B), r, float(lora_scale),
                                _ptr(_c(z, np.float32)), _ptr(dx), nthreads or default_threads())
    if rc != OK:
        raise ValueError(f"oracle dgrad status {rc}")
    return dx


def lora_grads(x_bits, dy_bits, a_bits, b_bits, lora_scale, z=None, nthreads=None):
    """(dA (r, K), dB (N, r)) float64: dA = s (dY B)^T X', dB = s dY^T (X' A^T),
    X' = bf16(X z)."""
    x = _c(x_bits, np.uint16)
    dy = _c(dy_bits, np.uint16)
    A = _c(a_bits, np.uint16)
    B = _c(b_bits, np.uint16)
    M, K = x.shape
    N = dy.shape[1]
    r = A.shape[0]
    if dy.shape[0] != M or A.shape[1] != K or B.shape != (N, r):
        raise ValueError("shapes do not match")
    da = np.zeros((r, K), np.float64)
    db = np.zeros((N, r), np.float64)
    rc = _load().orc_lora_grads(_ptr(x), _ptr(_c(z, np.float32)), _ptr(dy), M, N, K, _ptr(A), _ptr(B), r,
                                float(lora_scale), _ptr(da), _ptr(db), nthreads or default_threads())
    if rc != OK:
        raise ValueError(f"oracle lora_grads status {rc}")
    return da, db
