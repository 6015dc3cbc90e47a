"""Pins for the oracle's W4A16 GEMM with parallel LoRA and input noise (CPU).

Y = X' deq(W)^T + s (X' A^T) B^T with X' = bf16(X * z): weight-only
quantisation keeps activations 16-bit, the LoRA adapter runs in parallel as
in QLoRA, and the noise is applied through the RMSNorm gain, which equals
multiplicative weight noise ("RL with NVFP4 + LoRA" post, section "Метод").

Anchors: exact rational brute force on tiny shapes, an exact dyadic case,
power-of-two noise that must equal pre-scaled inputs and W diag(z), and the
degenerate cases (no LoRA, s = 0, z = 1, M = 1).
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

from nvfp4_weight_only_02_gb300 import synth

E2M1_MAG = [0, 0.5, 1, 1.5, 2, 3, 4, 6]


def _dec_e4m3(b):
    return float(torch.tensor([int(b)], dtype=torch.uint8).view(torch.float8_e4m3fn).float())


def _dequant_exact(codes, scales, st):
    """D = v(q) * dec(e) * s_t in float64 (exact: at most 30 significant bits)."""
    q = np.stack([codes & 15, codes >> 4], axis=-1).reshape(codes.shape[0], -1)
    v = np.where(q >= 8, -1.0, 1.0) * np.array(E2M1_MAG)[q & 7]
    dec = torch.from_numpy(scales).view(torch.float8_e4m3fn).double().numpy()
    return v * np.repeat(dec, 16, axis=1) * float(st)


def _xprime_torch(x_bits, z):
    x = torch.from_numpy(synth.bf16_bits_to_f32(x_bits))
    if z is None:
        return x.double().numpy()
    return (x * torch.from_numpy(z)).to(torch.bfloat16).double().numpy()


def _fraction_gemm(x_bits, codes, scales, st, a_bits, b_bits, s, z):
    xp = _xprime_torch(x_bits, z)
    M, K = xp.shape
    N = codes.shape[0]
    F = Fraction
    D = [[F(E2M1_MAG[((codes[n, k // 2] >> (4 * (k % 2))) & 7)])
          * (-1 if ((codes[n, k // 2] >> (4 * (k % 2))) & 8) else 1)
          * F(_dec_e4m3(scales[n, k // 16])) * F(float(st)) for k in range(K)] for n in range(N)]
    X = [[F(float(xp[m, k])) for k in range(K)] for m in range(M)]
    Y = [[sum(X[m][k] * D[n][k] for k in range(K)) for n in range(N)] for m in range(M)]
    if a_bits is not None:
        A = synth.bf16_bits_to_f32(a_bits)
        B = synth.bf16_bits_to_f32(b_bits)
        r = A.shape[0]
        T = [[sum(X[m][k] * F(float(A[j, k])) for k in range(K)) for j in range(r)] for m in range(M)]
        for m in range(M):
            for n in range(N):
                Y[m][n] += F(float(s)) * sum(T[m][j] * F(float(B[n, j])) for j in range(r))
    return np.array([[float(v) for v in row] for row in Y])


@pytest.mark.parametrize("M,N,K,r", [(1, 4, 16, 0), (3, 5, 32, 2), (2, 8, 48, 4)])
def test_gemm_vs_exact_rationals(orc, M, N, K, r):
    c = synth.small_case(M, N, K, r, seed=100 + M + N + K, with_lora=r > 0)
    rc, codes, scales, st = orc.quantize(c.w)
    y = orc.gemm(c.x, codes, scales, st, c.a, c.b, c.lora_scale, c.z)
    ref = _fraction_gemm(c.x, codes, scales, st, c.a, c.b, c.lora_scale, c.z)
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())


def test_gemm_dyadic_is_exact(orc):
    """Small-integer activations, power-of-two block scales and s_t = 1: every
    product and partial sum is an integer multiple of 2^-10, so double
    precision holds the exact result, checked with integer arithmetic."""
    g = np.random.default_rng(7)
    M, N, K = 4, 16, 64
    x = g.integers(-8, 9, size=(M, K)).astype(np.float32)
    q = g.integers(0, 16, size=(N, K))
    e = g.choice([0x20, 0x28, 0x30, 0x38, 0x40], size=(N, K // 16))  # 2^-3 .. 2^1
    codes = (q[:, 0::2] | (q[:, 1::2] << 4)).astype(np.uint8)
    y = orc.gemm(synth.to_bf16_bits(x), codes, e.astype(np.uint8), np.float32(1.0))
    v4 = np.where(q >= 8, -1, 1) * (np.array(E2M1_MAG)[q & 7] * 2).astype(np.int64)  # 2v
    dec_i = np.array([{0x20: 1, 0x28: 2, 0x30: 4, 0x38: 8, 0x40: 16}[b] for b in e.ravel()]).reshape(e.shape)
    d_int = v4 * np.repeat(dec_i, 16, axis=1)  # = D * 16
    ref = (x.astype(np.int64) @ d_int.T).astype(np.float64) / 16.0
    assert np.array_equal(y, ref)


def test_power_of_two_noise_equals_prescaled_input_and_scaled_weight(orc):
    c = synth.small_case(3, 12, 64, 4, seed=31)
    g = np.random.default_rng(32)
    z = (2.0 ** g.integers(-2, 3, size=64)).astype(np.float32)
    rc, codes, scales, st = orc.quantize(c.w)
    y_noise = orc.gemm(c.x, codes, scales, st, c.a, c.b, c.lora_scale, z)
    xz = synth.to_bf16_bits(synth.bf16_bits_to_f32(c.x) * z)  # exact: z is 2^j
    y_pre = orc.gemm(xz, codes, scales, st, c.a, c.b, c.lora_scale, None)
    assert np.array_equal(y_noise, y_pre)
    # multiplicative weight noise: X (W diag z)^T, base term, in float64
    D = _dequant_exact(codes, scales, st)
    xf = synth.bf16_bits_to_f32(c.x).astype(np.float64)
    y_base = orc.gemm(c.x, codes, scales, st, None, None, 0.0, z)
    assert np.allclose(y_base, xf @ (D * z).T, rtol=1e-12, atol=1e-14)


def test_degenerate_cases(orc):
    c = synth.small_case(4, 16, 64, 4, seed=41)
    rc, codes, scales, st = orc.quantize(c.w)
    base = orc.gemm(c.x, codes, scales, st)
    # LoRA off by A = 0, by s = 0, or by passing no adapter
    zero_a = np.zeros_like(c.a)
    assert np.array_equal(orc.gemm(c.x, codes, scales, st, zero_a, c.b, 2.0), base)
    assert np.array_equal(orc.gemm(c.x, codes, scales, st, c.a, c.b, 0.0), base)
    # z == 1 is the noiseless path
    ones = np.ones(64, np.float32)
    assert np.array_equal(orc.gemm(c.x, codes, scales, st, z=ones), base)
    # M = 1 is one row of the batched result
    full = orc.gemm(c.x, codes, scales, st, c.a, c.b, 2.0, c.z)
    for m in range(4):
        one = orc.gemm(c.x[m:m + 1], codes, scales, st, c.a, c.b, 2.0, c.z)
        assert np.array_equal(one[0], full[m])
    # the base term is linear in the dequantised weights
    ref = synth.bf16_bits_to_f32(c.x).astype(np.float64) @ _dequant_exact(codes, scales, st).T
    assert np.allclose(base, ref, rtol=1e-12, atol=1e-14)
