"""Pins for the oracle's input gradient of the W4A16 + LoRA + noise layer (CPU).

Only the LoRA factors are trained; the quantised weight is frozen and the
gradient flows through the layer to the layers below ("RL with NVFP4 + LoRA"
post, section "Метод").  For Y = X' deq(W)^T + s (X' A^T) B^T with
X' = X z, the input gradient is dX = (dY deq(W) + s (dY B) A) diag(z), the
bf16 rounding of X' taken as the identity.

Anchors, none of them the oracle's own formula:
  * the adjoint identity <dY, Y(X)> = <dX, X> between the (separately pinned)
    forward oracle and the gradient, on dyadic inputs where both are exact in
    double, compared in exact rationals;
  * float64 autograd of the same layer written with torch operations;
  * exact rational brute force on tiny shapes;
  * degenerate cases (no LoRA, s = 0, z = 1, one row of a batch).
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

from nvfp4_weight_only_02_gb300 import synth
from tests.test_oracle_gemm import E2M1_MAG, _dec_e4m3, _dequant_exact


def _dyadic_case(M, N, K, r, seed):
    """Small-integer X and dY, power-of-two block scales, s_t = 1, A and B in
    multiples of 1/8, z and s powers of two: every product and partial sum of
    both the forward and the gradient is exact in double."""
    g = np.random.default_rng(seed)
    x = g.integers(-8, 9, size=(M, K)).astype(np.float32)
    dy = g.integers(-8, 9, size=(M, N)).astype(np.float32)
    q = g.integers(0, 16, size=(N, K))
    e = g.choice([0x20, 0x28, 0x30, 0x38, 0x40], size=(N, K // 16)).astype(np.uint8)
    codes = (q[:, 0::2] | (q[:, 1::2] << 4)).astype(np.uint8)
    a = (g.integers(-8, 9, size=(r, K)) / 8.0).astype(np.float32)
    b = (g.integers(-8, 9, size=(N, r)) / 8.0).astype(np.float32)
    z = (2.0 ** g.integers(-2, 3, size=K)).astype(np.float32)
    bf = synth.to_bf16_bits
    return bf(x), bf(dy), codes, e, bf(a), bf(b), z


@pytest.mark.parametrize("M,N,K,r", [(3, 16, 64, 4), (5, 40, 128, 8), (1, 8, 32, 0)])
def test_adjoint_identity_exact(orc, M, N, K, r):
    x, dy, codes, e, a, b, z = _dyadic_case(M, N, K, r, seed=M * 100 + N + K)
    s = 2.0
    la, lb = (a, b) if r else (None, None)
    y = orc.gemm(x, codes, e, np.float32(1.0), la, lb, s, z)
    dx = orc.gemm_dgrad(dy, codes, e, np.float32(1.0), la, lb, s, z)
    F = Fraction
    dyf = synth.bf16_bits_to_f32(dy)
    xf = synth.bf16_bits_to_f32(x)
    lhs = sum(F(float(dyf[m, n])) * F(float(y[m, n])) for m in range(M) for n in range(N))
    rhs = sum(F(float(dx[m, k])) * F(float(xf[m, k])) for m in range(M) for k in range(K))
    assert lhs == rhs
    assert lhs != 0


@pytest.mark.parametrize("with_lora,with_noise", [(True, True), (True, False), (False, True)])
def test_matches_float64_autograd(orc, with_lora, with_noise):
    M, N, K, r = 4, 48, 96, 8
    c = synth.small_case(M, N, K, r, seed=77, with_lora=with_lora, with_noise=with_noise)
    rc, codes, scales, st = orc.quantize(c.w)
    dy = synth.activations(M, N, 78)
    dx = orc.gemm_dgrad(dy, codes, scales, st, c.a, c.b, c.lora_scale, c.z)

    X = torch.tensor(synth.bf16_bits_to_f32(c.x), dtype=torch.float64, requires_grad=True)
    D = torch.from_numpy(_dequant_exact(codes, scales, st))
    xp = X * torch.from_numpy(c.z).double() if c.z is not None else X
    Y = xp @ D.T
    if c.a is not None:
        A = torch.from_numpy(synth.bf16_bits_to_f32(c.a)).double()
        B = torch.from_numpy(synth.bf16_bits_to_f32(c.b)).double()
        Y = Y + c.lora_scale * (xp @ A.T) @ B.T
    Y.backward(torch.from_numpy(synth.bf16_bits_to_f32(dy)).double())
    ref = X.grad.numpy()
    assert np.allclose(dx, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())


def _fraction_dgrad(dy_bits, codes, scales, st, a_bits, b_bits, s, z):
    dyv = synth.bf16_bits_to_f32(dy_bits)
    M, N = dyv.shape
    K = codes.shape[1] * 2
    F = Fraction

    def w(n, k):
        q = (int(codes[n, k // 2]) >> (4 * (k % 2))) & 15
        v = F(E2M1_MAG[q & 7]) * (-1 if q & 8 else 1)
        return v * F(_dec_e4m3(scales[n, k // 16])) * F(float(st))

    G = [[F(float(dyv[m, n])) for n in range(N)] for m in range(M)]
    out = [[sum(G[m][n] * w(n, k) for n in range(N)) for k in range(K)] for m in range(M)]
    if a_bits is not None:
        A = synth.bf16_bits_to_f32(a_bits)
        B = synth.bf16_bits_to_f32(b_bits)
        r = A.shape[0]
        U = [[sum(G[m][n] * F(float(B[n, j])) for n in range(N)) for j in range(r)] for m in range(M)]
        for m in range(M):
            for k in range(K):
                out[m][k] += F(float(s)) * sum(U[m][j] * F(float(A[j, k])) for j in range(r))
    if z is not None:
        out = [[v * F(float(z[k])) for k, v in enumerate(row)] for row in out]
    return np.array([[float(v) for v in row] for row in out])


@pytest.mark.parametrize("M,N,K,r", [(1, 4, 16, 0), (2, 6, 32, 3), (3, 5, 48, 2)])
def test_vs_exact_rationals(orc, M, N, K, r):
    c = synth.small_case(M, N, K, r, seed=300 + M + N + K, with_lora=r > 0)
    rc, codes, scales, st = orc.quantize(c.w)
    dy = synth.activations(M, N, 301)
    dx = orc.gemm_dgrad(dy, codes, scales, st, c.a, c.b, c.lora_scale, c.z)
    ref = _fraction_dgrad(dy, codes, scales, st, c.a, c.b, c.lora_scale, c.z)
    assert np.allclose(dx, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())


def test_degenerate_cases(orc):
    M, N, K, r = 4, 32, 64, 4
    c = synth.small_case(M, N, K, r, seed=51)
    rc, codes, scales, st = orc.quantize(c.w)
    dy = synth.activations(M, N, 52)
    base = orc.gemm_dgrad(dy, codes, scales, st)
    assert np.array_equal(orc.gemm_dgrad(dy, codes, scales, st, np.zeros_like(c.a), c.b, 2.0), base)
    assert np.array_equal(orc.gemm_dgrad(dy, codes, scales, st, c.a, c.b, 0.0), base)
    assert np.array_equal(orc.gemm_dgrad(dy, codes, scales, st, z=np.ones(K, np.float32)), base)
    full = orc.gemm_dgrad(dy, codes, scales, st, c.a, c.b, 2.0, c.z)
    for m in range(M):
        one = orc.gemm_dgrad(dy[m:m + 1], codes, scales, st, c.a, c.b, 2.0, c.z)
        assert np.array_equal(one[0], full[m])
    # the base term is dY times the dequantised weight (not its transpose)
    ref = synth.bf16_bits_to_f32(dy).astype(np.float64) @ _dequant_exact(codes, scales, st)
    assert np.allclose(base, ref, rtol=1e-12, atol=1e-14)
