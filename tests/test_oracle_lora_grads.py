"""Pins for the oracle's LoRA gradients (CPU).

Only A and B are trained ("RL with NVFP4 + LoRA" post, section "Метод").  For
the LoRA term s (X' A^T) B^T of the layer, dB = s dY^T (X' A^T) and
dA = s (dY B)^T X', X' = bf16(X z).

Anchors, none of them the oracle's own formula:
  * the forward oracle (separately pinned) is linear in A and in B apart, so on
    dyadic inputs where everything is exact in double,
        <dY, Y(A + dA', B)> - <dY, Y(A, B)> = <dA, dA'>   and the same for B,
    compared in exact rationals;
  * float64 autograd of the LoRA term written with torch operations;
  * exact rational brute force on tiny shapes; degenerate cases.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

from nvfp4_weight_only_02_gb300 import synth


def _dyadic(M, N, K, r, seed):
    g = np.random.default_rng(seed)
    bf = synth.to_bf16_bits
    x = bf(g.integers(-8, 9, size=(M, K)).astype(np.float32))
    dy = bf(g.integers(-8, 9, size=(M, N)).astype(np.float32))
    a = bf((g.integers(-8, 9, size=(r, K)) / 8.0).astype(np.float32))
    b = bf((g.integers(-8, 9, size=(N, r)) / 8.0).astype(np.float32))
    da = bf((g.integers(-4, 5, size=(r, K)) / 4.0).astype(np.float32))
    db = bf((g.integers(-4, 5, size=(N, r)) / 4.0).astype(np.float32))
    z = (2.0 ** g.integers(-2, 3, size=K)).astype(np.float32)
    q = g.integers(0, 16, size=(N, K))
    codes = (q[:, 0::2] | (q[:, 1::2] << 4)).astype(np.uint8)
    e = g.choice([0x30, 0x38, 0x40], size=(N, K // 16)).astype(np.uint8)
    return x, dy, a, b, da, db, z, codes, e


def _inner(u, v):
    return sum(Fraction(float(p)) * Fraction(float(q)) for p, q in zip(u.ravel(), v.ravel()))


@pytest.mark.parametrize("M,N,K,r", [(3, 16, 64, 4), (5, 24, 96, 8)])
def test_linear_in_each_factor_exact(orc, M, N, K, r):
    x, dy, a, b, da, db, z, codes, e = _dyadic(M, N, K, r, seed=M * 10 + r)
    s = 2.0
    one = np.float32(1.0)
    ga, gb = orc.lora_grads(x, dy, a, b, s, z)
    f = lambda aa, bb: orc.gemm(x, codes, e, one, aa, bb, s, z)
    plus = lambda u, v: synth.to_bf16_bits(synth.bf16_bits_to_f32(u) + synth.bf16_bits_to_f32(v))
    dyf = synth.bf16_bits_to_f32(dy)
    base = _inner(dyf, f(a, b))
    lhs_a = _inner(dyf, f(plus(a, da), b)) - base
    lhs_b = _inner(dyf, f(a, plus(b, db))) - base
    assert lhs_a == _inner(ga, synth.bf16_bits_to_f32(da)) and lhs_a != 0
    assert lhs_b == _inner(gb, synth.bf16_bits_to_f32(db)) and lhs_b != 0


@pytest.mark.parametrize("noise", [True, False])
def test_matches_float64_autograd(orc, noise):
    M, N, K, r = 6, 40, 96, 8
    c = synth.small_case(M, N, K, r, seed=91, with_noise=noise)
    dy = synth.activations(M, N, 92)
    ga, gb = orc.lora_grads(c.x, dy, c.a, c.b, c.lora_scale, c.z)
    xp = torch.from_numpy(synth.bf16_bits_to_f32(c.x))
    if c.z is not None:
        xp = (xp * torch.from_numpy(c.z)).to(torch.bfloat16).float()
    xp = xp.double()
    A = torch.tensor(synth.bf16_bits_to_f32(c.a), dtype=torch.float64, requires_grad=True)
    B = torch.tensor(synth.bf16_bits_to_f32(c.b), dtype=torch.float64, requires_grad=True)
    Y = c.lora_scale * (xp @ A.T) @ B.T
    Y.backward(torch.from_numpy(synth.bf16_bits_to_f32(dy)).double())
    for got, ref in ((ga, A.grad.numpy()), (gb, B.grad.numpy())):
        assert np.allclose(got, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())


def test_vs_exact_rationals(orc):
    M, N, K, r = 2, 5, 32, 3
    c = synth.small_case(M, N, K, r, seed=93)
    dy = synth.activations(M, N, 94)
    ga, gb = orc.lora_grads(c.x, dy, c.a, c.b, c.lora_scale, c.z)
    F = Fraction
    xp = (torch.from_numpy(synth.bf16_bits_to_f32(c.x)) * torch.from_numpy(c.z)).to(torch.bfloat16).double()
    X = [[F(float(xp[m, k])) for k in range(K)] for m in range(M)]
    A = synth.bf16_bits_to_f32(c.a)
    B = synth.bf16_bits_to_f32(c.b)
    G = synth.bf16_bits_to_f32(dy)
    s = F(c.lora_scale)
    T = [[sum(X[m][k] * F(float(A[j, k])) for k in range(K)) for j in range(r)] for m in range(M)]
    U = [[sum(F(float(G[m, n])) * F(float(B[n, j])) for n in range(N)) for j in range(r)] for m in range(M)]
    rb = np.array([[float(s * sum(F(float(G[m, n])) * T[m][j] for m in range(M))) for j in range(r)]
                   for n in range(N)])
    ra = np.array([[float(s * sum(U[m][j] * X[m][k] for m in range(M))) for k in range(K)] for j in range(r)])
    assert np.allclose(ga, ra, rtol=1e-12, atol=1e-12 * np.abs(ra).max())
    assert np.allclose(gb, rb, rtol=1e-12, atol=1e-12 * np.abs(rb).max())


def test_degenerate_cases(orc):
    M, N, K, r = 4, 32, 64, 4
    c = synth.small_case(M, N, K, r, seed=95)
    dy = synth.activations(M, N, 96)
    ga, gb = orc.lora_grads(c.x, dy, c.a, c.b, 2.0, c.z)
    za, zb = orc.lora_grads(c.x, dy, c.a, c.b, 0.0, c.z)
    assert not za.any() and not zb.any()
    ha, hb = orc.lora_grads(c.x, dy, c.a, c.b, 4.0, c.z)
    assert np.array_equal(ha, 2 * ga) and np.array_equal(hb, 2 * gb)
    ya, yb = orc.lora_grads(c.x, np.zeros_like(dy), c.a, c.b, 2.0, c.z)
    assert not ya.any() and not yb.any()
    # dB with B's rows permuted follows the permutation; dA is the sum over tokens
    perm = np.random.default_rng(97).permutation(N)
    pa, pb = orc.lora_grads(c.x, dy[:, perm], c.a, c.b[perm], 2.0, c.z)
    assert np.allclose(pb, gb[perm], rtol=1e-13) and np.allclose(pa, ga, rtol=1e-12)
    parts = [orc.lora_grads(c.x[m:m + 1], dy[m:m + 1], c.a, c.b, 2.0, c.z) for m in range(M)]
    assert np.allclose(sum(p[0] for p in parts), ga, rtol=1e-12, atol=1e-15)
    assert np.allclose(sum(p[1] for p in parts), gb, rtol=1e-12, atol=1e-15)
