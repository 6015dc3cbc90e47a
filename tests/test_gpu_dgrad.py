"""Input gradient of the W4A16 + LoRA + noise layer on the GPU vs the oracle.

dX = (dY deq(W) + s (dY B) A) diag(z) ("RL with NVFP4 + LoRA" post, section
"Метод": the quantised weight is frozen, the gradient flows through it).  Same
gate as the forward GEMM tests: normwise max rel <= 1e-2 and mean rel <= 1e-3
against the FP64 oracle on FP32 output, plus the per-element FP32 accumulation
bound (N + r + 64) 2^-23 |dY| |deq(W)| (+ the LoRA magnitudes).  Full-size
layer shapes are compared on sampled rows, which the oracle computes one by
one.
"""
import dataclasses

import numpy as np
import pytest
import torch

from nvfp4_weight_only_02_gb300 import synth
from tests.test_gpu_gemm import _check, _dev, _quantize_both

pytestmark = pytest.mark.gpu


def _abs_bound(orc, dy, codes, scales, st, a, b, s, z):
    return orc.gemm_dgrad(dy & 0x7FFF, codes & 0x77, scales, st,
                          None if a is None else a & 0x7FFF, None if b is None else b & 0x7FFF,
                          abs(s), None if z is None else np.abs(z))


def _run(nv, dy, q, a, b, s, z, out_dtype=torch.float32):
    dx = nv.gemm_dgrad(_dev(dy), q, None if a is None else _dev(a), None if b is None else _dev(b), s,
                       None if z is None else torch.from_numpy(z).cuda(), out_dtype=out_dtype)
    torch.cuda.synchronize()
    return dx


CASES = [
    # M, N, K, r, lora, noise
    (1, 64, 64, 0, False, False),
    (5, 128, 192, 8, True, True),
    (64, 256, 512, 16, True, False),
    (200, 320, 1024, 32, True, True),
    (333, 512, 640, 64, True, True),
    (130, 192, 2048, 40, True, True),
    (17, 1024, 256, 5, True, True),
]


@pytest.mark.parametrize("M,N,K,r,lora,noise", CASES)
def test_dgrad_shapes(nv, orc, M, N, K, r, lora, noise):
    c = synth.small_case(M, N, K, r, seed=M + 3 * N + K, with_lora=lora, with_noise=noise)
    dy = synth.activations(M, N, M + N, std=0.1)
    q, codes, scales, st = _quantize_both(nv, orc, c.w)
    dx = _run(nv, dy, q, c.a, c.b, c.lora_scale, c.z).cpu().numpy()
    ref = orc.gemm_dgrad(dy, codes, scales, st, c.a, c.b, c.lora_scale, c.z)
    _check(dx, ref, _abs_bound(orc, dy, codes, scales, st, c.a, c.b, c.lora_scale, c.z), N, r if lora else 0)
    dxb = _run(nv, dy, q, c.a, c.b, c.lora_scale, c.z, torch.bfloat16)
    assert torch.equal(dxb.cpu(), torch.from_numpy(dx).to(torch.bfloat16))


@pytest.mark.parametrize("w_std", [1e-37, 1e-12, 1e30])
def test_dgrad_extreme_tensor_scale(nv, orc, w_std):
    M, N, K, r = 96, 256, 320, 16
    c = synth.small_case(M, N, K, r, seed=61, w_std=w_std)
    dy = synth.activations(M, N, 62)
    q, codes, scales, st = _quantize_both(nv, orc, c.w)
    dx = _run(nv, dy, q, c.a, c.b, c.lora_scale, c.z).cpu().numpy()
    assert np.isfinite(dx).all()
    ref = orc.gemm_dgrad(dy, codes, scales, st, c.a, c.b, c.lora_scale, c.z)
    _check(dx, ref, _abs_bound(orc, dy, codes, scales, st, c.a, c.b, c.lora_scale, c.z), N, r,
           floor=2.0 ** -140)


def test_dgrad_extreme_row_magnitudes(nv, orc):
    """Rows of dY scaled by 2^k from 2^-120 to 2^100 (and a zero row) take
    the rescaled path of the token-side kernel; each row is checked on its
    own scale."""
    M, N, K, r = 72, 384, 256, 8
    c = synth.small_case(M, N, K, r, seed=71)
    g = synth.bf16_bits_to_f32(synth.activations(M, N, 72)).astype(np.float64)
    exps = [None, -120, -70, -40, 0, 20, 40, 100]
    for i in range(M):
        e = exps[i % len(exps)]
        g[i] = 0.0 if e is None else g[i] * 2.0 ** e
    dy = synth.to_bf16_bits(g.astype(np.float32))
    q, codes, scales, st = _quantize_both(nv, orc, c.w)
    dx = _run(nv, dy, q, c.a, c.b, c.lora_scale, c.z).cpu().numpy()
    assert np.isfinite(dx).all()
    ref = orc.gemm_dgrad(dy, codes, scales, st, c.a, c.b, c.lora_scale, c.z)
    absref = _abs_bound(orc, dy, codes, scales, st, c.a, c.b, c.lora_scale, c.z)
    for i in range(M):
        if exps[i % len(exps)] is None:
            assert not dx[i].any()
        else:
            _check(dx[i:i + 1], ref[i:i + 1], absref[i:i + 1], N, r, floor=2.0 ** -140)


def test_dgrad_is_the_adjoint_of_the_forward(nv):
    """<dY, Y(X)> = <dX, X> up to FP32 rounding, both sides computed by the
    library (noise off, so X' = X exactly)."""
    M, N, K, r = 256, 512, 768, 16
    c = synth.small_case(M, N, K, r, seed=81, with_noise=False)
    dy = synth.activations(M, N, 82)
    q = nv.quantize(_dev(c.w))
    y = nv.gemm(_dev(c.x), q, _dev(c.a), _dev(c.b), c.lora_scale).double()
    dx = _run(nv, dy, q, c.a, c.b, c.lora_scale, None).double()
    x = _dev(c.x).double()
    dyd = _dev(dy).double()
    lhs, rhs = (dyd * y).sum().item(), (dx * x).sum().item()
    scale = (dyd.abs() * y.abs()).sum().item()
    assert abs(lhs - rhs) <= 1e-5 * scale


FULL = [
    # model, projection, M, rows checked
    ("7b", "up", 16384, 24),
    ("7b", "down", 4096, 16),
    ("32b", "up", 4096, 16),
    ("32b", "down", 2048, 12),
]


@pytest.mark.parametrize("model,proj,M,nrows", FULL)
def test_dgrad_full_size_sampled_rows(nv, orc, model, proj, M, nrows):
    shape = {("7b", "up"): synth.QWEN7B_UP, ("7b", "down"): synth.QWEN7B_DOWN,
             ("32b", "up"): synth.QWEN32B_UP, ("32b", "down"): synth.QWEN32B_DOWN}[(model, proj)]
    N, K = shape
    r = 32 if model == "7b" else 64
    w = synth.normal_weight((N, K), 0.02, 1, outlier_frac=1e-3)
    a, b = synth.lora_pair(N, K, r, 0.01, 3)
    z = synth.noise_vector(K, 5e-4, 4)
    dy = synth.activations(M, N, 5, std=1e-3)
    q, codes, scales, st = _quantize_both(nv, orc, w)
    dx = _run(nv, dy, q, a, b, 2.0, z).cpu().numpy()
    rows = np.sort(np.random.default_rng(6).choice(M, size=nrows, replace=False))
    rows[0] = 0
    rows[-1] = M - 1
    ref = orc.gemm_dgrad(dy[rows], codes, scales, st, a, b, 2.0, z)
    absref = _abs_bound(orc, dy[rows], codes, scales, st, a, b, 2.0, z)
    _check(dx[rows], ref, absref, N, r)
