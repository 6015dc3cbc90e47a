"""Gradients of the LoRA factors on the GPU vs the oracle.

dB = s dY^T (X' A^T) and dA = s (dY B)^T X', X' = bf16(X z): the parameters
the RL post trains on a frozen NVFP4 weight ("RL with NVFP4 + LoRA", section
"Метод").  Gate as for the GEMMs: normwise max rel <= 1e-2 and mean rel
<= 1e-3 against the FP64 oracle, plus a per-element bound of
(M + N + K + 256) 2^-23 times the same sums over magnitudes (the token sums and
the X' A^T, dY B rows both accumulate in FP32).
"""
import dataclasses

import numpy as np
import pytest
import torch

from nvfp4_weight_only_02_gb300 import synth
from tests.test_gpu_gemm import _check, _dev

pytestmark = pytest.mark.gpu


def _run_and_check(nv, orc, x, dy, a, b, s, z, floor=1e-30):
    M, K = x.shape
    N = dy.shape[1]
    zd = None if z is None else torch.from_numpy(z).cuda()
    ga, gb = nv.lora_grads(_dev(x), _dev(dy), _dev(a), _dev(b), s, zd)
    torch.cuda.synchronize()
    ra, rb = orc.lora_grads(x, dy, a, b, s, z)
    aa, ab = orc.lora_grads(x & 0x7FFF, dy & 0x7FFF, a & 0x7FFF, b & 0x7FFF, abs(s),
                            None if z is None else np.abs(z))
    n = M + N + K + 256 - 64  # _check adds 64 to its K + r
    _check(ga.cpu().numpy(), ra, aa, n, 0, floor)
    _check(gb.cpu().numpy(), rb, ab, n, 0, floor)
    return ga, gb


CASES = [
    # M, N, K, r, noise
    (1, 64, 64, 1, False),
    (5, 128, 192, 8, True),
    (70, 256, 320, 16, True),
    (200, 320, 1024, 32, True),
    (333, 512, 192, 64, False),
    (130, 192, 640, 40, True),
    (1000, 64, 128, 5, True),
]


@pytest.mark.parametrize("M,N,K,r,noise", CASES)
def test_lora_grads_shapes(nv, orc, M, N, K, r, noise):
    c = synth.small_case(M, N, K, r, seed=7 * M + N + K, with_noise=noise)
    dy = synth.activations(M, N, M + K, std=0.1)
    ga, gb = _run_and_check(nv, orc, c.x, dy, c.a, c.b, c.lora_scale, c.z)
    # a second call with the same workspace-free path gives the same bits
    ga2, gb2 = nv.lora_grads(_dev(c.x), _dev(dy), _dev(c.a), _dev(c.b), c.lora_scale,
                             None if c.z is None else torch.from_numpy(c.z).cuda())
    assert torch.equal(ga, ga2) and torch.equal(gb, gb2)


def test_lora_grads_extreme_token_magnitudes(nv, orc):
    """Tokens of X scaled by 2^k from 2^-120 to 2^40 and tokens of dY from
    2^-70 to 2^50 (and zero tokens) take the rescaled path of the token-side
    kernel on both sides; every true sum stays inside the FP32 range."""
    M, N, K, r = 72, 256, 320, 8
    c = synth.small_case(M, N, K, r, seed=301)
    xs = synth.bf16_bits_to_f32(c.x).astype(np.float64)
    gs = synth.bf16_bits_to_f32(synth.activations(M, N, 302)).astype(np.float64)
    ex_x = [None, -120, -70, -40, 0, 20, 40, 30]
    ex_dy = [0, 36, -30, 50, None, -70, 10, 40]
    for i in range(M):
        e1, e2 = ex_x[i % 8], ex_dy[(3 * i + 1) % 8]
        xs[i] = 0.0 if e1 is None else xs[i] * 2.0 ** e1
        gs[i] = 0.0 if e2 is None else gs[i] * 2.0 ** e2
    x = synth.to_bf16_bits(xs.astype(np.float32))
    dy = synth.to_bf16_bits(gs.astype(np.float32))
    ga, gb = nv.lora_grads(_dev(x), _dev(dy), _dev(c.a), _dev(c.b), c.lora_scale, torch.from_numpy(c.z).cuda())
    torch.cuda.synchronize()
    assert torch.isfinite(ga).all() and torch.isfinite(gb).all()
    ra, rb = orc.lora_grads(x, dy, c.a, c.b, c.lora_scale, c.z)
    # dominated by the largest tokens: compare normwise
    for got, ref in ((ga.cpu().numpy(), ra), (gb.cpu().numpy(), rb)):
        err = np.abs(got.astype(np.float64) - ref)
        assert err.max() <= 1e-2 * np.abs(ref).max() and err.sum() <= 1e-3 * np.abs(ref).sum()


@pytest.mark.parametrize("proj,r", [("up", 32), ("down", 32)])
def test_lora_grads_full_7b_shapes(nv, orc, proj, r):
    """4096 tokens x 7B MLP shapes: every element of dA (r x K) and dB (N x r)
    against the oracle."""
    N, K = synth.QWEN7B_UP if proj == "up" else synth.QWEN7B_DOWN
    M = 4096
    x = synth.activations(M, K, 11)
    dy = synth.activations(M, N, 12, std=1e-3)
    a, b = synth.lora_pair(N, K, r, 0.01, 13)
    z = synth.noise_vector(K, 5e-4, 14)
    _run_and_check(nv, orc, x, dy, a, b, 2.0, z)
