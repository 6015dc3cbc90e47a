"""Tensor scales far from the LoRA scale, through every GEMM path.

Weights near 1e-37 give s_t = amax / 2688 below the smallest normal FP32
number, and s / s_t beyond the FP32 range; weights near 1e30 give s / s_t
near 2^-90.  The prefill kernel then accumulates the LoRA term apart from the
weights' term and scales each by mantissa times an exact power of two; the
decode kernels scale the two terms apart already.  Every case is compared
with the FP64 oracle on FP32 output: normwise, and per element against the
FP32 accumulation bound with an absolute floor of a few subnormal units
(not 1e-30, which would hide outputs near 1e-35).
"""
import dataclasses

import numpy as np
import pytest
import torch

from nvfp4_weight_only_02_gb300 import synth
from tests.test_gpu_gemm import _abs_bound, _check, _quantize_both, _run_gpu

pytestmark = pytest.mark.gpu

# the three kernels: decode fallback (K % 256 != 0), streaming decode, prefill
SHAPES = [(8, 300, 1040, 16), (9, 1000, 3584, 32), (200, 300, 1024, 32)]
W_STD = [1e-37, 1e-12, 1e-6, 1e30]   # s / s_t: beyond FP32, ~2^46, ~2^26, ~2^-90


@pytest.mark.parametrize("w_std", W_STD)
@pytest.mark.parametrize("M,N,K,r", SHAPES)
@pytest.mark.parametrize("lora", [True, False])
def test_gemm_with_extreme_tensor_scale(nv, orc, M, N, K, r, w_std, lora):
    c = synth.small_case(M, N, K, r, seed=11 * M + K, w_std=w_std, with_lora=lora)
    q, codes, scales, st = _quantize_both(nv, orc, c.w)
    assert np.float32(st) == q.tensor_scale.cpu().numpy()[0]
    if w_std == 1e-37:
        assert 0 < st < np.finfo(np.float32).tiny      # a subnormal tensor scale
    y = _run_gpu(nv, c, q).cpu().numpy()
    assert np.isfinite(y).all()
    ref = orc.gemm(c.x, codes, scales, st, c.a, c.b, c.lora_scale, c.z)
    _check(y, ref, _abs_bound(orc, c, codes, scales, st), K, r if lora else 0, floor=2.0 ** -140)
    if M >= 64:
        yb = _run_gpu(nv, c, q, torch.bfloat16)
        assert torch.equal(yb.cpu(), torch.from_numpy(y).to(torch.bfloat16))


# tokens scaled by 2^k: zero, below 2^-113 (two-step power of two in the
# prefill), below 2^-64 and above 2^32 (rescaled tokens), and in between
ROW_EXP = [None, -120, -70, -40, 0, 20, 40, 100]


@pytest.mark.parametrize("noise", [True, False])
@pytest.mark.parametrize("M,N,K,r", SHAPES)
def test_gemm_with_extreme_token_magnitudes(nv, orc, M, N, K, r, noise):
    c = synth.small_case(M, N, K, r, seed=5 * M + K, with_noise=noise)
    x = synth.bf16_bits_to_f32(c.x).astype(np.float64)
    for i in range(M):
        e = ROW_EXP[i % len(ROW_EXP)]
        x[i] = 0.0 if e is None else x[i] * 2.0 ** e
    c = dataclasses.replace(c, x=synth.to_bf16_bits(x.astype(np.float32)))
    q, codes, scales, st = _quantize_both(nv, orc, c.w)
    y = _run_gpu(nv, c, q).cpu().numpy()
    assert np.isfinite(y).all()
    ref = orc.gemm(c.x, codes, scales, st, c.a, c.b, c.lora_scale, c.z)
    absref = _abs_bound(orc, c, codes, scales, st)
    for i in range(M):
        if ROW_EXP[i % len(ROW_EXP)] is None:
            assert not y[i].any()
        else:
            _check(y[i:i + 1], ref[i:i + 1], absref[i:i + 1], K, r, floor=2.0 ** -140)
