"""Tensor-core (tcgen05) W4A16 + LoRA + noise GEMM for many tokens vs the oracle.

Same gate as the decode tests: normwise max rel <= 1e-2 and mean rel <= 1e-3
against the FP64 oracle on FP32 output, plus the per-element FP32
accumulation bound.  The full prefill case (16384 tokens x 18944 x 3584)
is compared on sampled token rows, which the oracle computes one by one.
"""
import numpy as np
import pytest
import torch

from nvfp4_weight_only_02_gb300 import synth
from tests.test_gpu_gemm import _abs_bound, _check, _dev, _quantize_both, _run_gpu

pytestmark = pytest.mark.gpu


CASES = [
    # M, N, K, r, lora, noise
    (64, 256, 64, 0, False, False),
    (128, 256, 512, 8, True, True),
    (200, 300, 1024, 32, True, True),
    (333, 1000, 2048, 16, True, False),
    (512, 512, 3584, 64, True, True),
    (1000, 129, 640, 32, True, True),
]


@pytest.mark.parametrize("M,N,K,r,lora,noise", CASES)
def test_prefill_shapes(nv, orc, M, N, K, r, lora, noise):
    c = synth.small_case(M, N, K, r, seed=M + 7 * N + K, with_lora=lora, with_noise=noise)
    q, codes, scales, st = _quantize_both(nv, orc, c.w)
    y = _run_gpu(nv, c, q).cpu().numpy()
    ref = orc.gemm(c.x, codes, scales, st, c.a, c.b, c.lora_scale, c.z)
    _check(y, ref, _abs_bound(orc, c, codes, scales, st), K, r)
    yb = _run_gpu(nv, c, q, torch.bfloat16)
    assert torch.equal(yb.cpu(), torch.from_numpy(y).to(torch.bfloat16))


def test_prefill_dyadic_is_bit_exact(nv, orc):
    g = np.random.default_rng(17)
    M, N, K = 256, 512, 1024
    x = g.integers(-8, 9, size=(M, K)).astype(np.float32)
    x[:, 0] = 8.0  # every token's max is 8: one power of two per token
    qd = g.integers(0, 16, size=(N, K))
    e = g.choice([0x20, 0x28, 0x30, 0x38, 0x40], size=(N, K // 16)).astype(np.uint8)
    codes = (qd[:, 0::2] | (qd[:, 1::2] << 4)).astype(np.uint8)
    xb = synth.to_bf16_bits(x)
    qw = nv.QuantizedWeight(torch.from_numpy(codes).cuda(), torch.from_numpy(e).cuda(),
                            torch.ones(1, dtype=torch.float32, device="cuda"))
    y = nv.gemm(_dev(xb), qw).cpu().numpy()
    ref = orc.gemm(xb, codes, e, np.float32(1.0))
    assert np.array_equal(y.astype(np.float64), ref)


def test_prefill_matches_decode_path(nv, orc):
    """The same product through the tcgen05 path (M >= 64) and through the
    decode kernel (the same tokens 16 at a time) agrees to FP32 rounding."""
    c = synth.small_case(96, 384, 1024, 16, seed=5)
    q, codes, scales, st = _quantize_both(nv, orc, c.w)
    y = _run_gpu(nv, c, q)
    a, b, z = _dev(c.a), _dev(c.b), torch.from_numpy(c.z).cuda()
    x = _dev(c.x)
    parts = [nv.gemm(x[i:i + 16].contiguous(), q, a, b, c.lora_scale, z) for i in range(0, 96, 16)]
    yd = torch.cat(parts)
    assert torch.allclose(y, yd, rtol=1e-5, atol=1e-5 * y.abs().max().item())


def test_prefill_full_size_sampled_rows(nv, orc):
    """16384 tokens (batch 8 x 2048) x 7B-shaped W 18944 x 3584, LoRA r = 32,
    noise sigma 5e-4: FP32 output, 256 token rows checked against the oracle
    (normwise and per element), and every row against the decode kernel run
    16 tokens at a time."""
    M, (N, K), r = 16384, synth.QWEN7B_UP, 32
    w = synth.normal_weight((N, K), 0.02, 1, outlier_frac=1e-3)
    x = synth.activations(M, K, 2)
    a, b = synth.lora_pair(N, K, r, 0.01, 3)
    z = synth.noise_vector(K, 5e-4, 4)
    q, codes, scales, st = _quantize_both(nv, orc, w)
    y = nv.gemm(_dev(x), q, _dev(a), _dev(b), 2.0, torch.from_numpy(z).cuda(), out_dtype=torch.float32)
    torch.cuda.synchronize()
    rows = np.random.default_rng(5).choice(M, size=252, replace=False)
    rows = np.concatenate([rows, [0, 127, 128, M - 1]])
    ref = orc.gemm(x[rows], codes, scales, st, a, b, 2.0, z)
    got = y[torch.from_numpy(rows).cuda()].cpu().numpy()
    max_rel, mean_rel = _check(got, ref, _abs_bound(orc, synth.LinearCase("rows", w, x[rows], a, b, 2.0, z),
                                                    codes, scales, st), K, r)
    print(f"prefill 16384x18944x3584 sampled rows: max_rel {max_rel:.2e} mean_rel {mean_rel:.2e}")
    # every row against the decode kernel (pinned to the oracle on its own), 16 tokens per call
    xd, ad, bd, zd = _dev(x), _dev(a), _dev(b), torch.from_numpy(z).cuda()
    assert nv.gemm_kernel(16, N, K, r) == "decode_stream" and nv.gemm_kernel(M, N, K, r) == "prefill_tcgen05"
    yd = torch.cat([nv.gemm(xd[i:i + 16].contiguous(), q, ad, bd, 2.0, zd) for i in range(0, M, 16)])
    torch.cuda.synchronize()
    diff = (y - yd).abs()
    scale = y.abs().amax(dim=1, keepdim=True)
    assert (diff <= 1e-5 * scale + 1e-30).all(), (diff / scale).max().item()
