"""W4A16 + LoRA + noise GEMM on the GPU vs the CPU oracle (FP64).

Gate (normwise, on FP32 output): max|Y_gpu - Y| / max|Y| <= 1e-2 and
sum|Y_gpu - Y| / sum|Y| <= 1e-3.  In addition every element must sit within
the FP32 accumulation bound derived from the arithmetic,
|Y_gpu - Y| <= (K + r + 64) * 2^-23 * (|X'| |D|^T + |s| |T| |B|^T),
with the absolute-value product computed by the same oracle on |inputs|.
"""
import numpy as np
import pytest
import torch

from nvfp4_weight_only_02_gb300 import synth

pytestmark = pytest.mark.gpu

MAX_REL, MEAN_REL = 1e-2, 1e-3


def _dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def _quantize_both(nv, orc, w_bits):
    q = nv.quantize(_dev(w_bits))
    rc, codes, scales, st = orc.quantize(w_bits)
    assert np.array_equal(q.codes.cpu().numpy(), codes)
    return q, codes, scales, st


def _run_gpu(nv, c, q, out_dtype=torch.float32):
    a = _dev(c.a) if c.a is not None else None
    b = _dev(c.b) if c.b is not None else None
    z = torch.from_numpy(c.z).cuda() if c.z is not None else None
    y = nv.gemm(_dev(c.x), q, a, b, c.lora_scale if a is not None else 0.0, z, out_dtype=out_dtype)
    torch.cuda.synchronize()
    return y


def _abs_bound(orc, c, codes, scales, st):
    ax = c.x & 0x7FFF
    ac = codes & 0x77
    aa = None if c.a is None else c.a & 0x7FFF
    ab = None if c.b is None else c.b & 0x7FFF
    az = None if c.z is None else np.abs(c.z)
    return orc.gemm(ax, ac, scales, st, aa, ab, abs(c.lora_scale), az)


def _check(y_gpu, y_ref, absref=None, K=0, r=0, floor=1e-30):
    err = np.abs(y_gpu.astype(np.float64) - y_ref)
    max_rel = err.max() / max(np.abs(y_ref).max(), 1e-300)
    mean_rel = err.sum() / max(np.abs(y_ref).sum(), 1e-300)
    assert max_rel <= MAX_REL, max_rel
    assert mean_rel <= MEAN_REL, mean_rel
    if absref is not None:
        bound = (K + r + 64) * 2.0 ** -23 * absref + floor
        worst = (err / bound).max()
        assert worst <= 1.0, worst
    return max_rel, mean_rel


CASES = [
    # M, N, K, r, lora, noise
    (1, 1, 16, 0, False, False),
    (3, 17, 48, 4, True, True),
    (8, 300, 1040, 16, True, True),
    (16, 513, 2064, 8, True, False),
    (5, 256, 512, 32, False, True),
    (4, 512, 2048, 16, True, True),
    (9, 1000, 3584, 32, True, True),
    (2, 70, 8192, 24, True, True),
    (16, 2048, 640, 64, True, True),
    # K % 256 == 0 with a last 256-column chunk (half-chunk units)
    (7, 200, 1280, 16, True, True),
    (16, 129, 768, 8, True, True),
    (12, 640, 4096, 64, True, True),
    (1, 3, 256, 0, False, False),
    # more units than SMs: block ranges of one or two units that cross tile ends
    (6, 2000, 5632, 32, True, True),
    (8, 2000, 5376, 40, True, True),
    # LoRA ranks that are not multiples of 8 on the streaming kernel (K % 256 == 0)
    (8, 700, 2048, 1, True, True),
    (4, 300, 1536, 5, True, True),
    (16, 256, 2560, 12, True, True),
    (3, 1100, 1024, 20, True, True),
    (8, 513, 3072, 33, True, True),
]


@pytest.mark.parametrize("M,N,K,r,lora,noise", CASES)
def test_small_and_ragged(nv, orc, M, N, K, r, lora, noise):
    c = synth.small_case(M, N, K, r, seed=M * 1000 + N + K, with_lora=lora, with_noise=noise)
    q, codes, scales, st = _quantize_both(nv, orc, c.w)
    y = _run_gpu(nv, c, q).cpu().numpy()
    ref = orc.gemm(c.x, codes, scales, st, c.a, c.b, c.lora_scale, c.z)
    _check(y, ref, _abs_bound(orc, c, codes, scales, st), K, r)
    # bf16 output is the RNE rounding of the same FP32 result
    yb = _run_gpu(nv, c, q, torch.bfloat16)
    assert torch.equal(yb.cpu(), torch.from_numpy(y).to(torch.bfloat16))


def test_streaming_kernel_takes_ragged_lora_ranks(nv):
    """The odd-rank cases above really run the streaming kernel."""
    for M, N, K, r in ((8, 700, 2048, 1), (4, 300, 1536, 5), (16, 256, 2560, 12), (3, 1100, 1024, 20),
                       (8, 513, 3072, 33)):
        assert nv.gemm_kernel(M, N, K, r) == "decode_stream"


def test_kernel_selection(nv):
    """K % 256 == 0 (every Qwen2.5 projection) takes the bulk-copy streaming
    kernel, other K the register-streaming one, M >= 64 the tensor cores."""
    assert nv.gemm_kernel(8, 18944, 3584, 32) == "decode_stream"
    assert nv.gemm_kernel(16, 3584, 18944, 32) == "decode_stream"
    assert nv.gemm_kernel(1, 27648, 5120, 64) == "decode_stream"
    assert nv.gemm_kernel(8, 300, 1040, 16) == "decode_registers"
    assert nv.gemm_kernel(16, 2048, 640, 64) == "decode_registers"
    assert nv.gemm_kernel(16384, 18944, 3584, 32) == "prefill_tcgen05"
    assert nv.gemm_kernel(8, 300, 1000, 16) is None


def test_single_layer_case(nv, orc):
    c = synth.single_layer_case()
    q, codes, scales, st = _quantize_both(nv, orc, c.w)
    y = _run_gpu(nv, c, q).cpu().numpy()
    ref = orc.gemm(c.x, codes, scales, st, c.a, c.b, c.lora_scale, c.z)
    _check(y, ref, _abs_bound(orc, c, codes, scales, st), 2048, 16)


def test_dyadic_case_is_bit_exact(nv, orc):
    """Small-integer activations, power-of-two block scales, s_t = 1, no LoRA
    and no noise: every partial sum is exact in FP32, so the GPU result must
    equal the oracle exactly."""
    g = np.random.default_rng(7)
    M, N, K = 8, 384, 1024
    x = g.integers(-8, 9, size=(M, K)).astype(np.float32)
    q = g.integers(0, 16, size=(N, K))
    e = g.choice([0x20, 0x28, 0x30, 0x38, 0x40], size=(N, K // 16)).astype(np.uint8)
    codes = (q[:, 0::2] | (q[:, 1::2] << 4)).astype(np.uint8)
    xb = synth.to_bf16_bits(x)
    qw = nv.QuantizedWeight(torch.from_numpy(codes).cuda(), torch.from_numpy(e).cuda(),
                            torch.ones(1, dtype=torch.float32, device="cuda"))
    y = nv.gemm(_dev(xb), qw).cpu().numpy()
    ref = orc.gemm(xb, codes, e, np.float32(1.0))
    assert np.array_equal(y.astype(np.float64), ref)


def test_special_cases_reduce_to_base(nv, orc):
    c = synth.small_case(4, 512, 1024, 16, seed=5)
    q, codes, scales, st = _quantize_both(nv, orc, c.w)
    x = _dev(c.x)
    base = nv.gemm(x, q)
    a, b = _dev(c.a), _dev(c.b)
    assert torch.equal(nv.gemm(x, q, a, b, 0.0), base)                    # s = 0
    assert torch.equal(nv.gemm(x, q, torch.zeros_like(a), b, 2.0), base)  # A = 0
    ones = torch.ones(1024, dtype=torch.float32, device="cuda")
    assert torch.equal(nv.gemm(x, q, noise=ones), base)                  # z = 1
    # M = 1 rows agree with the batched result within FP32 rounding
    full = nv.gemm(x, q, a, b, 2.0, torch.from_numpy(c.z).cuda())
    for m in range(4):
        one = nv.gemm(x[m:m + 1].contiguous(), q, a, b, 2.0, torch.from_numpy(c.z).cuda())
        assert torch.allclose(one[0], full[m], rtol=1e-6, atol=1e-6)


def test_large_m_token_groups(nv, orc):
    c = synth.small_case(37, 300, 1024, 8, seed=77)
    q, codes, scales, st = _quantize_both(nv, orc, c.w)
    y = _run_gpu(nv, c, q).cpu().numpy()
    ref = orc.gemm(c.x, codes, scales, st, c.a, c.b, c.lora_scale, c.z)
    _check(y, ref, _abs_bound(orc, c, codes, scales, st), 1024, 8)


def test_activation_dynamic_range(nv, orc):
    """Token rows and 512-column chunks spanning 2^-60 .. 2^60: the f16
    re-expression with a power of two per token and chunk stays exact."""
    g = np.random.default_rng(9)
    M, N, K = 6, 256, 2048
    x = g.standard_normal((M, K)).astype(np.float32)
    x *= np.exp2(g.integers(-60, 60, size=(M, 1))).astype(np.float32)
    x[:, 512:1024] *= np.float32(2.0 ** 40)
    x[:, 1024:1536] *= np.float32(2.0 ** -40)
    c = synth.LinearCase("range", synth.normal_weight((N, K), 0.02, 3), synth.to_bf16_bits(x),
                         None, None, 0.0, None)
    q, codes, scales, st = _quantize_both(nv, orc, c.w)
    y = _run_gpu(nv, c, q).cpu().numpy()
    ref = orc.gemm(c.x, codes, scales, st)
    for m in range(M):  # each token row has its own magnitude: check rows separately
        _check(y[m:m + 1], ref[m:m + 1])


def _full_case(which, model, M):
    if model == "7b":
        return synth.qwen7b_case(which, M, seed=3)
    return synth.qwen32b_case(which, M, seed=4)


@pytest.mark.parametrize("model,which,M", [("7b", "up", 1), ("7b", "up", 16), ("7b", "down", 4),
                                           ("7b", "down", 8), ("32b", "up", 1), ("32b", "up", 8),
                                           ("32b", "down", 1), ("32b", "down", 8)])
def test_full_size_decode(nv, orc, model, which, M):
    c = _full_case(which, model, M)
    q, codes, scales, st = _quantize_both(nv, orc, c.w)
    y = _run_gpu(nv, c, q).cpu().numpy()
    ref = orc.gemm(c.x, codes, scales, st, c.a, c.b, c.lora_scale, c.z)
    max_rel, mean_rel = _check(y, ref)
    print(f"{model} {which} M={M}: max_rel {max_rel:.3e} mean_rel {mean_rel:.3e}")


def test_scale_qlora_forward(nv, orc):
    """Scale-QLoRA forward on 32B-shaped weights (W 27648 x 5120, 8 tokens,
    LoRA r = 64, noise): trainable FP32 block scales rounded on the way in,
    codes frozen.  The rounded scales are the CPU definition bit for bit, the
    output matches the FP64 oracle on the merged weights, and equals the plain
    GEMM on the merged weights exactly (the same kernels run)."""
    c = synth.qwen32b_case("up", 8, seed=41)
    q, codes, scales, st = _quantize_both(nv, orc, c.w)
    g = torch.Generator(device="cpu").manual_seed(42)
    dec = q.scales.view(torch.float8_e4m3fn).float()
    jitter = (torch.rand(dec.shape, generator=g) * 0.2 - 0.1).cuda()
    param = (dec * q.tensor_scale * (1 + jitter)).contiguous()
    x, a, b, z = _dev(c.x), _dev(c.a), _dev(c.b), torch.from_numpy(c.z).cuda()
    M, K = c.x.shape
    N = q.shape[0]
    rounded = torch.empty_like(q.scales)
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    ws = nv.new_workspace(nv.nvfp4_workspace_bytes(M, N, K, 64))
    nv.nvfp4_scale_qlora_gemm(x, q.codes, param, q.tensor_scale, rounded, a, b, c.lora_scale, z, y, ws)
    assert nv.nvfp4_get_device_status(ws) == nv.OK
    rc, ref_scales = orc.round_scales(param.cpu().numpy(), np.float32(q.tensor_scale.item()))
    assert rc == orc.OK and np.array_equal(rounded.cpu().numpy(), ref_scales)
    ref = orc.gemm(c.x, codes, ref_scales, st, c.a, c.b, c.lora_scale, c.z)
    _check(y.cpu().numpy(), ref)
    merged = nv.QuantizedWeight(q.codes, rounded, q.tensor_scale)
    y2 = nv.gemm(x, merged, a, b, c.lora_scale, z)
    assert torch.equal(y, y2)
