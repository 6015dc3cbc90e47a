"""Out-of-bounds writes (compute-sanitizer is closed on this machine): every
output buffer and the workspace sit between guard bytes holding a fixed
pattern, which must be untouched after each call, on ragged and tiled shapes
of every kernel family (quantiser both modes, dequantiser, scale update, the
GEMM's streaming, register-streaming and tcgen05 paths, and the input
gradient)."""
import numpy as np
import pytest
import torch

from nvfp4_weight_only_02_gb300 import synth

pytestmark = pytest.mark.gpu

GUARD = 4096  # bytes on each side (keeps the payload 16-byte aligned)
PATTERN = 0xA5


class Guarded:
    """nbytes of payload inside a buffer whose head and tail hold PATTERN."""

    def __init__(self, nbytes, fill=PATTERN):
        self.n = int(nbytes)
        self.buf = torch.full((self.n + 2 * GUARD,), PATTERN, dtype=torch.uint8, device="cuda")
        self.buf[GUARD:GUARD + self.n].fill_(fill)

    def view(self, dtype, shape):
        return self.buf[GUARD:GUARD + self.n].view(dtype).view(shape)

    def intact(self):
        torch.cuda.synchronize()
        return bool((self.buf[:GUARD] == PATTERN).all()) and bool((self.buf[GUARD + self.n:] == PATTERN).all())


def _dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


@pytest.mark.parametrize("N,K", [(1, 16), (17, 48), (129, 256), (300, 1040), (513, 2064), (1000, 3584)])
def test_quantize_dequantize_and_scale_update_stay_in_bounds(nv, N, K):
    w = _dev(synth.normal_weight((N, K), 0.02, N + K, outlier_frac=1e-3))
    for given in (False, True):
        codes, scales, ts = Guarded(N * K // 2), Guarded(N * K // 16), Guarded(4, fill=0)
        ws = Guarded(256, fill=0)
        t = ts.view(torch.float32, (1,))
        if given:
            t.fill_(0.01)
        nv.nvfp4_quantize(w, codes.view(torch.uint8, (N, K // 2)), scales.view(torch.uint8, (N, K // 16)), t,
                          given, ws.view(torch.uint8, (256,)))
        assert nv.nvfp4_get_device_status(ws.view(torch.uint8, (256,))) == nv.OK
        assert codes.intact() and scales.intact() and ts.intact() and ws.intact()
    q = nv.QuantizedWeight(codes.view(torch.uint8, (N, K // 2)), scales.view(torch.uint8, (N, K // 16)), t)
    for dt, es in ((torch.float32, 4), (torch.bfloat16, 2)):
        out = Guarded(N * K * es)
        nv.nvfp4_dequantize(q.codes, q.scales, q.tensor_scale, out.view(dt, (N, K)))
        assert out.intact()
    param = (q.scales.view(torch.float8_e4m3fn).float() * t * 1.03).contiguous()
    new = Guarded(N * K // 16)
    ws = Guarded(256, fill=0)
    nv.nvfp4_round_scales(param, t, new.view(torch.uint8, (N, K // 16)), ws.view(torch.uint8, (256,)))
    assert new.intact() and ws.intact()


# M, N, K, r: streaming decode (K % 256 == 0), register-streaming (other K),
# tcgen05 prefill (M >= 64), with ragged tiles, half chunks and LoRA ranks
GEMM_CASES = [
    (1, 3, 256, 0), (7, 200, 1280, 16), (16, 129, 768, 8), (12, 640, 4096, 64), (6, 2000, 5632, 32),
    (3, 17, 48, 4), (8, 300, 1040, 16), (16, 513, 2064, 8),
    (64, 256, 64, 0), (200, 300, 1024, 32), (1000, 129, 640, 64),
    # LoRA ranks that are not multiples of 8 on the streaming kernel
    (8, 700, 2048, 1), (4, 300, 1536, 5), (16, 256, 2560, 12), (3, 1100, 1024, 20), (8, 513, 3072, 33),
]


@pytest.mark.parametrize("M,N,K,r", GEMM_CASES)
def test_gemm_stays_in_bounds(nv, M, N, K, r):
    c = synth.small_case(M, N, K, max(r, 1), seed=M + N + K, with_lora=r > 0, with_noise=True)
    q = nv.quantize(_dev(c.w))
    a = _dev(c.a) if r > 0 else None
    b = _dev(c.b) if r > 0 else None
    z = torch.from_numpy(c.z).cuda()
    x = _dev(c.x)
    need = nv.nvfp4_workspace_bytes(M, N, K, r)
    for dt, es in ((torch.float32, 4), (torch.bfloat16, 2)):
        y = Guarded(M * N * es)
        ws = Guarded((need + 255) // 256 * 256, fill=0)
        for _ in range(2):  # a second call on the same workspace
            nv.nvfp4_w4a16_lora_gemm(x, q.codes, q.scales, q.tensor_scale, a, b, c.lora_scale if r else 0.0, z,
                                     y.view(dt, (M, N)), ws.view(torch.uint8, (ws.n,)))
        assert nv.nvfp4_get_device_status(ws.view(torch.uint8, (ws.n,))) == nv.OK
        assert y.intact(), "output guard overwritten"
        assert ws.intact(), "workspace guard overwritten"


# M, N, K, r for the input gradient (N, K multiples of 64): ragged tiles of
# tokens and of output columns, both extension widths, one rescaled token
DGRAD_CASES = [(1, 64, 64, 0), (5, 128, 320, 8), (130, 192, 640, 40), (200, 320, 1024, 32), (333, 512, 192, 64)]


@pytest.mark.parametrize("M,N,K,r", DGRAD_CASES)
def test_dgrad_stays_in_bounds(nv, M, N, K, r):
    c = synth.small_case(M, N, K, max(r, 1), seed=3 * M + N + K, with_lora=r > 0, with_noise=True)
    q = nv.quantize(_dev(c.w))
    a = _dev(c.a) if r > 0 else None
    b = _dev(c.b) if r > 0 else None
    z = torch.from_numpy(c.z).cuda()
    g = synth.bf16_bits_to_f32(synth.activations(M, N, M + 1))
    g[M // 2] *= 2.0 ** 50  # one token outside [2^-64, 2^32]: the rescaling kernel runs too
    dy = _dev(synth.to_bf16_bits(g))
    need = nv.nvfp4_dgrad_workspace_bytes(M, N, K, r)
    assert need > 0
    for dt, es in ((torch.float32, 4), (torch.bfloat16, 2)):
        dx = Guarded(M * K * es)
        ws = Guarded((need + 255) // 256 * 256, fill=0)
        for _ in range(2):  # a second call on the same workspace
            nv.nvfp4_w4a16_lora_gemm_dgrad(dy, q.codes, q.scales, q.tensor_scale, a, b, c.lora_scale if r else 0.0,
                                           z, dx.view(dt, (M, K)), ws.view(torch.uint8, (ws.n,)))
        assert nv.nvfp4_get_device_status(ws.view(torch.uint8, (ws.n,))) == nv.OK
        assert dx.intact(), "output guard overwritten"
        assert ws.intact(), "workspace guard overwritten"


@pytest.mark.parametrize("M,N,K,r", [(1, 64, 64, 1), (70, 192, 320, 40), (333, 512, 192, 64)])
def test_lora_grads_stay_in_bounds(nv, M, N, K, r):
    c = synth.small_case(M, N, K, r, seed=5 * M + N + K)
    g = synth.bf16_bits_to_f32(synth.activations(M, N, M + 2))
    g[M // 2] *= 2.0 ** 50  # a rescaled token
    dy = _dev(synth.to_bf16_bits(g))
    need = nv.nvfp4_lora_grads_workspace_bytes(M, N, K, r)
    assert need > 0
    ga, gb = Guarded(r * K * 4), Guarded(N * r * 4)
    ws = Guarded((need + 255) // 256 * 256, fill=0)
    for _ in range(2):
        nv.nvfp4_lora_grads(_dev(c.x), torch.from_numpy(c.z).cuda(), dy, _dev(c.a), _dev(c.b), c.lora_scale,
                            ga.view(torch.float32, (r, K)), gb.view(torch.float32, (N, r)),
                            ws.view(torch.uint8, (ws.n,)))
    assert ga.intact() and gb.intact(), "output guard overwritten"
    assert ws.intact(), "workspace guard overwritten"
