"""The fixed-scratch GEMM entry point, for callers that cannot allocate.

Some callers cannot allocate device memory at all: a host framework that owns
every device allocation and gives its plugins no scratch, or a latency-bound
loop that must not pay cudaMalloc's implicit synchronisation.  For them the
library offers nvfp4_w4a16_lora_gemm_static, which uses an 8 MiB scratch array
built into the library instead of a caller workspace.  This test calls it
through the C ABI twice in a row (the array keeps the previous call's
contents) and compares each result with the workspace entry point, within the
tolerance the other GEMM tests use; the device's free memory must not change
across those two calls.  The file is named so that pytest
collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

from nvfp4_weight_only_02_gb300 import synth

pytestmark = pytest.mark.gpu

MAX_REL, MEAN_REL = 1e-2, 1e-3


def _dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def _static_gemm(nv, x, q, a, b, s, z, y):
    lib = nv.load()
    M, K = x.shape
    N = q.codes.shape[0]
    r = 0 if a is None else a.shape[0]
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    st = lib.nvfp4_w4a16_lora_gemm_static(
        p(x), M, N, K, p(q.codes), p(q.scales), p(q.tensor_scale), p(a), p(b), r, float(s), p(z),
        p(y), nv.OUT_FP32, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return st


def _close(y, ref):
    err = (y.double() - ref.double()).abs()
    assert err.max().item() <= MAX_REL * ref.abs().max().item()
    assert err.sum().item() <= MEAN_REL * ref.abs().sum().item()


@pytest.mark.parametrize("case", ["small", "registers_K1040", "7b_up_M8", "7b_down_M16"])
def test_static_scratch_matches_workspace_entry_point(nv, case):
    if case == "small":
        c = synth.small_case(5, 300, 1024, 8, seed=3)
    elif case == "registers_K1040":
        # K % 256 != 0: the register-streaming decode kernel on the fixed scratch
        c = synth.small_case(8, 300, 1040, 16, seed=4)
        assert nv.gemm_kernel(8, 300, 1040, 16) == "decode_registers"
    elif case == "7b_up_M8":
        c = synth.qwen7b_case("up", 8, seed=5)
    else:
        c = synth.qwen7b_case("down", 16, seed=6)
    q = nv.quantize(_dev(c.w))
    x, a, b = _dev(c.x), _dev(c.a), _dev(c.b)
    z = torch.from_numpy(c.z).cuda()
    ref = nv.gemm(x, q, a, b, c.lora_scale, z)
    ys = [torch.full(ref.shape, float("nan"), dtype=torch.float32, device="cuda") for _ in range(3)]
    # a first call loads the library's device code and looks up the array
    assert _static_gemm(nv, x, q, a, b, c.lora_scale, z, ys.pop()) == nv.OK
    torch.cuda.synchronize()
    free_before, _ = torch.cuda.mem_get_info()
    for y in ys:
        assert _static_gemm(nv, x, q, a, b, c.lora_scale, z, y) == nv.OK
    torch.cuda.synchronize()
    free_after, _ = torch.cuda.mem_get_info()
    for y in ys:
        _close(y, ref)
    # the calls took no device memory (the device's free bytes are unchanged)
    assert free_after == free_before


def test_static_scratch_covers_qwen_projections(nv):
    """Every Qwen2.5-7B and -32B projection at up to 16 tokens, LoRA rank 32 or
    64, fits the fixed 8 MiB scratch."""
    shapes = list(synth.QWEN7B_LAYER.values()) + [synth.QWEN32B_UP, synth.QWEN32B_DOWN, (5120, 5120),
                                                  (1024, 5120)]
    for N, K in shapes:
        for M in (1, 8, 16):
            for r in (32, 64):
                assert 0 < nv.nvfp4_workspace_bytes(M, N, K, r) <= (8 << 20), (N, K, M, r)


def test_static_scratch_rejects_oversized_problems(nv):
    # a workspace beyond the 8 MiB scratch is refused before anything runs
    # (K % 256 != 0 takes the register-streaming kernel, whose f16 X' of
    # 16 tokens x 2^20 columns alone fills 32 MiB)
    N, K = 256, (1 << 20) + 16
    assert nv.nvfp4_workspace_bytes(16, N, K, 0) > (8 << 20)
    x = torch.zeros((16, K), dtype=torch.bfloat16, device="cuda")
    q = nv.QuantizedWeight(torch.zeros((N, K // 2), dtype=torch.uint8, device="cuda"),
                           torch.zeros((N, K // 16), dtype=torch.uint8, device="cuda"),
                           torch.ones(1, dtype=torch.float32, device="cuda"))
    y = torch.empty((16, N), dtype=torch.float32, device="cuda")
    assert _static_gemm(nv, x, q, None, None, 0.0, None, y) == nv.ERR_WORKSPACE
