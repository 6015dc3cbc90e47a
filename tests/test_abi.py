"""The C ABI library builds, loads and exports every declared symbol (CPU).

Also checks the host-side argument validation, which runs before any CUDA
call and so needs no GPU.
"""
import ctypes
import os
import re

import pytest

from nvfp4_weight_only_02_gb300 import binding, build

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "nvfp4.h")


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(nvfp4_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load()


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert "nvfp4_quantize" in names and "nvfp4_w4a16_lora_gemm" in names
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(binding.EXPORTS) == names


def test_status_strings(lib):
    for s in range(9):
        assert binding.status_string(s)
    assert "16" in binding.status_string(binding.ERR_SHAPE)


def test_host_checks_reject_before_launch(lib):
    P = ctypes.c_void_p
    good = P(4096)  # never dereferenced: the checks below fail first
    bad_align = P(4096 + 4)
    null = None
    # null pointer
    assert lib.nvfp4_quantize(null, 16, 32, good, good, good, 0, good, 256, null) == binding.ERR_INVALID_ARG
    # K not a multiple of 16, N < 1
    assert lib.nvfp4_quantize(good, 16, 24, good, good, good, 0, good, 256, null) == binding.ERR_SHAPE
    assert lib.nvfp4_quantize(good, 0, 32, good, good, good, 0, good, 256, null) == binding.ERR_SHAPE
    # misaligned pointer
    assert lib.nvfp4_quantize(bad_align, 16, 32, good, good, good, 0, good, 256, null) == binding.ERR_ALIGNMENT
    # workspace too small
    assert lib.nvfp4_quantize(good, 16, 32, good, good, good, 0, good, 64, null) == binding.ERR_WORKSPACE
    # gemm: bad dtype enum, r out of range, half a LoRA pair
    assert lib.nvfp4_w4a16_lora_gemm(good, 1, 16, 32, good, good, good, null, null, 0, 0.0, null, good,
                                     7, good, 1 << 20, null) == binding.ERR_INVALID_ARG
    assert lib.nvfp4_w4a16_lora_gemm(good, 1, 16, 32, good, good, good, good, good, 300, 1.0, null, good,
                                     0, good, 1 << 20, null) == binding.ERR_SHAPE
    assert lib.nvfp4_w4a16_lora_gemm(good, 1, 16, 32, good, good, good, good, null, 4, 1.0, null, good,
                                     0, good, 1 << 20, null) == binding.ERR_INVALID_ARG
    assert lib.nvfp4_w4a16_lora_gemm(good, 1, 16, 30, good, good, good, null, null, 0, 0.0, null, good,
                                     0, good, 1 << 20, null) == binding.ERR_SHAPE
    assert lib.nvfp4_dequantize(good, good, good, 4, 32, bad_align, 1, null) == binding.ERR_ALIGNMENT
    assert lib.nvfp4_round_scales(good, good, 4, 31, good, good, 256, null) == binding.ERR_SHAPE
    # Scale-QLoRA forward: both steps' host checks before any launch
    assert lib.nvfp4_scale_qlora_gemm(good, 1, 16, 32, good, null, good, good, null, null, 0, 0.0, null,
                                      good, 1, good, 1 << 20, null) == binding.ERR_INVALID_ARG
    assert lib.nvfp4_scale_qlora_gemm(good, 1, 16, 24, good, good, good, good, null, null, 0, 0.0, null,
                                      good, 1, good, 1 << 20, null) == binding.ERR_SHAPE
    assert lib.nvfp4_scale_qlora_gemm(good, 1, 16, 32, good, bad_align, good, good, null, null, 0, 0.0, null,
                                      good, 1, good, 1 << 20, null) == binding.ERR_ALIGNMENT
    # ... and every host check of the GEMM step too (these run before the
    # device query, so they fail here on a machine without a GPU)
    sq = lambda x, y, ydt, a, b, r, z=null: lib.nvfp4_scale_qlora_gemm(
        x, 1, 16, 32, good, good, good, good, a, b, r, 1.0, z, y, ydt, good, 1 << 20, null)
    assert sq(bad_align, good, 1, null, null, 0) == binding.ERR_ALIGNMENT        # x misaligned
    assert sq(good, bad_align, 1, null, null, 0) == binding.ERR_ALIGNMENT        # y misaligned
    assert sq(good, good, 7, null, null, 0) == binding.ERR_INVALID_ARG           # bad output dtype
    assert sq(good, good, 1, good, null, 4) == binding.ERR_INVALID_ARG           # half a LoRA pair
    assert sq(good, good, 1, null, null, 0, bad_align) == binding.ERR_ALIGNMENT  # noise misaligned
    assert sq(good, good, 1, good, bad_align, 4) == binding.ERR_ALIGNMENT        # LoRA B misaligned
    assert lib.nvfp4_scale_qlora_gemm(good, 1, 16, 32, bad_align, good, good, good, null, null, 0, 0.0, null,
                                      good, 1, good, 1 << 20, null) == binding.ERR_ALIGNMENT  # codes
    # the fixed-scratch variant checks its arguments before it queues anything
    st = lib.nvfp4_w4a16_lora_gemm_static(good, 1, 16, 32, good, good, good, good, null, 4, 1.0, null, good, 1,
                                          null)
    assert st in (binding.ERR_INVALID_ARG, binding.ERR_CUDA)  # ERR_CUDA: no device to look the array up on
    # the input gradient: every host check before the device query
    dg = lambda dy, dx, ddt, a, b, r, z=null, M=4, N=64, K=128: lib.nvfp4_w4a16_lora_gemm_dgrad(
        dy, M, N, K, good, good, good, a, b, r, 1.0, z, dx, ddt, good, 1 << 20, null)
    assert dg(null, good, 1, null, null, 0) == binding.ERR_INVALID_ARG           # no dY
    assert dg(good, good, 7, null, null, 0) == binding.ERR_INVALID_ARG           # bad output dtype
    assert dg(good, good, 1, null, null, 0, N=96) == binding.ERR_SHAPE           # N not a multiple of 64
    assert dg(good, good, 1, null, null, 0, K=80) == binding.ERR_SHAPE           # K not a multiple of 64
    assert dg(good, good, 1, null, null, 0, M=0) == binding.ERR_SHAPE
    assert dg(good, good, 1, good, good, 65) == binding.ERR_SHAPE                # rank above 64
    assert dg(good, good, 1, good, null, 4) == binding.ERR_INVALID_ARG           # half a LoRA pair
    assert dg(bad_align, good, 1, null, null, 0) == binding.ERR_ALIGNMENT        # dY misaligned
    assert dg(good, bad_align, 1, null, null, 0) == binding.ERR_ALIGNMENT        # dX misaligned
    assert dg(good, good, 1, null, null, 0, bad_align) == binding.ERR_ALIGNMENT  # noise misaligned
    assert dg(good, good, 1, bad_align, good, 4) == binding.ERR_ALIGNMENT        # LoRA A misaligned
    # the LoRA gradients
    lg = lambda x, dy, a, b, ga, gb, z=null, M=4, N=64, K=128, r=8: lib.nvfp4_lora_grads(
        x, z, dy, M, N, K, a, b, r, 1.0, ga, gb, good, 1 << 20, null)
    assert lg(null, good, good, good, good, good) == binding.ERR_INVALID_ARG
    assert lg(good, good, good, null, good, good) == binding.ERR_INVALID_ARG     # no B
    assert lg(good, good, good, good, good, null) == binding.ERR_INVALID_ARG     # no dB output
    assert lg(good, good, good, good, good, good, r=0) == binding.ERR_SHAPE
    assert lg(good, good, good, good, good, good, r=65) == binding.ERR_SHAPE
    assert lg(good, good, good, good, good, good, N=96) == binding.ERR_SHAPE
    assert lg(good, good, good, good, good, good, K=80) == binding.ERR_SHAPE
    assert lg(bad_align, good, good, good, good, good) == binding.ERR_ALIGNMENT
    assert lg(good, good, good, good, bad_align, good) == binding.ERR_ALIGNMENT  # dA misaligned
    assert lg(good, good, good, good, good, good, bad_align) == binding.ERR_ALIGNMENT
    assert lib.nvfp4_lora_grads_workspace_bytes(4, 64, 128, 0) == 0
    assert lib.nvfp4_lora_grads_workspace_bytes(4, 64, 128, 8) > 0
    assert lib.nvfp4_dgrad_workspace_bytes(4, 96, 128, 0) == 0
    assert lib.nvfp4_dgrad_workspace_bytes(4, 64, 128, 0) > 0
    assert lib.nvfp4_workspace_bytes(1, 16, 30, 0) == 0
    assert lib.nvfp4_gemm_kernel(1, 16, 30, 0) is None
    assert lib.nvfp4_encode_debug(good, 8, 5, good, null) == binding.ERR_INVALID_ARG
    assert lib.nvfp4_quotient_check(0, (1 << 23) + 1, good, null) == binding.ERR_INVALID_ARG


def test_list_host_checks_reject_before_launch(lib):
    P = ctypes.c_void_p
    good, bad = 4096, 4096 + 4

    def entry(x=good, codes=good, scales=good, ts=good, a=good, b=good, z=None, y=good, N=64, K=512):
        return binding.Projection(P(x) if x else None, P(codes) if codes else None, P(scales) if scales else None,
                                  P(ts) if ts else None, P(a) if a else None, P(b) if b else None,
                                  P(z) if z else None, P(y) if y else None, N, K, 2.0)

    def call(entries, M=4, r=8, ydt=1, ws=good, count=None):
        arr = (binding.Projection * max(1, len(entries)))(*entries)
        n = len(entries) if count is None else count
        return lib.nvfp4_w4a16_lora_gemm_list(arr, n, M, r, ydt, P(ws) if ws else None, 1 << 30, None)

    ok2 = [entry(), entry(N=3584, K=18944)]
    assert lib.nvfp4_w4a16_lora_gemm_list(None, 1, 4, 8, 1, P(good), 1 << 30, None) == binding.ERR_INVALID_ARG
    assert call(ok2, count=0) == binding.ERR_SHAPE
    assert call(ok2, count=65537) == binding.ERR_SHAPE
    assert call(ok2, M=0) == binding.ERR_SHAPE
    assert call(ok2, r=65) == binding.ERR_SHAPE
    assert call(ok2, ydt=7) == binding.ERR_INVALID_ARG
    assert call([entry(), entry(K=528)]) == binding.ERR_SHAPE           # K not a multiple of 256
    assert call([entry(K=0)]) == binding.ERR_SHAPE
    assert call([entry(), entry(N=0)]) == binding.ERR_SHAPE
    assert call([entry(N=1048577)]) == binding.ERR_SHAPE                # more tiles than the counters
    assert call([entry(), entry(codes=0)]) == binding.ERR_INVALID_ARG
    assert call([entry(b=0)]) == binding.ERR_INVALID_ARG                # half a LoRA pair with r > 0
    assert call([entry(a=0, b=0)], r=0) != binding.ERR_INVALID_ARG      # r = 0: A and B are ignored
    assert call([entry(x=bad)]) == binding.ERR_ALIGNMENT
    assert call([entry(), entry(y=bad)]) == binding.ERR_ALIGNMENT
    assert call([entry(z=bad)]) == binding.ERR_ALIGNMENT
    assert call([entry(a=bad)]) == binding.ERR_ALIGNMENT
    assert call(ok2, ws=0) == binding.ERR_INVALID_ARG
    assert call(ok2, ws=bad) == binding.ERR_ALIGNMENT
    # every check passed: the next step is the device query (no GPU here)
    assert call(ok2) in (binding.ERR_CUDA, binding.ERR_UNSUPPORTED_DEVICE)
    arr = (binding.Projection * 2)(entry(), entry(K=528))
    assert lib.nvfp4_gemm_list_workspace_bytes(arr, 2, 4, 8) == 0


def test_library_does_not_link_the_oracle():
    # the product library and the oracle share no code: no oracle symbol in it
    out = os.popen(f"nm -D --defined-only {build.LIB}").read()
    assert "orc_" not in out
    exported = set(re.findall(r"\b(nvfp4_[a-z0-9_]+)\b", out))
    assert exported == set(_declared())


def test_projection_struct_layout_matches_the_header(tmp_path):
    # the ctypes mirror of struct nvfp4_projection has the C layout of the header
    import shutil
    import subprocess
    if shutil.which("gcc") is None:
        pytest.skip("gcc not found")
    src = tmp_path / "layout.c"
    src.write_text('#include <stdio.h>\n#include <stddef.h>\n#include "nvfp4.h"\n'
                   'int main(void) { printf("%zu", sizeof(nvfp4_projection));\n'
                   '  const size_t o[] = {offsetof(nvfp4_projection, x_bf16), offsetof(nvfp4_projection, codes),\n'
                   '    offsetof(nvfp4_projection, scales_e4m3), offsetof(nvfp4_projection, tensor_scale),\n'
                   '    offsetof(nvfp4_projection, lora_a_bf16), offsetof(nvfp4_projection, lora_b_bf16),\n'
                   '    offsetof(nvfp4_projection, noise_fp32), offsetof(nvfp4_projection, y),\n'
                   '    offsetof(nvfp4_projection, N), offsetof(nvfp4_projection, K),\n'
                   '    offsetof(nvfp4_projection, lora_scale)};\n'
                   '  for (int i = 0; i < 11; i++) printf(" %zu", o[i]);\n  return 0; }\n')
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-I", os.path.dirname(HEADER), str(src), "-o", str(exe)], check=True)
    got = [int(v) for v in subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()]
    P = binding.Projection
    names = ["x_bf16", "codes", "scales_e4m3", "tensor_scale", "lora_a_bf16", "lora_b_bf16", "noise_fp32", "y",
             "N", "K", "lora_scale"]
    assert [f[0] for f in P._fields_] == names
    assert got == [ctypes.sizeof(P)] + [getattr(P, n).offset for n in names]
