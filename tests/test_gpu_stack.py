"""Whole-stack quantise + decode: the 28 layers of a Qwen2.5-7B-shaped model
(q/o 3584x3584, k/v 512x3584, gate/up 18944x3584, down 3584x18944), BF16
weights ~N(0, 0.02^2) drawn on the device from seeded generators, every one of
the 196 matrices quantised with its own dynamic tensor scale and multiplied by
the same 8 tokens, with a LoRA pair (r = 32, s = 2) of its own and the
multiplicative input noise (sigma 5e-4, one vector per input width).

Each matrix is checked against the oracle on sampled rows: the row holding the
matrix's largest |w| plus seven random rows, quantised by the oracle in
dynamic mode (so its tensor scale comes from the same amax), must give the
GPU's tensor scale, codes and block scales bit for bit, and the GPU's GEMM
outputs for those rows must match the oracle's FP64 GEMM within tolerance.
"""
import numpy as np
import pytest
import torch

from nvfp4_weight_only_02_gb300 import synth
from tests.test_gpu_gemm import _check

pytestmark = pytest.mark.gpu

LAYERS = 28
SHAPES = [("q", 3584, 3584), ("k", 512, 3584), ("v", 512, 3584), ("o", 3584, 3584),
          ("gate", 18944, 3584), ("up", 18944, 3584), ("down", 3584, 18944)]


def test_whole_stack_quantise_and_decode(nv, orc):
    M, r, s = 8, 32, 2.0
    xb = {K: synth.activations(M, K, 70 + K) for K in (3584, 18944)}
    xd = {K: torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).cuda() for K, b in xb.items()}
    zh = {K: synth.noise_vector(K, 5e-4, 90 + K) for K in (3584, 18944)}
    zd = {K: torch.from_numpy(v).cuda() for K, v in zh.items()}
    ws = nv.new_workspace(max(nv.nvfp4_workspace_bytes(M, N, K, r) for _, N, K in SHAPES))
    gen = torch.Generator(device="cuda")
    pick = np.random.default_rng(2048)
    checked = 0
    for layer in range(LAYERS):
        for j, (name, N, K) in enumerate(SHAPES):
            gen.manual_seed(1000 * layer + j)
            w = (torch.randn((N, K), generator=gen, device="cuda") * 0.02).to(torch.bfloat16)
            a = (torch.randn((r, K), generator=gen, device="cuda") * 0.01).to(torch.bfloat16)
            b = (torch.randn((N, r), generator=gen, device="cuda") * 0.01).to(torch.bfloat16)
            q = nv.quantize(w, workspace=ws)
            y = nv.gemm(xd[K], q, a, b, s, zd[K], workspace=ws)
            top = int(torch.argmax(w.abs().float()).item()) // K
            rows = [top] + [int(i) for i in pick.choice(np.delete(np.arange(N), top), size=7, replace=False)]
            wb = w[rows].view(torch.int16).cpu().numpy().view(np.uint16)
            rc, codes, scales, st = orc.quantize(wb)
            assert rc == orc.OK
            where = f"layer {layer} {name}"
            assert np.float32(q.tensor_scale.item()) == st, where
            assert np.array_equal(q.codes[rows].cpu().numpy(), codes), where
            assert np.array_equal(q.scales[rows].cpu().numpy(), scales), where
            bits = lambda t: t.view(torch.int16).cpu().numpy().view(np.uint16)
            ref = orc.gemm(xb[K], codes, scales, st, bits(a), bits(b[rows]), s, zh[K])
            _check(y[:, rows].cpu().numpy(), ref)
            checked += 1
            del w, a, b, q, y
    assert checked == LAYERS * len(SHAPES)
    assert nv.nvfp4_get_device_status(ws) == nv.OK


def test_whole_stack_as_projection_lists(nv, orc):
    """The same 196 matrices run three ways: single calls, lists grouped per
    layer as a decoder's dependencies allow ([q, k, v], [o], [gate, up],
    [down]) and lists of 64 in sweep order.  Every list output equals the
    single call's to FP32 summation order (only the split of K over blocks
    differs), and on sampled rows of every seventh matrix the list outputs
    match the oracle within tolerance."""
    M, r, s = 8, 32, 2.0
    xb = {K: synth.activations(M, K, 170 + K) for K in (3584, 18944)}
    xd = {K: torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).cuda() for K, b in xb.items()}
    zh = {K: synth.noise_vector(K, 5e-4, 190 + K) for K in (3584, 18944)}
    zd = {K: torch.from_numpy(v).cuda() for K, v in zh.items()}
    ws = nv.new_workspace(max(nv.nvfp4_workspace_bytes(M, N, K, r) for _, N, K in SHAPES))
    gen = torch.Generator(device="cuda")
    pick = np.random.default_rng(4096)
    bits = lambda t: t.view(torch.int16).cpu().numpy().view(np.uint16)
    items, samples = [], {}
    for layer in range(LAYERS):
        for j, (name, N, K) in enumerate(SHAPES):
            gen.manual_seed(5000 * layer + j)
            w = (torch.randn((N, K), generator=gen, device="cuda") * 0.02).to(torch.bfloat16)
            a = (torch.randn((r, K), generator=gen, device="cuda") * 0.01).to(torch.bfloat16)
            b = (torch.randn((N, r), generator=gen, device="cuda") * 0.01).to(torch.bfloat16)
            q = nv.quantize(w, workspace=ws)
            idx = len(items)
            if idx % 7 == 0:
                top = int(torch.argmax(w.abs().float()).item()) // K
                rows = [top] + [int(i) for i in pick.choice(np.delete(np.arange(N), top), size=7, replace=False)]
                samples[idx] = (rows, bits(w[rows]), bits(a), bits(b[rows]))
            items.append((xd[K], q, a, b, s, zd[K]))
            del w
    singles = [nv.gemm(*it, workspace=ws) for it in items]
    names = [n for n, _, _ in SHAPES]
    groups = [("q", "k", "v"), ("o",), ("gate", "up"), ("down",)]
    layer_lists = [[layer * len(SHAPES) + names.index(n) for n in grp] for layer in range(LAYERS) for grp in groups]
    flat = list(range(len(items)))
    longest = [flat[i:i + 64] for i in range(0, len(flat), 64)]
    for plan in (layer_lists, longest):
        outs = [None] * len(items)
        for ids in plan:
            for i, y in zip(ids, nv.gemm_list([items[i] for i in ids])):
                outs[i] = y
        torch.cuda.synchronize()
        for i, (y, y1) in enumerate(zip(outs, singles)):
            d = (y - y1).abs().max().item() / max(y1.abs().max().item(), 1e-30)
            assert d <= 1e-5, (i, d)
            if i in samples:
                rows, wb, ab, bb = samples[i]
                K = items[i][0].shape[1]
                rc, codes, scales, st = orc.quantize(wb)
                assert rc == orc.OK
                _check(y[:, rows].cpu().numpy(), orc.gemm(xb[K], codes, scales, st, ab, bb, s, zh[K]))
    assert nv.nvfp4_get_device_status(ws) == nv.OK
