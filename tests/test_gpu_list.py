"""Projection lists (nvfp4_w4a16_lora_gemm_list) on the GPU vs the CPU oracle.

A list is a batch of independent layers of the form of the RL post ("RL with
NVFP4 + LoRA", section "Метод"): each output must meet the GEMM's gate
against the FP64 oracle (normwise 1e-2 / 1e-3, and every element within the
FP32 accumulation bound), a one-entry list must equal the single call bit
for bit, and the lists exercise every way the host splits work: several
projections of mixed, ragged shapes in one launch, more entries than one
launch takes, more 128-row tiles than the tile counters, token groups of 16,
and entries that share one X.
"""
import numpy as np
import pytest
import torch

from nvfp4_weight_only_02_gb300 import synth

from .test_gpu_gemm import _abs_bound, _check, _dev, _quantize_both
from .test_gpu_guards import Guarded

pytestmark = pytest.mark.gpu


def _make(nv, orc, shapes, M, r, seed, shared_x=False, noise_every=2):
    """Cases, quantised weights and device inputs for a list of (N, K)."""
    items, cases = [], []
    xs = {}  # K -> (host bits, device tensor) when entries share X
    for i, (N, K) in enumerate(shapes):
        c = synth.small_case(M, N, K, max(r, 1), seed=seed + 7 * i, with_lora=r > 0,
                             with_noise=(i % noise_every) == 0)
        if shared_x and K in xs:
            c.x = xs[K][0]
        else:
            xs[K] = (c.x, _dev(c.x))
        dx = xs[K][1]
        c.lora_scale = 2.0 if i % 2 == 0 else 0.5
        q, codes, scales, st = _quantize_both(nv, orc, c.w)
        a = _dev(c.a) if r > 0 else None
        b = _dev(c.b) if r > 0 else None
        z = torch.from_numpy(c.z).cuda() if c.z is not None else None
        items.append((dx, q, a, b, c.lora_scale if r > 0 else 0.0, z))
        cases.append((c, codes, scales, st))
    return items, cases


def _check_all(orc, ys, cases, r):
    for y, (c, codes, scales, st) in zip(ys, cases):
        a = c.a if r > 0 else None
        b = c.b if r > 0 else None
        s = c.lora_scale if r > 0 else 0.0
        ref = orc.gemm(c.x, codes, scales, st, a, b, s, c.z)
        if r == 0:
            c.a = c.b = None
        absref = _abs_bound(orc, c, codes, scales, st)
        _check(y.float().cpu().numpy(), ref, absref, K=c.x.shape[1], r=r)


MIXED = [(200, 1280), (128, 256), (77, 768), (300, 1024), (1000, 3584), (513, 512)]


@pytest.mark.parametrize("M,r,dt", [(1, 0, torch.float32), (5, 8, torch.float32), (8, 32, torch.bfloat16),
                                    (13, 13, torch.float32), (16, 64, torch.float32), (3, 40, torch.bfloat16)])
def test_mixed_list_vs_oracle(nv, orc, M, r, dt):
    items, cases = _make(nv, orc, MIXED, M, r, seed=100 + M + r)
    ys = nv.gemm_list(items)
    torch.cuda.synchronize()
    _check_all(orc, ys, cases, r)
    if dt == torch.bfloat16:  # bf16 output is the RNE rounding of the same FP32 result
        yb = nv.gemm_list(items, out_dtype=dt)
        torch.cuda.synchronize()
        for y, y16 in zip(ys, yb):
            assert torch.equal(y16, y.to(torch.bfloat16))


@pytest.mark.parametrize("M,N,K,r", [(8, 1000, 3584, 32), (16, 2000, 5632, 32), (1, 300, 1280, 0),
                                     (4, 129, 768, 8)])
def test_one_entry_list_equals_single_call(nv, orc, M, N, K, r):
    items, _ = _make(nv, orc, [(N, K)], M, r, seed=7 + M)
    x, q, a, b, s, z = items[0]
    y_list = nv.gemm_list(items)[0]
    y_one = nv.gemm(x, q, a, b, s, z)
    torch.cuda.synchronize()
    assert torch.equal(y_list, y_one)


def test_long_list_with_shared_inputs(nv, orc):
    # 20 entries: one launch of the 32-entry kernel; entries of the same K read one X
    shapes = [(128 + 64 * (i % 5), 256 * (1 + i % 3)) for i in range(20)]
    items, cases = _make(nv, orc, shapes, 6, 16, seed=500, shared_x=True, noise_every=3)
    ys = nv.gemm_list(items)
    torch.cuda.synchronize()
    _check_all(orc, ys, cases, 16)


def test_list_longer_than_a_launch(nv, orc):
    # 72 entries: two launches (64 + 8), the second with the 16-entry kernel;
    # a 40-entry list takes the 64-entry kernel
    shapes = [(64 + 32 * (i % 7), 256 * (1 + i % 2)) for i in range(72)]
    items, cases = _make(nv, orc, shapes, 3, 8, seed=700, shared_x=True, noise_every=4)
    ys = nv.gemm_list(items)
    torch.cuda.synchronize()
    _check_all(orc, ys, cases, 8)


@pytest.mark.parametrize("n", [16, 17, 32, 33, 64, 65])
def test_list_length_boundaries(nv, orc, n):
    # the host takes the 16-, 32- or 64-entry kernel, the smallest that holds
    # the launch; 65 entries are a launch of 64 and a one-projection remainder
    shapes = [(64 + 16 * (i % 5), 256 * (1 + i % 3)) for i in range(n)]
    items, cases = _make(nv, orc, shapes, 2, 4, seed=1300 + n, shared_x=True, noise_every=5)
    ys = nv.gemm_list(items)
    torch.cuda.synchronize()
    _check_all(orc, ys, cases, 4)


@pytest.mark.parametrize("shapes", [[(128 + 32 * i, 16384) for i in range(5)], [(64, 81920)]])
def test_more_chunk_records_than_sms(nv, orc, shapes):
    # 160 chunks of 512 columns in one launch: the preparation kernel runs
    # with two blocks per SM (a list, then a single projection)
    items, cases = _make(nv, orc, shapes, 3, 8, seed=1500 + len(shapes), shared_x=True, noise_every=2)
    ys = nv.gemm_list(items)
    torch.cuda.synchronize()
    _check_all(orc, ys, cases, 8)


def test_list_split_by_tile_counters(nv, orc):
    # three entries of 3125 tiles each: more than the 8192 tile counters of
    # one launch, so the host splits them 2 + 1
    items, cases = _make(nv, orc, [(400000, 256), (400000, 256), (400000, 256)], 2, 0, seed=900)
    ys = nv.gemm_list(items)
    torch.cuda.synchronize()
    _check_all(orc, ys, cases, 0)


def test_token_groups(nv, orc):
    items, cases = _make(nv, orc, [(300, 1280), (96, 512)], 21, 8, seed=77)
    ys = nv.gemm_list(items)
    torch.cuda.synchronize()
    _check_all(orc, ys, cases, 8)


@pytest.mark.parametrize("M", [1, 8, 16])
def test_full_size_7b_mlp_list(nv, orc, M):
    """Two 18944 x 3584 projections reading one X (gate and up) and the
    3584 x 18944 one in one list, LoRA r = 32, noise: every output vs the
    oracle, and vs the single calls within the FP32 accumulation bound."""
    cs = [synth.qwen7b_case("up", M, seed=3), synth.qwen7b_case("up", M, seed=5),
          synth.qwen7b_case("down", M, seed=4)]
    cs[1].x, cs[1].z = cs[0].x, cs[0].z
    dx = [_dev(cs[0].x), None, _dev(cs[2].x)]
    dx[1] = dx[0]  # gate and up read the same device tensor
    items, cases = [], []
    for c, x in zip(cs, dx):
        q, codes, scales, st = _quantize_both(nv, orc, c.w)
        items.append((x, q, _dev(c.a), _dev(c.b), c.lora_scale, torch.from_numpy(c.z).cuda()))
        cases.append((c, codes, scales, st))
    ys = nv.gemm_list(items)
    singles = [nv.gemm(*it) for it in items]
    torch.cuda.synchronize()
    for y, y1, (c, codes, scales, st) in zip(ys, singles, cases):
        ref = orc.gemm(c.x, codes, scales, st, c.a, c.b, c.lora_scale, c.z)
        absref = _abs_bound(orc, c, codes, scales, st)
        _check(y.cpu().numpy(), ref, absref, K=c.x.shape[1], r=32)
        bound = 2 * (c.x.shape[1] + 32 + 64) * 2.0 ** -23 * absref + 1e-30
        assert (np.abs(y.cpu().numpy().astype(np.float64) - y1.cpu().numpy()) <= bound).all()


def test_list_stays_in_bounds(nv, orc):
    shapes = [(200, 1280), (77, 768), (513, 2048), (129, 256)]
    M, r = 7, 12
    items, _ = _make(nv, orc, shapes, M, r, seed=31)
    for dt, es in ((torch.float32, 4), (torch.bfloat16, 2)):
        outs = [Guarded(M * q.shape[0] * es) for _, q, *_ in items]
        entries = [(x, q.codes, q.scales, q.tensor_scale, a, b, s, z, g.view(dt, (M, q.shape[0])))
                   for (x, q, a, b, s, z), g in zip(items, outs)]
        need = nv.nvfp4_gemm_list_workspace_bytes(entries)
        assert need > 0
        ws = Guarded((need + 255) // 256 * 256, fill=0)
        for _ in range(2):  # a second call on the same workspace
            nv.nvfp4_w4a16_lora_gemm_list(entries, ws.view(torch.uint8, (ws.n,)))
        assert nv.nvfp4_get_device_status(ws.view(torch.uint8, (ws.n,))) == nv.OK
        assert all(g.intact() for g in outs), "output guard overwritten"
        assert ws.intact(), "workspace guard overwritten"
        # the tile counters are back at zero for the next call
        assert not ws.view(torch.uint8, (ws.n,))[256:256 + 4 * 8192].any()
