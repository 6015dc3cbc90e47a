"""Quantiser, dequantiser and scale-only update on the GPU vs the CPU oracle.

Codes, scales, tensor scales and dequantised values must match bit for bit.
"""
import os

import numpy as np
import pytest
import torch

from nvfp4_weight_only_02_gb300 import synth

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _dev_bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def _quant_gpu(nv, bits, tensor_scale=None):
    q = nv.quantize(_dev_bf16(bits), tensor_scale=tensor_scale)
    torch.cuda.synchronize()
    return q


def _assert_parity(nv, orc, bits, tensor_scale=None):
    ws = nv.new_workspace(256)
    w = _dev_bf16(bits)
    N, K = bits.shape
    codes = torch.empty((N, K // 2), dtype=torch.uint8, device="cuda")
    scales = torch.empty((N, K // 16), dtype=torch.uint8, device="cuda")
    ts = torch.tensor([0.0 if tensor_scale is None else tensor_scale], dtype=torch.float32,
                      device="cuda")
    nv.nvfp4_quantize(w, codes, scales, ts, tensor_scale is not None, ws)
    assert nv.nvfp4_get_device_status(ws) == nv.OK
    rc, c_ref, s_ref, st_ref = orc.quantize(bits, tensor_scale)
    assert rc == orc.OK
    assert ts.item() == st_ref or (np.float32(ts.item()).view(np.uint32) == st_ref.view(np.uint32))
    s_gpu = scales.cpu().numpy()
    c_gpu = codes.cpu().numpy()
    bad_s = np.argwhere(s_gpu != s_ref)
    assert bad_s.size == 0, f"{len(bad_s)} scale bytes differ, first {bad_s[:4].tolist()}"
    bad_c = np.argwhere(c_gpu != c_ref)
    assert bad_c.size == 0, f"{len(bad_c)} code bytes differ, first {bad_c[:4].tolist()}"
    # status, amax and arrival counters are left at zero for the next call
    # (word 4, the grid-barrier generation, only ever counts up)
    assert not ws[:16].any()
    return codes, scales, ts


def test_worked_example(nv, orc):
    d = {}
    for line in open(os.path.join(GOLDEN, "quant_worked_example.txt")):
        line = line.split("#")[0].strip()
        if line:
            k, *v = line.split()
            d[k] = v
    w = np.array([[float(v) for v in d[f"w_row{i}"]] for i in range(2)], np.float32)
    bits = synth.to_bf16_bits(w)
    codes, scales, ts = _assert_parity(nv, orc, bits)
    assert codes.cpu().numpy()[0].tolist() == [int(v, 16) for v in d["bytes_row0"]]
    assert ts.item() == 1.0


@pytest.mark.parametrize("N,K", [(1, 16), (3, 48), (17, 32), (129, 2048), (512, 2048), (7, 4096)])
def test_shapes_ragged(nv, orc, N, K):
    bits = synth.normal_weight((N, K), 0.02, seed=N * 7 + K, outlier_frac=1e-3)
    _assert_parity(nv, orc, bits)


@pytest.mark.parametrize("dist", ["normal", "student_t", "wide_range"])
def test_distributions(nv, orc, dist):
    N, K = 257, 1024
    if dist == "normal":
        bits = synth.normal_weight((N, K), 0.02, 1)
    elif dist == "student_t":
        bits = synth.student_t_weight((N, K), 0.02, 4.0, 2)
    else:
        g = np.random.default_rng(3)
        w = (g.standard_normal((N, K)) * np.exp(g.uniform(-30, 30, (N, 1)))).astype(np.float32)
        bits = synth.to_bf16_bits(w)
    _assert_parity(nv, orc, bits)


def test_frozen_scale_modes(nv, orc):
    bits = synth.normal_weight((64, 512), 0.02, 5)
    rc, _, _, st = orc.quantize(bits)
    for ts in [float(st), float(st) * 3.7, float(st) / 64, 1e-30, 1e20, 0.0]:
        _assert_parity(nv, orc, bits, tensor_scale=np.float32(ts))


def test_ties_at_every_scale(nv, orc):
    rows = []
    for e in range(0x08, 0x7F):
        dec = float(torch.tensor([e], dtype=torch.uint8).view(torch.float8_e4m3fn).float())
        for t in (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0):
            row = np.zeros(16, np.float64)
            row[0], row[1], row[2] = 6 * dec, t * dec, -t * dec
            rows.append(row)
    bits = synth.to_bf16_bits(np.array(rows, np.float32))
    _assert_parity(nv, orc, bits, tensor_scale=np.float32(1.0))
    _assert_parity(nv, orc, bits)


def test_subnormal_and_zero_blocks(nv, orc):
    w = np.zeros((4, 64), np.float32)
    w[0, 0] = 2688.0
    w[0, 16:32] = np.linspace(-0.03, 0.03, 16)
    w[1, :16] = 1e-4
    w[2, 16:32] = -0.0
    w[3, :] = np.float32(2.0 ** -133) * np.arange(64)
    _assert_parity(nv, orc, synth.to_bf16_bits(w))
    # all-zero tensor: s_t = 0, everything zero
    _assert_parity(nv, orc, np.zeros((8, 32), np.uint16))


def test_nonfinite_reported(nv, orc):
    ws = nv.new_workspace(256)
    for bad in (0x7F80, 0xFF80, 0x7FC1):
        bits = synth.normal_weight((8, 64), 0.02, 9)
        bits[5, 17] = bad
        w = _dev_bf16(bits)
        codes = torch.empty((8, 32), dtype=torch.uint8, device="cuda")
        scales = torch.empty((8, 4), dtype=torch.uint8, device="cuda")
        ts = torch.zeros(1, dtype=torch.float32, device="cuda")
        nv.nvfp4_quantize(w, codes, scales, ts, False, ws)
        assert nv.nvfp4_get_device_status(ws) == nv.ERR_NONFINITE
        assert nv.nvfp4_get_device_status(ws) == nv.OK  # reading clears it
        ts.fill_(1.0)
        nv.nvfp4_quantize(w, codes, scales, ts, True, ws)
        assert nv.nvfp4_get_device_status(ws) == nv.ERR_NONFINITE
    bits = synth.normal_weight((8, 64), 0.02, 9)
    for bad_ts in (float("nan"), float("inf"), -1.0):
        w = _dev_bf16(bits)
        ts = torch.tensor([bad_ts], dtype=torch.float32, device="cuda")
        codes = torch.empty((8, 32), dtype=torch.uint8, device="cuda")
        scales = torch.empty((8, 4), dtype=torch.uint8, device="cuda")
        nv.nvfp4_quantize(w, codes, scales, ts, True, ws)
        assert nv.nvfp4_get_device_status(ws) == nv.ERR_NONFINITE


@pytest.mark.parametrize("shape", [synth.QWEN7B_UP, synth.QWEN7B_DOWN])
def test_full_size_7b_layers(nv, orc, shape):
    bits = synth.normal_weight(shape, 0.02, seed=11, outlier_frac=1e-3, outlier_mult=20.0)
    _assert_parity(nv, orc, bits)


@pytest.mark.parametrize("shape", [synth.QWEN32B_UP])
def test_full_size_32b_layer(nv, orc, shape):
    bits = synth.student_t_weight(shape, 0.02, 4.0, seed=12)
    _assert_parity(nv, orc, bits)


@pytest.mark.parametrize("N,K", [(3, 48), (129, 2048), (18944, 3584)])
def test_dequantize_bit_exact(nv, orc, N, K):
    bits = synth.normal_weight((N, K), 0.02, seed=21, outlier_frac=1e-3)
    q = _quant_gpu(nv, bits)
    f32 = nv.dequantize(q, torch.float32).cpu().numpy()
    b16 = nv.dequantize(q, torch.bfloat16).view(torch.int16).cpu().numpy().view(np.uint16)
    rf, rb = orc.dequantize(q.codes.cpu().numpy(), q.scales.cpu().numpy(), np.float32(q.tensor_scale.item()))
    assert np.array_equal(f32.view(np.uint32), rf.view(np.uint32))
    assert np.array_equal(b16, rb)


@pytest.mark.parametrize("shape", [synth.QWEN32B_UP, synth.QWEN32B_DOWN])
def test_round_scales_and_scale_only_merge(nv, orc, shape):
    """Scale-QLoRA on 32B-shaped weights (both projections): codes untouched
    by the update, rounded scales bit-identical to the CPU definition, merged
    weights equal to the training-time fake-quantised weights."""
    bits = synth.student_t_weight(shape, 0.02, 4.0, seed=31 if shape == synth.QWEN32B_UP else 33)
    q = _quant_gpu(nv, bits)
    codes_before = q.codes.clone()
    st = q.tensor_scale
    g = torch.Generator(device="cpu").manual_seed(32)
    dec = q.scales.view(torch.float8_e4m3fn).float()
    param = (dec * st * (1 + (torch.rand(dec.shape, generator=g) * 0.2 - 0.1).cuda())).contiguous()
    new_scales = torch.empty_like(q.scales)
    ws = nv.new_workspace(256)
    nv.nvfp4_round_scales(param, st, new_scales, ws)
    assert nv.nvfp4_get_device_status(ws) == nv.OK
    assert torch.equal(q.codes, codes_before)
    rc, ref = orc.round_scales(param.cpu().numpy(), np.float32(st.item()))
    assert rc == orc.OK and np.array_equal(new_scales.cpu().numpy(), ref)
    merged = nv.QuantizedWeight(q.codes, new_scales, st)
    m_gpu = nv.dequantize(merged, torch.float32).cpu().numpy()
    m_ref, _ = orc.dequantize(q.codes.cpu().numpy(), ref, np.float32(st.item()))
    assert np.array_equal(m_gpu.view(np.uint32), m_ref.view(np.uint32))
    # edge parameters
    p = torch.tensor([[0.0, -1.0, 1e30, 1e-30] * 4], dtype=torch.float32, device="cuda")
    out = torch.empty((1, 16), dtype=torch.uint8, device="cuda")
    nv.nvfp4_round_scales(p, torch.ones(1, device="cuda"), out, ws)
    assert out.cpu().numpy().tolist()[0][:4] == [0, 0, 0x7E, 0]
    p[0, 5] = float("nan")
    nv.nvfp4_round_scales(p, torch.ones(1, device="cuda"), out, ws)
    assert nv.nvfp4_get_device_status(ws) == nv.ERR_NONFINITE
