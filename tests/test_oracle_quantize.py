"""Pins for the oracle's quantiser, dequantiser and scale-only update (CPU).

Anchors: a hand-worked example (tests/golden/quant_worked_example.txt), exact
grid round trips, the half-grid-step error bound, the code share of the file
("codes are about 90% of the file", Scale-QLoRA page), and the Scale-QLoRA
merge invariant (codes untouched, merged weights bit-identical to what the
training forward saw).
"""
import os

import numpy as np
import pytest
import torch

from nvfp4_weight_only_02_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
E2M1_MAG = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], np.float64)  # grid of the format


def _golden():
    d = {}
    with open(os.path.join(GOLDEN, "quant_worked_example.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                k, *v = line.split()
                d[k] = v
    return d


def _e4m3_torch(byte_arr):
    return torch.from_numpy(np.asarray(byte_arr, np.uint8)).view(torch.float8_e4m3fn).double().numpy()


def test_worked_example(orc):
    g = _golden()
    N, K = map(int, g["shape"])
    w = np.array([[float(v) for v in g[f"w_row{i}"]] for i in range(N)], np.float32)
    wb = synth.to_bf16_bits(w)
    assert np.array_equal(synth.bf16_bits_to_f32(wb), w)  # values are bf16-exact
    rc, codes, scales, st = orc.quantize(wb)
    assert rc == orc.OK
    assert st == np.float32(float(g["tensor_scale"][0]))
    for i in range(N):
        assert list(scales[i]) == [int(v, 16) for v in g[f"scales_row{i}"]]
        assert list(codes[i]) == [int(v, 16) for v in g[f"bytes_row{i}"]]
        nib = [int(v, 16) for v in g[f"codes_row{i}"]]
        unpacked = [(codes[i][k // 2] >> (4 * (k % 2))) & 15 for k in range(K)]
        assert unpacked == nib
    f32, _ = orc.dequantize(codes, scales, st)
    exp = np.array([[float(v) for v in g[f"deq_row{i}"]] for i in range(N)], np.float32)
    assert np.array_equal(f32.view(np.uint32), exp.view(np.uint32))  # incl. -0.0


def _grid_tensor(N, K, seed, s_t_log2=-10, dynamic=False):
    """Weights that sit exactly on the NVFP4 grid: w = v(q) * dec(e) * s_t with
    s_t a power of two and every block holding a +-6 code (so its scale is
    recovered exactly)."""
    g = np.random.default_rng(seed)
    nb = K // 16
    e = g.integers(0x08, 0x7F, size=(N, nb))  # normal E4M3 block scales
    q = g.integers(0, 16, size=(N, K))
    q[:, ::16] = np.where(g.random((N, nb)) < 0.5, 7, 15)  # block max code
    if dynamic:
        e[0, 0] = 0x7E  # the tensor max -> s_t recovered exactly
    st = 2.0 ** s_t_log2
    dec = _e4m3_torch(e)
    v = np.where(q >= 8, -1.0, 1.0) * E2M1_MAG[q & 7]
    w = v * np.repeat(dec, 16, axis=1) * st
    w = w.astype(np.float32)
    w[(q == 8)] = -0.0
    wb = synth.to_bf16_bits(w)
    assert np.array_equal(synth.bf16_bits_to_f32(wb).view(np.uint32), w.view(np.uint32))
    return wb, q.astype(np.uint8), e.astype(np.uint8), np.float32(st)


@pytest.mark.parametrize("dynamic", [False, True])
def test_grid_round_trip(orc, dynamic):
    wb, q, e, st = _grid_tensor(24, 128, seed=5, dynamic=dynamic)
    rc, codes, scales, st_out = orc.quantize(wb, tensor_scale=None if dynamic else st)
    assert rc == orc.OK and st_out == st
    assert np.array_equal(scales, e)
    packed = (q[:, 0::2] | (q[:, 1::2] << 4)).astype(np.uint8)
    assert np.array_equal(codes, packed)
    f32, b16 = orc.dequantize(codes, scales, st)
    assert np.array_equal(b16, wb)
    assert np.array_equal(f32.view(np.uint32), synth.bf16_bits_to_f32(wb).view(np.uint32))


TIES = {0.25: 0x0, 0.75: 0x2, 1.25: 0x2, 1.75: 0x4, 2.5: 0x4, 3.5: 0x6, 5.0: 0x6}


def test_exact_ties_resolve_to_even_code_at_every_scale(orc):
    """w / S_b landing exactly halfway between two grid values must take the
    even code, for every normal E4M3 block scale.  The quotient is exact here
    only when it is formed by one correctly rounded division."""
    rows = []
    expect = []
    for e in range(0x08, 0x7F):
        dec = float(_e4m3_torch([e])[0])
        for t, code in TIES.items():
            row = np.zeros(16, np.float64)
            row[0] = 6 * dec        # block max: recovers e exactly with s_t = 1
            row[1] = t * dec
            row[2] = -t * dec
            rows.append(row)
            expect.append((e, code))
    w = np.array(rows, np.float32)
    wb = synth.to_bf16_bits(w)
    assert np.array_equal(synth.bf16_bits_to_f32(wb), w)
    rc, codes, scales, st = orc.quantize(wb, tensor_scale=np.float32(1.0))
    assert rc == orc.OK
    for i, (e, code) in enumerate(expect):
        assert scales[i, 0] == e
        assert codes[i, 0] >> 4 == code, (e, i)
        assert codes[i, 1] & 15 == code | 8, (e, i)


def _half_step(vabs):
    """Half of the local E2M1 grid step at a grid magnitude."""
    return np.where(vabs < 2, 0.25, np.where(vabs < 4, 0.5, 1.0))


@pytest.mark.parametrize("kind", ["normal_outliers", "student_t"])
def test_error_bound(orc, kind):
    N, K = 64, 512
    if kind == "normal_outliers":
        wb = synth.normal_weight((N, K), 0.02, 11, outlier_frac=1e-3)
    else:
        wb = synth.student_t_weight((N, K), 0.02, 4.0, 12)
    rc, codes, scales, st = orc.quantize(wb)
    assert rc == orc.OK
    w = synth.bf16_bits_to_f32(wb).astype(np.float64)
    f32, _ = orc.dequantize(codes, scales, st)
    dec = np.repeat(_e4m3_torch(scales), 16, axis=1)
    S = dec * float(st)
    normal = np.repeat(scales >= 0x08, 16, axis=1)
    assert normal.mean() > 0.99  # subnormal-scale blocks are rare on these inputs
    q = np.stack([(codes >> 0) & 15, (codes >> 4) & 15], axis=-1).reshape(N, K)
    vabs = E2M1_MAG[q & 7]
    err = np.abs(w - f32.astype(np.float64))
    bound = _half_step(vabs) * S * (1 + 2.0 ** -22) + 1e-45
    assert np.all(err[normal] <= bound[normal])


def test_sign_symmetry(orc):
    """Negating W keeps the tensor scale (an amax of magnitudes) and every
    block scale, and flips exactly the sign bit of every code (the E2M1 code
    carries the sign of w, zeros included).  The largest magnitudes are made
    negative so a signed max would give a different tensor scale."""
    g = np.random.default_rng(7)
    w = g.standard_normal((24, 96)).astype(np.float32) * 0.02
    w[3, 5] = -0.5   # tensor amax, negative
    w[7, 40] = -0.3
    bits = synth.to_bf16_bits(w)
    rc, codes, scales, st = orc.quantize(bits)
    assert rc == orc.OK
    rcn, codes_n, scales_n, st_n = orc.quantize(bits ^ np.uint16(0x8000))
    assert rcn == orc.OK
    assert st_n == st
    assert np.array_equal(scales_n, scales)
    assert np.all(scales != 0)
    assert np.array_equal(codes_n, codes ^ np.uint8(0x88))


def test_code_share_is_eight_ninths(orc):
    # "codes are about 90% of the file": 16-element blocks with 1-byte scales
    for N, K in [(512, 2048), (18944, 3584), (27648, 5120)]:
        codes, scales = N * K // 2, N * K // 16
        assert codes * 9 == (codes + scales) * 8
        assert abs(codes / (codes + scales) - 0.9) < 0.012


def test_zero_tensor_and_zero_block(orc):
    wb = np.zeros((4, 32), np.uint16)
    wb[1, 3] = 0x8000  # -0.0
    rc, codes, scales, st = orc.quantize(wb)
    assert rc == orc.OK and st == 0.0
    assert not codes.any() and not scales.any()


def test_nonfinite_rejected(orc):
    for bad in (0x7F80, 0xFF80, 0x7FC0):
        wb = synth.normal_weight((4, 32), 0.02, 1)
        wb[2, 7] = bad
        assert orc.quantize(wb)[0] == orc.NONFINITE
        assert orc.quantize(wb, tensor_scale=1.0)[0] == orc.NONFINITE
    wb = synth.normal_weight((4, 32), 0.02, 1)
    for st in (np.nan, np.inf, -1.0):
        assert orc.quantize(wb, tensor_scale=st)[0] == orc.NONFINITE


def test_frozen_scale_used_verbatim(orc):
    wb = synth.normal_weight((8, 64), 0.02, 3)
    rc, c0, s0, st0 = orc.quantize(wb)
    rc1, c1, s1, st1 = orc.quantize(wb, tensor_scale=st0)
    assert rc1 == orc.OK and st1 == st0
    assert np.array_equal(c0, c1) and np.array_equal(s0, s1)
    # a larger frozen scale pushes every block scale down
    rc2, c2, s2, _ = orc.quantize(wb, tensor_scale=st0 * 4)
    assert np.all(s2 <= s0)
    # twice the tensor scale: every block target e_f halves, and halving is
    # exact on the E4M3 grid while the result stays normal, so each such block
    # scale byte drops by one exponent step (8) and S_b = dec(e) s_t, hence
    # every code, is unchanged
    rc3, c3, s3, st3 = orc.quantize(wb, tensor_scale=st0 * 2)
    assert rc3 == orc.OK and st3 == np.float32(st0 * 2)
    normal = s0 >= 16
    assert normal.mean() > 0.9
    assert np.array_equal(s3[normal], s0[normal] - 8)
    rows = np.repeat(normal, 8, axis=1)  # 8 code bytes per 16-element block
    assert np.array_equal(c3[rows], c0[rows])


def test_subnormal_scale_blocks_saturate(orc):
    """A block far below the tensor max gets a subnormal E4M3 scale; scaled
    values beyond 6 saturate to +-6, values whose scale rounds to 0 give
    code 0."""
    w = np.zeros((1, 48), np.float32)
    w[0, 0] = 2688.0                      # tensor max -> s_t = 1
    w[0, 16:32] = np.linspace(-0.03, 0.03, 16)
    w[0, 16] = 0.03125                    # a_b = 2^-5, e_f = 2^-5/6 = 0.0052
    w[0, 32:48] = 1e-4                    # e_f = 1.7e-5 < 2^-10 -> scale 0
    wb = synth.to_bf16_bits(w)
    rc, codes, scales, st = orc.quantize(wb)
    assert rc == orc.OK and st == 1.0
    # 0.0052 / 2^-9 = 2.67 -> m = 3 (0x03), S_b = 3 * 2^-9 = 0.00586
    assert scales[0, 1] == 0x03
    assert scales[0, 2] == 0x00 and not codes[0, 16:24].any()
    q = [(codes[0][k // 2] >> (4 * (k % 2))) & 15 for k in range(16, 32)]
    x = synth.bf16_bits_to_f32(wb)[0, 16:32].astype(np.float64) / (3 * 2.0 ** -9)
    for xi, qi in zip(x, q):
        if abs(xi) > 6:
            assert qi & 7 == 7  # saturated


def test_scale_only_update_merge_is_bit_identical(orc):
    """Scale-QLoRA: codes frozen, trained block-scale parameters rounded onto
    the E4M3 grid every forward; the merge writes only the scale bytes and the
    merged weights equal the training-time weights bit for bit."""
    wb = synth.student_t_weight((32, 256), 0.02, 4.0, 21)
    rc, codes, scales, st = orc.quantize(wb)
    codes_before = codes.copy()
    g = np.random.default_rng(22)
    # trainable parameter: the effective block scale in weight units
    param = (_e4m3_torch(scales) * float(st) * (1 + g.uniform(-0.1, 0.1, scales.shape)))
    param = param.astype(np.float32)
    rc, new_scales = orc.round_scales(param, st)
    assert rc == orc.OK
    assert np.array_equal(codes, codes_before)  # the update never sees the codes
    # training-time forward: v(q) * round_to_E4M3(param / s_t) * s_t, with the
    # rounding done by PyTorch's float8_e4m3fn conversion
    ratio = torch.from_numpy(param) / torch.tensor(float(st), dtype=torch.float32)
    e_train = ratio.to(torch.float8_e4m3fn)
    assert np.array_equal(e_train.view(torch.uint8).numpy(), new_scales)
    dec = np.repeat(e_train.float().numpy(), 16, axis=1)
    q = np.stack([codes & 15, codes >> 4], axis=-1).reshape(codes.shape[0], -1)
    v = np.where(q >= 8, -1.0, 1.0) * E2M1_MAG[q & 7]
    train_w = ((v * dec).astype(np.float32) * st).astype(np.float32)
    merged, _ = orc.dequantize(codes, new_scales, st)
    assert np.array_equal(merged.view(np.uint32), train_w.view(np.uint32))
    # rounding the unperturbed scales reproduces the original bytes
    rc, same = orc.round_scales(_e4m3_torch(scales).astype(np.float32) * st, st)
    assert np.array_equal(same, scales)


def test_round_scales_edge_values(orc):
    p = np.array([0.0, -1.0, 1e30, np.float32(2.0 ** -9) * 0.49], np.float32)
    rc, e = orc.round_scales(p, np.float32(1.0))
    assert rc == orc.OK and list(e) == [0, 0, 0x7E, 0]
    rc, e = orc.round_scales(np.array([np.nan], np.float32), np.float32(1.0))
    assert rc == orc.NONFINITE
