"""Device scalar encoders and the division-free quotient vs the CPU definition."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


def _sweep(lo_bits, hi_bits):
    return np.arange(lo_bits, hi_bits, dtype=np.uint32).view(np.float32)


@pytest.mark.parametrize("sign", [1.0, -1.0])
def test_e2m1_encoder_exhaustive_over_decision_range(nv, orc, sign):
    # every fp32 in +-[2^-4, 8): all thresholds 0.25 .. 5 and saturation at 6
    x = _sweep(0x3D800000, 0x41000000) * np.float32(sign)
    got = nv.nvfp4_encode_debug(torch.from_numpy(x).cuda(), 0).cpu().numpy()
    exp = orc.encode_array(x, 0)
    bad = np.nonzero(got != exp)[0]
    assert bad.size == 0, [(float(x[i]), got[i], exp[i]) for i in bad[:8]]


def test_e2m1_encoder_signs_zeros_and_extremes(nv, orc):
    g = np.random.default_rng(0)
    x = np.concatenate([
        np.array([0.0, -0.0, 1e-45, -1e-45, 0.25, -0.25, 5.0, -5.0, 6.0, -6.0, 7.9, 1e30, -1e30,
                  np.inf, -np.inf], np.float32),
        -_sweep(0x3D800000, 0x41000000)[::97],
        (g.standard_normal(200000) * 4).astype(np.float32),
        (g.standard_normal(100000) * 1e-3).astype(np.float32),
    ])
    got = nv.nvfp4_encode_debug(torch.from_numpy(x).cuda(), 0).cpu().numpy()
    exp = orc.encode_array(x, 0)
    bad = np.nonzero(got != exp)[0]
    assert bad.size == 0, [(float(x[i]), got[i], exp[i]) for i in bad[:8]]


def test_e4m3_encoder_exhaustive_over_grid_range(nv, orc):
    # every fp32 in [2^-11, 2^9): the whole E4M3 grid (subnormals from 2^-9,
    # max 448) and its saturation
    x = _sweep(0x3A000000, 0x44000000)
    got = nv.nvfp4_encode_debug(torch.from_numpy(x).cuda(), 1).cpu().numpy()
    exp = orc.encode_array(x, 1)
    bad = np.nonzero(got != exp)[0]
    assert bad.size == 0, [(float(x[i]), got[i], exp[i]) for i in bad[:8]]


def test_e4m3_encoder_extremes(nv, orc):
    x = np.array([0.0, 1e-45, 1e-30, 2.0 ** -10, 2.0 ** -10 * 1.0000001, 464.0, 464.1, 1e30, np.inf],
                 np.float32)
    got = nv.nvfp4_encode_debug(torch.from_numpy(x).cuda(), 1).cpu().numpy()
    assert list(got) == list(orc.encode_array(x, 1))


def test_fast_quotient_equals_ieee_division_everywhere(nv):
    # all 2^23 fp32 significands of the divisor x all 128 bf16 significands of
    # the dividend x both signs x quotient exponents -13..9
    assert nv.nvfp4_quotient_check(0, 1 << 23) == 0
