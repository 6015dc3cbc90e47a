"""Pins for the oracle's scalar codecs (CPU only).

Each check compares the oracle with something other than itself: a golden
table written by hand, a threshold encoder derived from round-to-nearest-even
on the grid, or PyTorch's own float8_e4m3fn / bfloat16 conversions.
"""
import os

import numpy as np
import pytest
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_pairs(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                rows.append(line.split())
    return rows


def test_e2m1_grid_matches_golden(orc):
    rows = _read_pairs("e2m1_grid.txt")
    assert len(rows) == 16
    for code_s, val_s in rows:
        code, val = int(code_s, 16), float(val_s)
        got = orc.e2m1_value(code)
        assert got == val and np.signbit(got) == np.signbit(val), (code, got, val)


def test_e2m1_ties_match_golden(orc):
    for x_s, code_s, val_s in _read_pairs("e2m1_ties.txt"):
        code = orc.e2m1_encode(float(x_s))
        assert code == int(code_s, 16), (x_s, code)
        assert orc.e2m1_value(code) == float(val_s)


def _threshold_e2m1(x):
    """Independent encoder: RNE decision thresholds written out per interval
    (midpoints 0.25 .75 1.25 1.75 2.5 3.5 5; ties go to the even code)."""
    s = 8 if np.signbit(x) else 0
    a = abs(float(x))
    if a <= 0.25:
        m = 0
    elif a < 0.75:
        m = 1
    elif a <= 1.25:
        m = 2
    elif a < 1.75:
        m = 3
    elif a <= 2.5:
        m = 4
    elif a < 3.5:
        m = 5
    elif a <= 5.0:
        m = 6
    else:
        m = 7
    return s | m


def test_e2m1_encoder_vs_thresholds(orc):
    rng = np.random.default_rng(1)
    pts = [0.0, -0.0, np.inf, -np.inf]
    for t in [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0, 0.5, 1, 1.5, 2, 3, 4]:
        t32 = np.float32(t)
        pts += [t32, np.nextafter(t32, np.float32(0)), np.nextafter(t32, np.float32(10))]
    pts += list(rng.uniform(-8, 8, 3000).astype(np.float32))
    pts += list((rng.standard_normal(1000) * 1e-3).astype(np.float32))
    for x in pts:
        x = np.float32(x)
        for v in (x, -x):
            assert orc.e2m1_encode(v) == _threshold_e2m1(v), v


def test_e4m3_decode_all_bytes_vs_torch(orc):
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy()
    for b in range(256):
        got = orc.e4m3_value(b)
        if np.isnan(ref[b]):
            assert np.isnan(got), b
        else:
            assert got == ref[b], (b, got, ref[b])
    # format landmarks: max 448, smallest subnormal 2^-9, NaN only at 0x7F/0xFF
    assert orc.e4m3_value(0x7E) == 448.0
    assert orc.e4m3_value(0x01) == 2.0 ** -9
    assert sum(np.isnan(orc.e4m3_value(b)) for b in range(256)) == 2


def test_e4m3_encoder_vs_torch_in_range(orc):
    rng = np.random.default_rng(2)
    grid = np.array([orc.e4m3_value(b) for b in range(127)], np.float64)
    mids = (grid[1:] + grid[:-1]) / 2
    xs = list(grid.astype(np.float32)) + list(mids.astype(np.float32))
    xs += [np.nextafter(np.float32(m), np.float32(0)) for m in mids]
    xs += [np.nextafter(np.float32(m), np.float32(1e9)) for m in mids]
    xs += list(np.exp(rng.uniform(np.log(1e-4), np.log(464), 20000)).astype(np.float32))
    xs += [np.float32(0.0), np.float32(1e-12), np.float32(464.0)]
    xs = np.array(xs, np.float32)
    xs = xs[xs <= 464.0]  # torch's conversion does not saturate above 464
    ref = torch.from_numpy(xs).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([orc.e4m3_encode(x) for x in xs], np.uint8)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, [(xs[i], got[i], ref[i]) for i in bad[:5]]


def test_e4m3_encoder_saturates(orc):
    for x in [464.0001, 480.0, 1e4, 3e38, np.inf]:
        assert orc.e4m3_encode(x) == 0x7E


def test_bf16_conversion_vs_torch(orc):
    rng = np.random.default_rng(3)
    xs = rng.standard_normal(4000).astype(np.float32) * np.float32(100)
    # exact ties between two bf16 values, both parities
    base = rng.integers(0, 2 ** 15, 200, dtype=np.uint32) << 16
    ties = (base | 0x8000).view(np.float32)
    ties = ties[np.isfinite(ties)]  # NaN payloads are not part of the format
    xs = np.concatenate([xs, ties, np.array([0.0, -0.0, 1e-40, -1e-40, 3.3895e38], np.float32)])
    ref = torch.from_numpy(xs).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = orc.f32_to_bf16(xs)
    assert np.array_equal(got, ref)
    bits = rng.integers(0, 2 ** 16, 3000, dtype=np.uint16)
    bits = bits[(bits & 0x7F80) != 0x7F80]
    back = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float().numpy()
    assert np.array_equal(orc.bf16_to_f32(bits).view(np.uint32), back.view(np.uint32))


def _threshold_e2m1_vec(x):
    """Vectorised form of the threshold encoder above (same midpoints and tie
    rule), written independently of the oracle's nearest-grid search."""
    x = np.asarray(x, np.float32)
    a = np.abs(x.astype(np.float64))
    m = np.select([a <= 0.25, a < 0.75, a <= 1.25, a < 1.75, a <= 2.5, a < 3.5, a <= 5.0],
                  [0, 1, 2, 3, 4, 5, 6], default=7)
    return (m | np.where(np.signbit(x), 8, 0)).astype(np.uint8)


@pytest.mark.parametrize("nthreads", [1, 5])
def test_encode_array_matches_independent_encoders(orc, nthreads):
    """The array encoder (the checker behind the device encoder sweeps) splits
    its input into 65,536-element pieces over threads; on lengths that are not
    a multiple of that piece, every byte must equal an independent encoder:
    the E2M1 thresholds for which == 0, PyTorch's float8_e4m3fn conversion
    (saturated at 448 first) for which == 1."""
    rng = np.random.default_rng(11)
    n = 3 * (1 << 16) + 12345
    x = np.concatenate([
        rng.uniform(-7, 7, n // 2).astype(np.float32),
        (rng.standard_normal(n - n // 2 - 6) * 0.3).astype(np.float32),
        np.array([0.25, -0.75, 5.0, -0.0, 6.5, 0.0], np.float32)])
    assert x.size == n and n % (1 << 16) != 0
    got = orc.encode_array(x, 0, nthreads=nthreads)
    ref = _threshold_e2m1_vec(x)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, [(x[i], got[i], ref[i]) for i in bad[:5]]

    y = np.concatenate([np.exp(rng.uniform(np.log(1e-4), np.log(600.0), n - 5)).astype(np.float32),
                        np.array([0.0, 448.0, 464.0, 470.0, 1e6], np.float32)])
    got = orc.encode_array(y, 1, nthreads=nthreads)
    ref = torch.from_numpy(np.minimum(y, np.float32(448.0))).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, [(y[i], got[i], ref[i]) for i in bad[:5]]
    # the tail piece (shorter than 65,536) is encoded too
    assert got[-1] == 0x7E and got[-5] == 0
