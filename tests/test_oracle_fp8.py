"""Pins of the oracle's FP8-E4M3 element format.

The decoder is pinned to code points of the format definition; the encoder to a
brute-force nearest search over every finite code (ties to the even mantissa,
saturating at 448), to torch's float8 cast on in-range values, and to the
slot-write rule e4m3(fl32(x) / scale).
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _points():
    with open(os.path.join(GOLDEN, "e4m3_points.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                code, val = line.split()
                yield int(code, 16), val


@pytest.mark.parametrize("code,val", list(_points()))
def test_decode_code_points(code, val):
    got = oracle.decode_bits(np.array([code], np.uint8), oracle.FP8_E4M3)[0]
    if val == "nan":
        assert math.isnan(got)
    else:
        assert got == float(val)
        assert math.copysign(1.0, got) == math.copysign(1.0, float(val))


def _finite_table():
    codes = np.arange(256, dtype=np.uint8)
    vals = oracle.decode_bits(codes, oracle.FP8_E4M3)
    keep = ~np.isnan(vals)
    return codes[keep], vals[keep]


def _brute_nearest(x: np.ndarray) -> np.ndarray:
    """Nearest finite code by a search over the full table of decoded codes: the
    neighbours of |x| among all non-negative finite values, compared exactly;
    exact ties go to the even mantissa; NaN -> S.1111.111; +-0 and +-inf keep the sign."""
    codes, vals = _finite_table()
    pos = ~np.signbit(vals)
    pcodes, pvals = codes[pos], vals[pos]
    order = np.argsort(pvals)
    pcodes, pvals = pcodes[order], pvals[order]
    assert np.all(np.diff(pvals) > 0)
    x = np.asarray(x, np.float64).ravel()
    neg = np.signbit(x)
    ax = np.abs(x)
    out = np.zeros(x.shape, np.uint8)
    hi = np.searchsorted(pvals, ax, side="left")           # first value >= |x|
    lo = np.clip(hi - 1, 0, pvals.size - 1)
    hi_c = np.clip(hi, 0, pvals.size - 1)
    d_lo = ax - pvals[lo]
    d_hi = np.where(hi < pvals.size, pvals[hi_c] - ax, np.inf)
    exact = (hi < pvals.size) & (pvals[hi_c] == ax)
    take_hi = exact | (d_hi < d_lo) | ((d_hi == d_lo) & (pcodes[hi_c] % 2 == 0))
    mag = np.where(take_hi, pcodes[hi_c], pcodes[lo])
    out[:] = mag | np.where(neg, 0x80, 0x00).astype(np.uint8)
    nan = np.isnan(x)
    out[nan] = np.where(neg[nan], 0xFF, 0x7F)
    return out


def test_encode_all_codes_roundtrip():
    codes, vals = _finite_table()
    got = oracle.e4m3_encode(vals.astype(np.float32))
    assert np.array_equal(got, codes)


@pytest.mark.filterwarnings("ignore::RuntimeWarning")
def test_encode_brute_force_dense_grid():
    # every bf16 bit pattern, as float32
    bits = np.arange(65536, dtype=np.uint32) << 16
    x = bits.view(np.float32)
    got = oracle.e4m3_encode(x)
    exp = _brute_nearest(x)
    mism = np.nonzero(got != exp)[0]
    assert mism.size == 0, [(float(x[i]), hex(got[i]), hex(exp[i])) for i in mism[:10]]


def test_encode_ties_and_saturation():
    cases = {
        0.5 * 2**-9: 0x00,         # tie between 0 and 2^-9 -> even (0)
        1.5 * 2**-9: 0x02,         # tie between codes 1 and 2 -> 2
        2.5 * 2**-9: 0x02,         # tie between 2 and 3 -> 2
        1.0625: 0x38,              # tie between 1.0 and 1.125 -> 1.0 (even)
        1.1875: 0x3A,              # tie between 1.125 and 1.25 -> 1.25 (even)
        448.0: 0x7E,
        463.99: 0x7E,
        464.0: 0x7E,               # tie with the unrepresentable 480 -> 448
        1e6: 0x7E,
        float("inf"): 0x7E,
        -float("inf"): 0xFE,
        -1e-30: 0x80,              # rounds to -0
    }
    x = np.array(list(cases.keys()), np.float32)
    got = oracle.e4m3_encode(x)
    assert [hex(c) for c in got] == [hex(c) for c in cases.values()]


def test_encode_nan_keeps_sign():
    x = np.array([np.nan, -np.nan], np.float32)
    x[1] = -np.abs(x[1])
    got = oracle.e4m3_encode(x)
    assert got[0] == 0x7F and got[1] == 0xFF


def test_encode_matches_torch_cast_in_range():
    g = torch.Generator().manual_seed(5)
    x = torch.randn(200000, generator=g) * 60
    x = x.clamp(-448, 448)
    ref = x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = oracle.e4m3_encode(x.numpy())
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("scale", [1.0, 5.9 / 448.0, 2.0**-4, 1e-3, 0.37])
@pytest.mark.filterwarnings("ignore::RuntimeWarning")
def test_quantize_rule_is_fl32_quotient_then_rne(scale):
    # the slot-write rule: the quotient is rounded once to binary32, then to E4M3
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    xf = (bits.astype(np.uint32) << 16).view(np.float32)
    q32 = (xf / np.float32(scale)).astype(np.float32)   # IEEE float32 division
    exp = _brute_nearest(q32)
    nan = np.isnan(q32)
    exp[nan] = np.where(np.signbit(xf[nan]), 0xFF, 0x7F)  # a NaN code takes the source element's sign
    got = oracle.quantize(bits, oracle.BF16, scale)
    mism = np.nonzero(got != exp)[0]
    assert mism.size == 0, [(float(xf[i]), hex(got[i]), hex(exp[i])) for i in mism[:10]]


def test_quantize_fp16_source():
    g = np.random.default_rng(3)
    x = (g.standard_normal(5000) * 3).astype(np.float16)
    scale = 0.02
    q32 = (x.astype(np.float32) / np.float32(scale)).astype(np.float32)
    assert np.array_equal(oracle.quantize(x.view(np.uint16), oracle.FP16, scale), _brute_nearest(q32))


def test_fp16_and_bf16_decode_match_numpy_torch():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    f16 = oracle.decode_bits(bits, oracle.FP16)
    ref16 = bits.view(np.float16).astype(np.float64)
    assert np.array_equal(np.isnan(f16), np.isnan(ref16))
    ok = ~np.isnan(ref16)
    assert np.array_equal(f16[ok], ref16[ok])
    bf = oracle.decode_bits(bits, oracle.BF16)
    refbf = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()
    ok = ~np.isnan(refbf)
    assert np.array_equal(bf[ok], refbf[ok]) and np.array_equal(np.isnan(bf), np.isnan(refbf))
