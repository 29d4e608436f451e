"""Pins for the oracle's binary16 rounding (fp16_rne), independent of the oracle.

The rounding is the one the laya.cpp Vulkan page fixes for the split
(docs/vulkan.md, split/merge paragraph: round to nearest with ties to even, and
subnormal binary16 results kept).  It is checked here against

* brute force: the nearest of all 63,488 finite binary16 values (plus +-2^16
  standing in for +-inf), ties to the even fraction, found by exhaustive search;
* numpy's float16 cast (a library routine) on large random sets of FP32 bit
  patterns and on doubles;
* the exact decode of every binary16 bit pattern.
"""
import numpy as np
import pytest


def _all_candidates():
    """Every finite binary16 value plus +-65536 (for +-inf), with its bits."""
    bits = np.arange(0x10000, dtype=np.uint32).astype(np.uint16)
    vals = bits.view(np.float16).astype(np.float64)
    finite = np.isfinite(vals)
    cand_bits = bits[finite]
    cand_vals = vals[finite]
    cand_bits = np.concatenate([cand_bits, np.array([0x7C00, 0xFC00], np.uint16)])
    cand_vals = np.concatenate([cand_vals, np.array([65536.0, -65536.0])])
    return cand_vals, cand_bits


def _brute_force(v, cand_vals, cand_bits):
    """Nearest candidate by exhaustive search, ties to the even fraction bit."""
    d = np.abs(cand_vals - v)
    best = d.min()
    idx = np.nonzero(d == best)[0]
    if len(idx) == 1:
        b = int(cand_bits[idx[0]])
    else:
        evens = [int(cand_bits[i]) for i in idx if (int(cand_bits[i]) & 1) == 0]
        assert len(evens) >= 1
        # +0 and -0 are both at distance |v|: keep the sign of v
        evens = [b for b in evens if ((b >> 15) & 1) == (1 if np.signbit(v) else 0)] or evens
        b = evens[0]
    if b & 0x7FFF == 0:  # zero result takes the sign of v
        b = 0x8000 if np.signbit(v) else 0
    return b


def test_decode_every_bit_pattern(orc):
    bits = np.arange(0x10000, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([orc.fp16_value(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def test_brute_force_nearest_even(orc):
    cand_vals, cand_bits = _all_candidates()
    rng = np.random.default_rng(1)
    # values of every kind: random FP32 below the overflow tie, subnormal range,
    # exact midpoints between neighbouring binary16 values, and the edges
    mid = (cand_vals[:-2][1:] + cand_vals[:-2][:-1]) / 2
    vals = np.concatenate(
        [
            rng.uniform(-65600, 65600, 400),
            rng.uniform(-1e-4, 1e-4, 300),
            rng.uniform(-1e-7, 1e-7, 100),
            rng.choice(mid[np.isfinite(mid)], 600),
            np.array([0.0, -0.0, 65504.0, 65519.99, 65520.0, 65535.9, -65520.0, 2**-24, 2**-25, 3 * 2**-26,
                      2**-14, 2**-14 - 2**-25, 32784.0, 32816.0, 1 + 2**-11, 1 + 3 * 2**-11]),
        ]
    ).astype(np.float32).astype(np.float64)
    for v in vals:
        want = _brute_force(v, cand_vals, cand_bits)
        got = orc.fp16_rne(v)
        assert got == want, (v, hex(got), hex(want))


def test_matches_numpy_cast_on_random_fp32_bits(orc):
    rng = np.random.default_rng(2)
    b = rng.integers(0, 2**32, 400_000, dtype=np.uint64).astype(np.uint32)
    x = b.view(np.float32)
    hi, _ = orc.split(x)
    with np.errstate(over="ignore", invalid="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    nan = np.isnan(x)
    assert np.all((hi[nan] & 0x7C00) == 0x7C00) and np.all((hi[nan] & 0x3FF) != 0)
    assert np.array_equal(hi[~nan], ref[~nan])


def test_matches_numpy_cast_on_fp32_near_fp16_range(orc):
    # dense sampling of the bit patterns whose values are near binary16's range
    lo_bits = np.float32(2.0**-30).view(np.uint32)
    hi_bits = np.float32(70000.0).view(np.uint32)
    b = np.arange(lo_bits, hi_bits, 97, dtype=np.uint32)
    x = np.concatenate([b.view(np.float32), -b.view(np.float32)])
    hi, _ = orc.split(x)
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(hi, ref)


def test_matches_numpy_cast_on_doubles(orc):
    rng = np.random.default_rng(3)
    v = np.concatenate([rng.normal(0, 1, 2000), rng.normal(0, 1e-5, 2000), rng.uniform(-7e4, 7e4, 2000)])
    got = np.array([orc.fp16_rne(float(t)) for t in v], np.uint16)
    with np.errstate(over="ignore"):
        ref = v.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, ref)


def test_nan_and_inf(orc):
    assert orc.fp16_rne(float("inf")) == 0x7C00
    assert orc.fp16_rne(float("-inf")) == 0xFC00
    n = orc.fp16_rne(float("nan"))
    assert (n & 0x7C00) == 0x7C00 and (n & 0x3FF) != 0
