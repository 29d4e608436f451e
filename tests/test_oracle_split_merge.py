"""Pins for the oracle's split and merge, independent of the oracle.

Split (laya.cpp, docs/vulkan.md, split/merge paragraph): hi = fp16_rne(x),
lo = fp16_rne((x - hi) * 1024), round-to-nearest-even including subnormals.
Merge: y = acc_hi + acc_lo * 2^-10 in FP32 (the "combines them in FP32" of the
compensated-FP32 paragraph, with the 1024 scale undone).

Pinned by: hand-derived bits (tests/golden), numpy's float16 cast and float32
arithmetic (library routines), and the reconstruction bound that follows from
the definition: for finite |x| < 65520,
    |x - (hi + lo/1024)| <= max(2^-23 |x|, 2^-35)   and   |lo| <= 2^14,
and the page's 2^-22 |x| form for |x| >= 2^-13.
"""
import numpy as np

from conftest import read_golden


def _f16(bits):
    return np.asarray(bits, np.uint16).view(np.float16).astype(np.float64)


def test_split_handset_golden(orc):
    rows = read_golden("split_handset.txt")
    xb = np.array([r[0] for r in rows], np.uint32)
    hi, lo = orc.split(xb.view(np.float32))
    for (x, h, l), gh, gl in zip(rows, hi, lo):
        assert (int(gh), int(gl)) == (h, l), (hex(x), hex(gh), hex(gl), hex(h), hex(l))


def test_split_golden_agrees_with_numpy():
    # the hand-derived table itself, re-checked with the library cast
    rows = read_golden("split_handset.txt")
    x = np.array([r[0] for r in rows], np.uint32).view(np.float32)
    with np.errstate(over="ignore", invalid="ignore"):
        hi = x.astype(np.float16)
        r = x.astype(np.float64) - hi.astype(np.float64)
        lo = (r * 1024).astype(np.float16)
    assert [int(v) for v in hi.view(np.uint16)] == [r[1] for r in rows]
    assert [int(v) for v in lo.view(np.uint16)] == [r[2] for r in rows]


def test_split_matches_library_cast(orc):
    rng = np.random.default_rng(11)
    b = rng.integers(0, 2**32, 300_000, dtype=np.uint64).astype(np.uint32)
    x = np.concatenate([b.view(np.float32), rng.normal(0, 1, 100_000).astype(np.float32),
                        rng.uniform(-65519, 65519, 100_000).astype(np.float32)])
    hi, lo = orc.split(x)
    with np.errstate(over="ignore", invalid="ignore"):
        hi_ref = x.astype(np.float16)
        r = x.astype(np.float64) - hi_ref.astype(np.float64)
        lo_ref = (r * 1024).astype(np.float16)
    nan = np.isnan(x) | np.isnan(lo_ref.astype(np.float64))
    assert np.array_equal(hi[~nan], hi_ref.view(np.uint16)[~nan])
    assert np.array_equal(lo[~nan], lo_ref.view(np.uint16)[~nan])
    # NaN inputs: both components are NaN
    xn = np.isnan(x)
    assert np.all(np.isnan(_f16(hi[xn]))) and np.all(np.isnan(_f16(lo[xn])))


def test_split_reconstruction_bound(orc):
    rng = np.random.default_rng(12)
    lo_b = np.float32(2.0**-149).view(np.uint32)
    hi_b = np.float32(65519.996).view(np.uint32)
    b = rng.integers(lo_b, hi_b + 1, 1_000_000, dtype=np.uint64).astype(np.uint32)
    x = b.view(np.float32)
    x = np.concatenate([x, -x])
    hi, lo = orc.split(x)
    xd = x.astype(np.float64)
    rec = _f16(hi) + _f16(lo) / 1024.0
    err = np.abs(xd - rec)
    assert np.all(err <= np.maximum(2.0**-23 * np.abs(xd), 2.0**-35))
    assert np.all(np.abs(_f16(lo)) <= 2.0**14)
    big = np.abs(xd) >= 2.0**-13
    assert np.all(err[big] <= 2.0**-22 * np.abs(xd[big]))
    # the residual is a genuine correction: it makes the error smaller than hi alone
    alone = np.abs(xd - _f16(hi))
    assert np.all(err <= alone)


def test_split_exact_fp16_inputs_have_zero_lo(orc):
    bits = np.arange(0x10000, dtype=np.uint32).astype(np.uint16)
    v = bits.view(np.float16)
    v = v[np.isfinite(v)].astype(np.float32)
    hi, lo = orc.split(v)
    assert np.array_equal(hi, v.astype(np.float16).view(np.uint16))
    assert np.all((lo & 0x7FFF) == 0)


def test_merge_golden(orc):
    rows = read_golden("merge_special.txt")
    a = np.array([r[0] for r in rows], np.uint32).view(np.float32)
    b = np.array([r[1] for r in rows], np.uint32).view(np.float32)
    y = orc.merge(a, b).view(np.uint32)
    for (ha, hb, hy), g in zip(rows, y):
        assert int(g) == hy, (hex(ha), hex(hb), hex(int(g)), hex(hy))


def test_merge_golden_agrees_with_numpy():
    rows = read_golden("merge_special.txt")
    a = np.array([r[0] for r in rows], np.uint32).view(np.float32)
    b = np.array([r[1] for r in rows], np.uint32).view(np.float32)
    with np.errstate(over="ignore", invalid="ignore"):
        y = a + b * np.float32(2.0**-10)
    assert [int(v) for v in y.view(np.uint32)] == [r[2] for r in rows]


def test_merge_matches_numpy_float32(orc):
    rng = np.random.default_rng(13)
    n = 500_000
    scale = 2.0 ** rng.integers(-140, 120, n)
    a = (rng.normal(0, 1, n) * scale).astype(np.float32)
    b = (rng.normal(0, 1, n) * scale * 2.0 ** rng.integers(-20, 20, n)).astype(np.float32)
    bits = rng.integers(0, 2**32, n, dtype=np.uint64).astype(np.uint32).view(np.float32)
    a = np.concatenate([a, bits, -b * np.float32(2.0**-10)])
    b = np.concatenate([b, bits[::-1].copy(), b])
    y = orc.merge(a, b)
    with np.errstate(over="ignore", invalid="ignore"):
        ref = a + b * np.float32(2.0**-10)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(y), nan)
    assert np.array_equal(y[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_merge_inverts_split_scale(orc):
    # merging the split components themselves reconstructs x to within the bound
    rng = np.random.default_rng(14)
    x = rng.normal(0, 100, 100_000).astype(np.float32)
    hi, lo = orc.split(x)
    y = orc.merge(_f16(hi).astype(np.float32), _f16(lo).astype(np.float32))
    xd = x.astype(np.float64)
    assert np.all(np.abs(y.astype(np.float64) - xd) <= 2.0**-22 * np.abs(xd) + 2.0**-35)
