"""Pins for the oracle's GEMMs, independent of the oracle's own loops.

The compensated product (laya.cpp, docs/vulkan.md, compensated-FP32 paragraph):
both FP16 components of x are multiplied by the exact FP16 weights and the two
results are combined, y = acc_hi + 2^-10 acc_lo.  The oracle sums in FP64.

Pinned by:
* the true product against numpy's float64 matmul (a library routine), which
  catches transposed operands and index mistakes in the shared loop structure;
* closed forms: inputs that are exact in FP16 (lo = 0, so the compensated, cast
  and true products coincide), one-hot rows (y is one weight times x), W = I
  (y reconstructs x within the split bound);
* the split's reconstruction bound carried through the sum:
  |y_comp - y_true| <= 2^-23 den + 2^-35 sum|w| + 2^-24 |y| (a dropped residual
  or a wrong scale fails this by orders of magnitude);
* the method's claim: at least 100x smaller max-normalised error than a single
  FP16 cast on the five projection shapes.
"""
import numpy as np
import pytest

from compensated_fp32_projection_gb300 import workloads


def _w64(W):
    return np.asarray(W, np.uint16).view(np.float16).astype(np.float64)


def _case(M, N, K, seed, scale=1.0):
    x, W = workloads.random_case(M, N, K, seed, scale)
    return x.numpy(), W.numpy().view(np.uint16)


def test_true_gemm_matches_numpy_matmul(orc):
    for (M, N, K, s) in [(7, 5, 3, 1), (33, 17, 65, 2), (64, 48, 200, 3)]:
        x, W = _case(M, N, K, s)
        y = orc.gemm_true(x, W)
        ref = (x.astype(np.float64) @ _w64(W).T)
        den = np.abs(x.astype(np.float64)) @ np.abs(_w64(W)).T
        assert y.shape == (M, N)
        assert np.all(np.abs(y - ref) <= 2.0**-24 * np.abs(ref) + 1e-12 * den)
        assert np.allclose(orc.gemm_den(x, W), den, rtol=1e-12, atol=0)


def test_cast_gemm_matches_numpy_fp16_cast_then_matmul(orc):
    # the single-FP16-cast product is numpy's round-to-nearest-even float16 cast
    # of x (a library routine) times W in float64, rounded once to binary32; a
    # cast that truncates or flushes subnormals, or a sum over the wrong
    # operand, fails this by orders of magnitude more than the bound
    for (M, N, K, s, scale) in [(9, 7, 5, 6, 1.0), (40, 24, 131, 7, 3.0), (16, 32, 520, 8, 1e-5)]:
        x, W = _case(M, N, K, s, scale)
        ref = x.astype(np.float16).astype(np.float64) @ _w64(W).T
        den = np.abs(x.astype(np.float64)) @ np.abs(_w64(W)).T
        y = orc.gemm_cast(x, W).astype(np.float64)
        assert np.all(np.abs(y - ref) <= 2.0**-24 * np.abs(ref) + 1e-15 * den + 2.0**-149)
        # and it is far from the compensated result wherever the cast loses bits
        yc = orc.gemm_comp(x, W).astype(np.float64)
        assert np.max(np.abs(y - yc) / (den + 1e-300)) > 1e-6


def test_exact_fp16_inputs_all_products_coincide(orc):
    x, W = _case(40, 30, 77, 4)
    x = x.astype(np.float16).astype(np.float32)  # every x is exact in FP16, so lo = 0
    yc = orc.gemm_comp(x, W)
    yt = orc.gemm_true(x, W)
    yk = orc.gemm_cast(x, W)
    assert np.array_equal(yc.view(np.uint32), yt.view(np.uint32))
    assert np.array_equal(yc.view(np.uint32), yk.view(np.uint32))
    ref = (x.astype(np.float64) @ _w64(W).T)
    assert np.all(np.abs(yc - ref) <= 2.0**-24 * np.abs(ref) + 1e-300)


def test_one_hot_rows(orc):
    K, N = 50, 20
    _, W = _case(1, N, K, 5)
    c = np.float32(1.0 / 3.0)
    x = np.zeros((K, K), np.float32)
    x[np.arange(K), np.arange(K)] = c
    y = orc.gemm_comp(x, W)
    # y[i, j] = fp32((hi_c + lo_c/1024) * w[j, i]); hi_c, lo_c of 1/3 from the hand table
    hi_c, lo_c = _w64(np.uint16(0x3555)), _w64(np.uint16(0x2D56))
    ref = ((hi_c + lo_c / 1024.0) * _w64(W).T).astype(np.float32)
    assert np.array_equal(y, ref)
    # an exact FP16 value: y is the weight times it exactly
    x2 = np.zeros((K, K), np.float32)
    x2[np.arange(K), np.arange(K)] = -2.5
    y2 = orc.gemm_comp(x2, W)
    assert np.array_equal(y2, (-2.5 * _w64(W).T).astype(np.float32))


def test_identity_weights_reconstruct_x(orc):
    K = 64
    W = np.eye(K, dtype=np.float16).view(np.uint16)
    rng = np.random.default_rng(6)
    x = np.concatenate([rng.normal(0, 1, (8, K)), rng.uniform(-65000, 65000, (8, K)),
                        rng.normal(0, 1e-6, (8, K))]).astype(np.float32)
    y = orc.gemm_comp(x, W)
    xd = x.astype(np.float64)
    assert np.all(np.abs(y.astype(np.float64) - xd) <= 2.0**-22 * np.abs(xd) + 2.0**-35)
    # and it is more accurate than the FP16 cast alone wherever the cast is inexact
    yc = orc.gemm_cast(x, W)
    inexact = yc.astype(np.float64) != xd
    assert np.all(np.abs(y - xd)[inexact] < np.abs(yc - xd)[inexact])


def test_comp_within_split_bound_of_true(orc):
    for (M, N, K, s, scale) in [(31, 29, 130, 7, 1.0), (16, 40, 300, 8, 1e4), (12, 9, 1027, 9, 1e-5)]:
        x, W = _case(M, N, K, s, scale)
        yc = orc.gemm_comp(x, W).astype(np.float64)
        yt_exact = x.astype(np.float64) @ _w64(W).T
        den = np.abs(x.astype(np.float64)) @ np.abs(_w64(W)).T
        wsum = np.abs(_w64(W)).sum(axis=1)[None, :]
        bound = 2.0**-23 * den + 2.0**-35 * wsum + 2.0**-24 * np.abs(yt_exact) + 1e-300
        assert np.all(np.abs(yc - yt_exact) <= bound)
        # a single FP16 cast is typically ~1000x worse; the bound must be tight
        # enough to tell the two apart
        yk = orc.gemm_cast(x, W).astype(np.float64)
        assert np.max(np.abs(yk - yt_exact) / bound) > 20


def test_sampled_equals_full(orc):
    x, W = _case(37, 45, 99, 10)
    full = orc.gemm_comp(x, W)
    rng = np.random.default_rng(0)
    r = rng.integers(0, 37, 200)
    c = rng.integers(0, 45, 200)
    order = np.argsort(r, kind="stable")
    r, c = r[order], c[order]
    for fn in (orc.gemm_comp, orc.gemm_true, orc.gemm_cast, orc.gemm_den):
        got = fn(x, W, r, c)
        ref = fn(x, W)[r, c]
        assert np.array_equal(got, ref)
    assert np.array_equal(orc.gemm_comp(x, W, r, c), full[r, c])


def test_weights_are_rne_of_the_fp32_draws(orc):
    import torch

    g = torch.Generator().manual_seed(123)
    w32 = torch.randn((64, 64), generator=g) * 0.02
    W = w32.half().numpy().view(np.uint16)
    hi, _ = orc.split(w32.numpy())
    assert np.array_equal(W, hi)


def _max_norm_err(y, y_true, den):
    return float(np.max(np.abs(y.astype(np.float64) - y_true.astype(np.float64)) / (den + 1e-30)))


@pytest.mark.parametrize("name", ["tiny", "encoder", "nonaligned"])
def test_hundredfold_over_fp16_cast_small_shapes(orc, name):
    x, W = workloads.make_inputs(name)
    x, W = x.numpy(), W.numpy().view(np.uint16)
    den = orc.gemm_den(x, W)
    y_true = orc.gemm_true(x, W)
    e_comp = _max_norm_err(orc.gemm_comp(x, W), y_true, den)
    e_cast = _max_norm_err(orc.gemm_cast(x, W), y_true, den)
    assert e_cast >= 100 * e_comp, (e_cast, e_comp)


@pytest.mark.parametrize("name", ["square", "skinny"])
def test_hundredfold_over_fp16_cast_sampled(orc, name):
    x, W = workloads.make_inputs(name)
    x, W = x.numpy(), W.numpy().view(np.uint16)
    rng = np.random.default_rng(1)
    M, N = x.shape[0], W.shape[0]
    r = np.sort(rng.integers(0, M, 400))
    c = rng.integers(0, N, 400)
    den = orc.gemm_den(x, W, r, c)
    y_true = orc.gemm_true(x, W, r, c)
    e_comp = _max_norm_err(orc.gemm_comp(x, W, r, c), y_true, den)
    e_cast = _max_norm_err(orc.gemm_cast(x, W, r, c), y_true, den)
    assert e_cast >= 100 * e_comp, (e_cast, e_comp)
