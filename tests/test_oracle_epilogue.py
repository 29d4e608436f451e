"""Pins of the oracle's GEGLU epilogue, out = gelu(gate) * (y + bias), gelu(g) =
g * Phi(g) (laya.cpp docs/vulkan.md, feed-forward paragraph: the gate activation
and multiplication fused into one dispatch).  Each pin is independent of the
oracle's own arithmetic: textbook values of the normal distribution function,
an identity of Phi, scipy's normal distribution function, numpy float32
arithmetic."""
import numpy as np
import pytest

import oracle

# Phi(1), Phi(2) to double precision (standard normal table values)
PHI_1 = 0.8413447460685429
PHI_2 = 0.9772498680518208


@pytest.fixture(scope="module", autouse=True)
def built():
    oracle.build()


def test_gelu_closed_forms():
    assert oracle.gelu(0.0) == 0.0
    assert oracle.gelu(1.0) == pytest.approx(PHI_1, rel=1e-15)
    assert oracle.gelu(2.0) == pytest.approx(2.0 * PHI_2, rel=1e-15)
    assert oracle.gelu(-1.0) == pytest.approx(-(1.0 - PHI_1), rel=1e-14)
    assert oracle.gelu(40.0) == 40.0  # Phi(40) is 1 in double
    assert oracle.gelu(-40.0) == 0.0  # -40 * Phi(-40) underflows


def test_gelu_identity_phi_plus_phi_minus_is_one():
    # Phi(g) + Phi(-g) = 1  =>  gelu(g) - gelu(-g) = g: fails for a wrong sign,
    # scale or argument of erf
    for g in np.linspace(-6.0, 6.0, 241):
        assert oracle.gelu(g) - oracle.gelu(-g) == pytest.approx(g, abs=4e-16 * max(1.0, abs(g)))


def test_against_scipy_normal_cdf():
    special = pytest.importorskip("scipy.special")
    rng = np.random.default_rng(7)
    M, N = 200, 1000
    y = rng.standard_normal((M, N)).astype(np.float32) * np.float32(3.0)
    b = rng.standard_normal(N).astype(np.float32)
    g = (rng.standard_normal((M, N)) * 2.5).astype(np.float32)
    out = oracle.epilogue(y, b, g)
    ref = ((y.astype(np.float64) + b.astype(np.float64)) * (g * special.ndtr(g.astype(np.float64)))).astype(np.float32)
    # two double evaluations of erf may differ in the last bit: at most one binary32 ulp apart after rounding
    diff = np.abs(out.view(np.int32).astype(np.int64) - ref.view(np.int32).astype(np.int64))
    assert diff.max() <= 1
    assert np.mean(diff == 0) > 0.999


def test_bias_only_is_a_float32_add_and_none_is_identity():
    rng = np.random.default_rng(3)
    y = rng.standard_normal((64, 300)).astype(np.float32)
    b = (rng.standard_normal(300) * 1e3).astype(np.float32)
    assert np.array_equal(oracle.epilogue(y, b).view(np.uint32), (y + b).view(np.uint32))
    assert np.array_equal(oracle.epilogue(y).view(np.uint32), y.view(np.uint32))


def test_zero_gate_gives_zero():
    y = np.full((3, 5), 7.5, np.float32)
    out = oracle.epilogue(y, None, np.zeros((3, 5), np.float32))
    assert np.all(out == 0.0)


def test_shape_checks():
    y = np.zeros((2, 3), np.float32)
    with pytest.raises(ValueError):
        oracle.epilogue(y, np.zeros(2, np.float32))
    with pytest.raises(ValueError):
        oracle.epilogue(y, None, np.zeros((3, 2), np.float32))
