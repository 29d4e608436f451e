"""The seeded input generators (no method arithmetic): they produce the value
classes the parity tests rely on."""
import numpy as np
import torch

from compensated_fp32_projection_gb300 import workloads


def test_special_values_cover_their_classes():
    n = 1 << 16
    x = workloads.special_values_f32(n, seed=3).numpy()
    assert x.dtype == np.float32 and x.size == n
    assert np.isfinite(x).all() and np.abs(x).max() <= 65504.0
    k = n // 4
    # first quarter: midpoints between neighbouring FP16 values, or the FP32 values beside them
    a = np.abs(x[:k]).astype(np.float64)
    lo16 = a.astype(np.float16)  # nearest FP16 (either neighbour)
    below = np.where(lo16.astype(np.float64) > a, np.nextafter(lo16, np.float16(0)), lo16).astype(np.float64)
    above = np.nextafter(below.astype(np.float16), np.float16(np.inf)).astype(np.float64)
    mid = ((below + above) / 2).astype(np.float32)
    ulp = np.abs(np.nextafter(mid, np.float32(np.inf)) - mid).astype(np.float64)
    assert np.all(np.abs(a - mid.astype(np.float64)) <= ulp + 0.0)
    exact_ties = np.mean(a == mid.astype(np.float64))
    assert 0.2 < exact_ties < 0.5  # a third are the ties themselves, the rest their neighbours
    # the block next to the FP16 maximum and the FP16-subnormal block
    assert np.all((x[k:k + 1000] >= 65000.0) & (x[k:k + 1000] <= 65504.0))
    tiny = np.abs(x[k + 1000:k + 2000])
    assert np.median(tiny) < 2.0**-14  # hi and lo mostly FP16-subnormal there
    # the rest: both FP16-subnormal and FP16-normal magnitudes, both signs
    rest = x[k + 2000:]
    assert np.mean(np.abs(rest) < 2.0**-14) > 0.1 and np.mean(np.abs(rest) >= 2.0**-14) > 0.5
    assert np.mean(rest < 0) > 0.4 and np.mean(rest > 0) > 0.4


def test_special_values_are_seeded():
    a = workloads.special_values_f32(4096, seed=1)
    b = workloads.special_values_f32(4096, seed=1)
    c = workloads.special_values_f32(4096, seed=2)
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))
    assert not torch.equal(a.view(torch.int32), c.view(torch.int32))
