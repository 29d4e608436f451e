"""What the chunked accumulation buys, measured (laya.cpp docs/vulkan.md, AMD
accumulation paragraph: the partial results of the tiles are summed by plain
FP32 additions instead of one long chain of cooperative-matrix multiply-adds,
which removes the accumulation drift of long dot products).

The product kernels restart the tensor-core accumulation every 128 of K and
add the pieces in FP32 registers.  comp_gemm_f16x2_variant 4 is the same
single-CTA product kernel compiled with one tensor-core chain per product over
all of K (hi and lo in separate accumulators, merged once at the tile end).
On x ~ N(0, 1), W ~ N(0, 0.02) with 256 x 512 outputs, at K = 4096 and 16384,
the test reports the max-normalised error E(y) = max |y - y_true| / sum|x||w|
of both (y_true the oracle's exact product) next to that of a single FP16 cast
of x, and the time of each kernel; it asserts that the chunked form meets the
gate and the 100x gain and is more accurate than the single chain.
"""
import json
import os
import statistics

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

from gemm_check import check_comp, w_bits  # noqa: E402


@pytest.fixture(scope="module")
def pkg():
    import __graft_entry__

    __graft_entry__.build()
    import compensated_fp32_projection_gb300 as p

    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return p


def _max_norm(y, y_true, den):
    return float(np.max(np.abs(y.astype(np.float64) - y_true) / (den + 1e-30)))


def _time(fn, reps=10):
    for _ in range(2):
        fn()
    ts = []
    for _ in range(reps):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        b.synchronize()
        ts.append(a.elapsed_time(b) * 1e3)
    return statistics.median(ts)


@pytest.mark.parametrize("K", [4096, 16384])
def test_chunked_promotion_against_one_chain(pkg, orc, K):
    from compensated_fp32_projection_gb300 import workloads

    M, N = 256, 512
    x, W = workloads.random_case(M, N, K, seed=K, scale=1.0)
    xd, Wd = x.cuda(), W.cuda()
    hi, lo = pkg.comp_split_f32(xd)
    y_chunk = pkg.comp_gemm_f16x2_variant(hi, lo, Wd, 1)
    y_chain = pkg.comp_gemm_f16x2_variant(hi, lo, Wd, 4)
    torch.cuda.synchronize()
    xn, wn = x.numpy(), w_bits(W)
    y_true = orc.gemm_true(xn, wn).astype(np.float64)
    den = orc.gemm_den(xn, wn)
    e_chunk = _max_norm(y_chunk.cpu().numpy(), y_true, den)
    e_chain = _max_norm(y_chain.cpu().numpy(), y_true, den)
    e_cast = _max_norm(orc.gemm_cast(xn, wn), y_true, den)
    t_chunk = _time(lambda: pkg.comp_gemm_f16x2_variant(hi, lo, Wd, 1, y=y_chunk))
    t_chain = _time(lambda: pkg.comp_gemm_f16x2_variant(hi, lo, Wd, 4, y=y_chain))
    figures = {"M": M, "N": N, "K": K, "E_chunked_128": e_chunk, "E_one_chain": e_chain, "E_fp16_cast": e_cast,
               "gain_chunked": e_cast / e_chunk, "gain_one_chain": e_cast / e_chain,
               "us_chunked": t_chunk, "us_one_chain": t_chain}
    print("\naccumulation " + json.dumps(figures))
    out = os.environ.get("COMP_ACCUMULATION_REPORT")
    if out:
        with open(out, "a") as f:
            f.write(json.dumps(figures) + "\n")
    check_comp(y_chunk, x, W, orc)
    assert e_cast >= 100 * e_chunk, figures
    assert e_chain > e_chunk, figures
