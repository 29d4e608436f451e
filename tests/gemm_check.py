"""The elementwise gate shared by the GPU projection tests.

Gate (the method's acceptance for the projection, laya.cpp docs/vulkan.md,
compensated-FP32 paragraph, with the stated tolerance): every element of y
satisfies |y - y_oracle| <= 4e-6 * sum_k |x_k||w_k| + 1e-30, where y_oracle is
the oracle's FP64 evaluation of the same formula; the max-normalised error
against the true product is returned beside that of a single FP16 cast of x so
that callers can also demand the 100x accuracy gain.
"""
import numpy as np
import torch

TOL = 4e-6


def w_bits(W):
    return W.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def check_comp(y, x, W, orc, rows=None, cols=None):
    """Elementwise gate against the oracle; returns (gpu error, cast error) max-normalised vs the true product."""
    xn, wn = x.cpu().numpy(), w_bits(W)
    yg = y.detach().cpu().numpy()
    if rows is not None:
        yg = yg[rows, cols]
    y_or = orc.gemm_comp(xn, wn, rows, cols).astype(np.float64)
    den = orc.gemm_den(xn, wn, rows, cols)
    err = np.abs(yg.astype(np.float64) - y_or)
    bound = TOL * den + 1e-30
    bad = np.argwhere(~(err <= bound))
    assert bad.size == 0, (
        f"{bad.shape[0]} elements over tolerance; first {bad[:3].tolist()}, "
        f"worst ratio {float(np.nanmax(err / bound))}"
    )
    y_true = orc.gemm_true(xn, wn, rows, cols).astype(np.float64)
    y_cast = orc.gemm_cast(xn, wn, rows, cols).astype(np.float64)
    e_gpu = float(np.max(np.abs(yg - y_true) / (den + 1e-30)))
    e_cast = float(np.max(np.abs(y_cast - y_true) / (den + 1e-30)))
    return e_gpu, e_cast


def sample_outputs(M, N, seed=5, count=3000):
    """Row-sorted (rows, cols): random outputs plus the corners and edges of an M x N result."""
    rng = np.random.default_rng(seed)
    r = np.concatenate([rng.integers(0, M, count), [0, 0, M - 1, M - 1], np.full(16, M - 1),
                        np.arange(min(M, 16))])
    c = np.concatenate([rng.integers(0, N, count), [0, N - 1, 0, N - 1], np.arange(N - 16, N),
                        np.full(min(M, 16), N - 1)])
    order = np.argsort(r, kind="stable")
    return r[order], c[order]
