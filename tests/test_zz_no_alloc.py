"""comp_gemm_f32x16_noalloc: the two-pass projection with the library's static
device workspace, for callers that cannot allocate device memory per call.

Called through the C ABI (ctypes on the library's symbol) and compared with
the existing workspace entry point comp_gemm_f32x16_ws within the projection
gate's tolerance, 4e-6 * sum|x||w| + 1e-30 per element, on two calls in a
row.  The file is named to be collected last, so that it also runs after
every other test in the same process; it builds and loads the library itself,
so it runs alone in a fresh process too.
"""
import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from gemm_check import TOL, w_bits  # noqa: E402

MAX_BYTES = 64 * 1024 * 1024


@pytest.fixture(scope="module")
def lib():
    from compensated_fp32_projection_gb300 import _native, build

    build.build()
    return _native.load()


@pytest.fixture(scope="module")
def pkg(lib):
    import compensated_fp32_projection_gb300 as p

    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return p


def noalloc(lib, x, W, y):
    stream = torch.cuda.current_stream(x.device).cuda_stream
    return lib.comp_gemm_f32x16_noalloc(x.data_ptr(), W.data_ptr(), y.data_ptr(), x.shape[0], W.shape[0],
                                        x.shape[1], ctypes.c_void_p(stream))


def test_size_limit_rejected_before_any_device_work(lib):
    P = ctypes.c_void_p
    # 4*M*K one element beyond 64 MiB, and overflowing products: rejected, never truncated
    assert lib.comp_gemm_f32x16_noalloc(P(4096), P(1 << 20), P(1 << 24), 4097, 8, 4096, None) == 1
    assert lib.comp_gemm_f32x16_noalloc(P(4096), P(1 << 20), P(1 << 24), 1, 8, MAX_BYTES // 4 + 1, None) == 1
    assert lib.comp_gemm_f32x16_noalloc(P(4096), P(1 << 20), P(1 << 24), 1 << 40, 8, 1 << 40, None) == 1
    assert lib.comp_gemm_f32x16_noalloc(P(4096), P(1 << 20), P(1 << 24), -1, 8, 8, None) == 1
    assert lib.comp_gemm_f32x16_noalloc(None, None, None, 0, 8, 8, None) == 0  # empty: no-op
    if not torch.cuda.is_available():
        # valid sizes without a usable device: an error, never a CPU path
        assert lib.comp_gemm_f32x16_noalloc(P(4096), P(1 << 20), P(1 << 24), 8, 8, 8, None) == 2


@pytest.mark.gpu
@pytest.mark.parametrize("shape", [(512, 1024, 1024), (130, 300, 72), (129, 257, 1027), (4096, 512, 4096)],
                         ids=lambda s: "x".join(map(str, s)))
def test_matches_workspace_entry_on_two_calls(pkg, lib, orc, shape):
    from compensated_fp32_projection_gb300 import workloads

    M, N, K = shape
    x, W = workloads.random_case(M, N, K, seed=M + 3 * N + 7 * K, scale=2.0)
    xd, Wd = x.cuda(), W.cuda()
    y_ref = pkg.comp_gemm_f32x16_ws(xd, Wd).cpu().numpy().astype(np.float64)
    den = orc.gemm_den(x.numpy(), w_bits(W))
    bound = TOL * den + 1e-30
    for _ in range(2):
        y = torch.full((M, N), float("nan"), device="cuda")
        assert noalloc(lib, xd, Wd, y) == 0
        torch.cuda.synchronize()
        err = np.abs(y.cpu().numpy().astype(np.float64) - y_ref)
        assert np.all(err <= bound), float(np.max(err / bound))


@pytest.mark.gpu
def test_largest_allowed_activation(pkg, lib):
    # M * K = 16 * 2^20 exactly fills the workspace
    M, N, K = 4096, 64, 4096
    g = torch.Generator().manual_seed(41)
    x = torch.randn((M, K), generator=g).cuda()
    W = (torch.randn((N, K), generator=g) * 0.02).half().cuda()
    y_ref = pkg.comp_gemm_f32x16_ws(x, W)
    y = torch.empty(M, N, device="cuda")
    assert noalloc(lib, x, W, y) == 0
    den = (x.double().abs() @ W.double().abs().t())
    assert torch.all((y.double() - y_ref.double()).abs() <= TOL * den + 1e-30)
    assert noalloc(lib, x[:, :-8].contiguous(), W[:, :-8].contiguous(), y) == 0
    big = torch.empty(M + 1, K, device="cuda")
    assert noalloc(lib, big, W, torch.empty(M + 1, N, device="cuda")) == 1


@pytest.mark.gpu
def test_device_status_clean(pkg):
    st, where = pkg.device_status()
    assert st == 0 and where == 0
