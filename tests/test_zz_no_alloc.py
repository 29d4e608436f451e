"""comp_gemm_f32x16_noalloc: the two-pass projection with the library's static
device workspace, for callers that cannot allocate device memory per call (a
plain C host with no device allocator of its own, or a serving loop that
cannot afford cudaFree's device synchronisation).

Called through the C ABI (ctypes on the library's symbol).  Given the same
inputs it runs the same kernels as the workspace entry point
comp_gemm_f32x16_ws, so on two calls in a row its output must equal that
entry point's bit for bit; one shape is also checked element by element
against the oracle within the projection gate, 4e-6 * sum|x||w| + 1e-30.  A
shape whose K is not a multiple of 8 and whose padded two-pass form does not
fit the static workspace (while 4 * M * K does) takes the fused kernel
instead, and is checked against the oracle on sampled outputs.  The file is
named to be collected last, so that it also runs after every other test in
the same process; it builds and loads the library itself, so it runs alone in
a fresh process too.
"""
import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from gemm_check import check_comp, sample_outputs  # noqa: E402

MAX_BYTES = 64 * 1024 * 1024
COMP_ERR_INVALID_VALUE = 1
COMP_ERR_UNSUPPORTED_DEVICE = 3


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


def bits(t):
    return t.detach().cpu().contiguous().view(torch.int32).numpy()


def test_size_limit_rejected_before_any_device_work(lib):
    P = ctypes.c_void_p
    # 4*M*K one element beyond 64 MiB, and overflowing products: rejected, never truncated
    assert lib.comp_gemm_f32x16_noalloc(P(4096), P(1 << 20), P(1 << 24), 4097, 8, 4096, None) == COMP_ERR_INVALID_VALUE
    assert lib.comp_gemm_f32x16_noalloc(P(4096), P(1 << 20), P(1 << 24), 1, 8, MAX_BYTES // 4 + 1,
                                        None) == COMP_ERR_INVALID_VALUE
    assert lib.comp_gemm_f32x16_noalloc(P(4096), P(1 << 20), P(1 << 24), 1 << 40, 8, 1 << 40,
                                        None) == COMP_ERR_INVALID_VALUE
    assert lib.comp_gemm_f32x16_noalloc(P(4096), P(1 << 20), P(1 << 24), -1, 8, 8, None) == COMP_ERR_INVALID_VALUE
    assert lib.comp_gemm_f32x16_noalloc(None, None, None, 0, 8, 8, None) == 0  # empty: no-op
    if not torch.cuda.is_available():
        # valid sizes without a usable device: an error, never a CPU path
        assert lib.comp_gemm_f32x16_noalloc(P(4096), P(1 << 20), P(1 << 24), 8, 8, 8,
                                            None) == COMP_ERR_UNSUPPORTED_DEVICE


@pytest.mark.gpu
@pytest.mark.parametrize("shape", [(512, 1024, 1024), (130, 300, 72), (129, 257, 1027), (4096, 512, 4096)],
                         ids=lambda s: "x".join(map(str, s)))
def test_matches_workspace_entry_on_two_calls(pkg, lib, shape):
    from compensated_fp32_projection_gb300 import workloads

    M, N, K = shape
    x, W = workloads.random_case(M, N, K, seed=M + 3 * N + 7 * K, scale=2.0)
    xd, Wd = x.cuda(), W.cuda()
    y_ref = bits(pkg.comp_gemm_f32x16_ws(xd, Wd))
    for _ in range(2):
        y = torch.full((M, N), float("nan"), device="cuda")
        assert noalloc(lib, xd, Wd, y) == 0
        torch.cuda.synchronize()
        assert np.array_equal(bits(y), y_ref)


@pytest.mark.gpu
def test_against_the_oracle(pkg, lib, orc):
    from compensated_fp32_projection_gb300 import workloads

    x, W = workloads.random_case(300, 520, 264, seed=17, scale=2.0)
    y = torch.full((300, 520), float("nan"), device="cuda")
    assert noalloc(lib, x.cuda(), W.cuda(), y) == 0
    e_gpu, e_cast = check_comp(y, x, W, orc)
    assert e_cast >= 100 * e_gpu, (e_cast, e_gpu)


@pytest.mark.gpu
def test_largest_allowed_activation(pkg, lib, orc):
    # M * K = 16 * 2^20 exactly fills the workspace
    M, N, K = 4096, 64, 4096
    g = torch.Generator().manual_seed(41)
    x = torch.randn((M, K), generator=g)
    W = (torch.randn((N, K), generator=g) * 0.02).half()
    xd, Wd = x.cuda(), W.cuda()
    y_ref = bits(pkg.comp_gemm_f32x16_ws(xd, Wd))
    y = torch.empty(M, N, device="cuda")
    assert noalloc(lib, xd, Wd, y) == 0
    assert np.array_equal(bits(y), y_ref)
    r, c = sample_outputs(M, N)
    check_comp(y, x, W, orc, r, c)
    # K = 4088 (fits), then one row too many (rejected before any work)
    x8, W8 = xd[:, :-8].contiguous(), Wd[:, :-8].contiguous()
    y8 = torch.full((M, N), float("nan"), device="cuda")
    assert noalloc(lib, x8, W8, y8) == 0
    assert np.array_equal(bits(y8), bits(pkg.comp_gemm_f32x16_ws(x8, W8)))
    check_comp(y8, x8.cpu(), W8.cpu(), orc, r, c)
    big = torch.empty(M + 1, K, device="cuda")
    assert noalloc(lib, big, Wd, torch.empty(M + 1, N, device="cuda")) == COMP_ERR_INVALID_VALUE


@pytest.mark.gpu
def test_padded_form_too_large_takes_the_fused_kernel(pkg, lib, orc):
    # K % 8 != 0: 4*M*K = 65,488,000 bytes fits the array, but the padded
    # two-pass form, 4*M*Kp + 2*N*Kp with Kp = 4096, is 67,633,152 bytes and
    # does not; the call runs the fused kernel (no workspace) instead
    from compensated_fp32_projection_gb300 import workloads

    M, N, K = 4000, 256, 4093
    assert 4 * M * K <= MAX_BYTES < pkg.comp_gemm_workspace_bytes_mnk(M, N, K)
    x, W = workloads.random_case(M, N, K, seed=23, scale=2.0)
    xd, Wd = x.cuda(), W.cuda()
    for _ in range(2):
        y = torch.full((M, N), float("nan"), device="cuda")
        assert noalloc(lib, xd, Wd, y) == 0
        torch.cuda.synchronize()
        r, c = sample_outputs(M, N)
        e_gpu, e_cast = check_comp(y, x, W, orc, r, c)
        assert e_cast >= 100 * e_gpu, (e_cast, e_gpu)
        assert torch.isfinite(y).all()
    # the same results as the fused entry point, bit for bit
    assert np.array_equal(bits(y), bits(pkg.comp_gemm_f32x16(xd, Wd)))


@pytest.mark.gpu
def test_device_status_clean(pkg):
    st, where = pkg.device_status()
    assert st == 0 and where == 0
