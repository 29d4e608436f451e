"""Failure reporting of the bounded waits, without faulting or hanging the GPU.

Every wait on an mbarrier inside the library's tensor-core kernels is bounded;
when one gives up, the kernel records a fault code in a device word and exits,
and comp_device_status reports COMP_ERR_TIMEOUT with the code.
comp_check_wait_timeout runs that same bounded wait on a barrier that nothing
completes (a flag that nothing sets), so the wait must give up after about a
second.  The test checks the reported status and code, that reading the status
clears it, and that the context is still usable afterwards.
"""
import ctypes

import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

COMP_ERR_TIMEOUT = 5
COMP_FAULT_CHECK_TIMEOUT = 0x0F01


@pytest.fixture(scope="module")
def pkg():
    import __graft_entry__

    __graft_entry__.build()
    import compensated_fp32_projection_gb300 as p

    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return p


def test_timeout_is_reported_and_the_context_stays_usable(pkg, orc):
    from compensated_fp32_projection_gb300 import _native, workloads
    from gemm_check import check_comp

    lib = _native.load()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert pkg.device_status() == (0, 0)
    assert lib.comp_check_wait_timeout(stream) == 0
    st, where = pkg.device_status(torch.cuda.current_stream().cuda_stream)
    assert (st, where) == (COMP_ERR_TIMEOUT, COMP_FAULT_CHECK_TIMEOUT)
    assert pkg.device_status() == (0, 0)  # read and cleared
    # the context is still usable: a projection afterwards is correct and clean
    x, W = workloads.random_case(130, 300, 72, seed=3)
    y = pkg.comp_gemm_f32x16_ws(x.cuda(), W.cuda())
    check_comp(y, x, W, orc)
    assert pkg.device_status() == (0, 0)
