"""Failure reporting of the bounded waits, without faulting or hanging the GPU.

Every wait on an mbarrier inside the library's tensor-core kernels is bounded;
when one gives up, the kernel records a fault code in a device word and exits,
and comp_device_status reports COMP_ERR_TIMEOUT with the code.
comp_check_wait_timeout runs that same bounded wait on a barrier that nothing
completes (a flag that nothing sets), so the wait must give up after about a
second.  comp_check_stalled_pipeline runs a real product kernel (CTA pairs, or
operands swapped) whose producer leaves out the loads of its first stage, so
that the MMA warp's wait for that stage gives up inside the pipeline: every
role then takes the abort path (bounded drains of the issued loads and MMAs,
tensor memory freed).  The tests check the reported status and code, that
reading the status clears it, and that the context is still usable afterwards.
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


PAIR_CODES = {0x701, 0x702, 0x703}
SWAP_CODES = {0x801, 0x802, 0x803, 0x804, 0x805}


# swapped-split: 32 tiles of W with 16 K blocks, K split over clusters of 4
# (every rank's first stage is left out; the ranks meet at the cluster barrier)
@pytest.mark.parametrize("variant,shape,codes", [(2, (256, 224, 128), PAIR_CODES), (3, (16, 4096, 128), SWAP_CODES),
                                                 (3, (16, 4096, 1024), SWAP_CODES)],
                         ids=["pairs", "swapped", "swapped-split"])
def test_stalled_pipeline_aborts_and_reports(pkg, orc, variant, shape, codes):
    from compensated_fp32_projection_gb300 import _native, workloads
    from gemm_check import check_comp

    M, N, K = shape
    lib = _native.load()
    x, W = workloads.random_case(M, N, K, seed=variant, scale=2.0)
    xd, Wd = x.cuda(), W.cuda()
    hi, lo = pkg.comp_split_f32(xd)
    y = torch.empty(M, N, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    assert pkg.device_status() == (0, 0)
    assert lib.comp_check_stalled_pipeline(hi.data_ptr(), lo.data_ptr(), Wd.data_ptr(), y.data_ptr(), M, N, K,
                                           variant, ctypes.c_void_p(stream)) == 0
    st, where = pkg.device_status(stream)
    assert st == COMP_ERR_TIMEOUT and where in codes, (st, hex(where))
    assert pkg.device_status() == (0, 0)  # read and cleared
    # the same kernel without the stall, right after on the same context: correct and clean
    y2 = pkg.comp_gemm_f16x2_variant(hi, lo, Wd, variant)
    check_comp(y2, x, W, orc)
    assert pkg.device_status() == (0, 0)


def test_stalled_pipeline_rejects(pkg):
    from compensated_fp32_projection_gb300 import _native

    lib = _native.load()
    h = torch.zeros(40, 64, dtype=torch.float16, device="cuda")
    W = torch.zeros(4096, 64, dtype=torch.float16, device="cuda")
    y = torch.empty(40, 4096, device="cuda")
    for variant in (0, 1, 4):  # only the pair and swapped kernels
        assert lib.comp_check_stalled_pipeline(h.data_ptr(), h.data_ptr(), W.data_ptr(), y.data_ptr(), 40, 4096, 64,
                                               variant, None) == 1
    # swapped operands take at most 32 rows
    assert lib.comp_check_stalled_pipeline(h.data_ptr(), h.data_ptr(), W.data_ptr(), y.data_ptr(), 40, 4096, 64, 3,
                                           None) == 1
