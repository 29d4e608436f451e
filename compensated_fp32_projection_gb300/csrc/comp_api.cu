// The C ABI entry points (include/compfp32.h): argument validation, the device
// check, and dispatch to the kernels' launchers.  Nothing here allocates
// device memory or synchronises, except comp_device_status.
#include <atomic>
#include <cstring>

#include "internal.h"

namespace compfp32 {

namespace {

constexpr int kMaxDevices = 64;
// 0 = unknown, 1 = supported, 2 = unsupported; SM count alongside.
std::atomic<int> g_dev_state[kMaxDevices];
std::atomic<int> g_dev_sms[kMaxDevices];

bool mul_ok(int64_t a, int64_t b, int64_t* out)
{
    if (a < 0 || b < 0)
        return false;
    if (a != 0 && b > INT64_MAX / a)
        return false;
    *out = a * b;
    return true;
}

// Byte ranges [a, a+na) and [b, b+nb) overlap.
bool overlap(const void* a, int64_t na, const void* b, int64_t nb)
{
    const uintptr_t pa = reinterpret_cast<uintptr_t>(a), pb = reinterpret_cast<uintptr_t>(b);
    return na > 0 && nb > 0 && pa < pb + static_cast<uintptr_t>(nb) && pb < pa + static_cast<uintptr_t>(na);
}

}  // namespace

comp_status_t current_device(DeviceInfo* info)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        (void)cudaGetLastError();
        return COMP_ERR_UNSUPPORTED_DEVICE;
    }
    int state = g_dev_state[dev].load(std::memory_order_acquire);
    if (state == 0) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            (void)cudaGetLastError();
            return COMP_ERR_UNSUPPORTED_DEVICE;
        }
        g_dev_sms[dev].store(sms, std::memory_order_relaxed);
        state = (major == 10 && minor == 3) ? 1 : 2;
        g_dev_state[dev].store(state, std::memory_order_release);
    }
    if (state != 1)
        return COMP_ERR_UNSUPPORTED_DEVICE;
    info->device = dev;
    info->sm_count = g_dev_sms[dev].load(std::memory_order_relaxed);
    return COMP_OK;
}

namespace {

// Shared checks of the GEMM entry points; x has x_elem bytes per element (4
// for FP32 activations, 2 for one FP16 split plane).  Sets *empty when there is
// nothing to launch (after writing y = 0 for K == 0).
comp_status_t check_gemm(const void* x, int64_t x_elem, const uint16_t* W, float* y, int64_t M, int64_t N,
                         int64_t K, cudaStream_t stream, DeviceInfo* dev, bool* empty)
{
    *empty = false;
    int64_t mk, nk, mn;
    if (M < 0 || N < 0 || K < 0 || !mul_ok(M, K, &mk) || !mul_ok(N, K, &nk) || !mul_ok(M, N, &mn))
        return COMP_ERR_INVALID_VALUE;
    if (M > INT32_MAX || N > INT32_MAX || K > INT32_MAX)
        return COMP_ERR_INVALID_VALUE;
    if (mk > INT64_MAX / 4 || nk > INT64_MAX / 2 || mn > INT64_MAX / 4)
        return COMP_ERR_INVALID_VALUE;
    if (mn == 0) {
        *empty = true;
        return COMP_OK;
    }
    if (!y || (K > 0 && (!x || !W)))
        return COMP_ERR_INVALID_VALUE;
    if (overlap(y, 4 * mn, x, x_elem * mk) || overlap(y, 4 * mn, W, 2 * nk))
        return COMP_ERR_INVALID_VALUE;
    const comp_status_t st = current_device(dev);
    if (st != COMP_OK)
        return st;
    if (K == 0) {
        *empty = true;
        return cudaMemsetAsync(y, 0, static_cast<size_t>(4 * mn), stream) == cudaSuccess ? COMP_OK : COMP_ERR_CUDA;
    }
    return COMP_OK;
}

// Epilogue operands: bias [N] and gate [M, N] FP32, either may be NULL; neither
// may overlap y (they are read while y is written).
bool epilogue_args_ok(const float* bias, const float* gate, const float* y, int64_t M, int64_t N)
{
    int64_t mn = 0;
    if (M < 0 || N < 0 || !mul_ok(M, N, &mn) || mn > INT64_MAX / 4)
        return false;
    if (bias && N > 0 && overlap(bias, 4 * N, y, 4 * mn))
        return false;
    if (gate && mn > 0 && overlap(gate, 4 * mn, y, 4 * mn))
        return false;
    return true;
}

comp_status_t gemm_ws_impl(const float* x, const uint16_t* W, float* y, int64_t M, int64_t N, int64_t K,
                           void* workspace, int64_t workspace_bytes, comp_stream_t stream, const Epilogue& epi)
{
    DeviceInfo dev;
    bool empty;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    const comp_status_t st = check_gemm(x, 4, W, y, M, N, K, s, &dev, &empty);
    if (st != COMP_OK || empty)
        return st;
    if (workspace_bytes < 0 || (workspace_bytes > 0 && !workspace))
        return COMP_ERR_INVALID_VALUE;
    if (workspace && workspace_bytes > 0 &&
        (overlap(workspace, workspace_bytes, x, 4 * M * K) || overlap(workspace, workspace_bytes, W, 2 * N * K) ||
         overlap(workspace, workspace_bytes, y, 4 * M * N)))
        return COMP_ERR_INVALID_VALUE;
    uint16_t* const ws = static_cast<uint16_t*>(workspace);
    const bool ws_aligned = (reinterpret_cast<uintptr_t>(workspace) & 15u) == 0;
    const int64_t need = comp_gemm_workspace_bytes(M, K);
    const bool planes_fit =
        ws && ws_aligned && need > 0 && workspace_bytes >= need && gemm_f16x2_supported(ws, ws + M * K, W, K);
    // at most 32 rows: one kernel with the split fused needs no workspace and
    // is as fast as the two-pass form or faster, except with 17 to 32 rows and
    // no split of K
    if (swap_fused_preferred(x, W, M, N, K) && !(planes_fit && swap_two_pass_better(M, N, K, dev)))
        return launch_swap_fused(x, W, y, M, N, K, dev, s, epi);
    // two-pass form on the caller's W: planes [M, K] in the workspace
    if (planes_fit) {
        const comp_status_t sp = launch_split(x, ws, ws + M * K, M * K, dev, s);
        if (sp != COMP_OK)
            return sp;
        return launch_gemm_f16x2(ws, ws + M * K, W, y, M, N, K, 0, dev, s, epi);
    }
    // two-pass form with K padded to a multiple of 8 (any K, any alignment):
    // planes [M, Kp] and a zero-padded copy of W [N, Kp] in the workspace
    const int64_t need_p = comp_gemm_workspace_bytes_mnk(M, N, K);
    if (ws && ws_aligned && need_p > 0 && workspace_bytes >= need_p) {
        const int64_t Kp = (K + 7) / 8 * 8;
        uint16_t* hi = ws;
        uint16_t* lo = ws + M * Kp;
        uint16_t* wp = ws + 2 * M * Kp;
        const comp_status_t r = launch_prep_padded(x, W, hi, lo, wp, M, N, K, Kp, dev, s);
        if (r != COMP_OK)
            return r;
        return launch_gemm_f16x2(hi, lo, wp, y, M, N, Kp, 0, dev, s, epi);
    }
    return launch_gemm_tc(x, W, y, M, N, K, 0, dev, s, epi);
}

comp_status_t gemm_f16x2_impl(const uint16_t* hi, const uint16_t* lo, const uint16_t* W, float* y, int64_t M,
                              int64_t N, int64_t K, int variant, comp_stream_t stream, const Epilogue& epi)
{
    DeviceInfo dev;
    bool empty;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (variant < 0 || variant > 4 || (variant == 3 && M > 32))
        return COMP_ERR_INVALID_VALUE;
    const comp_status_t st = check_gemm(hi, 2, W, y, M, N, K, s, &dev, &empty);
    if (st != COMP_OK || empty)
        return st;
    // check_gemm has bounded M*N and M*K
    if (!lo || overlap(y, 4 * M * N, lo, 2 * M * K))
        return COMP_ERR_INVALID_VALUE;
    if (!gemm_f16x2_supported(hi, lo, W, K))
        return COMP_ERR_INVALID_VALUE;
    return launch_gemm_f16x2(hi, lo, W, y, M, N, K, variant, dev, s, epi);
}

}  // namespace
}  // namespace compfp32

using namespace compfp32;

extern "C" {

comp_status_t comp_split_f32(const float* x, uint16_t* hi, uint16_t* lo, int64_t n, comp_stream_t stream)
{
    if (n < 0 || n > INT64_MAX / 4)
        return COMP_ERR_INVALID_VALUE;
    if (n == 0)
        return COMP_OK;
    if (!x || !hi || !lo)
        return COMP_ERR_INVALID_VALUE;
    if (overlap(x, 4 * n, hi, 2 * n) || overlap(x, 4 * n, lo, 2 * n) || overlap(hi, 2 * n, lo, 2 * n))
        return COMP_ERR_INVALID_VALUE;
    DeviceInfo dev;
    const comp_status_t st = current_device(&dev);
    if (st != COMP_OK)
        return st;
    return launch_split(x, hi, lo, n, dev, static_cast<cudaStream_t>(stream));
}

comp_status_t comp_merge_f32(const float* acc_hi, const float* acc_lo, float* y, int64_t n, comp_stream_t stream)
{
    if (n < 0 || n > INT64_MAX / 4)
        return COMP_ERR_INVALID_VALUE;
    if (n == 0)
        return COMP_OK;
    if (!acc_hi || !acc_lo || !y)
        return COMP_ERR_INVALID_VALUE;
    if ((y != acc_hi && overlap(y, 4 * n, acc_hi, 4 * n)) || (y != acc_lo && overlap(y, 4 * n, acc_lo, 4 * n)))
        return COMP_ERR_INVALID_VALUE;
    DeviceInfo dev;
    const comp_status_t st = current_device(&dev);
    if (st != COMP_OK)
        return st;
    return launch_merge(acc_hi, acc_lo, y, n, dev, static_cast<cudaStream_t>(stream));
}

comp_status_t comp_geglu_f32(const float* gate, const float* up, float* out, int64_t n, comp_stream_t stream)
{
    if (n < 0 || n > INT64_MAX / 4)
        return COMP_ERR_INVALID_VALUE;
    if (n == 0)
        return COMP_OK;
    if (!gate || !up || !out)
        return COMP_ERR_INVALID_VALUE;
    if ((out != gate && overlap(out, 4 * n, gate, 4 * n)) || (out != up && overlap(out, 4 * n, up, 4 * n)))
        return COMP_ERR_INVALID_VALUE;
    DeviceInfo dev;
    const comp_status_t st = current_device(&dev);
    if (st != COMP_OK)
        return st;
    return launch_geglu(gate, up, out, n, dev, static_cast<cudaStream_t>(stream));
}

comp_status_t comp_gemm_f32x16_variant(const float* x, const uint16_t* W, float* y, int64_t M, int64_t N, int64_t K,
                                       int variant, comp_stream_t stream)
{
    if (variant < 0 || variant > 4)
        return COMP_ERR_INVALID_VALUE;
    // the fused swapped-operand kernel (at most 32 rows) and the fused kernel
    // on CTA pairs: TMA-legal W and x
    const bool tma_legal = K % 8 == 0 && (reinterpret_cast<uintptr_t>(x) & 15u) == 0 &&
                           (reinterpret_cast<uintptr_t>(W) & 15u) == 0;
    if ((variant == 3 && (M > 32 || !tma_legal)) || (variant == 4 && !tma_legal))
        return COMP_ERR_INVALID_VALUE;
    DeviceInfo dev;
    bool empty;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    const comp_status_t st = check_gemm(x, 4, W, y, M, N, K, s, &dev, &empty);
    if (st != COMP_OK || empty)
        return st;
    return launch_gemm_tc(x, W, y, M, N, K, variant, dev, s);
}

comp_status_t comp_gemm_f32x16(const float* x, const uint16_t* W, float* y, int64_t M, int64_t N, int64_t K,
                               comp_stream_t stream)
{
    return comp_gemm_f32x16_variant(x, W, y, M, N, K, 0, stream);
}

comp_status_t comp_gemm_f32_simt(const float* x, const uint16_t* W, float* y, int64_t M, int64_t N, int64_t K,
                                 comp_stream_t stream)
{
    DeviceInfo dev;
    bool empty;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    const comp_status_t st = check_gemm(x, 4, W, y, M, N, K, s, &dev, &empty);
    if (st != COMP_OK || empty)
        return st;
    return launch_gemm_simt(x, W, y, M, N, K, dev, s);
}

comp_status_t comp_gemm_f16x2_variant(const uint16_t* hi, const uint16_t* lo, const uint16_t* W, float* y, int64_t M,
                                      int64_t N, int64_t K, int variant, comp_stream_t stream)
{
    return gemm_f16x2_impl(hi, lo, W, y, M, N, K, variant, stream, Epilogue{});
}

comp_status_t comp_gemm_f16x2(const uint16_t* hi, const uint16_t* lo, const uint16_t* W, float* y, int64_t M,
                              int64_t N, int64_t K, comp_stream_t stream)
{
    return comp_gemm_f16x2_variant(hi, lo, W, y, M, N, K, 0, stream);
}

int64_t comp_gemm_workspace_bytes(int64_t M, int64_t K)
{
    int64_t mk = 0;
    if (!mul_ok(M, K, &mk) || mk > INT64_MAX / 4)
        return 0;
    return 4 * mk;
}

int64_t comp_gemm_workspace_bytes_mnk(int64_t M, int64_t N, int64_t K)
{
    if (M < 0 || N < 0 || K < 0 || K > INT64_MAX - 8)
        return 0;
    const int64_t Kp = (K + 7) / 8 * 8;
    int64_t mk = 0, nk = 0;
    if (!mul_ok(M, Kp, &mk) || !mul_ok(N, Kp, &nk) || mk > INT64_MAX / 8 || nk > INT64_MAX / 8 ||
        4 * mk > INT64_MAX - 2 * nk)
        return 0;
    return 4 * mk + 2 * nk;
}

comp_status_t comp_gemm_f32x16_ws(const float* x, const uint16_t* W, float* y, int64_t M, int64_t N, int64_t K,
                                  void* workspace, int64_t workspace_bytes, comp_stream_t stream)
{
    return gemm_ws_impl(x, W, y, M, N, K, workspace, workspace_bytes, stream, Epilogue{});
}

comp_status_t comp_gemm_f32x16_epilogue(const float* x, const uint16_t* W, const float* bias, const float* gate,
                                        float* y, int64_t M, int64_t N, int64_t K, void* workspace,
                                        int64_t workspace_bytes, comp_stream_t stream)
{
    if (!epilogue_args_ok(bias, gate, y, M, N))
        return COMP_ERR_INVALID_VALUE;
    // the bias in the product kernel's epilogue; the gate by the GEGLU dispatch
    // on y in place right after, on the same stream (on GB300 the gate's erfc
    // work stalls the tensor pipe when the product kernel does it)
    comp_status_t st = gemm_ws_impl(x, W, y, M, N, K, workspace, workspace_bytes, stream, Epilogue{bias, nullptr});
    if (st != COMP_OK || !gate || M == 0 || N == 0)
        return st;
    DeviceInfo dev;
    st = current_device(&dev);
    if (st != COMP_OK)
        return st;
    return launch_geglu(gate, y, y, M * N, dev, static_cast<cudaStream_t>(stream));
}

comp_status_t comp_gemm_f16x2_epilogue(const uint16_t* hi, const uint16_t* lo, const uint16_t* W, const float* bias,
                                       const float* gate, float* y, int64_t M, int64_t N, int64_t K, int variant,
                                       comp_stream_t stream)
{
    if (!epilogue_args_ok(bias, gate, y, M, N))
        return COMP_ERR_INVALID_VALUE;
    return gemm_f16x2_impl(hi, lo, W, y, M, N, K, variant, stream, Epilogue{bias, gate});
}



comp_status_t comp_check_stalled_pipeline(const uint16_t* hi, const uint16_t* lo, const uint16_t* W, float* y,
                                          int64_t M, int64_t N, int64_t K, int variant, comp_stream_t stream)
{
    DeviceInfo dev;
    bool empty;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (variant != 2 && variant != 3)
        return COMP_ERR_INVALID_VALUE;
    if (variant == 3 && M > 32)
        return COMP_ERR_INVALID_VALUE;
    const comp_status_t st = check_gemm(hi, 2, W, y, M, N, K, s, &dev, &empty);
    if (st != COMP_OK || empty)
        return st;
    if (!lo || overlap(y, 4 * M * N, lo, 2 * M * K) || !gemm_f16x2_supported(hi, lo, W, K))
        return COMP_ERR_INVALID_VALUE;
    return launch_gemm_f16x2(hi, lo, W, y, M, N, K, variant, dev, s, Epilogue{}, true);
}

comp_status_t comp_check_wait_timeout(comp_stream_t stream)
{
    DeviceInfo dev;
    const comp_status_t st = current_device(&dev);
    if (st != COMP_OK)
        return st;
    return launch_check_wait_timeout(static_cast<cudaStream_t>(stream));
}

comp_status_t comp_device_status(comp_stream_t stream, uint32_t* where)
{
    if (where)
        *where = 0;
    DeviceInfo dev;
    const comp_status_t st = current_device(&dev);
    if (st != COMP_OK)
        return st;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) {
        (void)cudaGetLastError();
        return COMP_ERR_CUDA;
    }
    return read_and_clear_fault(s, where);
}

const char* comp_status_string(comp_status_t status)
{
    switch (status) {
    case COMP_OK:
        return "COMP_OK";
    case COMP_ERR_INVALID_VALUE:
        return "COMP_ERR_INVALID_VALUE: bad pointer, size or aliasing";
    case COMP_ERR_MISALIGNED:
        return "COMP_ERR_MISALIGNED: reserved (no call returns it)";
    case COMP_ERR_UNSUPPORTED_DEVICE:
        return "COMP_ERR_UNSUPPORTED_DEVICE: the current device is not an sm_103 GPU";
    case COMP_ERR_LAUNCH:
        return "COMP_ERR_LAUNCH: kernel launch failed";
    case COMP_ERR_TIMEOUT:
        return "COMP_ERR_TIMEOUT: a kernel gave up a bounded wait";
    case COMP_ERR_CUDA:
        return "COMP_ERR_CUDA: a CUDA runtime call failed";
    }
    return "unknown comp_status_t";
}

int comp_version(void)
{
    return 100;  // 0.1.0
}

}  // extern "C"
