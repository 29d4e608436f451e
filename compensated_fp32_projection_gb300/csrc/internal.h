// Internal declarations shared by the translation units of the library.
#pragma once

#include <cuda_runtime.h>
#include <cstdint>

#include "compfp32.h"

namespace compfp32 {

// Properties of the current device, checked once per device.
struct DeviceInfo {
    int device;
    int sm_count;
};

// COMP_OK and fills `info` if the current device is compute capability 10.3.
comp_status_t current_device(DeviceInfo* info);

// Launchers (arguments already validated; sizes > 0).
comp_status_t launch_split(const float* x, uint16_t* hi, uint16_t* lo, int64_t n, const DeviceInfo& dev,
                           cudaStream_t stream);
// One launch: x [M, K] split into planes [M, Kp] (Kp >= K, a multiple of 8)
// and W [N, K] copied into wp [N, Kp], all zero-padded past K.
comp_status_t launch_prep_padded(const float* x, const uint16_t* W, uint16_t* hi, uint16_t* lo, uint16_t* wp,
                                 int64_t M, int64_t N, int64_t K, int64_t Kp, const DeviceInfo& dev,
                                 cudaStream_t stream);
comp_status_t launch_geglu(const float* gate, const float* up, float* out, int64_t n, const DeviceInfo& dev,
                           cudaStream_t stream);
comp_status_t launch_merge(const float* acc_hi, const float* acc_lo, float* y, int64_t n, const DeviceInfo& dev,
                           cudaStream_t stream);
comp_status_t launch_gemm_simt(const float* x, const uint16_t* W, float* y, int64_t M, int64_t N, int64_t K,
                               const DeviceInfo& dev, cudaStream_t stream);
// Optional FP32 operations on the merged projection in the product kernels'
// epilogue (GEGLU feed-forward step): y = gelu(gate) * (y + bias).
struct Epilogue {
    const float* bias = nullptr;  // [N] (nullptr: none)
    const float* gate = nullptr;  // [M, N] row-major (nullptr: factor 1)
};

// Fused split and swapped-operand product for at most 32 rows of x (K a
// multiple of 8, x and W 16-byte aligned), with K split over a cluster when W
// has few tiles of 128 rows.
bool swap_fused_preferred(const float* x, const uint16_t* W, int64_t M, int64_t N, int64_t K);
// Given a workspace, whether the two-pass form beats the fused swapped kernel
// for a shape that swap_fused_preferred accepts (17 to 32 rows, no split of K).
bool swap_two_pass_better(int64_t M, int64_t N, int64_t K, const DeviceInfo& dev);
comp_status_t launch_swap_fused(const float* x, const uint16_t* W, float* y, int64_t M, int64_t N, int64_t K,
                                const DeviceInfo& dev, cudaStream_t stream, const Epilogue& epi = Epilogue{});
// Fused split and product on CTA pairs (K a multiple of 8, x and W 16-byte
// aligned); preferred for more than 128 rows once the output fills about a
// wave of tiles.
bool fused_pair_preferred(const float* x, const uint16_t* W, int64_t M, int64_t N, int64_t K, const DeviceInfo& dev);
comp_status_t launch_fused_pair(const float* x, const uint16_t* W, float* y, int64_t M, int64_t N, int64_t K,
                                const DeviceInfo& dev, cudaStream_t stream, const Epilogue& epi = Epilogue{});
// variant: 0 automatic, 1 TMA loads, 2 plain loads (both one CTA per tile),
// 3 operands swapped with the split fused (M <= 32), 4 CTA pairs with the
// split fused.
comp_status_t launch_gemm_tc(const float* x, const uint16_t* W, float* y, int64_t M, int64_t N, int64_t K,
                             int variant, const DeviceInfo& dev, cudaStream_t stream, const Epilogue& epi = Epilogue{});

// The two products and the merge from split planes (hi, lo: [M, K] FP16).
// Needs 16-byte aligned hi, lo, W and K % 8 == 0 (else COMP_ERR_INVALID_VALUE).
bool gemm_f16x2_supported(const void* hi, const void* lo, const void* W, int64_t K);
// variant: 0 automatic, 1 one CTA per 128-row tile, 2 CTA pairs on 256-row
// tiles, 3 operands swapped (M <= 32).
// stall: diagnostic run of the CTA-pair (variant 2) or swapped (variant 3)
// kernel whose producer leaves out its first stage's loads (see
// comp_check_stalled_pipeline).
comp_status_t launch_gemm_f16x2(const uint16_t* hi, const uint16_t* lo, const uint16_t* W, float* y, int64_t M,
                                int64_t N, int64_t K, int variant, const DeviceInfo& dev, cudaStream_t stream,
                                const Epilogue& epi = Epilogue{}, bool stall = false);

// One thread runs a bounded wait that cannot succeed (comp_check_wait_timeout).
comp_status_t launch_check_wait_timeout(cudaStream_t stream);

// Reads and clears the fault word of the tensor-core kernels (after the stream
// has been synchronised).
comp_status_t read_and_clear_fault(cudaStream_t stream, uint32_t* where);

inline comp_status_t launch_status()
{
    return cudaGetLastError() == cudaSuccess ? COMP_OK : COMP_ERR_LAUNCH;
}

}  // namespace compfp32
