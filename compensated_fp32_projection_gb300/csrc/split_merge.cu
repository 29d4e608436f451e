// The standalone split and merge kernels (laya.cpp docs/vulkan.md, split/merge
// paragraph: the split of an input and the merge of an output are one dispatch
// each).  Both are streaming,
// HBM-bound kernels: 128-bit coalesced loads, 64/128-bit coalesced stores,
// evict-first cache hints, grid-stride loops over a grid sized to the SM count.
//
// Bit-exactness: conversions use the hardware round-to-nearest-even
// instructions (cvt.rn.f16x2.f32 / cvt.f32.f16) and the residual arithmetic
// uses __fsub_rn / __fmul_rn / __fadd_rn, which are never contracted into a
// fused multiply-add; the library is built without flush-to-zero.
#include <cuda_fp16.h>

#include "internal.h"

namespace compfp32 {
namespace {

constexpr int kThreads = 256;
constexpr int kBlocksPerSm = 8;
constexpr int kUnroll = 4;

__device__ __forceinline__ uint32_t h2_bits(__half2 h)
{
    return *reinterpret_cast<uint32_t*>(&h);
}

// Split two FP32 values into packed (hi, lo) FP16 pairs; element a lands in the
// low 16 bits, as it is first in memory.
__device__ __forceinline__ void split2(float a, float b, uint32_t& hi, uint32_t& lo)
{
    const __half2 h = __floats2half2_rn(a, b);
    const float2 hf = __half22float2(h);
    const float ra = __fmul_rn(__fsub_rn(a, hf.x), 1024.0f);
    const float rb = __fmul_rn(__fsub_rn(b, hf.y), 1024.0f);
    hi = h2_bits(h);
    lo = h2_bits(__floats2half2_rn(ra, rb));
}

__device__ __forceinline__ void split4(const float4 v, uint2& hi, uint2& lo)
{
    split2(v.x, v.y, hi.x, lo.x);
    split2(v.z, v.w, hi.y, lo.y);
}

// Vector body: n4 groups of four elements, x 16-byte aligned, hi/lo 8-byte aligned.
__global__ void __launch_bounds__(kThreads) split_vec_kernel(const float4* __restrict__ x, uint2* __restrict__ hi,
                                                             uint2* __restrict__ lo, int64_t n4)
{
    // a product kernel launched after this one may start its set-up now; it
    // waits for this grid's completion before it reads hi and lo
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    for (; i + (kUnroll - 1) * stride < n4; i += kUnroll * stride) {
        float4 v[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u)
            v[u] = __ldcs(x + i + u * stride);
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            uint2 h, l;
            split4(v[u], h, l);
            __stcs(hi + i + u * stride, h);
            __stcs(lo + i + u * stride, l);
        }
    }
    for (; i < n4; i += stride) {
        uint2 h, l;
        split4(__ldcs(x + i), h, l);
        __stcs(hi + i, h);
        __stcs(lo + i, l);
    }
}

// Scalar body for [begin, n): any alignment.
__global__ void __launch_bounds__(kThreads) split_scalar_kernel(const float* __restrict__ x, uint16_t* __restrict__ hi,
                                                                uint16_t* __restrict__ lo, int64_t begin, int64_t n)
{
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = begin + static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride) {
        const float v = x[i];
        const __half h = __float2half_rn(v);
        const float r = __fmul_rn(__fsub_rn(v, __half2float(h)), 1024.0f);
        const __half l = __float2half_rn(r);
        hi[i] = __half_as_ushort(h);
        lo[i] = __half_as_ushort(l);
    }
}

// Split of a row-major x [rows, K] into planes with a wider row stride Kp >= K
// (a multiple of 8, so that their rows start on 16-byte boundaries); the
// columns K..Kp-1 of both planes are +0, which adds exact zeros to every dot
// product.  Any alignment of x.
__global__ void __launch_bounds__(kThreads) split_pad_kernel(const float* __restrict__ x, uint16_t* __restrict__ hi,
                                                             uint16_t* __restrict__ lo, int64_t rows, int64_t K,
                                                             int64_t Kp)
{
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const int64_t n = rows * Kp;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride) {
        const int64_t r = i / Kp, k = i - r * Kp;
        uint16_t h = 0, l = 0;
        if (k < K) {
            const float v = x[r * K + k];
            const __half hh = __float2half_rn(v);
            h = __half_as_ushort(hh);
            l = __half_as_ushort(__float2half_rn(__fmul_rn(__fsub_rn(v, __half2float(hh)), 1024.0f)));
        }
        hi[i] = h;
        lo[i] = l;
    }
}

// Copy of a row-major binary16 matrix [rows, K] into rows of Kp >= K elements,
// zero-filled past K.
__global__ void __launch_bounds__(kThreads) pad_rows_kernel(const uint16_t* __restrict__ src, uint16_t* __restrict__ dst,
                                                            int64_t rows, int64_t K, int64_t Kp)
{
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const int64_t n = rows * Kp;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride) {
        const int64_t r = i / Kp, k = i - r * Kp;
        dst[i] = k < K ? src[r * K + k] : static_cast<uint16_t>(0);
    }
}

__device__ __forceinline__ float merge1(float a, float b)
{
    return __fadd_rn(a, __fmul_rn(b, 0x1p-10f));
}

// y may alias acc_hi or acc_lo element for element, so no __restrict__ and
// coherent (non read-only-path) loads.
__global__ void __launch_bounds__(kThreads) merge_vec_kernel(const float4* a, const float4* b, float4* y, int64_t n4)
{
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    for (; i + (kUnroll - 1) * stride < n4; i += kUnroll * stride) {
        float4 va[kUnroll], vb[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            va[u] = __ldcs(a + i + u * stride);
            vb[u] = __ldcs(b + i + u * stride);
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const float4 r = make_float4(merge1(va[u].x, vb[u].x), merge1(va[u].y, vb[u].y),
                                         merge1(va[u].z, vb[u].z), merge1(va[u].w, vb[u].w));
            __stcs(y + i + u * stride, r);
        }
    }
    for (; i < n4; i += stride) {
        const float4 va = __ldcs(a + i), vb = __ldcs(b + i);
        __stcs(y + i, make_float4(merge1(va.x, vb.x), merge1(va.y, vb.y), merge1(va.z, vb.z), merge1(va.w, vb.w)));
    }
}

__global__ void __launch_bounds__(kThreads) merge_scalar_kernel(const float* a, const float* b, float* y, int64_t begin,
                                                                int64_t n)
{
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = begin + static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride)
        y[i] = merge1(a[i], b[i]);
}

inline unsigned grid_for(int64_t work, const DeviceInfo& dev)
{
    const int64_t cap = static_cast<int64_t>(dev.sm_count) * kBlocksPerSm;
    int64_t g = (work + kThreads - 1) / kThreads;
    if (g > cap)
        g = cap;
    return static_cast<unsigned>(g < 1 ? 1 : g);
}

inline bool aligned(const void* p, uintptr_t a)
{
    return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0;
}

}  // namespace

comp_status_t launch_split(const float* x, uint16_t* hi, uint16_t* lo, int64_t n, const DeviceInfo& dev,
                           cudaStream_t stream)
{
    int64_t done = 0;
    if (aligned(x, 16) && aligned(hi, 8) && aligned(lo, 8)) {
        const int64_t n4 = n / 4;
        if (n4 > 0) {
            split_vec_kernel<<<grid_for(n4, dev), kThreads, 0, stream>>>(
                reinterpret_cast<const float4*>(x), reinterpret_cast<uint2*>(hi), reinterpret_cast<uint2*>(lo), n4);
            if (launch_status() != COMP_OK)
                return COMP_ERR_LAUNCH;
        }
        done = n4 * 4;
    }
    if (done < n) {
        split_scalar_kernel<<<grid_for(n - done, dev), kThreads, 0, stream>>>(x, hi, lo, done, n);
        if (launch_status() != COMP_OK)
            return COMP_ERR_LAUNCH;
    }
    return COMP_OK;
}

comp_status_t launch_split_padded(const float* x, uint16_t* hi, uint16_t* lo, int64_t rows, int64_t K, int64_t Kp,
                                  const DeviceInfo& dev, cudaStream_t stream)
{
    split_pad_kernel<<<grid_for(rows * Kp, dev), kThreads, 0, stream>>>(x, hi, lo, rows, K, Kp);
    return launch_status();
}

comp_status_t launch_pad_rows(const uint16_t* src, uint16_t* dst, int64_t rows, int64_t K, int64_t Kp,
                              const DeviceInfo& dev, cudaStream_t stream)
{
    pad_rows_kernel<<<grid_for(rows * Kp, dev), kThreads, 0, stream>>>(src, dst, rows, K, Kp);
    return launch_status();
}

comp_status_t launch_merge(const float* acc_hi, const float* acc_lo, float* y, int64_t n, const DeviceInfo& dev,
                           cudaStream_t stream)
{
    int64_t done = 0;
    if (aligned(acc_hi, 16) && aligned(acc_lo, 16) && aligned(y, 16)) {
        const int64_t n4 = n / 4;
        if (n4 > 0) {
            merge_vec_kernel<<<grid_for(n4, dev), kThreads, 0, stream>>>(reinterpret_cast<const float4*>(acc_hi),
                                                                         reinterpret_cast<const float4*>(acc_lo),
                                                                         reinterpret_cast<float4*>(y), n4);
            if (launch_status() != COMP_OK)
                return COMP_ERR_LAUNCH;
        }
        done = n4 * 4;
    }
    if (done < n) {
        merge_scalar_kernel<<<grid_for(n - done, dev), kThreads, 0, stream>>>(acc_hi, acc_lo, y, done, n);
        if (launch_status() != COMP_OK)
            return COMP_ERR_LAUNCH;
    }
    return COMP_OK;
}

}  // namespace compfp32
