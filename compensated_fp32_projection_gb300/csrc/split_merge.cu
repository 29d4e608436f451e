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

// The two-pass form's operands for any K: x [M, K] split into planes of row
// stride Kp >= K (a multiple of 8, so that their rows start on 16-byte
// boundaries), and W [N, K] copied into rows of Kp elements; columns K..Kp-1
// are +0 in all three, which adds exact zeros to every dot product.  One
// launch: block rows 0..M-1 split x, rows M..M+N-1 copy W.  Each thread
// writes 8 consecutive elements of a row (16-byte stores), reading its
// inputs with element loads (any alignment of x and W).
__global__ void __launch_bounds__(kThreads) prep_padded_kernel(const float* __restrict__ x,
                                                               const uint16_t* __restrict__ W,
                                                               uint16_t* __restrict__ hi, uint16_t* __restrict__ lo,
                                                               uint16_t* __restrict__ wp, int64_t M, int64_t N,
                                                               int64_t K, int64_t Kp)
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int64_t c8 = Kp / 8;  // 8-element pieces per row
    for (int64_t r = blockIdx.x; r < M + N; r += gridDim.x) {
        if (r < M) {
            const float* xr = x + r * K;
            for (int64_t c = threadIdx.x; c < c8; c += blockDim.x) {
                const int64_t k0 = 8 * c;
                float v[8];
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    v[e] = k0 + e < K ? xr[k0 + e] : 0.0f;
                uint4 h, l;
                split2(v[0], v[1], h.x, l.x);
                split2(v[2], v[3], h.y, l.y);
                split2(v[4], v[5], h.z, l.z);
                split2(v[6], v[7], h.w, l.w);
                *reinterpret_cast<uint4*>(hi + r * Kp + k0) = h;
                *reinterpret_cast<uint4*>(lo + r * Kp + k0) = l;
            }
        } else {
            const int64_t n = r - M;
            const uint16_t* wr = W + n * K;
            for (int64_t c = threadIdx.x; c < c8; c += blockDim.x) {
                const int64_t k0 = 8 * c;
                uint32_t h[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const uint32_t a = k0 + 2 * e < K ? wr[k0 + 2 * e] : 0u;
                    const uint32_t b = k0 + 2 * e + 1 < K ? wr[k0 + 2 * e + 1] : 0u;
                    h[e] = a | (b << 16);
                }
                *reinterpret_cast<uint4*>(wp + n * Kp + k0) = make_uint4(h[0], h[1], h[2], h[3]);
            }
        }
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

comp_status_t launch_prep_padded(const float* x, const uint16_t* W, uint16_t* hi, uint16_t* lo, uint16_t* wp,
                                 int64_t M, int64_t N, int64_t K, int64_t Kp, const DeviceInfo& dev,
                                 cudaStream_t stream)
{
    const int64_t rows = M + N;
    const int64_t cap = static_cast<int64_t>(dev.sm_count) * kBlocksPerSm;
    const unsigned grid = static_cast<unsigned>(rows < cap ? rows : cap);
    prep_padded_kernel<<<grid, kThreads, 0, stream>>>(x, W, hi, lo, wp, M, N, K, Kp);
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
