// The GEGLU step of the FP32 feed-forward layers as one dispatch (laya.cpp
// docs/vulkan.md, feed-forward paragraph: a fused GEGLU shader, with no
// separate gate copy, activation or multiplication dispatches):
//   out[i] = gelu(gate[i]) * up[i],  gelu(g) = g * Phi(g),
//   Phi(g) = erfc(-g / sqrt 2) / 2  (the exact GELU; erfc has no cancellation
//   for negative g),
// each operation a binary32 operation rounded to nearest even, in the same
// order as the product kernels' epilogue, so that both give the same bits.
// A streaming kernel, bound by HBM at 12 bytes per element: 128-bit loads and
// stores, grid-stride loops over a grid sized to the SM count; a scalar kernel
// takes a misaligned head or tail.
#include "internal.h"

namespace compfp32 {
namespace {

constexpr int kThreads = 256;
constexpr int kBlocksPerSm = 8;
constexpr int kUnroll = 4;

__device__ __forceinline__ float geglu1(float g, float u)
{
    const float phi = __fmul_rn(0.5f, erfcf(__fmul_rn(-g, 0.70710678118654752f)));  // 1 / sqrt 2
    return __fmul_rn(u, __fmul_rn(g, phi));
}

__device__ __forceinline__ float4 geglu4(float4 g, float4 u)
{
    return make_float4(geglu1(g.x, u.x), geglu1(g.y, u.y), geglu1(g.z, u.z), geglu1(g.w, u.w));
}

// out may be gate or up element for element, so no __restrict__ and coherent
// (non read-only-path) loads.
__global__ void __launch_bounds__(kThreads) geglu_vec_kernel(const float4* gate, const float4* up, float4* out,
                                                             int64_t n4)
{
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    for (; i + (kUnroll - 1) * stride < n4; i += kUnroll * stride) {
        float4 g[kUnroll], u[kUnroll];
#pragma unroll
        for (int k = 0; k < kUnroll; ++k) {
            g[k] = __ldcs(gate + i + k * stride);
            u[k] = __ldcs(up + i + k * stride);
        }
#pragma unroll
        for (int k = 0; k < kUnroll; ++k)
            __stcs(out + i + k * stride, geglu4(g[k], u[k]));
    }
    for (; i < n4; i += stride)
        __stcs(out + i, geglu4(__ldcs(gate + i), __ldcs(up + i)));
}

__global__ void __launch_bounds__(kThreads) geglu_scalar_kernel(const float* gate, const float* up, float* out,
                                                                int64_t begin, int64_t n)
{
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = begin + static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride)
        out[i] = geglu1(gate[i], up[i]);
}

inline unsigned grid_for(int64_t work, const DeviceInfo& dev)
{
    const int64_t cap = static_cast<int64_t>(dev.sm_count) * kBlocksPerSm;
    int64_t g = (work + kThreads - 1) / kThreads;
    if (g > cap)
        g = cap;
    return static_cast<unsigned>(g < 1 ? 1 : g);
}

}  // namespace

comp_status_t launch_geglu(const float* gate, const float* up, float* out, int64_t n, const DeviceInfo& dev,
                           cudaStream_t stream)
{
    int64_t done = 0;
    const auto a16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    if (a16(gate) && a16(up) && a16(out)) {
        const int64_t n4 = n / 4;
        if (n4 > 0) {
            geglu_vec_kernel<<<grid_for(n4, dev), kThreads, 0, stream>>>(
                reinterpret_cast<const float4*>(gate), reinterpret_cast<const float4*>(up),
                reinterpret_cast<float4*>(out), n4);
            if (launch_status() != COMP_OK)
                return COMP_ERR_LAUNCH;
        }
        done = n4 * 4;
    }
    if (done < n) {
        geglu_scalar_kernel<<<grid_for(n - done, dev), kThreads, 0, stream>>>(gate, up, out, done, n);
        if (launch_status() != COMP_OK)
            return COMP_ERR_LAUNCH;
    }
    return COMP_OK;
}

}  // namespace compfp32
