// The true-FP32 reference product (laya.cpp docs/vulkan.md, paragraph on the
// true FP32 matrix kernels that keep explicitly FP32 operands from being
// converted to FP16): y = x * float(W)^T with binary32 fused multiply-adds on
// the CUDA cores, summed in increasing k.  W is widened to FP32 exactly.
//
// Shared-memory tiled: a 128x128 output tile per 256-thread block, 8x8
// outputs per thread (multiply-adds issued two at a time as packed
// fma.rn.f32x2, each lane an ordinary binary32 fused multiply-add), K step
// 16, operands staged k-major in shared memory (rows padded to 132 floats)
// and double-buffered through registers.  A warp
// covers 4 x 8 threads of the 16 x 16 thread grid, so that its operand loads
// from shared memory are one wavefront each.
// Global loads: with K % 8 == 0 and 16-byte aligned x and W, coalesced
// 16-byte loads (four threads read a row's 16 values of x, two threads its 16
// values of W); otherwise bounds-checked scalar loads (any size and
// alignment).  Both load paths stage the same values, and the order of the
// multiply-adds does not depend on them.
#include <cuda_fp16.h>

#include "internal.h"

namespace compfp32 {
namespace {

constexpr int TBM = 128, TBN = 128, TBK = 16, kThreads = 256;
constexpr int kLd = TBM + 4;  // padded row of a k-major operand tile (floats)

__device__ __forceinline__ uint64_t f2_pack(float lo, float hi)
{
    return static_cast<uint64_t>(__float_as_uint(lo)) | (static_cast<uint64_t>(__float_as_uint(hi)) << 32);
}

// c0 = fma(a, b0, c0), c1 = fma(a, b1, c1): two independent binary32 fused
// multiply-adds, each rounded to nearest even, in one packed instruction
// (the same results as two scalar fmaf; half the issue slots).
__device__ __forceinline__ void fma2(float& c0, float& c1, float a, float b0, float b1)
{
    uint64_t c;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(c) : "l"(f2_pack(a, a)), "l"(f2_pack(b0, b1)), "l"(f2_pack(c0, c1)));
    c0 = __uint_as_float(static_cast<uint32_t>(c));
    c1 = __uint_as_float(static_cast<uint32_t>(c >> 32));
}

template <bool kVec>
__global__ void __launch_bounds__(kThreads, 2) gemm_simt_kernel(const float* __restrict__ x,
                                                                const uint16_t* __restrict__ W,
                                                                float* __restrict__ y, int64_t M, int64_t N,
                                                                int64_t K, int vec_y)
{
    __shared__ __align__(16) float As[2][TBK][kLd];
    __shared__ __align__(16) float Bs[2][TBK][kLd];

    const int tid = threadIdx.x;
    const int warp = tid / 32;
    const int tx = (tid % 8) + 8 * (warp % 2);  // 0..15: output columns tx*4.. and 64+tx*4..
    const int ty = ((tid / 8) % 4) + 4 * (warp / 2);  // 0..15: output rows ty*4.. and 64+ty*4..
    const int64_t m0 = static_cast<int64_t>(blockIdx.y) * TBM;
    const int64_t n0 = static_cast<int64_t>(blockIdx.x) * TBN;

    // Staged values of one K step: 8 of x and 8 of W per thread.
    //   vector path: x rows xr0 = tid/4 and xr0 + 64, k = 4*(tid%4) .. +3;
    //                W row tid/2, k = 8*(tid%2) .. +7
    //   scalar path: x and W row tid/2, k = 8*(tid%2) .. +7
    float ra[8], rb[8];
    const int xr0 = kVec ? tid / 4 : tid / 2;
    const int xk = kVec ? 4 * (tid % 4) : 8 * (tid % 2);
    const int wr = tid / 2, wk = 8 * (tid % 2);

    auto load = [&](int64_t k0) {
        if constexpr (kVec) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int64_t m = m0 + xr0 + 64 * h;
                const int64_t k = k0 + xk;
                float4 v = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                if (m < M && k < K)
                    v = __ldg(reinterpret_cast<const float4*>(x + m * K + k));
                ra[4 * h] = v.x;
                ra[4 * h + 1] = v.y;
                ra[4 * h + 2] = v.z;
                ra[4 * h + 3] = v.w;
            }
            const int64_t n = n0 + wr;
            const int64_t k = k0 + wk;
            uint4 u = make_uint4(0u, 0u, 0u, 0u);
            if (n < N && k < K)
                u = __ldg(reinterpret_cast<const uint4*>(W + n * K + k));
            const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w4[i]));
                rb[2 * i] = f.x;
                rb[2 * i + 1] = f.y;
            }
        } else {
            const int64_t gm = m0 + xr0, gn = n0 + wr;
            const float* xrow = x + (gm < M ? gm : 0) * K;
            const uint16_t* wrow = W + (gn < N ? gn : 0) * K;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int64_t k = k0 + xk + i;
                ra[i] = (gm < M && k < K) ? xrow[k] : 0.0f;
                rb[i] = (gn < N && k < K) ? __half2float(__ushort_as_half(wrow[k])) : 0.0f;
            }
        }
    };
    auto stage = [&](int buf) {
        if constexpr (kVec) {
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    As[buf][xk + i][xr0 + 64 * h] = ra[4 * h + i];
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i)
                As[buf][xk + i][xr0] = ra[i];
        }
#pragma unroll
        for (int i = 0; i < 8; ++i)
            Bs[buf][wk + i][wr] = rb[i];
    };

    float acc[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j)
            acc[i][j] = 0.0f;

    const int64_t nk = (K + TBK - 1) / TBK;
    load(0);
    stage(0);
    __syncthreads();
    for (int64_t kt = 0; kt < nk; ++kt) {
        const int buf = static_cast<int>(kt & 1);
        if (kt + 1 < nk)
            load((kt + 1) * TBK);
#pragma unroll
        for (int kk = 0; kk < TBK; ++kk) {
            const float4 a0 = *reinterpret_cast<const float4*>(&As[buf][kk][ty * 4]);
            const float4 a1 = *reinterpret_cast<const float4*>(&As[buf][kk][64 + ty * 4]);
            const float4 b0 = *reinterpret_cast<const float4*>(&Bs[buf][kk][tx * 4]);
            const float4 b1 = *reinterpret_cast<const float4*>(&Bs[buf][kk][64 + tx * 4]);
            const float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
            const float b[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int j = 0; j < 8; j += 2)
                    fma2(acc[i][j], acc[i][j + 1], a[i], b[j], b[j + 1]);
        }
        if (kt + 1 < nk)
            stage(buf ^ 1);
        __syncthreads();
    }

#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int64_t m = m0 + (i < 4 ? ty * 4 + i : 64 + ty * 4 + (i - 4));
        if (m >= M)
            continue;
        float* yrow = y + m * N;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int64_t n = n0 + 64 * h + tx * 4;
            if (vec_y && n + 3 < N) {
                *reinterpret_cast<float4*>(yrow + n) =
                    make_float4(acc[i][4 * h], acc[i][4 * h + 1], acc[i][4 * h + 2], acc[i][4 * h + 3]);
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (n + j < N)
                        yrow[n + j] = acc[i][4 * h + j];
            }
        }
    }
}

}  // namespace

comp_status_t launch_gemm_simt(const float* x, const uint16_t* W, float* y, int64_t M, int64_t N, int64_t K,
                               const DeviceInfo& dev, cudaStream_t stream)
{
    (void)dev;
    const dim3 grid(static_cast<unsigned>((N + TBN - 1) / TBN), static_cast<unsigned>((M + TBM - 1) / TBM));
    const bool vec = K % 8 == 0 && (reinterpret_cast<uintptr_t>(x) & 15u) == 0 &&
                     (reinterpret_cast<uintptr_t>(W) & 15u) == 0;
    const int vec_y = (N % 4 == 0 && (reinterpret_cast<uintptr_t>(y) & 15u) == 0) ? 1 : 0;
    if (vec)
        gemm_simt_kernel<true><<<grid, kThreads, 0, stream>>>(x, W, y, M, N, K, vec_y);
    else
        gemm_simt_kernel<false><<<grid, kThreads, 0, stream>>>(x, W, y, M, N, K, vec_y);
    return launch_status();
}

}  // namespace compfp32
