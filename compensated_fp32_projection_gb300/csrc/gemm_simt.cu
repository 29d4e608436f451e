// The true-FP32 reference product (laya.cpp docs/vulkan.md, paragraph on the
// true FP32 matrix kernels that keep explicitly FP32 operands from being
// converted to FP16): y = x * float(W)^T with binary32 fused multiply-adds on
// the CUDA cores, summed in increasing k.  W is widened to FP32 exactly.
//
// Shared-memory tiled: a 128x128 output tile per 256-thread block, 8x8
// outputs per thread, K step 16, operands staged k-major in shared memory and
// double-buffered through registers.  Any sizes and alignments (scalar,
// bounds-checked global loads).
#include <cuda_fp16.h>

#include "internal.h"

namespace compfp32 {
namespace {

constexpr int TBM = 128, TBN = 128, TBK = 16, kThreads = 256;

__global__ void __launch_bounds__(kThreads) gemm_simt_kernel(const float* __restrict__ x,
                                                             const uint16_t* __restrict__ W, float* __restrict__ y,
                                                             int64_t M, int64_t N, int64_t K)
{
    __shared__ __align__(16) float As[2][TBK][TBM];
    __shared__ __align__(16) float Bs[2][TBK][TBN];

    const int tid = threadIdx.x;
    const int tx = tid % 16, ty = tid / 16;
    const int64_t m0 = static_cast<int64_t>(blockIdx.y) * TBM;
    const int64_t n0 = static_cast<int64_t>(blockIdx.x) * TBN;

    // loader: thread stages 8 consecutive k of one row of x and one row of W
    const int lrow = tid >> 1, lk = (tid & 1) * 8;
    const int64_t gm = m0 + lrow, gn = n0 + lrow;
    const float* xrow = x + (gm < M ? gm : 0) * K;
    const uint16_t* wrow = W + (gn < N ? gn : 0) * K;
    float ra[8], rb[8];

    auto load = [&](int64_t k0) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int64_t k = k0 + lk + i;
            ra[i] = (gm < M && k < K) ? xrow[k] : 0.0f;
            rb[i] = (gn < N && k < K) ? __half2float(__ushort_as_half(wrow[k])) : 0.0f;
        }
    };
    auto stage = [&](int buf) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            As[buf][lk + i][lrow] = ra[i];
            Bs[buf][lk + i][lrow] = rb[i];
        }
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
                for (int j = 0; j < 8; ++j)
                    acc[i][j] = __fmaf_rn(a[i], b[j], acc[i][j]);
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
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int64_t n = n0 + (j < 4 ? tx * 4 + j : 64 + tx * 4 + (j - 4));
            if (n < N)
                y[m * N + n] = acc[i][j];
        }
    }
}

}  // namespace

comp_status_t launch_gemm_simt(const float* x, const uint16_t* W, float* y, int64_t M, int64_t N, int64_t K,
                               const DeviceInfo& dev, cudaStream_t stream)
{
    (void)dev;
    const dim3 grid(static_cast<unsigned>((N + TBN - 1) / TBN), static_cast<unsigned>((M + TBM - 1) / TBM));
    gemm_simt_kernel<<<grid, kThreads, 0, stream>>>(x, W, y, M, N, K);
    return launch_status();
}

}  // namespace compfp32
