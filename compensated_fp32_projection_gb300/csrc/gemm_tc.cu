// The fused compensated-FP32 projection on the fifth-generation tensor cores
// (laya.cpp docs/vulkan.md: the compensated-FP32 paragraph — two FP16
// components per input, both products with FP32 accumulators, combined in FP32
// — and "The fused split/merge build" paragraph — split and merge fused into
// the projection).
//
// One CTA computes a 128 x 256 tile of y = acc_hi + acc_lo * 2^-10:
//   warp 0      TMA producer: per K block of 64, one 256x64 FP16 box of W and
//               two 128x32 FP32 boxes of x into a pipeline stage (128-byte
//               swizzle), completion counted on the stage's `full` barrier;
//   warp 1      allocates 512 TMEM columns (two 128x256 FP32 accumulators) and,
//               from one thread, issues per K block 4 x 2 tcgen05.mma
//               (M=128, N=256, K=16): D_hi += hi*W^T, D_lo += lo*W^T, both
//               reading the same W descriptor; a commit frees the stage;
//   warps 2..5  split: each thread owns one row of the stage's x tile, reads
//               its 64 FP32 values, and writes hi = fp16_rne(x) and
//               lo = fp16_rne((x - hi) * 1024) in place, in the K-major
//               128-byte-swizzled layout the MMA reads (hi over the first 16
//               KB of the x area, lo over the second); then they run the
//               epilogue: tcgen05.ld of both accumulators, the merge
//               y = D_hi + D_lo * 2^-10 (two rounded FP32 operations), store.
// The plain-load variant (any alignment / K) has no producer warp: the split
// warps stage x and W with coalesced, bounds-checked loads into the same
// layout and then split as above.
//
// Every mbarrier wait is bounded: past about a second the waiting thread
// records a fault code, raises the CTA's abort flag, and all roles skip to the
// end, drain what they issued (also bounded) and free TMEM.
#include <cuda_fp16.h>

#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace compfp32 {
namespace {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 64;
constexpr int kStages = 3;
constexpr int kSplitWarps = 4;
constexpr int kThreads = 64 + 32 * kSplitWarps;
constexpr uint32_t kWBytes = BN * BK * 2;             // 32 KB: W box, FP16
constexpr uint32_t kABytes = BM * BK * 4;             // 32 KB: x as FP32, later hi | lo as FP16
constexpr uint32_t kHalfA = kABytes / 2;              // 16 KB: one 128x32 FP32 box / one 128x64 FP16 plane
constexpr uint32_t kStageBytes = kWBytes + kABytes;   // 64 KB
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kIdesc = idesc_f16_f32(BM, BN);
constexpr size_t kSmemBytes = 1024 /* alignment slack */ + kStages * kStageBytes + 256 /* barriers */;
constexpr long long kWaitLimit = 1ll << 31;  // cycles (about a second)

// Fault codes (the wait that gave up).
constexpr uint32_t kFaultProducerEmpty = 0x101;
constexpr uint32_t kFaultSplitFull = 0x201;
constexpr uint32_t kFaultSplitEmpty = 0x202;
constexpr uint32_t kFaultMmaReady = 0x301;
constexpr uint32_t kFaultEpilogue = 0x401;

__device__ uint32_t g_fault_word;

struct Barriers {
    uint64_t full[kStages];   // TMA bytes landed (count 1 + tx)
    uint64_t ready[kStages];  // hi/lo written (count kSplitWarps)
    uint64_t empty[kStages];  // MMAs of the stage completed (tcgen05.commit)
    uint64_t acc;             // all MMAs of the tile completed
    uint64_t drain;           // MMA drain on abort
    uint32_t tmem_base;
    int abort;
};

__device__ __forceinline__ bool wait_bounded(uint64_t* bar, uint32_t parity, Barriers* b, uint32_t code)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const long long start = clock64();
    while (true) {
        if (mbar_try_wait(bar, parity))
            return true;
        if (*reinterpret_cast<volatile int*>(&b->abort))
            return false;
        if (clock64() - start > kWaitLimit) {
            atomicCAS(&g_fault_word, 0u, code);
            *reinterpret_cast<volatile int*>(&b->abort) = 1;
            return false;
        }
    }
}

__device__ __forceinline__ bool aborted(Barriers* b)
{
    return *reinterpret_cast<volatile int*>(&b->abort) != 0;
}

// Barrier over the kSplitWarps split warps (named barrier 1) that also returns
// the AND of `v` over all of them.
__device__ __forceinline__ bool split_warps_all(bool v)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 q, %1, 0;\n\t"
        "bar.red.and.pred p, 1, %2, q;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(v)), "n"(32 * kSplitWarps)
        : "memory");
    return r != 0;
}

__device__ __forceinline__ uint32_t pack_h2(__half2 h)
{
    return *reinterpret_cast<uint32_t*>(&h);
}

// Byte offset of the 16-byte chunk `chunk` of row `row` in a tile of 128-byte
// rows with the 128-byte swizzle (the tile base is 1024-byte aligned).
__device__ __forceinline__ uint32_t sw128(uint32_t row, uint32_t chunk)
{
    return row * 128u + ((chunk ^ (row & 7u)) << 4);
}

// In-place split of one row of the stage's A area: reads the 64 FP32 values of
// row r (two 128x32 boxes), writes 64 hi values to plane 0 and 64 lo values to
// plane 1, each plane a 128x64 FP16 tile.  A thread only touches the bytes of
// its own row, so no other synchronisation is needed.
__device__ __forceinline__ void split_row_inplace(uint8_t* A, uint32_t r)
{
    float v[64];
#pragma unroll
    for (int c = 0; c < 16; ++c) {  // 16 chunks of 4 FP32: chunk c is k = 4c .. 4c+3
        const float4 q = *reinterpret_cast<const float4*>(A + (c >> 3) * kHalfA + sw128(r, c & 7));
        v[4 * c + 0] = q.x;
        v[4 * c + 1] = q.y;
        v[4 * c + 2] = q.z;
        v[4 * c + 3] = q.w;
    }
#pragma unroll
    for (int c = 0; c < 8; ++c) {  // 8 chunks of 8 FP16: chunk c is k = 8c .. 8c+7
        uint32_t h[4], l[4];
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            const float a = v[8 * c + 2 * p], b = v[8 * c + 2 * p + 1];
            const __half2 hh = __floats2half2_rn(a, b);
            const float2 hf = __half22float2(hh);
            const float ra = __fmul_rn(__fsub_rn(a, hf.x), 1024.0f);
            const float rb = __fmul_rn(__fsub_rn(b, hf.y), 1024.0f);
            h[p] = pack_h2(hh);
            l[p] = pack_h2(__floats2half2_rn(ra, rb));
        }
        *reinterpret_cast<uint4*>(A + sw128(r, c)) = make_uint4(h[0], h[1], h[2], h[3]);
        *reinterpret_cast<uint4*>(A + kHalfA + sw128(r, c)) = make_uint4(l[0], l[1], l[2], l[3]);
    }
}

// Plain-load staging of one K block by the split warps (128 threads):
// x rows m0..m0+127, k0..k0+63 as FP32 into the two 128x32 swizzled boxes,
// W rows n0..n0+255 as FP16 into the 256x64 swizzled tile; zero outside.
__device__ __forceinline__ void stage_plain(uint8_t* Wt, uint8_t* A, const float* __restrict__ x,
                                            const uint16_t* __restrict__ W, int64_t M, int64_t N, int64_t K,
                                            int64_t m0, int64_t n0, int64_t k0, int sw, int lane)
{
    // x: warp sw handles rows sw, sw+4, ...; lane covers k0+lane and k0+32+lane
#pragma unroll 4
    for (int r = sw; r < BM; r += kSplitWarps) {
        const int64_t m = m0 + r;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int64_t k = k0 + h * 32 + lane;
            const float v = (m < M && k < K) ? x[m * K + k] : 0.0f;
            *reinterpret_cast<float*>(A + h * kHalfA + sw128(r, lane >> 2) + (lane & 3) * 4) = v;
        }
    }
    // W: lane covers the FP16 pair k0+2*lane, k0+2*lane+1
#pragma unroll 4
    for (int r = sw; r < BN; r += kSplitWarps) {
        const int64_t n = n0 + r;
        const int64_t k = k0 + 2 * lane;
        uint32_t lo16 = 0, hi16 = 0;
        if (n < N) {
            const uint16_t* row = W + n * K;
            if (k < K)
                lo16 = row[k];
            if (k + 1 < K)
                hi16 = row[k + 1];
        }
        *reinterpret_cast<uint32_t*>(Wt + sw128(r, lane >> 2) + (lane & 3) * 4) = lo16 | (hi16 << 16);
    }
}

template <bool kTma>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmap_x, const __grid_constant__ CUtensorMap tmap_w,
                   const float* __restrict__ x, const uint16_t* __restrict__ W, float* __restrict__ y, int64_t M,
                   int64_t N, int64_t K, int vec_y)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Barriers* bars = reinterpret_cast<Barriers*>(smem + kStages * kStageBytes);
    auto stage_w = [&](int s) { return smem + s * kStageBytes; };
    auto stage_a = [&](int s) { return smem + s * kStageBytes + kWBytes; };

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const int64_t m0 = static_cast<int64_t>(blockIdx.y) * BM;
    const int64_t n0 = static_cast<int64_t>(blockIdx.x) * BN;
    const int num_kb = static_cast<int>((K + BK - 1) / BK);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&bars->full[s], 1);
            mbar_init(&bars->ready[s], kSplitWarps);
            mbar_init(&bars->empty[s], 1);
        }
        mbar_init(&bars->acc, 1);
        mbar_init(&bars->drain, 1);
        bars->abort = 0;
        fence_mbar_init();
        fence_proxy_async_smem();
        if (kTma) {
            tma_prefetch_desc(&tmap_x);
            tma_prefetch_desc(&tmap_w);
        }
    }
    if (warp == 1) {
        tmem_alloc(&bars->tmem_base, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;

    if (warp == 0) {
        // ---------------- TMA producer ----------------
        if (kTma && lane == 0) {
            int issued = 0;
            for (int kb = 0; kb < num_kb; ++kb) {
                const int s = kb % kStages;
                const uint32_t round = static_cast<uint32_t>(kb / kStages);
                if (kb >= kStages && !wait_bounded(&bars->empty[s], (round - 1) & 1, bars, kFaultProducerEmpty))
                    break;
                mbar_arrive_expect_tx(&bars->full[s], kStageBytes);
                tma_load_2d(stage_w(s), &tmap_w, &bars->full[s], kb * BK, static_cast<int32_t>(n0));
                tma_load_2d(stage_a(s), &tmap_x, &bars->full[s], kb * BK, static_cast<int32_t>(m0));
                tma_load_2d(stage_a(s) + kHalfA, &tmap_x, &bars->full[s], kb * BK + 32, static_cast<int32_t>(m0));
                issued = kb + 1;
            }
            if (aborted(bars)) {
                // let the copies still in flight land before the CTA exits
                for (int kb = issued - kStages < 0 ? 0 : issued - kStages; kb < issued; ++kb) {
                    const int s = kb % kStages;
                    const uint32_t round = static_cast<uint32_t>(kb / kStages);
                    const long long start = clock64();
                    while (!mbar_try_wait(&bars->full[s], round & 1) && clock64() - start < kWaitLimit) {
                    }
                }
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            int kb = 0;
            for (; kb < num_kb; ++kb) {
                const int s = kb % kStages;
                const uint32_t round = static_cast<uint32_t>(kb / kStages);
                if (!wait_bounded(&bars->ready[s], round & 1, bars, kFaultMmaReady))
                    break;
                tc_fence_after();
                const uint32_t a_base = smem_u32(stage_a(s));
                const uint32_t w_base = smem_u32(stage_w(s));
#pragma unroll
                for (int j = 0; j < BK / 16; ++j) {
                    const uint64_t bdesc = sw128_kmajor_desc(w_base + 32 * j);
                    const uint64_t hdesc = sw128_kmajor_desc(a_base + 32 * j);
                    const uint64_t ldesc = sw128_kmajor_desc(a_base + kHalfA + 32 * j);
                    const uint32_t accum = (kb > 0 || j > 0) ? 1u : 0u;
                    umma_f16(tmem, hdesc, bdesc, kIdesc, accum);
                    umma_f16(tmem + BN, ldesc, bdesc, kIdesc, accum);
                }
                umma_commit(&bars->empty[s]);
            }
            if (kb == num_kb) {
                umma_commit(&bars->acc);
            } else {
                // aborted: wait for the MMAs already issued before TMEM is freed
                umma_commit(&bars->drain);
                const long long start = clock64();
                while (!mbar_try_wait(&bars->drain, 0) && clock64() - start < kWaitLimit) {
                }
            }
        }
        __syncwarp();
    } else {
        // ---------------- split, then epilogue ----------------
        const int sw = warp - 2;                       // 0..3
        const uint32_t row = static_cast<uint32_t>(sw * 32 + lane);  // split row, 0..127
        bool ok = true;
        for (int kb = 0; kb < num_kb; ++kb) {
            const int s = kb % kStages;
            const uint32_t round = static_cast<uint32_t>(kb / kStages);
            if (kTma) {
                ok = wait_bounded(&bars->full[s], round & 1, bars, kFaultSplitFull);
                ok = __all_sync(0xffffffffu, ok);  // uniform per warp
            } else {
                if (kb >= kStages)
                    ok = wait_bounded(&bars->empty[s], (round - 1) & 1, bars, kFaultSplitEmpty);
                if (__all_sync(0xffffffffu, ok))
                    stage_plain(stage_w(s), stage_a(s), x, W, M, N, K, m0, n0, static_cast<int64_t>(kb) * BK, sw,
                                lane);
                ok = split_warps_all(ok);  // barrier over the split warps; uniform across them
            }
            if (!ok)
                break;
            split_row_inplace(stage_a(s), row);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&bars->ready[s]);
        }

        if (ok)
            ok = __all_sync(0xffffffffu, wait_bounded(&bars->acc, 0, bars, kFaultEpilogue));
        if (ok) {
            tc_fence_after();
            const int q = warp & 3;  // TMEM lane quarter this warp may access
            const int64_t m = m0 + q * 32 + lane;
            const uint32_t t_lane = tmem + (static_cast<uint32_t>(q * 32) << 16);
#pragma unroll 1
            for (int j = 0; j < BN / 32; ++j) {
                uint32_t rh[32], rl[32];
                tmem_ld_32x32b_x32(t_lane + 32 * j, rh);
                tmem_ld_32x32b_x32(t_lane + BN + 32 * j, rl);
                tmem_ld_wait();
                if (m < M) {
                    const int64_t nb = n0 + 32 * j;
                    float* yrow = y + m * N;
                    float out[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        out[i] = __fadd_rn(__uint_as_float(rh[i]), __fmul_rn(__uint_as_float(rl[i]), 0x1p-10f));
                    if (vec_y && nb + 32 <= N) {
#pragma unroll
                        for (int i = 0; i < 32; i += 4)
                            *reinterpret_cast<float4*>(yrow + nb + i) =
                                make_float4(out[i], out[i + 1], out[i + 2], out[i + 3]);
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            if (nb + i < N)
                                yrow[nb + i] = out[i];
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
        else
            (void)cudaGetLastError();
    });
    return fn;
}

bool encode_2d(CUtensorMap* map, CUtensorMapDataType dtype, size_t elem, const void* base, int64_t inner,
               int64_t outer, uint32_t box_inner, uint32_t box_outer)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn)
        return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(outer)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(inner) * elem};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, dtype, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <bool kTma>
bool configure_once(int device)
{
    static std::mutex mu;
    static bool done[64] = {};
    std::lock_guard<std::mutex> lock(mu);
    if (device < 0 || device >= 64)
        return false;
    if (!done[device]) {
        if (cudaFuncSetAttribute(gemm_tc_kernel<kTma>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kSmemBytes)) != cudaSuccess) {
            (void)cudaGetLastError();
            return false;
        }
        done[device] = true;
    }
    return true;
}

inline bool aligned16(const void* p)
{
    return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

}  // namespace

comp_status_t launch_gemm_tc(const float* x, const uint16_t* W, float* y, int64_t M, int64_t N, int64_t K,
                             int variant, const DeviceInfo& dev, cudaStream_t stream)
{
    const bool tma_ok = aligned16(x) && aligned16(W) && (K % 8 == 0);
    bool use_tma;
    if (variant == 1) {
        if (!tma_ok)
            return COMP_ERR_INVALID_VALUE;
        use_tma = true;
    } else if (variant == 2) {
        use_tma = false;
    } else {
        use_tma = tma_ok;
    }
    const int64_t grid_y = (M + BM - 1) / BM;
    const int64_t grid_x = (N + BN - 1) / BN;
    if (grid_y > 65535 || grid_x > 0x7FFFFFFF)
        return COMP_ERR_INVALID_VALUE;
    const int vec_y = (N % 4 == 0) && aligned16(y);

    CUtensorMap tx{}, tw{};
    if (use_tma && !(encode_2d(&tx, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, x, K, M, 32, BM) &&
                     encode_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, W, K, N, BK, BN))) {
        if (variant == 1)
            return COMP_ERR_CUDA;
        use_tma = false;  // the driver refused the descriptors: take the plain-load kernel
    }
    if (use_tma) {
        if (!configure_once<true>(dev.device))
            return COMP_ERR_CUDA;
        gemm_tc_kernel<true><<<dim3(static_cast<unsigned>(grid_x), static_cast<unsigned>(grid_y)), kThreads,
                               kSmemBytes, stream>>>(tx, tw, x, W, y, M, N, K, vec_y);
    } else {
        if (!configure_once<false>(dev.device))
            return COMP_ERR_CUDA;
        gemm_tc_kernel<false><<<dim3(static_cast<unsigned>(grid_x), static_cast<unsigned>(grid_y)), kThreads,
                                kSmemBytes, stream>>>(tx, tw, x, W, y, M, N, K, vec_y);
    }
    return launch_status();
}

comp_status_t read_and_clear_fault(cudaStream_t stream, uint32_t* where)
{
    uint32_t word = 0;
    const uint32_t zero = 0;
    if (cudaMemcpyFromSymbolAsync(&word, g_fault_word, sizeof(word), 0, cudaMemcpyDeviceToHost, stream) !=
            cudaSuccess ||
        cudaMemcpyToSymbolAsync(g_fault_word, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, stream) !=
            cudaSuccess ||
        cudaStreamSynchronize(stream) != cudaSuccess) {
        (void)cudaGetLastError();
        return COMP_ERR_CUDA;
    }
    if (where)
        *where = word;
    return word == 0 ? COMP_OK : COMP_ERR_TIMEOUT;
}

}  // namespace compfp32
