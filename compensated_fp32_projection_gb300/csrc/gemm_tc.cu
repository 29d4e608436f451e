// The fused compensated-FP32 projection on the fifth-generation tensor cores.
//
// Method (laya.cpp, docs/vulkan.md):
//   - compensated-FP32 paragraph: each FP32 input is split into two FP16
//     components, both products with the exact FP16 weights accumulate in FP32,
//     and the two are combined in FP32;
//   - fused-build paragraph: split and merge folded into the projection;
//   - AMD paragraph: partial results of the tiles are summed by plain FP32
//     additions instead of one long chain of cooperative-matrix multiply-adds,
//     which removes the accumulation drift of long dot products.
//
// The kernels of this file, in order:
//   comp_gemm_kernel         fused, one CTA per 128 x BN tile (below; also
//                            the plain-load form for any alignment and K);
//   comp_f16x2_kernel,       the products and merge from split planes (the
//   comp_f16x2_splitk_kernel second pass of the two-pass form), one CTA per
//                            tile, or K split over a cluster for <= 32 rows;
//   comp_f16x2_pair_kernel   the same on CTA pairs (256-row tiles);
//   comp_f32x16_pair_kernel  fused on CTA pairs: FP32 x split in place in
//                            the pair product's stages;
//   comp_f16x2_swap_kernel   operands swapped for <= 32 rows, optionally with
//                            the split fused.
//
// comp_gemm_kernel: a persistent CTA computes 128 x BN tiles of y.  Per tile
// and K block of 64:
//   1. TMA brings the 128 x 64 FP32 block of x (two 128x32 boxes, 128-byte
//      swizzle) into a 4-deep shared-memory ring, and the BN x 64 FP16 box of W
//      into another 4-deep ring;
//   2. eight split warps (two per 32-row quarter, one half of the K block
//      each), one thread per row, read their part of the row of x, form
//      hi = fp16_rne(x) and lo = fp16_rne((x - hi) * 1024), and store both
//      into tensor memory (tcgen05.st), where the MMA reads its A operand;
//   3. one thread issues 8 tcgen05.mma (M=128, N=BN, K=16, A from tensor
//      memory, B = W from shared memory) into a fresh accumulator D: four for
//      lo*W^T (the first overwrites D), then four for hi*W^T, the first of
//      which scales the accumulator by 2^-10 on input, so that
//      D = hi*W^T + 2^-10 * (lo*W^T) for the block; both products read the
//      same W descriptor.  D is double-buffered, the A operand triple-buffered;
//   4. eight promotion warps read D (tcgen05.ld, all of a warp's columns in
//      one round trip) and add it to an FP32 register accumulator R with
//      round-to-nearest-even adds, one FP32 add per K block outside the tensor
//      core; after the tile's last block R is y.
// Tensor memory: D buffers at columns [0, 2*BN), A stages at [320, 512)
// (64 columns each: hi in the first 32, lo in the next 32).
//
// The plain-load variant (any alignment, any K) stages W and x with ordinary
// bounds-checked loads done by the split warps instead of TMA.
//
// Every mbarrier wait is bounded: after about a second the waiting thread
// records a fault code, raises the CTA's abort flag, and every role skips to
// the end, drains what it issued (bounded) and frees tensor memory.
#include <cuda_fp16.h>

#include <mutex>
#include <utility>

#include "internal.h"
#include "ptx.cuh"

namespace compfp32 {
namespace {

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int kPromoters = 8;  // warpgroups 1-2: promote the accumulator, store y
constexpr int kSplitters = 8;  // warpgroups 3-4: split x into hi/lo in tensor memory
constexpr int kThreads = 128 + 32 * (kPromoters + kSplitters);  // warpgroup 0: W and x producers, MMA issuer
// Register split between warpgroups (setmaxnreg).  The launch gives every
// thread 96 registers (640 threads, one CTA per SM), a pool of 61440; the
// control warpgroup drops to 24, the promotion warpgroups rise to 168 and the
// split warpgroups drop to 56: 128*24 + 256*168 + 256*56 = 60416 <= 61440.
// The build checks the 96.
constexpr int kLaunchRegs = 96;
constexpr int kCtrlRegs = 24;
constexpr int kPromoRegs = 168;
constexpr int kSplitRegs = 56;
static_assert(128 * kCtrlRegs + 32 * kPromoters * kPromoRegs + 32 * kSplitters * kSplitRegs <=
                  kThreads * kLaunchRegs,
              "register split");
constexpr int kWStages = 4;
constexpr int kXStages = 4;
constexpr uint32_t kXBytes = BM * BK * 4;  // 32 KB: two 128x32 FP32 boxes
constexpr uint32_t kXBox = kXBytes / 2;
constexpr uint32_t kTmemCols = 512;
constexpr int kAStageCols = 64;            // one A stage: hi (32 columns) + lo (32 columns)
constexpr long long kWaitLimit = 1ll << 31;  // cycles (about a second)

template <int BN>
struct Cfg {
    static_assert(BN % 32 == 0 && BN >= 64 && BN <= 160, "BN");
    static constexpr uint32_t kWBytes = BN * BK * 2;
    static constexpr size_t kSmem = 1024 + kWStages * kWBytes + kXStages * kXBytes + 512;
    static_assert(kSmem <= 232448, "shared memory");
    static constexpr uint32_t kIdesc = idesc_f16_f32(BM, BN);
    static constexpr int kHalf = BN / 2;  // accumulator columns per promotion warp
    // Tensor memory: two accumulator buffers, then as many A stages as fit.
    static constexpr uint32_t kACol = 2 * BN;
    static constexpr int kAStages = static_cast<int>((kTmemCols - kACol) / kAStageCols) > 4
                                        ? 4
                                        : static_cast<int>((kTmemCols - kACol) / kAStageCols);
    static_assert(kAStages >= 2, "A stages");
};

// Fault codes (the wait that gave up).
constexpr uint32_t kFaultWProducer = 0x101;
constexpr uint32_t kFaultXProducer = 0x102;
constexpr uint32_t kFaultMmaW = 0x301;
constexpr uint32_t kFaultMmaA = 0x302;
constexpr uint32_t kFaultMmaD = 0x303;
constexpr uint32_t kFaultSplitX = 0x201;
constexpr uint32_t kFaultSplitA = 0x202;
constexpr uint32_t kFaultSplitW = 0x203;
constexpr uint32_t kFaultPromote = 0x401;

__device__ uint32_t g_fault_word;

struct Barriers {
    uint64_t wfull[kWStages];   // W box landed (TMA bytes) / staged (plain path: split warps)
    uint64_t wempty[kWStages];  // MMAs reading the W stage completed
    uint64_t xfull[kXStages];   // x block landed (TMA bytes)
    uint64_t xempty[kXStages];  // split warps have read the x stage
    uint64_t aready[4];         // hi/lo of a K block are in tensor memory
    uint64_t aempty[4];         // MMAs reading the A stage completed
    uint64_t dfull[2];          // accumulator buffer holds a finished K block
    uint64_t dfree[2];          // promotion warps have read the accumulator buffer
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
};

// Suspend-time hint (ns) of the polling waits; 0 polls with the plain
// try_wait, whose own bounded wait window is the only pause.
#ifndef COMP_WAIT_SUSPEND_NS
#define COMP_WAIT_SUSPEND_NS 20000
#endif

__device__ __forceinline__ bool wait_bounded(uint64_t* bar, uint32_t parity, int* abort_flag, uint32_t code)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const long long start = clock64();
    while (true) {
        if (COMP_WAIT_SUSPEND_NS > 0 ? mbar_try_wait_sleep(bar, parity, COMP_WAIT_SUSPEND_NS)
                                     : mbar_try_wait(bar, parity))
            return true;
        if (*reinterpret_cast<volatile int*>(abort_flag))
            return false;
        if (clock64() - start > kWaitLimit) {
            atomicCAS(&g_fault_word, 0u, code);
            *reinterpret_cast<volatile int*>(abort_flag) = 1;
            return false;
        }
    }
}

// Warp-wide bounded wait: lane 0 polls, the verdict is broadcast, and on
// success every lane performs one (immediately successful) try_wait so that it
// observes the phase completion itself.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, int* abort_flag, uint32_t code)
{
    bool ok = true;
    if ((threadIdx.x & 31) == 0)
        ok = wait_bounded(bar, parity, abort_flag, code);
    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    if (ok)
        (void)mbar_try_wait(bar, parity);
    return ok;
}

// Bounded wait for the copies or MMAs a role already issued before the CTA
// exits after an abort; no fault code (the first failure has one).
// Lane 0 waits and the warp takes its verdict; for consumers whose reads are
// ordered by tcgen05.fence::after_thread_sync after this warp synchronisation
// (tensor-memory loads), so the other lanes need not touch the barrier.
__device__ __forceinline__ bool lane0_wait(uint64_t* bar, uint32_t parity, int* abort_flag, uint32_t code)
{
    bool ok = true;
    if ((threadIdx.x & 31) == 0)
        ok = wait_bounded(bar, parity, abort_flag, code);
    return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
}

__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity)
{
    const long long start = clock64();
    while (!mbar_try_wait(bar, parity) && clock64() - start < kWaitLimit) {
    }
}

// 16-byte load from shared memory at a 32-bit shared-window address.
__device__ __forceinline__ float4 lds128(uint32_t addr)
{
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr));
    return v;
}

__device__ __forceinline__ uint32_t pack_h2(__half2 h)
{
    return *reinterpret_cast<uint32_t*>(&h);
}

// Byte offset of 16-byte chunk `chunk` of row `row` in a tile of 128-byte rows
// with the 128-byte swizzle (tile base 1024-byte aligned).
__device__ __forceinline__ uint32_t sw128(uint32_t row, uint32_t chunk)
{
    return row * 128u + ((chunk ^ (row & 7u)) << 4);
}

__device__ __forceinline__ uint64_t f2_bits(float a, float b)
{
    return static_cast<uint64_t>(__float_as_uint(a)) | (static_cast<uint64_t>(__float_as_uint(b)) << 32);
}

__device__ __forceinline__ float lo_f(uint64_t v)
{
    return __uint_as_float(static_cast<uint32_t>(v));
}

__device__ __forceinline__ float hi_f(uint64_t v)
{
    return __uint_as_float(static_cast<uint32_t>(v >> 32));
}

// Split two consecutive values (a first): packed FP16 pairs hi and lo.
// The residual (a - hi) * 1024 is computed on both lanes at once, each
// operation rounded to nearest even and never fused (exact here: the
// difference and the scaling by a power of two are representable).
__device__ __forceinline__ void split2(float a, float b, uint32_t& hi, uint32_t& lo)
{
    const __half2 h = __floats2half2_rn(a, b);
    const float2 hf = __half22float2(h);
    uint64_t d, r;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(f2_bits(a, b)), "l"(f2_bits(hf.x, hf.y)));
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(d), "l"(f2_bits(1024.0f, 1024.0f)));
    hi = pack_h2(h);
    lo = pack_h2(__floats2half2_rn(lo_f(r), hi_f(r)));
}

// Two element-wise RNE FP32 additions: r0 += v0, r1 += v1.
__device__ __forceinline__ void add2(float& r0, float& r1, uint32_t v0, uint32_t v1)
{
    uint64_t s;
    asm("add.rn.f32x2 %0, %1, %2;"
        : "=l"(s)
        : "l"(f2_bits(r0, r1)), "l"(f2_bits(__uint_as_float(v0), __uint_as_float(v1))));
    r0 = lo_f(s);
    r1 = hi_f(s);
}

// Warp-wide: 32 TMEM lanes x 16 consecutive 32-bit columns.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
                 "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
                 : "memory");
}

__device__ __forceinline__ void tmem_st_wait()
{
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// D (+)= A * B^T with A (128 x 16 FP16) in tensor memory and B in shared memory.
__device__ __forceinline__ void umma_f16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// D = A * B^T + D * 2^-10 (accumulator input scaled by 2^-10), A in tensor memory.
__device__ __forceinline__ void umma_f16_ta_scale10(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, 1, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p, 10;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc)
        : "memory");
}

struct Problem {
    const float* x;
    const uint16_t* W;
    float* y;
    int M, N, K;
    int tiles_m, tiles_n, nk;
    int vec_y;
    int tma_y;                     // y is written with tensor-map stores (kernels that support it)
    const float* bias = nullptr;   // epilogue: [N], added to y (nullptr: none)
    const float* gate = nullptr;   // epilogue: [M, N], y times gelu(gate) (nullptr: factor 1)
    int stall = 0;                 // diagnostic: the producer leaves out its first stage's loads
};

// Epilogue of a GEGLU feed-forward step (laya.cpp docs/vulkan.md, feed-forward
// paragraph: gate activation and multiplication fused into one dispatch), on
// element (m, n) of the merged projection: gelu(gate) * (y + bias), with the
// exact GELU g * Phi(g), Phi(g) = erfc(-g / sqrt 2) / 2 (no cancellation for
// negative g).  Each operation rounds to nearest even; never contracted.
__device__ __forceinline__ float epilogue_at(float v, int64_t m, int64_t n, const Problem& P)
{
    if (P.bias)
        v = __fadd_rn(v, __ldg(P.bias + n));
    if (P.gate) {
        const float g = __ldg(P.gate + m * static_cast<int64_t>(P.N) + n);
        const float phi = __fmul_rn(0.5f, erfcf(__fmul_rn(-g, 0.70710678118654752f)));  // 1 / sqrt 2
        v = __fmul_rn(v, __fmul_rn(g, phi));
    }
    return v;
}

// The epilogue on 16 consecutive columns n0.. of row m, held in v[0..15];
// columns >= N are left as they are.  The bias and gate values are all loaded
// first (16-byte loads where the row segment allows), then combined, so that
// a thread waits for one round of loads per 16 columns.  Same operations as
// epilogue_at.
__device__ __forceinline__ void epilogue16(float* v, int64_t m, int64_t n0, const Problem& P)
{
    float b[16], f[16];  // bias, then the gate's gelu factors
    const bool full = n0 + 16 <= P.N;
    const float* grow = P.gate ? P.gate + m * static_cast<int64_t>(P.N) + n0 : nullptr;
    if (P.bias) {
        if (full && (reinterpret_cast<uintptr_t>(P.bias + n0) & 15u) == 0) {
#pragma unroll
            for (int i = 0; i < 16; i += 4)
                *reinterpret_cast<float4*>(b + i) = __ldg(reinterpret_cast<const float4*>(P.bias + n0 + i));
        } else {
#pragma unroll
            for (int i = 0; i < 16; ++i)
                b[i] = n0 + i < P.N ? __ldg(P.bias + n0 + i) : 0.0f;
        }
    }
    if (grow) {
        if (full && (reinterpret_cast<uintptr_t>(grow) & 15u) == 0) {
#pragma unroll
            for (int i = 0; i < 16; i += 4)
                *reinterpret_cast<float4*>(f + i) = __ldg(reinterpret_cast<const float4*>(grow + i));
        } else {
#pragma unroll
            for (int i = 0; i < 16; ++i)
                f[i] = n0 + i < P.N ? __ldg(grow + i) : 0.0f;
        }
        // one copy of the GELU arithmetic: a loop kept rolled over the 16 factors
#pragma unroll 1
        for (int i = 0; i < 16; ++i) {
            const float g = f[i];
            f[i] = __fmul_rn(g, __fmul_rn(0.5f, erfcf(__fmul_rn(-g, 0.70710678118654752f))));  // 1 / sqrt 2
        }
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        if (n0 + i < P.N) {
            float x = v[i];
            if (P.bias)
                x = __fadd_rn(x, b[i]);
            if (grow)
                x = __fmul_rn(x, f[i]);
            v[i] = x;
        }
    }
}

// Tile t covers rows (t / tiles_n) * 128 .. and columns (t % tiles_n) * BN ..;
// N runs fastest so that CTAs working at the same time share rows of x.
__device__ __forceinline__ int tile_m(int t, const Problem& P)
{
    return t / P.tiles_n;
}
__device__ __forceinline__ int tile_n(int t, const Problem& P)
{
    return t % P.tiles_n;
}

// Walks this CTA's K blocks in order (tiles blockIdx.x, + gridDim.x, ...; K
// blocks 0 .. nk-1 of each), dividing only when the tile changes.
template <int BN>
struct Cursor {
    int t, kb, m0, n0;  // tile, K block, first row, first column
    __device__ __forceinline__ void start(const Problem& P)
    {
        t = static_cast<int>(blockIdx.x);
        kb = 0;
        m0 = tile_m(t, P) * BM;
        n0 = tile_n(t, P) * BN;
    }
    __device__ __forceinline__ void next(const Problem& P)
    {
        if (++kb == P.nk) {
            kb = 0;
            t += static_cast<int>(gridDim.x);
            m0 = tile_m(t, P) * BM;
            n0 = tile_n(t, P) * BN;
        }
    }
};

template <int BN, bool kVec, bool EPI>
__global__ void __launch_bounds__(kThreads, 1)
    comp_gemm_kernel(const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ CUtensorMap tmap_x,
                     const Problem P)
{
    using C = Cfg<BN>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* wring = smem;                          // kWStages x BN x 128 B
    uint8_t* xring = smem + kWStages * C::kWBytes;  // kXStages x 32 KB
    Barriers* bars = reinterpret_cast<Barriers*>(xring + kXStages * kXBytes);

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const int num_tiles = P.tiles_m * P.tiles_n;
    const int my_tiles =
        static_cast<int>(blockIdx.x) < num_tiles ? (num_tiles - 1 - static_cast<int>(blockIdx.x)) / gridDim.x + 1 : 0;
    const int total = my_tiles * P.nk;  // K blocks this CTA processes

    if (threadIdx.x == 0) {
        for (int s = 0; s < kWStages; ++s) {
            mbar_init(&bars->wfull[s], kVec ? 1 : kSplitters);
            mbar_init(&bars->wempty[s], 1);
        }
        for (int s = 0; s < kXStages; ++s) {
            mbar_init(&bars->xfull[s], 1);
            mbar_init(&bars->xempty[s], kSplitters);
        }
        for (int a = 0; a < C::kAStages; ++a) {
            mbar_init(&bars->aready[a], kSplitters);
            mbar_init(&bars->aempty[a], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&bars->dfull[b], 1);
            mbar_init(&bars->dfree[b], kPromoters);
        }
        mbar_init(&bars->drain, 1);
        bars->abort = 0;
        fence_mbar_init();
        fence_proxy_async_smem();
        if (kVec) {
            tma_prefetch_desc(&tmap_w);
            tma_prefetch_desc(&tmap_x);
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

    if (warp < 4) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kCtrlRegs));
        if (kVec && (warp == 0 || warp == 2) && lane == 0) {
            // ---------------- TMA producers: W (warp 0) and x (warp 2) ----------------
            const bool is_w = warp == 0;
            const int depth = is_w ? kWStages : kXStages;
            uint64_t* full = is_w ? bars->wfull : bars->xfull;
            uint64_t* empty = is_w ? bars->wempty : bars->xempty;
            int issued = 0;
            Cursor<BN> cur;
            cur.start(P);
            for (int g = 0; g < total; ++g, cur.next(P)) {
                const int s = g % depth;
                if (g >= depth &&
                    !wait_bounded(&empty[s], ((g / depth) - 1) & 1, &bars->abort, is_w ? kFaultWProducer : kFaultXProducer))
                    break;
                const int k0 = cur.kb * BK;
                if (is_w) {
                    mbar_arrive_expect_tx(&full[s], C::kWBytes);
                    tma_load_2d(wring + s * C::kWBytes, &tmap_w, &full[s], k0, cur.n0);
                } else {
                    mbar_arrive_expect_tx(&full[s], kXBytes);
                    uint8_t* dst = xring + s * kXBytes;
                    tma_load_2d(dst, &tmap_x, &full[s], k0, cur.m0);
                    tma_load_2d(dst + kXBox, &tmap_x, &full[s], k0 + 32, cur.m0);
                }
                issued = g + 1;
            }
            if (*reinterpret_cast<volatile int*>(&bars->abort))
                for (int g = issued - depth < 0 ? 0 : issued - depth; g < issued; ++g)
                    drain_wait(&full[g % depth], (g / depth) & 1);
        } else if (warp == 1 && lane == 0) {
            // ---------------- MMA issuer ----------------
            // B descriptors: stage s, K step j = desc of stage 0 + (s * stage bytes + 32 j) / 16 in the
            // start-address field (no carry: shared addresses stay below 2^18).
            const uint64_t wdesc0 = sw128_kmajor_desc(smem_u32(wring));
            bool ok = true;
            for (int g = 0; g < total && ok; ++g) {
                const int sw = g % kWStages;
                const int sa = g % C::kAStages;  // A stage
                const int b = g & 1;          // accumulator buffer
                ok = wait_bounded(&bars->wfull[sw], (g / kWStages) & 1, &bars->abort, kFaultMmaW) &&
                     wait_bounded(&bars->aready[sa], (g / C::kAStages) & 1, &bars->abort, kFaultMmaA) &&
                     (g < 2 || wait_bounded(&bars->dfree[b], ((g >> 1) - 1) & 1, &bars->abort, kFaultMmaD));
                if (!ok)
                    break;
                tc_fence_after();
                const uint32_t d = tmem + b * BN;
                const uint32_t a_hi = tmem + C::kACol + sa * 64;
                const uint32_t a_lo = a_hi + 32;
                const uint64_t bd = wdesc0 + static_cast<uint64_t>(sw * (C::kWBytes >> 4));
#pragma unroll
                for (int j = 0; j < BK / 16; ++j)  // lo * W^T, the first overwrites D
                    umma_f16_ta(d, a_lo + 8 * j, bd + 2 * j, C::kIdesc, j > 0 ? 1u : 0u);
                // D = hi*W^T + 2^-10 * D, then the rest of hi*W^T
                umma_f16_ta_scale10(d, a_hi, bd, C::kIdesc);
#pragma unroll
                for (int j = 1; j < BK / 16; ++j)
                    umma_f16_ta(d, a_hi + 8 * j, bd + 2 * j, C::kIdesc, 1u);
                umma_commit(&bars->wempty[sw]);
                umma_commit(&bars->aempty[sa]);
                umma_commit(&bars->dfull[b]);
            }
            if (!ok) {
                umma_commit(&bars->drain);
                drain_wait(&bars->drain, 0);
            }
        }
    } else if (warp < 12) {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kPromoRegs));
        // ---------------- promotion: R (+)= D per K block, then store y ----------------
        const int wq = warp & 3;         // TMEM lane quarter this warp may access
        const int wh = (warp - 4) >> 2;  // column half of the tile
        float R[C::kHalf];
#pragma unroll
        for (int i = 0; i < C::kHalf; ++i)
            R[i] = 0.0f;
        Cursor<BN> cur;
        cur.start(P);
        for (int j = 0; j < total; ++j, cur.next(P)) {
            const int b = j & 1;
            if (!warp_wait(&bars->dfull[b], (j >> 1) & 1, &bars->abort, kFaultPromote))
                break;
            tc_fence_after();
            const uint32_t taddr = tmem + (static_cast<uint32_t>(wq * 32) << 16) + b * BN + wh * C::kHalf;
            uint32_t v[C::kHalf];  // the whole half row in one round trip
#pragma unroll
            for (int c = 0; c < C::kHalf; c += 16)
                tmem_ld16(taddr + c, *reinterpret_cast<uint32_t(*)[16]>(v + c));
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < C::kHalf; i += 2)
                add2(R[i], R[i + 1], v[i], v[i + 1]);
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&bars->dfree[b]);

            if (cur.kb == P.nk - 1) {
                // tile finished: R holds y[m, nb .. nb + BN/2) for this thread's row m
                const int64_t m = static_cast<int64_t>(cur.m0) + wq * 32 + lane;
                const int64_t nb = static_cast<int64_t>(cur.n0) + wh * C::kHalf;
                if (m < P.M) {
                    if constexpr (EPI) {
                        static_assert(C::kHalf % 16 == 0, "epilogue in pieces of 16 columns");
#pragma unroll
                        for (int p = 0; p < C::kHalf; p += 16)
                            epilogue16(R + p, m, nb + p, P);
                    }
                    float* yrow = P.y + m * P.N;
                    if (P.vec_y && nb + C::kHalf <= P.N) {
#pragma unroll
                        for (int i = 0; i < C::kHalf; i += 4)
                            *reinterpret_cast<float4*>(yrow + nb + i) = make_float4(R[i], R[i + 1], R[i + 2], R[i + 3]);
                    } else {
#pragma unroll
                        for (int i = 0; i < C::kHalf; ++i)
                            if (nb + i < P.N)
                                yrow[nb + i] = R[i];
                    }
                }
#pragma unroll
                for (int i = 0; i < C::kHalf; ++i)
                    R[i] = 0.0f;  // the next tile starts from +0 (0 + D = D exactly, except -0 -> +0)
            }
        }
    } else {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kSplitRegs));
        // ---------------- split: half a row of x -> hi/lo in tensor memory ----------------
        const int q = warp & 3;               // TMEM lane quarter
        const int kh = (warp - 12) >> 2;      // half of the K block: elements 32*kh .. 32*kh+31
        const uint32_t row = q * 32 + lane;   // row of the tile this thread splits
        const int st = threadIdx.x - 384;     // 0..255 (plain-path W staging)
        const uint32_t xring_s = smem_u32(xring);
        // byte offsets of this thread's 16-byte chunks of its row in an x box
        uint32_t xoff[8];
#pragma unroll
        for (int c = 0; c < 8; ++c)
            xoff[c] = sw128(row, c);
        Cursor<BN> cur;
        cur.start(P);
        for (int g = 0; g < total; ++g, cur.next(P)) {
            const int sx = g % kXStages;
            const int sa = g % C::kAStages;
            const int64_t k0 = static_cast<int64_t>(cur.kb) * BK;
            if (kVec) {
                if (!warp_wait(&bars->xfull[sx], (g / kXStages) & 1, &bars->abort, kFaultSplitX))
                    break;
            } else {
                // plain path: stage the W box with bounds-checked loads (BN rows x 8 chunks of 8 FP16)
                const int sw = g % kWStages;
                if (g >= kWStages && !warp_wait(&bars->wempty[sw], ((g / kWStages) - 1) & 1, &bars->abort, kFaultSplitW))
                    break;
                const int64_t n0 = cur.n0;
                uint8_t* Wt = wring + sw * C::kWBytes;
#pragma unroll 1
                for (int cid = st; cid < BN * 8; cid += 32 * kSplitters) {
                    const int r = cid >> 3, c = cid & 7;
                    const int64_t n = n0 + r;
                    uint32_t h[4] = {0, 0, 0, 0};
                    if (n < P.N) {
                        const uint16_t* wrow = P.W + n * P.K;
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const int64_t k = k0 + 8 * c + e;
                            const uint32_t v = k < P.K ? wrow[k] : 0u;
                            h[e >> 1] |= v << (16 * (e & 1));
                        }
                    }
                    *reinterpret_cast<uint4*>(Wt + sw128(r, c)) = make_uint4(h[0], h[1], h[2], h[3]);
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&bars->wfull[sw]);
            }
            if (g >= C::kAStages && !warp_wait(&bars->aempty[sa], ((g / C::kAStages) - 1) & 1, &bars->abort, kFaultSplitA))
                break;
            tc_fence_after();
            const uint32_t X = xring_s + sx * kXBytes + kh * kXBox;
            const int64_t m = static_cast<int64_t>(cur.m0) + row;
            // TMEM columns of this thread's part: hi at 16*kh .., lo at 32 + 16*kh ..
            const uint32_t a_row = tmem + (static_cast<uint32_t>(q * 32) << 16) + C::kACol + sa * 64 + 16 * kh;
#pragma unroll
            for (int qr = 0; qr < 2; ++qr) {  // 16 elements: k = 32*kh + 16*qr .. +15 -> 8 TMEM columns
                float v[16];
                if (kVec) {
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const float4 f = lds128(X + xoff[4 * qr + c]);
                        v[4 * c] = f.x;
                        v[4 * c + 1] = f.y;
                        v[4 * c + 2] = f.z;
                        v[4 * c + 3] = f.w;
                    }
                } else {
                    const float* xrow = P.x + (m < P.M ? m : 0) * static_cast<int64_t>(P.K);
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const int64_t k = k0 + 32 * kh + 16 * qr + e;
                        v[e] = (m < P.M && k < P.K) ? __ldg(xrow + k) : 0.0f;
                    }
                }
                uint32_t hi[8], lo[8];
#pragma unroll
                for (int p = 0; p < 8; ++p)
                    split2(v[2 * p], v[2 * p + 1], hi[p], lo[p]);
                tmem_st8(a_row + 8 * qr, hi);
                tmem_st8(a_row + 32 + 8 * qr, lo);
            }
            tmem_st_wait();
            if (kVec) {
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&bars->xempty[sx]);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&bars->aready[sa]);
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
// The two products and the merge from split planes (comp_gemm_f16x2): the
// second half of the two-pass form, in which comp_split_f32 writes hi and lo
// once and this kernel reads both planes by TMA, so no split work is repeated
// per output tile.  Per 128 x BN tile and chunk of two K blocks of 64:
//   lo*W^T of both blocks into a fresh TMEM accumulator, then hi*W^T of both
//   blocks, the first of which scales the accumulator by 2^-10 on input:
//   D = hi*W^T + 2^-10 (lo*W^T) over the chunk; eight promotion warps add each
//   chunk's D into FP32 registers (one FP32 addition per 128 of K).
// ---------------------------------------------------------------------------
namespace x2 {
constexpr int kPromoters = 8;
constexpr int kThreads = 128 + 32 * kPromoters;  // warpgroup 0: producer, MMA issuer, two idle warps
// 384 threads launch with 168 registers each (pool 64512): control 40,
// promotion 232: 128*40 + 256*232 = 64512.  The build checks the 168.
constexpr int kLaunchRegs = 168;
constexpr int kCtrlRegs = 40;
constexpr int kPromoRegs = 232;
static_assert(128 * kCtrlRegs + 32 * kPromoters * kPromoRegs <= kThreads * kLaunchRegs, "register split");
// BN: tile width; NS: pipeline stages; CH: K blocks per accumulation chunk
// (tensor-core accumulation restarts every CH * 64 of K; CH = 0 is the
// measurement option of one tensor-core chain per product over all of K, hi
// and lo in separate accumulators merged once at the tile end); AR: rows of the hi
// and lo boxes.  AR < 128 serves problems of at most AR rows: only AR rows of
// each plane are loaded, so a stage is small and many stages stay in flight
// while W streams.  The MMA still reads 128 rows from each plane's offset;
// rows AR..127 read whatever follows inside the same stage, and since each
// output row depends only on its own A row, those garbage rows only produce
// outputs that are never stored.
// KS: CTAs of a cluster that split K for the same tile (1: no split).  With
// AR = 32 their partial sums are added in rank order through the leader's
// shared memory (rows 0..31 only); with AR = 128 every rank keeps its partial
// tile in its own shared memory and reduces 1/KS of the tile's rows, reading
// all ranks' partials through distributed shared memory and adding them in
// rank order (reduce-scatter).
template <int BN, int NS, int CH, int AR = BM, int KS = 1>
struct Cfg {
    static_assert(BN % 32 == 0 && BN >= 64 && BN <= 256, "BN");
    static_assert(NS >= 2 && CH >= 0 && CH <= NS, "stages");
    static_assert(CH > 0 || (KS == 1 && 2 * BN <= 512), "one chain per product: two accumulators, no split K");
    static_assert(AR == BM || AR == 32, "box rows");
    static constexpr uint32_t kPlaneBytes = AR * BK * 2;  // an AR x 64 FP16 box
    static constexpr uint32_t kWBytes = BN * BK * 2;
    static constexpr uint32_t kStageBytes = 2 * kPlaneBytes + kWBytes;  // hi | lo | W
    static_assert(kStageBytes % 1024 == 0, "stage alignment of the 128-byte swizzle");
    static_assert(kPlaneBytes + BM * BK * 2 <= kStageBytes, "the 128-row read of the lo plane stays in its stage");
    static_assert(KS == 1 || (KS <= 8 && AR == 32) || (AR == BM && (KS == 2 || KS == 4)), "split K");
    static constexpr bool kScatter = KS > 1 && AR == BM;  // reduce-scatter of full 128-row tiles
    static constexpr int kRedStride = kScatter ? BN + 4 : BN / 2 + 4;  // floats per buffer row (padded)
    static constexpr uint32_t kRedBytes =
        KS == 1 ? 0u : (kScatter ? static_cast<uint32_t>(BM) * kRedStride * 4u : 2u * 32u * kRedStride * 4u);
    static_assert(!kScatter || (BN % 16 == 0 && (BM / KS) * (BN / 16) % 32 == 0), "reduce-scatter segments");
    static constexpr uint32_t kBarBytes = 512;
    static constexpr size_t kSmem = 1024 + NS * kStageBytes + kBarBytes + kRedBytes;
    static_assert(kSmem <= 232448, "shared memory");
    static constexpr uint32_t kIdesc = idesc_f16_f32(BM, BN);
    static constexpr int kHalf = BN / 2;
};

constexpr int kMaxStages = 12;
struct Barriers {
    uint64_t full[kMaxStages];   // hi, lo and W boxes landed (TMA bytes)
    uint64_t empty[kMaxStages];  // MMAs reading the stage completed
    uint64_t dfull[2];        // accumulator buffer holds a finished chunk
    uint64_t dfree[2];        // promotion warps have read the accumulator buffer
    uint64_t drain;
    uint64_t red_full[2];  // leader: a peer's partial sums for one column half are in the buffer
    uint64_t red_go[2];    // peer: the leader's buffer for one column half is free for this peer
    uint64_t rs_full;      // reduce-scatter: every rank's sums for this rank's rows are in its buffer
    uint64_t rs_done;      // reduce-scatter: every rank has read the sums this rank sent it
    uint32_t tmem_base;
    int abort;
};
}  // namespace x2

// Fault codes of the two-pass product kernel.
constexpr uint32_t kFaultX2Producer = 0x501;
constexpr uint32_t kFaultX2MmaFull = 0x502;
constexpr uint32_t kFaultX2MmaFree = 0x503;
constexpr uint32_t kFaultX2Promote = 0x504;
constexpr uint32_t kFaultX2Reduce = 0x505;

// The body of the single-CTA-tile product kernels.  With KS > 1 the CTAs of a
// cluster of KS split K for the same tile: rank r takes the contiguous K blocks
// [r nk / KS, (r + 1) nk / KS), and at the tile end the ranks' FP32 partial
// sums are added in rank order (deterministic, no atomics, no global scratch).
// For problems of at most 32 rows (AR = 32), whose valid rows all sit in TMEM
// lanes 0..31 (promotion warps 4 and 8), the peers send their sums to the
// leader, which adds them.  For 128-row tiles (AR = 128) the ranks reduce the
// tile between them (reduce-scatter through distributed shared memory): the
// laya.cpp page's ordered reduction of split projection products (Vulkan
// page, fused-build paragraph), here across the SMs of a cluster.
template <int BN, int NS, int CH, int AR, int KS, bool EPI>
__device__ __forceinline__ void f16x2_tile_body(const CUtensorMap& tmap_hi, const CUtensorMap& tmap_lo,
                                                const CUtensorMap& tmap_w, const Problem& P)
{
    using C = x2::Cfg<BN, NS, CH, AR, KS>;
    static_assert(NS <= x2::kMaxStages, "stages");
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    x2::Barriers* bars = reinterpret_cast<x2::Barriers*>(smem + NS * C::kStageBytes);
    static_assert(sizeof(x2::Barriers) <= C::kBarBytes, "barrier area");
    float* redbuf = reinterpret_cast<float*>(smem + NS * C::kStageBytes + C::kBarBytes);

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const int rank = KS > 1 ? static_cast<int>(cluster_ctarank()) : 0;
    const int group = static_cast<int>(blockIdx.x) / KS;  // this CTA's cluster (its tiles)
    const int groups = static_cast<int>(gridDim.x) / KS;
    const int kb_lo = rank * P.nk / KS;                    // this CTA's K blocks of every tile
    const int nkr = (rank + 1) * P.nk / KS - kb_lo;
    const int num_tiles = P.tiles_m * P.tiles_n;
    const int my_tiles = group < num_tiles ? (num_tiles - 1 - group) / groups + 1 : 0;
    const int total = my_tiles * nkr;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(&bars->full[s], 1);
            mbar_init(&bars->empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&bars->dfull[b], 1);
            mbar_init(&bars->dfree[b], x2::kPromoters);
        }
        mbar_init(&bars->drain, 1);
        for (int h = 0; h < 2; ++h) {
            mbar_init(&bars->red_full[h], 1);
            mbar_init(&bars->red_go[h], 1);
        }
        mbar_init(&bars->rs_full, x2::kPromoters);  // the warps of all ranks that hold this rank's rows
        mbar_init(&bars->rs_done, KS * x2::kPromoters);
        bars->abort = 0;
        fence_mbar_init();
        fence_proxy_async_smem();
        tma_prefetch_desc(&tmap_hi);
        tma_prefetch_desc(&tmap_lo);
        tma_prefetch_desc(&tmap_w);
    }
    if (warp == 1) {
        tmem_alloc(&bars->tmem_base, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    if (KS > 1)
        cluster_sync();  // every CTA's barriers initialised before any remote arrival
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;

    if (warp < 4) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(x2::kCtrlRegs));
        if (warp == 0 && lane == 0) {
            // ---------------- TMA producer: hi, lo and W boxes per K block ----------------
            int issued = 0;
            grid_dependency_wait();  // the planes come from the previous kernel of the stream
            int t = group, kb = 0;
            for (int g = 0; g < total; ++g) {
                const int s = g % NS;
                if (g >= NS && !wait_bounded(&bars->empty[s], ((g / NS) - 1) & 1, &bars->abort, kFaultX2Producer))
                    break;
                uint8_t* st = smem + s * C::kStageBytes;
                const int k0 = (kb_lo + kb) * BK;
                const int m0 = tile_m(t, P) * BM, n0 = tile_n(t, P) * BN;
                mbar_arrive_expect_tx(&bars->full[s], C::kStageBytes);
                tma_load_2d(st, &tmap_hi, &bars->full[s], k0, m0);
                tma_load_2d(st + C::kPlaneBytes, &tmap_lo, &bars->full[s], k0, m0);
                tma_load_2d(st + 2 * C::kPlaneBytes, &tmap_w, &bars->full[s], k0, n0);
                issued = g + 1;
                if (++kb == nkr) {
                    kb = 0;
                    t += groups;
                }
            }
            if (*reinterpret_cast<volatile int*>(&bars->abort))
                for (int g = issued - NS < 0 ? 0 : issued - NS; g < issued; ++g)
                    drain_wait(&bars->full[g % NS], (g / NS) & 1);
        } else if (warp == 1 && CH == 0) {
            // ---------------- MMA issuer, one tensor-core chain per product (CH = 0) ----------------
            // hi * W^T into columns [0, BN), lo * W^T into [BN, 2 BN), over all K
            // blocks of the tile; the promotion warps merge them once at the
            // tile end and hand the accumulators back before the next tile.
            const uint32_t leader = lane == 0 ? 1u : 0u;
            const uint64_t desc0 = sw128_kmajor_desc(smem_u32(smem));
            int tt = 0;
            bool ok = true;
            for (int g = 0; g < total; ++g) {
                const int s = g % NS;
                const int kbi = g % nkr;
                bool r = true;
                if (lane == 0) {
                    if (kbi == 0 && tt > 0)
                        r = wait_bounded(&bars->dfree[0], (tt - 1) & 1, &bars->abort, kFaultX2MmaFree);
                    r = r && wait_bounded(&bars->full[s], (g / NS) & 1, &bars->abort, kFaultX2MmaFull);
                }
                ok = __shfl_sync(0xffffffffu, r ? 1 : 0, 0) != 0;
                if (!ok)
                    break;
                tc_fence_after();
                const uint64_t st = desc0 + static_cast<uint64_t>((s * C::kStageBytes) >> 4);
                const uint64_t a_hi = st, a_lo = st + (C::kPlaneBytes >> 4), w = st + ((2 * C::kPlaneBytes) >> 4);
#pragma unroll
                for (int j = 0; j < BK / 16; ++j)
                    umma_f16_by(leader, tmem + BN, a_lo + 2 * j, w + 2 * j, C::kIdesc, (kbi > 0 || j > 0) ? 1u : 0u);
#pragma unroll
                for (int j = 0; j < BK / 16; ++j)
                    umma_f16_by(leader, tmem, a_hi + 2 * j, w + 2 * j, C::kIdesc, (kbi > 0 || j > 0) ? 1u : 0u);
                umma_commit_by(leader, &bars->empty[s]);
                if (kbi == nkr - 1) {
                    umma_commit_by(leader, &bars->dfull[0]);
                    ++tt;
                }
            }
            if (!ok) {
                umma_commit_by(leader, &bars->drain);
                if (lane == 0)
                    drain_wait(&bars->drain, 0);
                __syncwarp();
            }
        } else if (warp == 1) {
            // ---------------- MMA issuer, one chunk of CH K blocks at a time ----------------
            // The whole warp runs the loop, so descriptors are warp-uniform;
            // lane 0 observes the barriers and issues the MMAs and commits.
            const uint32_t leader = lane == 0 ? 1u : 0u;
            const uint64_t desc0 = sw128_kmajor_desc(smem_u32(smem));
            // Everything chunk (g, c) of n blocks needs: the full barriers of its
            // stages and, from the third chunk on, its accumulator buffer back from
            // promotion.  The whole warp tests them with non-blocking phase tests
            // (one broadcast access each, identical results in every lane).  The
            // tests for the next chunk are issued before the current chunk's last
            // block of MMAs and read after it, so that their shared-memory round
            // trips overlap queued tensor work; only resources still pending are
            // then waited for, after all of the current chunk is issued.
            auto test_chunk = [&](int g, int c, int n) -> bool {
                bool r = c < 2 || mbar_test_wait(&bars->dfree[c & 1], ((c >> 1) - 1) & 1);
#pragma unroll
                for (int i = 0; i < CH; ++i)
                    if (i < n)
                        r = mbar_test_wait(&bars->full[(g + i) % NS], ((g + i) / NS) & 1) && r;
                return r;
            };
            auto wait_chunk = [&](int g, int c, int n) -> bool {
                bool ok = true;
                if (lane == 0) {
#pragma unroll
                    for (int i = 0; i < CH; ++i)
                        if (ok && i < n)
                            ok = wait_bounded(&bars->full[(g + i) % NS], ((g + i) / NS) & 1, &bars->abort,
                                              kFaultX2MmaFull);
                    if (ok && c >= 2)
                        ok = wait_bounded(&bars->dfree[c & 1], ((c >> 1) - 1) & 1, &bars->abort, kFaultX2MmaFree);
                }
                return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
            };
            int g = 0, c = 0, kb = 0;
            int n = (nkr < CH) ? nkr : CH;  // blocks in this chunk (chunks stay inside a tile)
            bool ok = total == 0 || wait_chunk(0, 0, n);
            while (g < total && ok) {
                const int b = c & 1;
                tc_fence_after();
                const uint32_t d = tmem + b * BN;
                // descriptor of stage s: hi at +0, lo at +16 KB, W at +32 KB (start field counts 16 bytes)
                auto sdesc = [&](int blk, uint32_t off) {
                    return desc0 + static_cast<uint64_t>(((blk % NS) * C::kStageBytes + off) >> 4);
                };
                for (int i = 0; i < n; ++i) {  // lo * W^T of the chunk; the very first overwrites D
                    const uint64_t a = sdesc(g + i, C::kPlaneBytes), w = sdesc(g + i, 2 * C::kPlaneBytes);
#pragma unroll
                    for (int j = 0; j < BK / 16; ++j)
                        umma_f16_by(leader, d, a + 2 * j, w + 2 * j, C::kIdesc, (i > 0 || j > 0) ? 1u : 0u);
                }
                // the next chunk's coordinates
                const int g2 = g + n, c2 = c + 1;
                const int kb2 = (kb + n == nkr) ? 0 : kb + n;
                const int n2 = (nkr - kb2 < CH) ? nkr - kb2 : CH;
                bool ready2 = true;
                for (int i = 0; i < n; ++i) {  // hi * W^T; the first scales D by 2^-10 on input
                    const uint64_t a = sdesc(g + i, 0), w = sdesc(g + i, 2 * C::kPlaneBytes);
                    if (i == n - 1 && g2 < total)
                        ready2 = test_chunk(g2, c2, n2);
#pragma unroll
                    for (int j = 0; j < BK / 16; ++j) {
                        if (i == 0 && j == 0)
                            umma_f16_scale10_by(leader, d, a, w, C::kIdesc);
                        else
                            umma_f16_by(leader, d, a + 2 * j, w + 2 * j, C::kIdesc, 1u);
                    }
                    umma_commit_by(leader, &bars->empty[(g + i) % NS]);
                }
                umma_commit_by(leader, &bars->dfull[b]);
                g = g2;
                c = c2;
                kb = kb2;
                n = n2;
                if (g < total && !ready2)
                    ok = wait_chunk(g, c, n);
            }
            if (!ok) {
                umma_commit_by(leader, &bars->drain);
                if (lane == 0)
                    drain_wait(&bars->drain, 0);
                __syncwarp();
            }
        }
    } else if (CH == 0) {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(x2::kPromoRegs));
        // ---------------- promotion, one chain per product: y = D_hi + 2^-10 D_lo per tile ----------------
        const int wq = warp & 3;
        const int wh = (warp - 4) >> 2;
        int t = group;
        for (int g0 = 0, tt = 0; g0 < total; g0 += nkr, ++tt, t += groups) {
            if (warp == 4)
                (void)lane0_wait(&bars->dfull[0], tt & 1, &bars->abort, kFaultX2Promote);
            // one verdict for all promotion warps: a flag read by each warp after a
            // plain barrier could change between their reads
            if (bar_red_or(1, 32 * x2::kPromoters, *reinterpret_cast<volatile int*>(&bars->abort) != 0))
                break;
            tc_fence_after();
            const uint32_t taddr = tmem + (static_cast<uint32_t>(wq * 32) << 16) + wh * C::kHalf;
            float R[C::kHalf];
#pragma unroll
            for (int c0 = 0; c0 < C::kHalf; c0 += 16) {
                uint32_t vh[16], vl[16];
                tmem_ld16(taddr + c0, vh);
                tmem_ld16(taddr + BN + c0, vl);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    R[c0 + i] = __fadd_rn(__uint_as_float(vh[i]), __fmul_rn(__uint_as_float(vl[i]), 0x1p-10f));
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&bars->dfree[0]);
            const int64_t m = static_cast<int64_t>(tile_m(t, P)) * BM + wq * 32 + lane;
            const int64_t nb = static_cast<int64_t>(tile_n(t, P)) * BN + wh * C::kHalf;
            if (m < P.M) {
                if constexpr (EPI) {
#pragma unroll
                    for (int p = 0; p < C::kHalf; p += 16)
                        epilogue16(R + p, m, nb + p, P);
                }
                float* yrow = P.y + m * P.N;
#pragma unroll
                for (int i = 0; i < C::kHalf; ++i)
                    if (nb + i < P.N)
                        yrow[nb + i] = R[i];
            }
        }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(x2::kPromoRegs));
        // ---------------- promotion: R += D per chunk, then store y ----------------
        const int wq = warp & 3;         // TMEM lane quarter
        const int wh = (warp - 4) >> 2;  // column half of the tile
        float R[C::kHalf];
#pragma unroll
        for (int i = 0; i < C::kHalf; ++i)
            R[i] = 0.0f;
        // Split-K reduction of one finished tile, for the warps of lane quarter 0
        // (one per column half).  Peers, in rank order, wait for the leader's go,
        // store their sums into the leader's buffer and publish them (release at
        // cluster scope); the leader adds each peer's sums in rank order.
        auto reduce_tile = [&](int tt) -> bool {
            float* buf = redbuf + wh * 32 * C::kRedStride + lane * C::kRedStride;
            if (rank == 0) {
                for (int p = 1; p < KS; ++p) {
                    if (lane == 0)
                        mbar_arrive_release_cluster(mapa_shared(&bars->red_go[wh], static_cast<uint32_t>(p)));
                    bool ok = true;
                    if (lane == 0) {
                        const uint32_t parity = static_cast<uint32_t>(tt * (KS - 1) + p - 1) & 1u;
                        const long long start = clock64();
                        while (!mbar_try_wait_acquire_cluster(&bars->red_full[wh], parity)) {
                            if (*reinterpret_cast<volatile int*>(&bars->abort) || clock64() - start > kWaitLimit) {
                                atomicCAS(&g_fault_word, 0u, kFaultX2Reduce);
                                *reinterpret_cast<volatile int*>(&bars->abort) = 1;
                                ok = false;
                                break;
                            }
                        }
                    }
                    if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0))
                        return false;
                    (void)mbar_try_wait_acquire_cluster(&bars->red_full[wh], static_cast<uint32_t>(tt * (KS - 1) + p - 1) & 1u);
#pragma unroll
                    for (int i = 0; i < C::kHalf; i += 4) {
                        const float4 v = *reinterpret_cast<const float4*>(buf + i);
                        R[i] = __fadd_rn(R[i], v.x);
                        R[i + 1] = __fadd_rn(R[i + 1], v.y);
                        R[i + 2] = __fadd_rn(R[i + 2], v.z);
                        R[i + 3] = __fadd_rn(R[i + 3], v.w);
                    }
                    __syncwarp();
                }
            } else {
                bool ok = true;
                if (lane == 0) {
                    const long long start = clock64();
                    while (!mbar_try_wait_acquire_cluster(&bars->red_go[wh], static_cast<uint32_t>(tt) & 1u)) {
                        if (*reinterpret_cast<volatile int*>(&bars->abort) || clock64() - start > kWaitLimit) {
                            atomicCAS(&g_fault_word, 0u, kFaultX2Reduce);
                            *reinterpret_cast<volatile int*>(&bars->abort) = 1;
                            ok = false;
                            break;
                        }
                    }
                }
                if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0))
                    return false;
                (void)mbar_try_wait_acquire_cluster(&bars->red_go[wh], static_cast<uint32_t>(tt) & 1u);
                const uint32_t dst = mapa_shared(buf, 0);
#pragma unroll
                for (int i = 0; i < C::kHalf; i += 4)
                    st_cluster_v4(dst + 4u * i, R[i], R[i + 1], R[i + 2], R[i + 3]);
                __syncwarp();
                if (lane == 0)
                    mbar_arrive_release_cluster(mapa_shared(&bars->red_full[wh], 0));
            }
            return true;
        };
        // Reduce-scatter of one finished 128-row tile over the cluster (AR = 128):
        // rank r owns rows [r 128/KS, (r+1) 128/KS) of the tile.  Every
        // promotion warp stores its partial sums straight into the owner's
        // receive buffer (slot of the sending rank; remote stores through
        // distributed shared memory) and arrives on the owner's barrier; the
        // owner's 256 promotion threads then add the KS slots of each element
        // in rank order (binary32 RNE additions), apply the epilogue and store
        // y in pieces of 16 columns.  Before a rank sends the next tile's sums,
        // every owner has finished reading its buffer (rs_done).
        auto scatter_tile = [&](int tt, int tile) -> bool {
            auto wait_cluster = [&](uint64_t* bar, uint32_t parity) -> bool {
                bool ok = true;
                if (lane == 0) {
                    const long long start = clock64();
                    while (!mbar_try_wait_acquire_cluster(bar, parity)) {
                        if (*reinterpret_cast<volatile int*>(&bars->abort) || clock64() - start > kWaitLimit) {
                            atomicCAS(&g_fault_word, 0u, kFaultX2Reduce);
                            *reinterpret_cast<volatile int*>(&bars->abort) = 1;
                            ok = false;
                            break;
                        }
                    }
                }
                ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
                if (ok)
                    (void)mbar_try_wait_acquire_cluster(bar, parity);
                return ok;
            };
            constexpr int kRows = BM / KS;  // rows owned by one rank
            if (tt > 0 && !wait_cluster(&bars->rs_done, static_cast<uint32_t>(tt - 1) & 1u))
                return false;
            {
                const int row = wq * 32 + lane;           // this thread's row of the tile
                const uint32_t owner = static_cast<uint32_t>(row / kRows);
                const int slot_row = rank * kRows + row % kRows;  // receive buffer: [sender][row of the owner]
                const uint32_t dst = mapa_shared(redbuf + slot_row * C::kRedStride + wh * C::kHalf, owner);
#pragma unroll
                for (int i = 0; i < C::kHalf; i += 4)
                    st_cluster_v4(dst + 4u * i, R[i], R[i + 1], R[i + 2], R[i + 3]);
                __syncwarp();
                // the warp's 32 rows share one owner
                if (lane == 0)
                    mbar_arrive_release_cluster(mapa_shared(&bars->rs_full, owner));
            }
            if (!wait_cluster(&bars->rs_full, static_cast<uint32_t>(tt) & 1u))
                return false;
            constexpr int kSegsPerRow = BN / 16;
            const int tid = (warp - 4) * 32 + lane;
            const int64_t mt = static_cast<int64_t>(tile_m(tile, P)) * BM + rank * kRows;
            const int64_t nt = static_cast<int64_t>(tile_n(tile, P)) * BN;
            for (int sidx = tid; sidx < kRows * kSegsPerRow; sidx += 32 * x2::kPromoters) {
                const int rl = sidx / kSegsPerRow;
                const int c0 = (sidx % kSegsPerRow) * 16;
                float acc[16];
#pragma unroll
                for (int p = 0; p < KS; ++p) {
                    const float* src = redbuf + (p * kRows + rl) * C::kRedStride + c0;
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const float4 v = *reinterpret_cast<const float4*>(src + 4 * q);
                        if (p == 0) {
                            acc[4 * q] = v.x;
                            acc[4 * q + 1] = v.y;
                            acc[4 * q + 2] = v.z;
                            acc[4 * q + 3] = v.w;
                        } else {
                            acc[4 * q] = __fadd_rn(acc[4 * q], v.x);
                            acc[4 * q + 1] = __fadd_rn(acc[4 * q + 1], v.y);
                            acc[4 * q + 2] = __fadd_rn(acc[4 * q + 2], v.z);
                            acc[4 * q + 3] = __fadd_rn(acc[4 * q + 3], v.w);
                        }
                    }
                }
                const int64_t m = mt + rl, n0 = nt + c0;
                if (m < P.M && n0 < P.N) {
                    if constexpr (EPI)
                        epilogue16(acc, m, n0, P);
                    float* yrow = P.y + m * P.N;
                    if (P.vec_y && n0 + 16 <= P.N) {
#pragma unroll
                        for (int i = 0; i < 16; i += 4)
                            *reinterpret_cast<float4*>(yrow + n0 + i) =
                                make_float4(acc[i], acc[i + 1], acc[i + 2], acc[i + 3]);
                    } else {
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            if (n0 + i < P.N)
                                yrow[n0 + i] = acc[i];
                    }
                }
            }
            __syncwarp();
            if (lane == 0) {
                fence_release_smem_cta_cluster();  // the reads of the receive buffer, before the senders reuse it
                for (int p = 0; p < KS; ++p)
                    mbar_arrive_relaxed_cluster(mapa_shared(&bars->rs_done, static_cast<uint32_t>(p)));
            }
            return true;
        };
        int g = 0, c = 0, kb = 0;
        int t = group;
        int tt = 0;  // tiles finished by this CTA
        while (g < total) {
            const int n = (nkr - kb < CH) ? nkr - kb : CH;
            const int b = c & 1;
            // one warp polls the barrier; the others wait at a named barrier
            // (no shared-memory traffic) and read the verdict from the abort flag
            if (warp == 4)
                (void)lane0_wait(&bars->dfull[b], (c >> 1) & 1, &bars->abort, kFaultX2Promote);
            // one verdict for all promotion warps: a flag read by each warp after a
            // plain barrier could change between their reads
            if (bar_red_or(1, 32 * x2::kPromoters, *reinterpret_cast<volatile int*>(&bars->abort) != 0))
                break;
            tc_fence_after();
            const uint32_t taddr = tmem + (static_cast<uint32_t>(wq * 32) << 16) + b * BN + wh * C::kHalf;
            // all of this thread's columns in one round trip; the buffer goes back
            // to the MMA warp before the additions
            uint32_t v[C::kHalf];
#pragma unroll
            for (int q = 0; q < C::kHalf / 16; ++q)
                tmem_ld16(taddr + 16 * q, *reinterpret_cast<uint32_t(*)[16]>(v + 16 * q));
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&bars->dfree[b]);
#pragma unroll
            for (int i = 0; i < C::kHalf; i += 2)
                add2(R[i], R[i + 1], v[i], v[i + 1]);
            g += n;
            ++c;
            kb += n;
            if (kb == nkr) {
                // tile finished: R holds this CTA's sums for y[m, nb .. nb + BN/2), m this thread's row
                if constexpr (C::kScatter) {
                    // a failed wait leaves the abort flag raised; every promotion
                    // warp then leaves at the next chunk's wait
                    (void)scatter_tile(tt, t);
                } else if (KS > 1 && wq == 0) {
                    // rows 0..31 (the only valid rows here) are in lane quarter 0.  A
                    // failed reduction leaves the abort flag raised; every promotion
                    // warp then leaves at the next chunk's wait, together.
                    (void)reduce_tile(tt);
                }
                if (!C::kScatter && (KS == 1 || (rank == 0 && wq == 0))) {
                    const int64_t m = static_cast<int64_t>(tile_m(t, P)) * BM + wq * 32 + lane;
                    const int64_t nb = static_cast<int64_t>(tile_n(t, P)) * BN + wh * C::kHalf;
                    if (m < P.M && *reinterpret_cast<volatile int*>(&bars->abort) == 0) {
                        if constexpr (EPI) {
                            static_assert(C::kHalf % 16 == 0, "epilogue in pieces of 16 columns");
#pragma unroll
                            for (int p = 0; p < C::kHalf; p += 16)
                                epilogue16(R + p, m, nb + p, P);
                        }
                        float* yrow = P.y + m * P.N;
                        if (P.vec_y && nb + C::kHalf <= P.N) {
#pragma unroll
                            for (int i = 0; i < C::kHalf; i += 4)
                                *reinterpret_cast<float4*>(yrow + nb + i) =
                                    make_float4(R[i], R[i + 1], R[i + 2], R[i + 3]);
                        } else {
#pragma unroll
                            for (int i = 0; i < C::kHalf; ++i)
                                if (nb + i < P.N)
                                    yrow[nb + i] = R[i];
                        }
                    }
                }
#pragma unroll
                for (int i = 0; i < C::kHalf; ++i)
                    R[i] = 0.0f;
                ++tt;
                kb = 0;
                t += groups;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (KS > 1)
        cluster_sync();  // no CTA leaves while another may still write its buffer or barriers
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

template <int BN, int NS, int CH, int AR, bool EPI>
__global__ void __launch_bounds__(x2::kThreads, 1)
    comp_f16x2_kernel(const __grid_constant__ CUtensorMap tmap_hi, const __grid_constant__ CUtensorMap tmap_lo,
                      const __grid_constant__ CUtensorMap tmap_w, const Problem P)
{
    f16x2_tile_body<BN, NS, CH, AR, 1, EPI>(tmap_hi, tmap_lo, tmap_w, P);
}

template <int BN, int NS, int CH, int AR, int KS, bool EPI>
__global__ void __cluster_dims__(KS, 1, 1) __launch_bounds__(x2::kThreads, 1)
    comp_f16x2_splitk_kernel(const __grid_constant__ CUtensorMap tmap_hi, const __grid_constant__ CUtensorMap tmap_lo,
                             const __grid_constant__ CUtensorMap tmap_w, const Problem P)
{
    f16x2_tile_body<BN, NS, CH, AR, KS, EPI>(tmap_hi, tmap_lo, tmap_w, P);
}

// ---------------------------------------------------------------------------
// Two-pass product on CTA pairs.  A cluster of two CTAs computes a 256 x BN
// tile with one tcgen05 instruction stream (.cta_group::2, M = 256) issued by
// the leader CTA (rank 0): each CTA holds its own 128 rows of the hi and lo
// planes and half of the tile's W rows (BN / 2) in shared memory, and its 128
// rows x BN columns of the accumulator in tensor memory.  Each SM thus reads
// half of W per MMA and loads half of W per stage, which keeps the tensor
// core's operand reads plus the TMA writes within the SM's shared-memory
// bandwidth.  The accumulation is that of comp_f16x2_kernel: per chunk of CH
// K blocks, lo * W^T fresh, then hi * W^T with the chunk's first MMA scaling
// the lo sums by 2^-10, promoted into FP32 registers in both CTAs.
// Synchronisation: each CTA's producer waits on its own empty barriers (the
// leader's commits multicast to both CTAs) and counts its TMA bytes on the
// leader's full barrier; both CTAs' promotion warps hand the accumulator back
// by arriving on the leader's dfree barrier.
// ---------------------------------------------------------------------------
namespace pair {
constexpr int kPromoters = 8;
constexpr int kThreads = 128 + 32 * kPromoters;  // warpgroup 0: producer, MMA issuer, its waiter, one idle warp
// 384 threads launch with 168 registers each (pool 64512): control 40,
// promotion 232: 128*40 + 256*232 = 64512.  The build checks the 168.
constexpr int kLaunchRegs = 168;
constexpr int kCtrlRegs = 40;
constexpr int kPromoRegs = 232;
static_assert(128 * kCtrlRegs + 32 * kPromoters * kPromoRegs <= kThreads * kLaunchRegs, "register split");
constexpr uint32_t kPlaneBytes = BM * BK * 2;  // one CTA's 128 rows x 64 of K, FP16
constexpr int kMaxStages = 8;
constexpr int kRows = 2 * BM;  // rows of a pair tile
// y epilogue: each promotion warp stages 32 rows x 16 columns of FP32 (2 KB,
// 64-byte swizzle) in one of two buffers and writes it with a TMA store.
constexpr uint32_t kYPiece = 32 * 16 * 4;
constexpr uint32_t kYStage = kPromoters * 2 * kYPiece;  // 32 KB
constexpr uint32_t kBarBytes = 1024;

// BN: the pair's tile width (each CTA holds BN / 2 rows of W); NS: stages;
// CH: K blocks per accumulation chunk.
template <int BN, int NS, int CH>
struct Cfg {
    static_assert(BN % 32 == 0 && BN >= 64 && BN <= 256, "BN");
    static_assert(NS >= 2 && NS <= kMaxStages && CH >= 1 && CH <= NS, "stages");
    static_assert(2 * BN <= 512, "tensor memory: two accumulator buffers");
    static constexpr uint32_t kWBytes = (BN / 2) * BK * 2;
    static constexpr uint32_t kStageBytes = 2 * kPlaneBytes + kWBytes;  // hi | lo | W half
    static_assert(kStageBytes % 1024 == 0, "stage alignment of the 128-byte swizzle");
    static constexpr uint32_t kTxBytes = 2 * kStageBytes;  // both CTAs' loads count on the leader's barrier
    static constexpr size_t kSmem = 1024 + NS * kStageBytes + kBarBytes + kYStage;
    static_assert(kSmem <= 232448, "shared memory");
    static constexpr uint32_t kIdesc = idesc_f16_f32(kRows, BN);
    static constexpr int kHalf = BN / 2;  // columns per promotion thread
    static_assert(kHalf % 16 == 0, "promotion loads 16 columns at a time");
};

struct Barriers {
    uint64_t full[kMaxStages];   // leader: both CTAs' hi, lo and W boxes landed
    uint64_t empty[kMaxStages];  // the stage's MMAs completed (commit multicast to both CTAs)
    uint64_t dfull[2];           // accumulator buffer holds a finished chunk (multicast)
    uint64_t dfree[2];           // leader: both CTAs' promotion warps have read the buffer
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
};
}  // namespace pair

// Fault codes of the CTA-pair product kernel.
constexpr uint32_t kFaultPairProducer = 0x701;
constexpr uint32_t kFaultPairMma = 0x702;
constexpr uint32_t kFaultPairPromote = 0x703;


// Bounded wait on a barrier that the other CTA of the cluster arrives on after
// a shared-memory release fence at cluster scope: relaxed polls at cluster
// scope, then the matching acquire fence.
__device__ __forceinline__ bool wait_bounded_cluster(uint64_t* bar, uint32_t parity, int* abort_flag, uint32_t code)
{
    const long long start = clock64();
    while (!mbar_try_wait_relaxed_cluster(bar, parity)) {
        if (*reinterpret_cast<volatile int*>(abort_flag))
            return false;
        if (clock64() - start > kWaitLimit) {
            atomicCAS(&g_fault_word, 0u, code);
            *reinterpret_cast<volatile int*>(abort_flag) = 1;
            return false;
        }
    }
    fence_acquire_smem_cluster();
    return true;
}

// Descriptor offset, in 16-byte units from the stage base, of K slice j
// (16 of K) of the hi or lo operand of a stage of the fused kernel: line r of
// box h (h = 0, 1) holds the hi values of K 32h .. 32h+31 of row r in its
// first 64 bytes and their lo values in its last 64 bytes, 128-byte rows with
// the 128-byte swizzle like the planes' boxes.
__device__ __forceinline__ constexpr uint32_t fused_a_slice(int j, bool lo)
{
    return static_cast<uint32_t>((j >> 1) * (pair::kPlaneBytes >> 4) + (lo ? 4 : 0) + 2 * (j & 1));
}

// The chunk sequence of one CTA pair of the two-pass product: chunk c starts
// at block g (block kb of its tile), in stage s with full-barrier parity ph,
// and has n blocks (CH, or fewer at a tile's end).  The waiter and the MMA
// issuer walk it in step.  Stage, parity and position advance by additions.
template <int NS, int CH>
struct PairChunkWalk {
    int g = 0, c = 0, kb = 0, s = 0, n = 0;
    uint32_t ph = 0;
    int nk = 0;
    __device__ __forceinline__ explicit PairChunkWalk(int nk_) : n(nk_ < CH ? nk_ : CH), nk(nk_) {}
    __device__ __forceinline__ static void stage_of(int s0, uint32_t ph0, int i, int& si, uint32_t& pi)
    {
        si = s0 + i;
        pi = ph0;
        if (si >= NS) {
            si -= NS;
            pi ^= 1u;
        }
    }
    __device__ __forceinline__ void next()
    {
        g += n;
        ++c;
        kb += n;
        if (kb == nk)
            kb = 0;
        int s2;
        uint32_t ph2;
        stage_of(s, ph, n, s2, ph2);
        s = s2;
        ph = ph2;
        n = nk - kb < CH ? nk - kb : CH;
    }
};

// Waiter of the two-pass pair product (warp 2 of the leader CTA): for each
// chunk in turn, waits until its stages have landed and its accumulator
// buffer is back from promotion, then hands the chunk to the MMA warp through
// a reduction at named barrier 2 + (chunk & 1) (64 threads: this warp and
// the MMA warp).  A failed wait passes false, which ends both loops at the
// same chunk.  The issuing thread's own mbarrier operations took hundreds of
// cycles each while the tensor cores streamed operands through shared
// memory; a named barrier does not go through shared memory, so the MMA warp
// now spends its time issuing.  A hand-off completes only when both warps
// have arrived, so neither can be more than one hand-off ahead of the other.
// Ordering: the waiter observes the stages' and the accumulator's barriers,
// the named barrier orders that before the MMA warp's
// tcgen05.fence::after_thread_sync, and the MMAs follow the fence.
template <int BN, int NS, int CH>
__device__ __forceinline__ void pair_wait_role(pair::Barriers* bars, int total, const Problem& P, int lane)
{
    PairChunkWalk<NS, CH> w(P.nk);
    bool ok = true;
    while (w.g < total) {
        if (ok && lane == 0) {
#pragma unroll
            for (int i = 0; i < CH; ++i)
                if (ok && i < w.n) {
                    int si;
                    uint32_t pi;
                    PairChunkWalk<NS, CH>::stage_of(w.s, w.ph, i, si, pi);
                    ok = wait_bounded(&bars->full[si], pi, &bars->abort, kFaultPairMma);
                }
            if (ok && w.c >= 2)
                ok = wait_bounded(&bars->dfree[w.c & 1], ((w.c >> 1) - 1) & 1, &bars->abort, kFaultPairMma);
        }
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (!bar_red_and(2 + (w.c & 1), 64, ok))
            break;
        w.next();
    }
}

// The MMA issuer of the two-pass pair product (leader CTA, warp 1; the whole
// warp runs the loop, lane 0 issues), one chunk of CH K blocks at a time,
// each handed over by the waiter warp: lo * W^T of the chunk into a fresh
// accumulator, then hi * W^T, whose first MMA scales the accumulator by
// 2^-10 on input.  Stage s holds, in both CTAs, the CTA's 128 rows of the hi
// plane (16 KB), then of the lo plane, then its half of the W rows.  The
// tensor pipe takes 112 cycles per 256 x 224 x 16 pair MMA and issuing one
// takes this thread 60 to 70, so the loop does nothing else between MMAs:
// descriptors are 32-bit words advanced by additions, and the commits that
// give the stages and the accumulator back are its only mbarrier accesses.
template <int BN, int NS, int CH>
__device__ __forceinline__ void pair_mma_role(pair::Barriers* bars, uint8_t* smem, uint32_t tmem, int total,
                                              const Problem& P, int lane)
{
    using C = pair::Cfg<BN, NS, CH>;
    const uint32_t leader = lane == 0 ? 1u : 0u;
    const uint64_t desc0 = sw128_kmajor_desc(smem_u32(smem));
    const uint32_t dlo0 = static_cast<uint32_t>(desc0);
    const uint32_t dhi = static_cast<uint32_t>(desc0 >> 32);
    constexpr uint32_t kSW = C::kStageBytes >> 4;
    constexpr uint32_t kPW = pair::kPlaneBytes >> 4;
    PairChunkWalk<NS, CH> w(P.nk);
    bool ok = true;
    while (w.g < total) {
        ok = bar_red_and(2 + (w.c & 1), 64, true);
        if (!ok)
            break;
        const uint32_t d = tmem + (w.c & 1) * BN;
        tc_fence_after();
        uint32_t st[CH];
        int sidx[CH];
#pragma unroll
        for (int i = 0; i < CH; ++i) {
            uint32_t pi;
            PairChunkWalk<NS, CH>::stage_of(w.s, w.ph, i, sidx[i], pi);
            st[i] = dlo0 + static_cast<uint32_t>(sidx[i]) * kSW;
        }
        const int n = w.n;
#pragma unroll
        for (int i = 0; i < CH; ++i)  // lo * W^T of the chunk; the very first overwrites D
            if (i < n) {
#pragma unroll
                for (int j = 0; j < BK / 16; ++j)
                    umma_pair_w_by(leader, d, st[i] + kPW + 2 * j, st[i] + 2 * kPW + 2 * j, dhi, C::kIdesc,
                                   (i > 0 || j > 0) ? 1u : 0u);
            }
#pragma unroll
        for (int i = 0; i < CH; ++i)  // hi * W^T; the first scales D by 2^-10 on input
            if (i < n) {
#pragma unroll
                for (int j = 0; j < BK / 16; ++j) {
                    if (i == 0 && j == 0)
                        umma_pair_w_scale10_by(leader, d, st[0], st[0] + 2 * kPW, dhi, C::kIdesc);
                    else
                        umma_pair_w_by(leader, d, st[i] + 2 * j, st[i] + 2 * kPW + 2 * j, dhi, C::kIdesc, 1u);
                }
                umma_commit_pair_by(leader, &bars->empty[sidx[i]], 0x3);
            }
        umma_commit_pair_by(leader, &bars->dfull[w.c & 1], 0x3);
        w.next();
    }
    if (!ok) {
        umma_commit_pair_by(leader, &bars->drain, 0x1);
        if (lane == 0)
            drain_wait(&bars->drain, 0);
        __syncwarp();
    }
}

// The MMA issuer of the fused pair kernel, in the same chunk order.  Stage s
// holds, in both CTAs, hi and lo of the CTA's 128 rows (first 32 KB, laid
// out as fused_a_slice says) and the CTA's half of the W rows.
// bars->full[s] counts the W bytes and split[s] the split warps of both CTAs
// (the other CTA's after a shared-memory release at cluster scope: relaxed
// polls at cluster scope, then the acquire fence).  A chunk starts once its
// first stage is ready, and each later stage is waited for just before its
// first MMA, so the products of a stage overlap the split of the next.  The
// bookkeeping is kept short as in the two-pass issuer (stages, parities and
// 32-bit descriptor words advanced by additions); the test for the next
// chunk stays before the last stage's hi products (testing it while the
// first hi product waits, as the two-pass issuer does, measured slower here).
template <int BN, int NS, int CH>
__device__ __forceinline__ void pair_mma_role_fused(pair::Barriers* bars, uint64_t* split, uint8_t* smem,
                                                    uint32_t tmem, int total, const Problem& P, int lane)
{
    using C = pair::Cfg<BN, NS, CH>;
    const uint32_t leader = lane == 0 ? 1u : 0u;
    const uint64_t desc0 = sw128_kmajor_desc(smem_u32(smem));
    const uint32_t dlo0 = static_cast<uint32_t>(desc0);
    const uint32_t dhi = static_cast<uint32_t>(desc0 >> 32);
    constexpr uint32_t kSW = C::kStageBytes >> 4;
    constexpr uint32_t kPW = pair::kPlaneBytes >> 4;
    const int nk = P.nk;
    auto stage_of = [](int s, uint32_t ph, int i, int& si, uint32_t& pi) {
        si = s + i;
        pi = ph;
        if (si >= NS) {
            si -= NS;
            pi ^= 1u;
        }
    };
    auto test_stage = [&](int si, uint32_t pi) -> bool {
        if (!(mbar_test_wait(&bars->full[si], pi) && mbar_test_wait_relaxed_cluster(&split[si], pi)))
            return false;
        fence_acquire_smem_cluster();
        return true;
    };
    auto wait_stage = [&](int si, uint32_t pi) -> bool {  // lane 0
        return wait_bounded(&bars->full[si], pi, &bars->abort, kFaultPairMma) &&
               wait_bounded_cluster(&split[si], pi, &bars->abort, kFaultPairMma);
    };
    auto test_chunk = [&](int s, uint32_t ph, int c) -> bool {
        return (c < 2 || mbar_test_wait(&bars->dfree[c & 1], ((c >> 1) - 1) & 1)) && test_stage(s, ph);
    };
    auto wait_chunk = [&](int s, uint32_t ph, int c) -> bool {
        bool ok = true;
        if (lane == 0) {
            ok = wait_stage(s, ph);
            if (ok && c >= 2)
                ok = wait_bounded(&bars->dfree[c & 1], ((c >> 1) - 1) & 1, &bars->abort, kFaultPairMma);
        }
        return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    };
    int g = 0, c = 0, kb = 0, s = 0;
    uint32_t ph = 0;
    int n = nk < CH ? nk : CH;
    bool ok = total == 0 || wait_chunk(s, ph, c);
    while (g < total && ok) {
        const uint32_t d = tmem + (c & 1) * BN;
        tc_fence_after();
        uint32_t st[CH];
        int sidx[CH];
        uint32_t spar[CH];
#pragma unroll
        for (int i = 0; i < CH; ++i) {
            stage_of(s, ph, i, sidx[i], spar[i]);
            st[i] = dlo0 + static_cast<uint32_t>(sidx[i]) * kSW;
        }
#pragma unroll
        for (int i = 0; i < CH; ++i)  // lo * W^T; each later stage is waited for before its first MMA
            if (i < n) {
                if (i >= 1) {
                    bool r = true;
                    if (lane == 0)
                        r = test_stage(sidx[i], spar[i]) || wait_stage(sidx[i], spar[i]);
                    ok = __shfl_sync(0xffffffffu, r ? 1 : 0, 0) != 0;
                    if (!ok)
                        break;
                    tc_fence_after();
                }
#pragma unroll
                for (int j = 0; j < BK / 16; ++j)
                    umma_pair_w_by(leader, d, st[i] + fused_a_slice(j, true), st[i] + 2 * kPW + 2 * j, dhi, C::kIdesc,
                                   (i > 0 || j > 0) ? 1u : 0u);
            }
        if (!ok)
            break;
        const int g2 = g + n, c2 = c + 1;
        int kb2 = kb + n;
        if (kb2 == nk)
            kb2 = 0;
        const int n2 = nk - kb2 < CH ? nk - kb2 : CH;
        int s2;
        uint32_t ph2;
        stage_of(s, ph, n, s2, ph2);
        bool ready2 = true;
#pragma unroll
        for (int i = 0; i < CH; ++i)  // hi * W^T; the first scales D by 2^-10 on input
            if (i < n) {
                if (i == n - 1 && g2 < total)
                    ready2 = test_chunk(s2, ph2, c2);
#pragma unroll
                for (int j = 0; j < BK / 16; ++j) {
                    if (i == 0 && j == 0)
                        umma_pair_w_scale10_by(leader, d, st[0] + fused_a_slice(0, false), st[0] + 2 * kPW, dhi,
                                               C::kIdesc);
                    else
                        umma_pair_w_by(leader, d, st[i] + fused_a_slice(j, false), st[i] + 2 * kPW + 2 * j, dhi,
                                       C::kIdesc, 1u);
                }
                umma_commit_pair_by(leader, &bars->empty[sidx[i]], 0x3);
            }
        umma_commit_pair_by(leader, &bars->dfull[c & 1], 0x3);
        g = g2;
        c = c2;
        kb = kb2;
        n = n2;
        s = s2;
        ph = ph2;
        if (g < total && !ready2)
            ok = wait_chunk(s, ph, c);
    }
    if (!ok) {
        umma_commit_pair_by(leader, &bars->drain, 0x1);
        if (lane == 0)
            drain_wait(&bars->drain, 0);
        __syncwarp();
    }
}

// Promotion in both CTAs of a pair (warps 4 .. 4 + kPromoters - 1): R += D per
// chunk in FP32 registers, RT accumulator columns per tensor-memory round
// trip; at the tile end the optional epilogue, then y.  Warp w owns TMEM lane
// quarter w % 4 (32 rows of the CTA's 128) and one column half of the tile.
template <int BN, int NS, int CH, bool EPI, int RT>
__device__ __forceinline__ void pair_promote_role(pair::Barriers* bars, const CUtensorMap* tmap_y, uint8_t* ystage,
                                                  uint32_t tmem, int total, const Problem& P, uint32_t rank,
                                                  int pair_id, int num_pairs, int warp, int lane)
{
    using C = pair::Cfg<BN, NS, CH>;
    static_assert(RT % 16 == 0 && RT <= 64, "round trip");
    const int wq = warp & 3;         // TMEM lane quarter
    const int wh = (warp - 4) >> 2;  // column half of the tile
    const uint32_t dfree0 = mapa_shared(&bars->dfree[0], 0);  // the leader's dfree barriers
    float R[C::kHalf];
#pragma unroll
    for (int i = 0; i < C::kHalf; ++i)
        R[i] = 0.0f;
    int g = 0, c = 0, kb = 0;
    int t = pair_id;
    uint8_t* ybuf = ystage + (warp - 4) * (2 * pair::kYPiece);
    int ng = 0;  // y pieces stored by this warp (its bulk groups, alternating buffers)
    while (g < total) {
        const int n = (P.nk - kb < CH) ? P.nk - kb : CH;
        const int b = c & 1;
        // one warp polls the barrier; the others wait at a named barrier
        if (warp == 4)
            (void)lane0_wait(&bars->dfull[b], (c >> 1) & 1, &bars->abort, kFaultPairPromote);
        // one verdict for all promotion warps: a flag read by each warp after a
        // plain barrier could change between their reads
        if (bar_red_or(1, 32 * pair::kPromoters, *reinterpret_cast<volatile int*>(&bars->abort) != 0))
            break;
        tc_fence_after();
        const uint32_t taddr = tmem + (static_cast<uint32_t>(wq * 32) << 16) + b * BN + wh * C::kHalf;
#pragma unroll
        for (int c0 = 0; c0 < C::kHalf; c0 += RT) {  // RT columns per round trip
            uint32_t v[RT];
#pragma unroll
            for (int q = 0; q < RT / 16; ++q)
                if (c0 + 16 * q < C::kHalf)
                    tmem_ld16(taddr + c0 + 16 * q, *reinterpret_cast<uint32_t(*)[16]>(v + 16 * q));
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < RT; i += 2)
                if (c0 + i < C::kHalf)
                    add2(R[c0 + i], R[c0 + i + 1], v[i], v[i + 1]);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0)
            mbar_arrive_cluster(dfree0 + static_cast<uint32_t>(b) * 8u);
        g += n;
        ++c;
        kb += n;
        if (kb == P.nk) {
            // tile finished: R holds y[m, nb .. nb + BN/2) for this thread's row m
            const int64_t row0 = static_cast<int64_t>(tile_m(t, P)) * pair::kRows + rank * BM + wq * 32;
            const int64_t m = row0 + lane;
            const int64_t nb = static_cast<int64_t>(tile_n(t, P)) * BN + wh * C::kHalf;
            if constexpr (EPI) {
                static_assert(C::kHalf % 16 == 0, "epilogue in pieces of 16 columns");
                if (m < P.M) {
#pragma unroll
                    for (int p = 0; p < C::kHalf; p += 16)
                        epilogue16(R + p, m, nb + p, P);
                }
            }
            if (P.tma_y) {
                // 16-column pieces through shared memory; the tensor-map store
                // clips rows >= M and columns >= N
#pragma unroll
                for (int p = 0; p < C::kHalf / 16; ++p) {
                    if (row0 >= P.M || nb + 16 * p >= P.N)
                        continue;
                    uint8_t* buf = ybuf + (ng & 1) * pair::kYPiece;
                    if (ng >= 2) {  // the store that last read this buffer has finished reading it
                        if (lane == 0)
                            bulk_wait_group_read1();
                        __syncwarp();
                    }
#pragma unroll
                    for (int j = 0; j < 4; ++j)  // 64-byte swizzle: 16-byte chunk j of row `lane`
                        st_shared_v4(buf + lane * 64 + ((j ^ ((lane >> 1) & 3)) << 4), R[16 * p + 4 * j],
                                     R[16 * p + 4 * j + 1], R[16 * p + 4 * j + 2], R[16 * p + 4 * j + 3]);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(tmap_y, buf, static_cast<int32_t>(nb + 16 * p), static_cast<int32_t>(row0));
                        bulk_commit_group();
                    }
                    ++ng;
                }
            } else if (m < P.M) {
                float* yrow = P.y + m * P.N;
                if (P.vec_y && nb + C::kHalf <= P.N) {
#pragma unroll
                    for (int i = 0; i < C::kHalf; i += 4)
                        *reinterpret_cast<float4*>(yrow + nb + i) = make_float4(R[i], R[i + 1], R[i + 2], R[i + 3]);
                } else {
#pragma unroll
                    for (int i = 0; i < C::kHalf; ++i)
                        if (nb + i < P.N)
                            yrow[nb + i] = R[i];
                }
            }
#pragma unroll
            for (int i = 0; i < C::kHalf; ++i)
                R[i] = 0.0f;
            kb = 0;
            t += num_pairs;
        }
    }
    if (lane == 0)
        bulk_wait_group0();  // y stores complete
    __syncwarp();
}

template <int BN, int NS, int CH, bool EPI>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(pair::kThreads, 1)
    comp_f16x2_pair_kernel(const __grid_constant__ CUtensorMap tmap_hi, const __grid_constant__ CUtensorMap tmap_lo,
                           const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ CUtensorMap tmap_y,
                           const Problem P)
{
    using C = pair::Cfg<BN, NS, CH>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    pair::Barriers* bars = reinterpret_cast<pair::Barriers*>(smem + NS * C::kStageBytes);
    static_assert(sizeof(pair::Barriers) <= pair::kBarBytes, "barrier area");
    uint8_t* ystage = smem + NS * C::kStageBytes + pair::kBarBytes;  // 1024-aligned

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const uint32_t rank = cluster_ctarank();
    const bool leader_cta = rank == 0;
    const int pair_id = static_cast<int>(blockIdx.x >> 1);
    const int num_pairs = static_cast<int>(gridDim.x >> 1);
    const int num_tiles = P.tiles_m * P.tiles_n;  // pair tiles of 256 x BN
    const int my_tiles = pair_id < num_tiles ? (num_tiles - 1 - pair_id) / num_pairs + 1 : 0;
    const int total = my_tiles * P.nk;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(&bars->full[s], 1);
            mbar_init(&bars->empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&bars->dfull[b], 1);
            mbar_init(&bars->dfree[b], 2 * pair::kPromoters);
        }
        mbar_init(&bars->drain, 1);
        bars->abort = 0;
        fence_mbar_init();
        fence_proxy_async_smem();
        tma_prefetch_desc(&tmap_hi);
        tma_prefetch_desc(&tmap_lo);
        tma_prefetch_desc(&tmap_w);
        if (P.tma_y)
            tma_prefetch_desc(&tmap_y);
    }
    if (warp == 1) {
        tmem_alloc_pair(&bars->tmem_base, kTmemCols);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // both CTAs' barriers initialised before any remote arrival
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;

    if (warp < 4) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(pair::kCtrlRegs));
        if (warp == 0 && lane == 0) {
            // ---------------- TMA producer (both CTAs): own rows of hi and lo, own half of W ----------------
            grid_dependency_wait();  // the planes come from the previous kernel of the stream
            const uint32_t full0 = mapa_shared(&bars->full[0], 0);  // the leader's full barriers
            int issued = 0;
            int t = pair_id, kb = 0;
            for (int g = 0; g < total; ++g) {
                const int s = g % NS;
                if (g >= NS && !wait_bounded(&bars->empty[s], ((g / NS) - 1) & 1, &bars->abort, kFaultPairProducer))
                    break;
                const int m0 = tile_m(t, P) * pair::kRows + static_cast<int>(rank) * BM;
                const int n0 = tile_n(t, P) * BN + static_cast<int>(rank) * (BN / 2);
                const int k0 = kb * BK;
                uint8_t* st = smem + s * C::kStageBytes;
                const uint32_t fb = full0 + static_cast<uint32_t>(s) * 8u;
                if (leader_cta)
                    mbar_arrive_expect_tx(&bars->full[s], C::kTxBytes);
                // diagnostic (comp_check_stalled_pipeline): the leader's first
                // stage never lands, so the MMA warp's bounded wait gives up
                if (!(P.stall && leader_cta && g == 0)) {
                    tma_load_2d_pair(st, &tmap_hi, fb, k0, m0);
                    tma_load_2d_pair(st + pair::kPlaneBytes, &tmap_lo, fb, k0, m0);
                    tma_load_2d_pair(st + 2 * pair::kPlaneBytes, &tmap_w, fb, k0, n0);
                }
                issued = g + 1;
                if (++kb == P.nk) {
                    kb = 0;
                    t += num_pairs;
                }
            }
            if (*reinterpret_cast<volatile int*>(&bars->abort)) {
                if (leader_cta) {
                    // the leader's full barriers count both CTAs' loads
                    for (int g = issued - NS < 0 ? 0 : issued - NS; g < issued; ++g)
                        drain_wait(&bars->full[g % NS], (g / NS) & 1);
                } else {
                    // this CTA's loads complete on the leader's barriers: give them time to land
                    const long long start = clock64();
                    while (clock64() - start < (1ll << 22)) {
                    }
                }
            }
        } else if (warp == 1 && leader_cta) {
            // ---------------- MMA issuer (leader CTA) ----------------
            pair_mma_role<BN, NS, CH>(bars, smem, tmem, total, P, lane);
        } else if (warp == 2 && leader_cta) {
            // ---------------- waiter for the MMA issuer (leader CTA) ----------------
            pair_wait_role<BN, NS, CH>(bars, total, P, lane);
        }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(pair::kPromoRegs));
        // ---------------- promotion (both CTAs): R += D per chunk, then store y ----------------
        pair_promote_role<BN, NS, CH, EPI, 64>(bars, &tmap_y, ystage, tmem, total, P, rank, pair_id, num_pairs, warp,
                                               lane);
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync();  // neither CTA leaves while the other may still signal its barriers
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem, kTmemCols);
    }
}

// ---------------------------------------------------------------------------
// The fused projection on CTA pairs (comp_gemm_f32x16 for outputs of about a
// wave of 256-row tiles or more): the pair product above, reading FP32 x
// instead of the split planes, so nothing but y leaves the kernel.
//
// Each CTA's producer loads its 128 rows of the K block of x by TMA, as two
// 128 x 32 FP32 boxes with the 128-byte swizzle, into the 32 KB of the stage
// where the pair product keeps its hi and lo boxes (the FP32 block has exactly
// their size).  Four split warps, one thread per row, then split each
// 128-byte line in place with the arithmetic of comp_split_f32: line r of box
// h holds x[r, 32h .. 32h+31]; afterwards its first 64 bytes hold their hi
// values and its last 64 bytes their lo values.  A line is read whole before
// it is written, and no line depends on another, so a thread orders only its
// own accesses.  The MMA reads hi and lo K slices at their offsets within the
// same 128-byte swizzled rows (fused_a_slice), in the order of the pair
// product, so both forms give identical bits.
//
// Signalling.  The TMA bytes of x count on a barrier of the CTA that loads
// them (xfull), which its split warps wait on.  A stage is ready for the MMA,
// issued by the leader CTA, when both CTAs' W halves have landed (bytes on
// the leader's `full`) and all eight split warps have written hi and lo
// (sfull).  The split warps publish their generic-proxy writes to the tensor
// cores with fence.proxy.async; the leader's split warps arrive on the
// leader's sfull, the other CTA's after a release fence at cluster scope
// restricted to shared memory, with a relaxed arrival.  The MMA lane polls
// sfull relaxed at cluster scope and then takes the matching acquire fence.
// ---------------------------------------------------------------------------
namespace fpair {
constexpr int kSplitters = 4;  // warps 12-15: split x in place, one thread per row
constexpr int kThreads = 128 + 32 * (pair::kPromoters + kSplitters);
// 512 threads launch with 128 registers each (pool 65536): control 40,
// promotion 208, split 56: 128*40 + 256*208 + 128*56 = 65536.  The build
// checks the 128.
constexpr int kLaunchRegs = 128;
constexpr int kCtrlRegs = 40;
constexpr int kPromoRegs = 208;
constexpr int kSplitRegs = 56;
static_assert(128 * kCtrlRegs + 32 * pair::kPromoters * kPromoRegs + 32 * kSplitters * kSplitRegs <=
                  kThreads * kLaunchRegs,
              "register split");
constexpr int kRoundTrip = 32;  // accumulator columns per tensor-memory round trip (fits 208 registers)

struct Barriers : pair::Barriers {
    uint64_t xfull[pair::kMaxStages];  // this CTA's FP32 x boxes landed (TMA bytes)
    uint64_t sfull[pair::kMaxStages];  // leader: the split warps of both CTAs wrote hi and lo
};
}  // namespace fpair

// Fault codes of the fused CTA-pair kernel (its MMA and promotion roles report
// the pair product's codes).
constexpr uint32_t kFaultFpairProducer = 0x901;
constexpr uint32_t kFaultFpairSplit = 0x903;

__device__ __forceinline__ void sts128(uint32_t addr, const uint32_t (&v)[4])
{
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3])
                 : "memory");
}

// Splits 8 consecutive values (two 16-byte chunks a, b of x) into one 16-byte
// chunk of hi and one of lo.
__device__ __forceinline__ void split8(const float4& a, const float4& b, uint32_t (&h)[4], uint32_t (&l)[4])
{
    split2(a.x, a.y, h[0], l[0]);
    split2(a.z, a.w, h[1], l[1]);
    split2(b.x, b.y, h[2], l[2]);
    split2(b.z, b.w, h[3], l[3]);
}

// One 128-byte line of a stage (32 FP32 values of a row, 16-byte chunk c at
// (c ^ sw) << 4) split in place: hi of the 32 values into chunks 0..3, lo
// into chunks 4..7.  All eight chunks are read before the first write.
__device__ __forceinline__ void split_line_in_place(uint32_t line, uint32_t sw)
{
    float4 v[8];
#pragma unroll
    for (uint32_t c = 0; c < 8; ++c)
        v[c] = lds128(line + ((c ^ sw) << 4));
#pragma unroll
    for (uint32_t c = 0; c < 4; ++c) {  // values 8c .. 8c+7
        uint32_t h[4], l[4];
        split8(v[2 * c], v[2 * c + 1], h, l);
        sts128(line + ((c ^ sw) << 4), h);
        sts128(line + (((4 + c) ^ sw) << 4), l);
    }
}

template <int BN, int NS, int CH, bool EPI>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(fpair::kThreads, 1)
    comp_f32x16_pair_kernel(const __grid_constant__ CUtensorMap tmap_x, const __grid_constant__ CUtensorMap tmap_w,
                            const __grid_constant__ CUtensorMap tmap_y, const Problem P)
{
    using C = pair::Cfg<BN, NS, CH>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    fpair::Barriers* bars = reinterpret_cast<fpair::Barriers*>(smem + NS * C::kStageBytes);
    static_assert(sizeof(fpair::Barriers) <= pair::kBarBytes, "barrier area");
    uint8_t* ystage = smem + NS * C::kStageBytes + pair::kBarBytes;  // 1024-aligned

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const uint32_t rank = cluster_ctarank();
    const bool leader_cta = rank == 0;
    const int pair_id = static_cast<int>(blockIdx.x >> 1);
    const int num_pairs = static_cast<int>(gridDim.x >> 1);
    const int num_tiles = P.tiles_m * P.tiles_n;  // pair tiles of 256 x BN
    const int my_tiles = pair_id < num_tiles ? (num_tiles - 1 - pair_id) / num_pairs + 1 : 0;
    const int total = my_tiles * P.nk;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(&bars->full[s], 1);  // leader: W bytes of both CTAs
            mbar_init(&bars->empty[s], 1);
            mbar_init(&bars->xfull[s], 1);
            mbar_init(&bars->sfull[s], 2 * fpair::kSplitters);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&bars->dfull[b], 1);
            mbar_init(&bars->dfree[b], 2 * pair::kPromoters);
        }
        mbar_init(&bars->drain, 1);
        bars->abort = 0;
        fence_mbar_init();
        fence_proxy_async_smem();
        tma_prefetch_desc(&tmap_x);
        tma_prefetch_desc(&tmap_w);
        if (P.tma_y)
            tma_prefetch_desc(&tmap_y);
    }
    if (warp == 1) {
        tmem_alloc_pair(&bars->tmem_base, kTmemCols);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // both CTAs' barriers initialised before any remote arrival
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;

    if (warp < 4) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(fpair::kCtrlRegs));
        if (warp == 0 && lane == 0) {
            // ---------------- TMA producer (both CTAs): own 128 rows of x, own half of W ----------------
            grid_dependency_wait();  // x may come from the previous kernel of the stream
            const uint32_t full0 = mapa_shared(&bars->full[0], 0);  // the leader's W barriers
            int issued = 0;
            int t = pair_id, kb = 0;
            for (int g = 0; g < total; ++g) {
                const int s = g % NS;
                if (g >= NS && !wait_bounded(&bars->empty[s], ((g / NS) - 1) & 1, &bars->abort, kFaultFpairProducer))
                    break;
                const int m0 = tile_m(t, P) * pair::kRows + static_cast<int>(rank) * BM;
                const int n0 = tile_n(t, P) * BN + static_cast<int>(rank) * (BN / 2);
                const int k0 = kb * BK;
                uint8_t* st = smem + s * C::kStageBytes;
                mbar_arrive_expect_tx(&bars->xfull[s], 2 * pair::kPlaneBytes);
                tma_load_2d(st, &tmap_x, &bars->xfull[s], k0, m0);
                tma_load_2d(st + pair::kPlaneBytes, &tmap_x, &bars->xfull[s], k0 + 32, m0);
                if (leader_cta)
                    mbar_arrive_expect_tx(&bars->full[s], 2 * C::kWBytes);
                tma_load_2d_pair(st + 2 * pair::kPlaneBytes, &tmap_w, full0 + static_cast<uint32_t>(s) * 8u, k0, n0);
                issued = g + 1;
                if (++kb == P.nk) {
                    kb = 0;
                    t += num_pairs;
                }
            }
            if (*reinterpret_cast<volatile int*>(&bars->abort)) {
                for (int g = issued - NS < 0 ? 0 : issued - NS; g < issued; ++g)
                    drain_wait(&bars->xfull[g % NS], (g / NS) & 1);
                if (leader_cta) {
                    // the leader's W barriers count both CTAs' W loads
                    for (int g = issued - NS < 0 ? 0 : issued - NS; g < issued; ++g)
                        drain_wait(&bars->full[g % NS], (g / NS) & 1);
                } else {
                    // this CTA's W loads complete on the leader's barriers: give them time to land
                    const long long start = clock64();
                    while (clock64() - start < (1ll << 22)) {
                    }
                }
            }
        } else if (warp == 1 && leader_cta) {
            // ---------------- MMA issuer (leader CTA) ----------------
            pair_mma_role_fused<BN, NS, CH>(bars, bars->sfull, smem, tmem, total, P, lane);
        }
    } else if (warp < 4 + pair::kPromoters) {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(fpair::kPromoRegs));
        // ---------------- promotion (both CTAs): R += D per chunk, then store y ----------------
        pair_promote_role<BN, NS, CH, EPI, fpair::kRoundTrip>(bars, &tmap_y, ystage, tmem, total, P, rank, pair_id,
                                                              num_pairs, warp, lane);
    } else {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(fpair::kSplitRegs));
        // ---------------- split (both CTAs): each stage's x rows -> hi and lo in place ----------------
        const uint32_t row = static_cast<uint32_t>(warp - 4 - pair::kPromoters) * 32u + lane;
        const uint32_t sfull0 = mapa_shared(&bars->sfull[0], 0);  // the leader's split barriers
        const uint32_t smem_s = smem_u32(smem);
        for (int g = 0; g < total; ++g) {
            const int s = g % NS;
            if (!warp_wait(&bars->xfull[s], (g / NS) & 1, &bars->abort, kFaultFpairSplit))
                break;
            const uint32_t line = smem_s + static_cast<uint32_t>(s) * C::kStageBytes + row * 128u;
            split_line_in_place(line, row & 7u);                       // K 0 .. 31 of the row
            split_line_in_place(line + pair::kPlaneBytes, row & 7u);  // K 32 .. 63
            fence_proxy_async_smem();  // generic-proxy stores, read next by the tensor cores
            __syncwarp();
            if (lane == 0) {
                if (leader_cta)
                    mbar_arrive(&bars->sfull[s]);
                else
                    mbar_arrive_release_smem_cluster(sfull0 + static_cast<uint32_t>(s) * 8u);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync();  // neither CTA leaves while the other may still signal its barriers
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem, kTmemCols);
    }
}

// ---------------------------------------------------------------------------
// Two-pass product for problems of at most 32 rows, with the operands swapped.
// The tensor cores compute y^T = W x^T.  The A operand is a 128-row tile of W,
// so the MMA rows are all used however small M is.  The B operand is the x rows
// padded to Mp (16 or 32): Mp hi rows, then Mp lo rows, N = 2 Mp.  One MMA
// therefore reads its 4 KB of W once for both products.  TMEM lane n of a
// tile holds, for output column n, the hi sums in columns 0..Mp-1 and the lo
// sums in Mp..2Mp-1.
//
// The kernel streams W, about 4 bytes of W per FLOP-pair of output, so its
// bound is DRAM.  A stage holds BPS consecutive 64-wide K blocks of the tile:
// the BPS W boxes, then per block its hi and lo boxes side by side (one
// 2 Mp-row B operand).  Asking for several K blocks of the same W rows at
// once reads more of each DRAM page per visit than one block per stage.  One
// stage is one accumulation chunk: it accumulates fresh in one of two TMEM
// buffers and promotion adds both halves into FP32 registers.  The epilogue
// merges y = R_hi + rn(2^-10 R_lo); a warp stores 32 consecutive columns of
// one row of y per instruction.
//
// FX (fused split): the kernel reads FP32 x instead of the planes.  The
// producer loads the stage's FP32 x boxes (L2-resident: every CTA reads all of
// x) into a staging area of the stage by TMA, with their own barrier, at the
// same time as the W boxes, so their latency hides behind that of W.  Two
// warps then split the staged values with the arithmetic of comp_split_f32
// and store hi and lo where the planes' TMA boxes would have put them.  TMA
// fills rows >= M and columns >= K with zeros, so the split needs no bounds.
// One kernel then does the whole projection, with no planes in HBM.
// ---------------------------------------------------------------------------
namespace swp {
constexpr int kPromoters = 4;
constexpr int kThreads = 128 + 32 * kPromoters;  // warpgroup 0: producer, MMA issuer, two idle warps
constexpr int kTileN = 128;                       // W rows per tile (the MMA's M)
constexpr int kMaxStages = 8;

template <int MP, int BPS, int NS, bool FX, int KS = 1>
struct Cfg {
    static_assert(MP == 16 || MP == 32, "padded rows of x");
    static_assert(BPS >= 1 && BPS <= 8 && NS >= 2 && NS <= kMaxStages, "pipeline");
    static_assert(KS == 1 || KS == 2 || KS == 4, "split K over a cluster of 1, 2 or 4 CTAs");
    static constexpr uint32_t kWBox = kTileN * BK * 2;  // 16 KB: one K block of the W tile
    static constexpr uint32_t kXBox = MP * BK * 2;      // one plane's Mp rows of one K block
    static constexpr uint32_t kXF = MP * BK * 4;        // FX: the FP32 x rows of one K block
    static constexpr uint32_t kXFOff = BPS * (kWBox + 2 * kXBox);
    static constexpr uint32_t kStageBytes = kXFOff + (FX ? BPS * kXF : 0u);
    static_assert(kXBox % 1024 == 0, "128-byte swizzle atoms");
    // split K: the partial sums of the columns this rank owns, one slot per
    // rank of the cluster: (4 / KS) warps x 32 lanes x (Mp hi, then Mp lo)
    static constexpr uint32_t kRedBytes = KS > 1 ? static_cast<uint32_t>(KS * (4 / KS) * 32 * 2 * MP * 4) : 0u;
    static constexpr size_t kSmem = 1024 + NS * kStageBytes + 512 + kRedBytes;
    static_assert(kSmem <= 232448, "shared memory");
    static constexpr int kCols = 2 * MP;               // accumulator columns per buffer
    static constexpr uint32_t kTmemCols = 2 * kCols;  // two buffers (64 or 128 columns)
    static constexpr uint32_t kIdesc = idesc_f16_f32(kTileN, kCols);
};

struct Barriers {
    uint64_t full[kMaxStages];
    uint64_t empty[kMaxStages];
    uint64_t xfull[kMaxStages];  // FX: the FP32 x boxes of the stage landed
    uint64_t dfull[2];
    uint64_t dfree[2];
    uint64_t drain;
    uint64_t rs_full[4];  // split K, owner: the other ranks' partial sums of warp w's columns landed
    uint64_t rs_done[4];  // split K, other ranks: the owner has read warp w's slot of the previous tile
    uint32_t tmem_base;
    int abort;
};
}  // namespace swp

// Fault codes of the swapped-operand product kernel.
constexpr uint32_t kFaultSwpProducer = 0x801;
constexpr uint32_t kFaultSwpMma = 0x802;
constexpr uint32_t kFaultSwpPromote = 0x803;
constexpr uint32_t kFaultSwpSplit = 0x804;
constexpr uint32_t kFaultSwpReduce = 0x805;

// Bounded wait, by lane 0 of a warp, for a barrier that other CTAs of the
// cluster arrive on with release at cluster scope; then every lane takes the
// phase with acquire at cluster scope itself, so that each may read what the
// arrivals published.
__device__ __forceinline__ bool warp_wait_acquire_cluster(uint64_t* bar, uint32_t parity, int* abort_flag,
                                                          uint32_t code)
{
    bool ok = true;
    if ((threadIdx.x & 31) == 0) {
        const long long start = clock64();
        while (!mbar_try_wait_acquire_cluster(bar, parity)) {
            if (*reinterpret_cast<volatile int*>(abort_flag) || clock64() - start > kWaitLimit) {
                atomicCAS(&g_fault_word, 0u, code);
                *reinterpret_cast<volatile int*>(abort_flag) = 1;
                ok = false;
                break;
            }
        }
    }
    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    if (ok)
        (void)mbar_try_wait_acquire_cluster(bar, parity);
    return ok;
}

// FX: tmap_hi is the map of FP32 x (boxes of 64 x Mp, no swizzle); tmap_lo is unused.
// KS > 1: a cluster of KS CTAs per tile, rank r taking the r-th of KS
// contiguous ranges of the K blocks; at the tile end rank r owns the tile's
// columns 128 r / KS .. 128 (r + 1) / KS - 1: the other ranks' promotion warps
// store their partial hi and lo sums of those columns into its receive buffer
// (distributed shared memory, st.async counting the bytes on its barrier,
// which the owner arms with the bytes due); the owner adds the KS partial sums
// in rank order (binary32, round to nearest even), so reruns give identical
// bits, then merges and stores y, and gives each slot back.
template <int MP, int BPS, int NS, bool FX, bool EPI, int KS>
__device__ __forceinline__ void swap_kernel_body(const CUtensorMap& tmap_hi, const CUtensorMap& tmap_lo,
                                                 const CUtensorMap& tmap_w, const Problem& P)
{
    using C = swp::Cfg<MP, BPS, NS, FX, KS>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    swp::Barriers* bars = reinterpret_cast<swp::Barriers*>(smem + NS * C::kStageBytes);
    static_assert(sizeof(swp::Barriers) <= 512, "barrier area");

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const int rank = KS > 1 ? static_cast<int>(cluster_ctarank()) : 0;
    const int cid = static_cast<int>(blockIdx.x) / KS;  // the cluster (one tile at a time)
    const int ncl = static_cast<int>(gridDim.x) / KS;
    const int num_tiles = P.tiles_n;  // tiles of 128 columns of y (rows of W)
    const int my_tiles = cid < num_tiles ? (num_tiles - 1 - cid) / ncl + 1 : 0;
    // this rank's K blocks of every tile: [kb_lo, kb_hi), at least one (the host
    // splits K only when every rank gets some)
    const int kb_lo = static_cast<int>(static_cast<int64_t>(P.nk) * rank / KS);
    const int kb_hi = static_cast<int>(static_cast<int64_t>(P.nk) * (rank + 1) / KS);
    const int spt = (kb_hi - kb_lo + BPS - 1) / BPS;  // stages per tile; the last may hold fewer blocks
    const int total = my_tiles * spt;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(&bars->full[s], FX ? 3 : 1);  // FX: the W bytes and both split warps
            mbar_init(&bars->empty[s], 1);
            mbar_init(&bars->xfull[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&bars->dfull[b], 1);
            mbar_init(&bars->dfree[b], swp::kPromoters);
        }
        mbar_init(&bars->drain, 1);
        for (int w = 0; w < 4; ++w) {
            mbar_init(&bars->rs_full[w], 1);  // the owner's expect_tx; the other ranks' bytes complete the phase
            mbar_init(&bars->rs_done[w], 1);
        }
        bars->abort = 0;
        fence_mbar_init();
        fence_proxy_async_smem();
        tma_prefetch_desc(&tmap_hi);
        if (!FX)
            tma_prefetch_desc(&tmap_lo);
        tma_prefetch_desc(&tmap_w);
    }
    if (warp == 1) {
        tmem_alloc(&bars->tmem_base, C::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    if (KS > 1)
        cluster_sync();  // every rank's barriers initialised before any remote arrival
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;

    if (warp == 0 && lane == 0) {
        // ---------------- TMA producer: per stage, BPS K blocks of the W tile and of both planes ----------------
        int issued = 0;
        grid_dependency_wait();  // the planes come from the previous kernel of the stream
        int t = cid, sk = 0;
        for (int g = 0; g < total; ++g) {
            const int s = g % NS;
            if (g >= NS && !wait_bounded(&bars->empty[s], ((g / NS) - 1) & 1, &bars->abort, kFaultSwpProducer))
                break;
            const int kb0 = kb_lo + sk * BPS;
            const int n = kb_hi - kb0 < BPS ? kb_hi - kb0 : BPS;
            uint8_t* st = smem + s * C::kStageBytes;
            if (FX) {  // the FP32 x rows first: the split warps need them before the MMA needs W
                mbar_arrive_expect_tx(&bars->xfull[s], n * C::kXF);
                for (int i = 0; i < n; ++i)
                    tma_load_2d(st + C::kXFOff + i * C::kXF, &tmap_hi, &bars->xfull[s], (kb0 + i) * BK, 0);
            }
            mbar_arrive_expect_tx(&bars->full[s], n * (C::kWBox + (FX ? 0u : 2 * C::kXBox)));
            // diagnostic (comp_check_stalled_pipeline): the first stage's W never
            // lands, so the MMA warp's bounded wait gives up
            for (int i = 0; i < n && !(P.stall && g == 0); ++i)
                tma_load_2d(st + i * C::kWBox, &tmap_w, &bars->full[s], (kb0 + i) * BK, t * swp::kTileN);
            for (int i = 0; i < n && !FX; ++i) {  // rows >= M read as 0
                uint8_t* xb = st + BPS * C::kWBox + i * 2 * C::kXBox;
                tma_load_2d(xb, &tmap_hi, &bars->full[s], (kb0 + i) * BK, 0);
                tma_load_2d(xb + C::kXBox, &tmap_lo, &bars->full[s], (kb0 + i) * BK, 0);
            }
            issued = g + 1;
            if (++sk == spt) {
                sk = 0;
                t += ncl;
            }
        }
        if (*reinterpret_cast<volatile int*>(&bars->abort))
            for (int g = issued - NS < 0 ? 0 : issued - NS; g < issued; ++g) {
                if (FX)
                    drain_wait(&bars->xfull[g % NS], (g / NS) & 1);
                drain_wait(&bars->full[g % NS], (g / NS) & 1);
            }
    } else if (warp == 1) {
        // ---------------- MMA issuer, one stage (= one accumulation chunk) at a time ----------------
        // The whole warp runs the loop (warp-uniform descriptors); lane 0 waits and issues.
        const uint32_t leader = lane == 0 ? 1u : 0u;
        const uint64_t desc0 = sw128_kmajor_desc(smem_u32(smem));
        int sk = 0;
        bool ok = true;
        for (int g = 0; g < total; ++g) {
            const int s = g % NS, b = g & 1;
            const int n = kb_hi - (kb_lo + sk * BPS) < BPS ? kb_hi - (kb_lo + sk * BPS) : BPS;
            // the stage's data, and from the third stage on its accumulator buffer back from promotion
            bool r = true;
            if (lane == 0) {
                r = wait_bounded(&bars->full[s], (g / NS) & 1, &bars->abort, kFaultSwpMma);
                if (r && g >= 2)
                    r = wait_bounded(&bars->dfree[b], ((g >> 1) - 1) & 1, &bars->abort, kFaultSwpMma);
            }
            ok = __shfl_sync(0xffffffffu, r ? 1 : 0, 0) != 0;
            if (!ok)
                break;
            tc_fence_after();
            const uint32_t d = tmem + b * C::kCols;
            const uint64_t st = desc0 + static_cast<uint64_t>((s * C::kStageBytes) >> 4);
            for (int i = 0; i < n; ++i) {
                const uint64_t a = st + static_cast<uint64_t>((i * C::kWBox) >> 4);  // A: W tile
                const uint64_t bx = st + static_cast<uint64_t>((BPS * C::kWBox + i * 2 * C::kXBox) >> 4);  // B: hi, lo
#pragma unroll
                for (int j = 0; j < BK / 16; ++j)
                    umma_f16_by(leader, d, a + 2 * j, bx + 2 * j, C::kIdesc, (i > 0 || j > 0) ? 1u : 0u);
            }
            umma_commit_by(leader, &bars->empty[s]);
            umma_commit_by(leader, &bars->dfull[b]);
            if (++sk == spt)
                sk = 0;
        }
        if (!ok) {
            umma_commit_by(leader, &bars->drain);
            if (lane == 0)
                drain_wait(&bars->drain, 0);
            __syncwarp();
        }
    } else if (FX && (warp == 2 || warp == 3)) {
        // ---------------- split: staged FP32 x of each stage -> hi and lo in the stage ----------------
        // Item (block i, row m, 16-byte chunk c): 8 consecutive x of row m,
        // stored where a 128-byte-swizzled TMA box of the planes would put them.
        constexpr int kItems = BPS * MP * 8;
        constexpr int kPer = (kItems + 63) / 64;
        const int lt = static_cast<int>(threadIdx.x) - 64;
        int sk = 0;
        for (int g = 0; g < total; ++g) {
            const int s = g % NS;
            if (!warp_wait(&bars->xfull[s], (g / NS) & 1, &bars->abort, kFaultSwpSplit))
                break;
            const int n = kb_hi - (kb_lo + sk * BPS) < BPS ? kb_hi - (kb_lo + sk * BPS) : BPS;
            uint8_t* st = smem + s * C::kStageBytes;
#pragma unroll
            for (int u = 0; u < kPer; ++u) {
                const int it = lt + 64 * u;
                const int i = it / (MP * 8), m = (it / 8) % MP, c = it % 8;
                if (it < kItems && i < n) {
                    const float4* src = reinterpret_cast<const float4*>(st + C::kXFOff + i * C::kXF + m * (BK * 4) + c * 32);
                    const float4 va = src[0], vb = src[1];
                    uint32_t h[4], l[4];
                    split2(va.x, va.y, h[0], l[0]);
                    split2(va.z, va.w, h[1], l[1]);
                    split2(vb.x, vb.y, h[2], l[2]);
                    split2(vb.z, vb.w, h[3], l[3]);
                    uint8_t* hb = st + BPS * C::kWBox + i * 2 * C::kXBox + m * 128 + ((c ^ (m & 7)) << 4);
                    st_shared_v4(hb, __uint_as_float(h[0]), __uint_as_float(h[1]), __uint_as_float(h[2]),
                                 __uint_as_float(h[3]));
                    st_shared_v4(hb + C::kXBox, __uint_as_float(l[0]), __uint_as_float(l[1]), __uint_as_float(l[2]),
                                 __uint_as_float(l[3]));
                }
            }
            fence_proxy_async_smem();  // generic-proxy stores, read next by the tensor cores
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&bars->full[s]);
            if (++sk == spt)
                sk = 0;
        }
    } else if (warp >= 4) {
        // ---------------- promotion and epilogue (lane quarter wq = rows 32 wq .. of the tile) ----------------
        const int wq = warp - 4;
        float Rh[MP], Rl[MP];
#pragma unroll
        for (int i = 0; i < MP; ++i) {
            Rh[i] = 0.0f;
            Rl[i] = 0.0f;
        }
        int sk = 0;
        int t = cid;
        int tt = 0;  // tiles finished by this CTA
        for (int g = 0; g < total; ++g) {
            const int b = g & 1;
            if (warp == 4)
                (void)lane0_wait(&bars->dfull[b], (g >> 1) & 1, &bars->abort, kFaultSwpPromote);
            // one verdict for all promotion warps: a flag read by each warp after a
            // plain barrier could change between their reads
            if (bar_red_or(1, 32 * swp::kPromoters, *reinterpret_cast<volatile int*>(&bars->abort) != 0))
                break;
            tc_fence_after();
            uint32_t v[C::kCols];
#pragma unroll
            for (int q = 0; q < C::kCols / 16; ++q)
                tmem_ld16(tmem + (static_cast<uint32_t>(wq * 32) << 16) + b * C::kCols + 16 * q,
                          *reinterpret_cast<uint32_t(*)[16]>(v + 16 * q));
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&bars->dfree[b]);
#pragma unroll
            for (int i = 0; i < MP; ++i) {
                Rh[i] = __fadd_rn(Rh[i], __uint_as_float(v[i]));
                Rl[i] = __fadd_rn(Rl[i], __uint_as_float(v[MP + i]));
            }
            if (++sk == spt) {
                // tile finished: this thread holds column col of y for rows 0..M-1
                // (with split K, the partial sums of its rank's K range)
                const int64_t col = static_cast<int64_t>(t) * swp::kTileN + wq * 32 + lane;
                bool store = true;
                if constexpr (KS > 1) {
                    const int owner = wq * KS / 4;              // the rank that owns this warp's 32 columns
                    const int lw = wq - owner * (4 / KS);       // the warp's index among the owner's
                    float* redbuf = reinterpret_cast<float*>(smem + NS * C::kStageBytes + 512);
                    auto slot = [&](int p) { return redbuf + ((p * (4 / KS) + lw) * 32 + lane) * (2 * MP); };
                    // float offset of value v (a multiple of 4) in a lane's slot: the
                    // 16-byte chunks rotated by lane, so that eight lanes' 16-byte
                    // accesses at the same offset fall in eight different bank groups
                    auto SW = [&](int v) { return ((v >> 2) ^ (lane & 7)) << 2; };
                    // a failed wait sets the abort flag and skips the rest of the tile;
                    // the promotion warps leave the loop together at the next
                    // chunk's barrier reduction
                    if (owner == rank && lane == 0)  // the other ranks' partial sums due this tile
                        mbar_arrive_expect_tx(&bars->rs_full[wq], (KS - 1) * 32 * 2 * MP * 4);
                    if (owner != rank) {
                        // the owner must have read this slot for the previous tile
                        if (tt > 0 && !warp_wait_acquire_cluster(&bars->rs_done[wq], static_cast<uint32_t>(tt - 1) & 1u,
                                                                 &bars->abort, kFaultSwpReduce)) {
                            store = false;
                        } else {
                            // asynchronous stores that count their bytes on the owner's
                            // barrier (no fence or arrival here)
                            const uint32_t dst = mapa_shared(slot(rank), static_cast<uint32_t>(owner));
                            const uint32_t rbar = mapa_shared(&bars->rs_full[wq], static_cast<uint32_t>(owner));
#pragma unroll
                            for (int i = 0; i < MP; i += 4) {
                                st_async_v4(dst + 4u * SW(i), Rh[i], Rh[i + 1], Rh[i + 2], Rh[i + 3], rbar);
                                st_async_v4(dst + 4u * SW(MP + i), Rl[i], Rl[i + 1], Rl[i + 2], Rl[i + 3], rbar);
                            }
                            store = false;
                        }
                    } else if (!warp_wait_acquire_cluster(&bars->rs_full[wq], static_cast<uint32_t>(tt) & 1u, &bars->abort,
                                                          kFaultSwpReduce)) {
                        store = false;
                    } else {
                        // rank order, ranks 0 .. KS-1: this rank's own sums go to its
                        // own slot, then one pass adds the KS slots starting from -0
                        // (-0 + v == v for every v, so the first addition is exact)
                        {
                            float* own = slot(rank);
#pragma unroll
                            for (int i = 0; i < MP; i += 4) {
                                st_shared_v4(own + SW(i), Rh[i], Rh[i + 1], Rh[i + 2], Rh[i + 3]);
                                st_shared_v4(own + SW(MP + i), Rl[i], Rl[i + 1], Rl[i + 2], Rl[i + 3]);
                            }
                        }
#pragma unroll
                        for (int i = 0; i < MP; ++i) {
                            Rh[i] = -0.0f;
                            Rl[i] = -0.0f;
                        }
#pragma unroll 1
                        for (int p = 0; p < KS; ++p) {
                            const float* src = slot(p);
#pragma unroll
                            for (int i = 0; i < MP; i += 4) {
                                const float4 a = *reinterpret_cast<const float4*>(src + SW(i));
                                const float4 c = *reinterpret_cast<const float4*>(src + SW(MP + i));
                                Rh[i] = __fadd_rn(Rh[i], a.x);
                                Rh[i + 1] = __fadd_rn(Rh[i + 1], a.y);
                                Rh[i + 2] = __fadd_rn(Rh[i + 2], a.z);
                                Rh[i + 3] = __fadd_rn(Rh[i + 3], a.w);
                                Rl[i] = __fadd_rn(Rl[i], c.x);
                                Rl[i + 1] = __fadd_rn(Rl[i + 1], c.y);
                                Rl[i + 2] = __fadd_rn(Rl[i + 2], c.z);
                                Rl[i + 3] = __fadd_rn(Rl[i + 3], c.w);
                            }
                        }
                        __syncwarp();
                        if (lane == 0) {
                            fence_release_smem_cta_cluster();  // the slots' reads, before the senders reuse them
                            for (int p = 0; p < KS; ++p)
                                if (p != rank)
                                    mbar_arrive_relaxed_cluster(mapa_shared(&bars->rs_done[wq], static_cast<uint32_t>(p)));
                        }
                    }
                    ++tt;
                }
                if (store && col < P.N) {
#pragma unroll
                    for (int m = 0; m < MP; ++m)
                        if (m < P.M)
                        {
                            const float v = __fadd_rn(Rh[m], __fmul_rn(Rl[m], 0x1p-10f));
                            P.y[m * static_cast<int64_t>(P.N) + col] = EPI ? epilogue_at(v, m, col, P) : v;
                        }
                }
#pragma unroll
                for (int i = 0; i < MP; ++i) {
                    Rh[i] = 0.0f;
                    Rl[i] = 0.0f;
                }
                sk = 0;
                t += ncl;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (KS > 1)
        cluster_sync();  // no CTA leaves while another may still write its buffer or arrive on its barriers
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, C::kTmemCols);
    }
}

template <int MP, int BPS, int NS, bool FX, bool EPI>
__global__ void __launch_bounds__(swp::kThreads, 1)
    comp_f16x2_swap_kernel(const __grid_constant__ CUtensorMap tmap_hi, const __grid_constant__ CUtensorMap tmap_lo,
                           const __grid_constant__ CUtensorMap tmap_w, const Problem P)
{
    swap_kernel_body<MP, BPS, NS, FX, EPI, 1>(tmap_hi, tmap_lo, tmap_w, P);
}

// The swapped-operand kernel with K split over a cluster of KS CTAs per tile.
template <int MP, int BPS, int NS, bool FX, bool EPI, int KS>
__global__ void __cluster_dims__(KS, 1, 1) __launch_bounds__(swp::kThreads, 1)
    comp_f16x2_swap_splitk_kernel(const __grid_constant__ CUtensorMap tmap_hi,
                                  const __grid_constant__ CUtensorMap tmap_lo,
                                  const __grid_constant__ CUtensorMap tmap_w, const Problem P)
{
    swap_kernel_body<MP, BPS, NS, FX, EPI, KS>(tmap_hi, tmap_lo, tmap_w, P);
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

// A 2-D row-major tensor (inner extent `inner` contiguous, `outer` rows) as a
// tensor map with box_inner x box_outer boxes and the 128-byte swizzle.
bool encode_2d(CUtensorMap* map, CUtensorMapDataType dtype, size_t elem, const void* base, int64_t inner,
               int64_t outer, uint32_t box_inner, uint32_t box_outer,
               CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn)
        return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(outer)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(inner) * elem};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, dtype, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int BN, bool kVec, bool EPI>
comp_status_t launch_bn_t(const CUtensorMap& tw, const CUtensorMap& tx, const Problem& P, const DeviceInfo& dev,
                          cudaStream_t stream)
{
    static std::mutex mu;
    static bool done[64] = {};
    {
        std::lock_guard<std::mutex> lock(mu);
        if (dev.device < 0 || dev.device >= 64)
            return COMP_ERR_CUDA;
        if (!done[dev.device]) {
            if (cudaFuncSetAttribute(comp_gemm_kernel<BN, kVec, EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(Cfg<BN>::kSmem)) != cudaSuccess) {
                (void)cudaGetLastError();
                return COMP_ERR_CUDA;
            }
            done[dev.device] = true;
        }
    }
    const int tiles = P.tiles_m * P.tiles_n;
    const int grid = tiles < dev.sm_count ? tiles : dev.sm_count;
    comp_gemm_kernel<BN, kVec, EPI><<<grid, kThreads, Cfg<BN>::kSmem, stream>>>(tw, tx, P);
    return launch_status();
}

// The instance with the epilogue compiled in only when the call has one.
template <int BN, bool kVec>
comp_status_t launch_bn(const CUtensorMap& tw, const CUtensorMap& tx, const Problem& P, const DeviceInfo& dev,
                        cudaStream_t stream)
{
    return (P.bias || P.gate) ? launch_bn_t<BN, kVec, true>(tw, tx, P, dev, stream)
                              : launch_bn_t<BN, kVec, false>(tw, tx, P, dev, stream);
}

// The N tile width expected to finish first: rounds of tiles over the SMs
// times the per-tile cost, modelled as BN plus a fixed 64 for the per-block
// split and promotion work; ties go to the wider tile.
int pick_bn(int64_t M, int64_t N, int sms)
{
    static const int cands[] = {160, 128};
    int best = 128;
    int64_t best_cost = INT64_MAX;
    for (int bn : cands) {
        const int64_t tiles = ((M + BM - 1) / BM) * ((N + bn - 1) / bn);
        const int64_t rounds = (tiles + sms - 1) / sms;
        const int64_t cost = rounds * (bn + 64);
        if (cost < best_cost) {
            best_cost = cost;
            best = bn;
        }
    }
    return best;
}

inline bool aligned16(const void* p)
{
    return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

template <bool kVec>
comp_status_t dispatch(int bn, const CUtensorMap& tw, const CUtensorMap& tx, const Problem& P, const DeviceInfo& dev,
                       cudaStream_t s)
{
    switch (bn) {
    case 160:
        return launch_bn<160, kVec>(tw, tx, P, dev, s);
    default:
        return launch_bn<128, kVec>(tw, tx, P, dev, s);
    }
}

}  // namespace

comp_status_t launch_gemm_tc(const float* x, const uint16_t* W, float* y, int64_t M, int64_t N, int64_t K,
                             int variant, const DeviceInfo& dev, cudaStream_t stream, const Epilogue& epi)
{
    const bool vec_ok = aligned16(x) && aligned16(W) && (K % 8 == 0);
    // at most 32 rows: the swapped-operand kernel with the split fused (variant
    // 3, or automatically once W spans at least 32 tiles of 128 rows)
    if (variant == 3 || (variant == 0 && swap_fused_preferred(x, W, M, N, K))) {
        if (!vec_ok || M > 32)
            return COMP_ERR_INVALID_VALUE;
        return launch_swap_fused(x, W, y, M, N, K, dev, stream, epi);
    }
    // more than 128 rows and about a wave of pair tiles: the fused kernel on
    // CTA pairs (variant 4, or automatically with TMA-legal operands)
    if (variant == 4 || (variant == 0 && fused_pair_preferred(x, W, M, N, K, dev))) {
        if (!vec_ok)
            return COMP_ERR_INVALID_VALUE;
        return launch_fused_pair(x, W, y, M, N, K, dev, stream, epi);
    }
    if (variant == 1 && !vec_ok)
        return COMP_ERR_INVALID_VALUE;
    bool use_vec = variant == 2 ? false : vec_ok;

    Problem P;
    P.x = x;
    P.W = W;
    P.y = y;
    P.M = static_cast<int>(M);
    P.N = static_cast<int>(N);
    P.K = static_cast<int>(K);
    P.nk = static_cast<int>((K + BK - 1) / BK);
    P.vec_y = (N % 4 == 0) && aligned16(y);
    P.tma_y = 0;
    P.bias = epi.bias;
    P.gate = epi.gate;
    const int bn = pick_bn(M, N, dev.sm_count);
    P.tiles_m = static_cast<int>((M + BM - 1) / BM);
    P.tiles_n = static_cast<int>((N + bn - 1) / bn);
    if (static_cast<int64_t>(P.tiles_m) * P.tiles_n > INT32_MAX / 2 ||
        static_cast<int64_t>(P.tiles_m) * P.tiles_n * P.nk > INT32_MAX / 2)
        return COMP_ERR_INVALID_VALUE;

    CUtensorMap tw{}, tx{};
    if (use_vec && !(encode_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, W, K, N, BK, static_cast<uint32_t>(bn)) &&
                     encode_2d(&tx, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, x, K, M, 32, BM))) {
        if (variant == 1)
            return COMP_ERR_CUDA;
        use_vec = false;  // the driver refused a descriptor: plain loads
    }
    return use_vec ? dispatch<true>(bn, tw, tx, P, dev, stream) : dispatch<false>(bn, tw, tx, P, dev, stream);
}

namespace {

// Launch with programmatic stream serialisation: the kernel's set-up overlaps
// the end of the previous kernel on the stream; its producer waits
// (griddepcontrol.wait) before it reads what that kernel wrote.
template <typename... KArgs, typename... Args>
comp_status_t launch_pdl(void (*kernel)(KArgs...), int grid, int threads, size_t smem, cudaStream_t stream,
                         Args&&... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(static_cast<unsigned>(threads), 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...) != cudaSuccess) {
        (void)cudaGetLastError();
        return COMP_ERR_LAUNCH;
    }
    return COMP_OK;
}

// Clusters of KS CTAs of the split-K instance that run at once on the device
// (the occupancy API's count: clusters must fit inside one GPC, so it can be
// below sm_count / KS); the first call per device also sets the kernel's
// shared-memory limit.  0 on a CUDA error.
template <int BN, int NS, int CH, int AR, int KS, bool EPI>
int x2_resident_clusters(const DeviceInfo& dev)
{
    using C = x2::Cfg<BN, NS, CH, AR, KS>;
    static std::mutex mu;
    static int clusters[64] = {};  // per device, 0 = not yet known
    std::lock_guard<std::mutex> lock(mu);
    if (dev.device < 0 || dev.device >= 64)
        return 0;
    if (clusters[dev.device] == 0) {
        if (cudaFuncSetAttribute(comp_f16x2_splitk_kernel<BN, NS, CH, AR, KS, EPI>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(C::kSmem)) != cudaSuccess) {
            (void)cudaGetLastError();
            return 0;
        }
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(dev.sm_count / KS * KS), 1, 1);
        cfg.blockDim = dim3(x2::kThreads, 1, 1);
        cfg.dynamicSmemBytes = C::kSmem;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, comp_f16x2_splitk_kernel<BN, NS, CH, AR, KS, EPI>, &cfg) != cudaSuccess ||
            n <= 0) {
            (void)cudaGetLastError();
            n = dev.sm_count / KS;
        }
        clusters[dev.device] = n;
    }
    return clusters[dev.device];
}

template <int BN, int NS, int CH, int AR, int KS, bool EPI>
comp_status_t launch_x2_splitk_t(const CUtensorMap& th, const CUtensorMap& tl, const CUtensorMap& tw, const Problem& P,
                                 const DeviceInfo& dev, cudaStream_t stream)
{
    using C = x2::Cfg<BN, NS, CH, AR, KS>;
    const int nc = x2_resident_clusters<BN, NS, CH, AR, KS, EPI>(dev);
    if (nc <= 0)
        return COMP_ERR_CUDA;
    const int tiles = P.tiles_m * P.tiles_n;
    const int grid = KS * (tiles < nc ? tiles : nc);
    return launch_pdl(comp_f16x2_splitk_kernel<BN, NS, CH, AR, KS, EPI>, grid, x2::kThreads, C::kSmem, stream, th, tl, tw,
                      P);
}

template <int BN, int NS, int CH, int AR, int KS>
comp_status_t launch_x2_splitk(const CUtensorMap& th, const CUtensorMap& tl, const CUtensorMap& tw, const Problem& P,
                               const DeviceInfo& dev, cudaStream_t stream)
{
    return (P.bias || P.gate) ? launch_x2_splitk_t<BN, NS, CH, AR, KS, true>(th, tl, tw, P, dev, stream)
                              : launch_x2_splitk_t<BN, NS, CH, AR, KS, false>(th, tl, tw, P, dev, stream);
}

template <int MP, int BPS, int NS, bool FX, bool EPI, int KS>
auto swap_kernel_of()
{
    void (*kern)(CUtensorMap, CUtensorMap, CUtensorMap, Problem);
    if constexpr (KS == 1)
        kern = comp_f16x2_swap_kernel<MP, BPS, NS, FX, EPI>;
    else
        kern = comp_f16x2_swap_splitk_kernel<MP, BPS, NS, FX, EPI, KS>;
    return kern;
}

// Units of the swapped kernel instance that run at once on the device: CTAs
// for KS = 1 (one per SM), else clusters of KS CTAs as the occupancy API
// counts them.  Clusters must fit inside one GPC, so fewer than sm_count / KS
// may be resident (36 clusters of 4 on a 152-SM GB300, not 38); a grid sized
// past that runs its last clusters as a second wave.  The first call per
// device also sets the kernel's shared-memory limit.  0 on a CUDA error.
template <int MP, int BPS, int NS, bool FX, bool EPI, int KS>
int swap_resident_units(const DeviceInfo& dev)
{
    using C = swp::Cfg<MP, BPS, NS, FX, KS>;
    static std::mutex mu;
    static int units[64] = {};  // per device, 0 = not yet known
    std::lock_guard<std::mutex> lock(mu);
    if (dev.device < 0 || dev.device >= 64)
        return 0;
    if (units[dev.device] == 0) {
        const auto kern = swap_kernel_of<MP, BPS, NS, FX, EPI, KS>();
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(C::kSmem)) !=
            cudaSuccess) {
            (void)cudaGetLastError();
            return 0;
        }
        int n = dev.sm_count / KS;
        if (KS > 1) {
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(static_cast<unsigned>(dev.sm_count / KS * KS), 1, 1);
            cfg.blockDim = dim3(swp::kThreads, 1, 1);
            cfg.dynamicSmemBytes = C::kSmem;
            int q = 0;
            if (cudaOccupancyMaxActiveClusters(&q, kern, &cfg) == cudaSuccess && q > 0)
                n = q < n ? q : n;
            else
                (void)cudaGetLastError();
        }
        units[dev.device] = n;
    }
    return units[dev.device];
}

template <int MP, int BPS, int NS, bool FX, bool EPI, int KS>
comp_status_t launch_swap_t(const CUtensorMap& th, const CUtensorMap& tl, const CUtensorMap& tw, const Problem& P,
                          const DeviceInfo& dev, cudaStream_t stream)
{
    using C = swp::Cfg<MP, BPS, NS, FX, KS>;
    const int units = swap_resident_units<MP, BPS, NS, FX, EPI, KS>(dev);
    if (units <= 0)
        return COMP_ERR_CUDA;
    const int grid = KS * (P.tiles_n < units ? P.tiles_n : units);
    return launch_pdl(swap_kernel_of<MP, BPS, NS, FX, EPI, KS>(), grid, swp::kThreads, C::kSmem, stream, th, tl, tw, P);
}

// K split of the swapped kernel: clusters of 4 CTAs per tile when every tile
// gets a resident cluster of 4 at once and K has at least 16 blocks (4 or more
// per rank), of 2 likewise with at least 8 blocks, else none.  With few tiles
// of W this puts several CTAs on each tile's stream of W.  Several rounds of
// split tiles do not pay: with 144 CTAs in clusters of 4 each CTA's stream of
// W slowed to about half the rate of one CTA per tile.
int swap_split_ks(int tiles, int nk, int clusters2, int clusters4)
{
    if (tiles <= clusters4 && nk >= 16)
        return 4;
    if (tiles <= clusters2 && nk >= 8)
        return 2;
    return 1;
}

template <int MP, int BPS, int NS, bool FX>
int swap_split_ks_for(const Problem& P, const DeviceInfo& dev, bool epi)
{
    const int c2 = epi ? swap_resident_units<MP, BPS, NS, FX, true, 2>(dev)
                       : swap_resident_units<MP, BPS, NS, FX, false, 2>(dev);
    const int c4 = epi ? swap_resident_units<MP, BPS, NS, FX, true, 4>(dev)
                       : swap_resident_units<MP, BPS, NS, FX, false, 4>(dev);
    return swap_split_ks(P.tiles_n, P.nk, c2, c4);
}

template <int MP, int BPS, int NS, bool FX = false>
comp_status_t launch_swap(const CUtensorMap& th, const CUtensorMap& tl, const CUtensorMap& tw, const Problem& P,
                          const DeviceInfo& dev, cudaStream_t stream)
{
    const bool epi = P.bias || P.gate;
    switch (swap_split_ks_for<MP, BPS, NS, FX>(P, dev, epi)) {
    case 4:
        return epi ? launch_swap_t<MP, BPS, NS, FX, true, 4>(th, tl, tw, P, dev, stream)
                   : launch_swap_t<MP, BPS, NS, FX, false, 4>(th, tl, tw, P, dev, stream);
    case 2:
        return epi ? launch_swap_t<MP, BPS, NS, FX, true, 2>(th, tl, tw, P, dev, stream)
                   : launch_swap_t<MP, BPS, NS, FX, false, 2>(th, tl, tw, P, dev, stream);
    default:
        return epi ? launch_swap_t<MP, BPS, NS, FX, true, 1>(th, tl, tw, P, dev, stream)
                   : launch_swap_t<MP, BPS, NS, FX, false, 1>(th, tl, tw, P, dev, stream);
    }
}

template <int BN, int NS, int CH, int AR, bool EPI>
comp_status_t launch_x2_bn_t(const CUtensorMap& th, const CUtensorMap& tl, const CUtensorMap& tw, const Problem& P,
                             const DeviceInfo& dev, cudaStream_t stream)
{
    using C = x2::Cfg<BN, NS, CH, AR>;
    static std::mutex mu;
    static bool done[64] = {};
    {
        std::lock_guard<std::mutex> lock(mu);
        if (dev.device < 0 || dev.device >= 64)
            return COMP_ERR_CUDA;
        if (!done[dev.device]) {
            if (cudaFuncSetAttribute(comp_f16x2_kernel<BN, NS, CH, AR, EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(C::kSmem)) != cudaSuccess) {
                (void)cudaGetLastError();
                return COMP_ERR_CUDA;
            }
            done[dev.device] = true;
        }
    }
    const int tiles = P.tiles_m * P.tiles_n;
    const int grid = tiles < dev.sm_count ? tiles : dev.sm_count;
    return launch_pdl(comp_f16x2_kernel<BN, NS, CH, AR, EPI>, grid, x2::kThreads, C::kSmem, stream, th, tl, tw, P);
}

template <int BN, int NS, int CH, int AR = BM>
comp_status_t launch_x2_bn(const CUtensorMap& th, const CUtensorMap& tl, const CUtensorMap& tw, const Problem& P,
                           const DeviceInfo& dev, cudaStream_t stream)
{
    return (P.bias || P.gate) ? launch_x2_bn_t<BN, NS, CH, AR, true>(th, tl, tw, P, dev, stream)
                              : launch_x2_bn_t<BN, NS, CH, AR, false>(th, tl, tw, P, dev, stream);
}

template <int BN, int NS, int CH, bool EPI>
comp_status_t launch_pair_bn_t(const CUtensorMap& th, const CUtensorMap& tl, const CUtensorMap& tw, const CUtensorMap& ty,
                             const Problem& P, const DeviceInfo& dev, cudaStream_t stream)
{
    using C = pair::Cfg<BN, NS, CH>;
    static std::mutex mu;
    static int pairs[64] = {};  // co-resident CTA pairs per device, 0 = not yet known
    int np;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (dev.device < 0 || dev.device >= 64)
            return COMP_ERR_CUDA;
        if (pairs[dev.device] == 0) {
            if (cudaFuncSetAttribute(comp_f16x2_pair_kernel<BN, NS, CH, EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(C::kSmem)) != cudaSuccess) {
                (void)cudaGetLastError();
                return COMP_ERR_CUDA;
            }
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(static_cast<unsigned>(dev.sm_count & ~1), 1, 1);
            cfg.blockDim = dim3(pair::kThreads, 1, 1);
            cfg.dynamicSmemBytes = C::kSmem;
            int clusters = 0;
            if (cudaOccupancyMaxActiveClusters(&clusters, comp_f16x2_pair_kernel<BN, NS, CH, EPI>, &cfg) != cudaSuccess ||
                clusters <= 0) {
                (void)cudaGetLastError();
                clusters = dev.sm_count / 2;
            }
            pairs[dev.device] = clusters;
        }
        np = pairs[dev.device];
    }
    const int tiles = P.tiles_m * P.tiles_n;
    const int grid = 2 * (tiles < np ? tiles : np);
    return launch_pdl(comp_f16x2_pair_kernel<BN, NS, CH, EPI>, grid, pair::kThreads, C::kSmem, stream, th, tl, tw, ty, P);
}

template <int BN, int NS, int CH>
comp_status_t launch_pair_bn(const CUtensorMap& th, const CUtensorMap& tl, const CUtensorMap& tw, const CUtensorMap& ty,
                             const Problem& P, const DeviceInfo& dev, cudaStream_t stream)
{
    return (P.bias || P.gate) ? launch_pair_bn_t<BN, NS, CH, true>(th, tl, tw, ty, P, dev, stream)
                              : launch_pair_bn_t<BN, NS, CH, false>(th, tl, tw, ty, P, dev, stream);
}

template <int BN, int NS, int CH, bool EPI>
comp_status_t launch_fpair_bn_t(const CUtensorMap& tx, const CUtensorMap& tw, const CUtensorMap& ty, const Problem& P,
                                const DeviceInfo& dev, cudaStream_t stream)
{
    using C = pair::Cfg<BN, NS, CH>;
    static std::mutex mu;
    static int pairs[64] = {};  // co-resident CTA pairs per device, 0 = not yet known
    int np;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (dev.device < 0 || dev.device >= 64)
            return COMP_ERR_CUDA;
        if (pairs[dev.device] == 0) {
            if (cudaFuncSetAttribute(comp_f32x16_pair_kernel<BN, NS, CH, EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(C::kSmem)) != cudaSuccess) {
                (void)cudaGetLastError();
                return COMP_ERR_CUDA;
            }
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(static_cast<unsigned>(dev.sm_count & ~1), 1, 1);
            cfg.blockDim = dim3(fpair::kThreads, 1, 1);
            cfg.dynamicSmemBytes = C::kSmem;
            int clusters = 0;
            if (cudaOccupancyMaxActiveClusters(&clusters, comp_f32x16_pair_kernel<BN, NS, CH, EPI>, &cfg) !=
                    cudaSuccess ||
                clusters <= 0) {
                (void)cudaGetLastError();
                clusters = dev.sm_count / 2;
            }
            pairs[dev.device] = clusters;
        }
        np = pairs[dev.device];
    }
    const int tiles = P.tiles_m * P.tiles_n;
    const int grid = 2 * (tiles < np ? tiles : np);
    return launch_pdl(comp_f32x16_pair_kernel<BN, NS, CH, EPI>, grid, fpair::kThreads, C::kSmem, stream, tx, tw, ty, P);
}

template <int BN, int NS, int CH>
comp_status_t launch_fpair_bn(const CUtensorMap& tx, const CUtensorMap& tw, const CUtensorMap& ty, const Problem& P,
                              const DeviceInfo& dev, cudaStream_t stream)
{
    return (P.bias || P.gate) ? launch_fpair_bn_t<BN, NS, CH, true>(tx, tw, ty, P, dev, stream)
                              : launch_fpair_bn_t<BN, NS, CH, false>(tx, tw, ty, P, dev, stream);
}

// N tile width for the two-pass product (tiles are all tensor work there).
int pick_bn_x2(int64_t M, int64_t N, int sms)
{
    static const int cands[] = {192, 128, 96};
    if (M <= BM) {
        // one row of tiles: the product streams W, so the tile width that keeps
        // the most SMs busy per round wins (ties: the wider tile)
        int best = 192;
        double best_busy = -1.0;
        for (int bn : cands) {
            const int64_t tiles = (N + bn - 1) / bn;
            const int64_t rounds = (tiles + sms - 1) / sms;
            const double busy = static_cast<double>(tiles) / static_cast<double>(rounds);
            if (busy > best_busy + 0.5) {
                best_busy = busy;
                best = bn;
            }
        }
        return best;
    }
    int best = 128;
    int64_t best_cost = INT64_MAX;
    for (int bn : {192, 128}) {  // narrower MMAs would be issue-bound
        const int64_t tiles = ((M + BM - 1) / BM) * ((N + bn - 1) / bn);
        const int64_t cost = ((tiles + sms - 1) / sms) * (bn + 32);
        if (cost < best_cost) {
            best_cost = cost;
            best = bn;
        }
    }
    return best;
}

// Pair-tile width for the CTA-pair product: fewest rounds of pair tiles over
// the co-resident pairs, weighted by the tile width.
int pick_bn_pair(int64_t M, int64_t N, int pairs)
{
    static const int cands[] = {224, 256};
    int best = 256;
    int64_t best_cost = INT64_MAX;
    for (int bn : cands) {
        const int64_t tiles = ((M + pair::kRows - 1) / pair::kRows) * ((N + bn - 1) / bn);
        const int64_t cost = ((tiles + pairs - 1) / pairs) * (bn + 32);
        if (cost < best_cost) {
            best_cost = cost;
            best = bn;
        }
    }
    return best;
}

}  // namespace

bool gemm_f16x2_supported(const void* hi, const void* lo, const void* W, int64_t K)
{
    return aligned16(hi) && aligned16(lo) && aligned16(W) && (K % 8 == 0);
}

comp_status_t launch_gemm_f16x2(const uint16_t* hi, const uint16_t* lo, const uint16_t* W, float* y, int64_t M,
                                int64_t N, int64_t K, int variant, const DeviceInfo& dev, cudaStream_t stream,
                                const Epilogue& epi, bool stall)
{
    if (!gemm_f16x2_supported(hi, lo, W, K) || variant < 0 || variant > 4 || (variant == 3 && M > 32))
        return COMP_ERR_INVALID_VALUE;
    // CTA pairs once the output fills about one wave of single-CTA tiles: below
    // that, pipeline fill dominates and the 128-row tiles spread over more SMs.
    const bool pairs = variant == 2 || (variant == 0 && M > BM && M * N >= static_cast<int64_t>(dev.sm_count) * BM * 192);
    Problem P;
    P.x = nullptr;
    P.W = W;
    P.y = y;
    P.M = static_cast<int>(M);
    P.N = static_cast<int>(N);
    P.K = static_cast<int>(K);
    P.nk = static_cast<int>((K + BK - 1) / BK);
    P.vec_y = (N % 4 == 0) && aligned16(y);
    P.tma_y = 0;
    P.bias = epi.bias;
    P.gate = epi.gate;
    P.stall = stall ? 1 : 0;
    CUtensorMap th{}, tl{}, tw{};
    // at most 32 rows: operands swapped, W streams through full 128-row MMAs,
    // with K split over a cluster of 2 or 4 CTAs per tile when W has few tiles
    // (each CTA streams about 40-50 GB/s of W)
    const int64_t t128 = (N + swp::kTileN - 1) / swp::kTileN;
    if (variant == 3 || (variant == 0 && M <= 32)) {
        const uint32_t mp = M <= 16 ? 16u : 32u;
        P.tiles_m = 1;
        P.tiles_n = static_cast<int>(t128);
        if (static_cast<int64_t>(P.tiles_n) * P.nk > INT32_MAX / 2)
            return COMP_ERR_INVALID_VALUE;
        if (!encode_2d(&th, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, hi, K, M, BK, mp) ||
            !encode_2d(&tl, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, lo, K, M, BK, mp) ||
            !encode_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, W, K, N, BK, static_cast<uint32_t>(swp::kTileN)))
            return COMP_ERR_CUDA;
        // two K blocks per stage: with 2 or 3 per stage W streams at 4.1 TB/s
        // on GB300 at 16 x 14336 x 4096 (one per stage: 3.0-3.8).  The fused
        // kernel has the same stages (fewer of them, for its FP32 staging),
        // hence the same chunks: both forms give identical bits.
        return mp == 16 ? launch_swap<16, 2, 5>(th, tl, tw, P, dev, stream)
                        : launch_swap<32, 2, 4>(th, tl, tw, P, dev, stream);
    }
    if (variant == 4) {
        // measurement option: one tensor-core chain per product over all of K,
        // one CTA per 128 x 128 tile
        P.tiles_m = static_cast<int>((M + BM - 1) / BM);
        P.tiles_n = static_cast<int>((N + 127) / 128);
        if (static_cast<int64_t>(P.tiles_m) * P.tiles_n * P.nk > INT32_MAX / 2)
            return COMP_ERR_INVALID_VALUE;
        if (!encode_2d(&th, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, hi, K, M, BK, BM) ||
            !encode_2d(&tl, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, lo, K, M, BK, BM) ||
            !encode_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, W, K, N, BK, 128))
            return COMP_ERR_CUDA;
        return launch_x2_bn<128, 4, 0>(th, tl, tw, P, dev, stream);
    }
    if (pairs) {
        // CTA pairs on 256-row tiles
        const int bn = pick_bn_pair(M, N, dev.sm_count / 2);
        P.tiles_m = static_cast<int>((M + pair::kRows - 1) / pair::kRows);
        P.tiles_n = static_cast<int>((N + bn - 1) / bn);
        if (static_cast<int64_t>(P.tiles_m) * P.tiles_n * P.nk > INT32_MAX / 2)
            return COMP_ERR_INVALID_VALUE;
        CUtensorMap ty{};
        if (!encode_2d(&th, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, hi, K, M, BK, BM) ||
            !encode_2d(&tl, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, lo, K, M, BK, BM) ||
            !encode_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, W, K, N, BK, static_cast<uint32_t>(bn / 2)))
            return COMP_ERR_CUDA;
        if (P.vec_y)
            P.tma_y = encode_2d(&ty, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, y, N, M, 16, 32, CU_TENSOR_MAP_SWIZZLE_64B)
                          ? 1
                          : 0;
        return bn == 224 ? launch_pair_bn<224, 4, 2>(th, tl, tw, ty, P, dev, stream)
                         : launch_pair_bn<256, 4, 2>(th, tl, tw, ty, P, dev, stream);
    }
    // few tiles: split K over clusters of 2 or 4 CTAs (at most 32 rows:
    // 192-wide tiles reduced in the leader; otherwise 128 x 128 tiles, or
    // 128 x 64 tiles with a short K, reduced across the cluster), when every
    // tile gets a resident cluster at once
    int ks = 1;
    bool narrow = false;  // 128 x 64 tiles
    if (M <= 32) {
        const int64_t t192 = (N + 191) / 192;
        if (t192 <= x2_resident_clusters<192, 6, 2, 32, 4, false>(dev) && P.nk >= 16)
            ks = 4;
        else if (t192 <= x2_resident_clusters<192, 6, 2, 32, 2, false>(dev) && P.nk >= 8)
            ks = 2;
    } else {
        const int64_t t128 = ((M + BM - 1) / BM) * ((N + 127) / 128);
        const int64_t t64 = ((M + BM - 1) / BM) * ((N + 63) / 64);
        if (t128 * 2 <= dev.sm_count && P.nk <= 32) {
            // few tiles and K at most 2048: twice as many 64-wide tiles, with K
            // split over pairs if they fit one wave, else unsplit.  Each rank
            // then has half the partial sums to send, or none (GB300, product
            // from the planes, cold / back to back: 512 x 1024 x 1024 16.4 /
            // 12.3 us against 18.4 / 13.8 for 128-wide tiles split over 4;
            // 1000 x 776 x 1032 unsplit 20.5 / 15.1 against 22.5 / 17.3 split
            // over 2).  With a longer K the narrow MMAs lose (512 x 512 x 4096:
            // 30.7 against 28.7 us).
            if (t64 <= x2_resident_clusters<64, 4, 2, BM, 2, false>(dev) && P.nk >= 8) {
                ks = 2;
                narrow = true;
            } else if (t64 <= dev.sm_count) {
                narrow = true;
            }
        }
        if (!narrow) {
            if (t128 <= x2_resident_clusters<128, 3, 2, BM, 4, false>(dev) && P.nk >= 16)
                ks = 4;
            else if (t128 <= x2_resident_clusters<128, 3, 2, BM, 2, false>(dev) && P.nk >= 8)
                ks = 2;
        }
    }
    const int bn = narrow ? 64 : ks > 1 ? (M <= 32 ? 192 : 128) : pick_bn_x2(M, N, dev.sm_count);
    P.tiles_m = static_cast<int>((M + BM - 1) / BM);
    P.tiles_n = static_cast<int>((N + bn - 1) / bn);
    if (static_cast<int64_t>(P.tiles_m) * P.tiles_n * P.nk > INT32_MAX / 2)
        return COMP_ERR_INVALID_VALUE;
    // at most 32 rows (decode-like shapes): 32-row boxes, 7 to 10 stages in flight
    const uint32_t box_rows = M <= 32 ? 32u : static_cast<uint32_t>(BM);
    if (!encode_2d(&th, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, hi, K, M, BK, box_rows) ||
        !encode_2d(&tl, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, lo, K, M, BK, box_rows) ||
        !encode_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, W, K, N, BK, static_cast<uint32_t>(bn)))
        return COMP_ERR_CUDA;
    if (narrow)
        return ks == 2 ? launch_x2_splitk<64, 4, 2, BM, 2>(th, tl, tw, P, dev, stream)
                       : launch_x2_bn<64, 4, 2>(th, tl, tw, P, dev, stream);
    if (ks == 4)
        return M <= 32 ? launch_x2_splitk<192, 6, 2, 32, 4>(th, tl, tw, P, dev, stream)
                       : launch_x2_splitk<128, 3, 2, BM, 4>(th, tl, tw, P, dev, stream);
    if (ks == 2)
        return M <= 32 ? launch_x2_splitk<192, 6, 2, 32, 2>(th, tl, tw, P, dev, stream)
                       : launch_x2_splitk<128, 3, 2, BM, 2>(th, tl, tw, P, dev, stream);
    if (M <= 32) {
        if (bn == 192)
            return launch_x2_bn<192, 7, 2, 32>(th, tl, tw, P, dev, stream);
        if (bn == 128)
            return launch_x2_bn<128, 9, 2, 32>(th, tl, tw, P, dev, stream);
        return launch_x2_bn<96, 10, 2, 32>(th, tl, tw, P, dev, stream);
    }
    if (bn == 192)
        return launch_x2_bn<192, 4, 2>(th, tl, tw, P, dev, stream);
    if (bn == 128)
        return launch_x2_bn<128, 4, 2>(th, tl, tw, P, dev, stream);
    return launch_x2_bn<96, 4, 2>(th, tl, tw, P, dev, stream);
}

bool swap_two_pass_better(int64_t M, int64_t N, int64_t K, const DeviceInfo& dev)
{
    // given a workspace: with 17 to 32 rows and no split of K the one-launch
    // kernel holds three 64 KB stages (x in FP32 beside W) against the
    // two-pass swapped product's four (32 x 4096 x 4096 without the split:
    // 36.9 us one launch, 26.6 us product + 6.1 us split, cold).  A short K
    // stays on the one-launch kernel.
    const int tiles = static_cast<int>((N + swp::kTileN - 1) / swp::kTileN);
    const int nk = static_cast<int>((K + BK - 1) / BK);
    if (M <= 16 || nk <= 8)
        return false;
    // the fused kernel for 17 to 32 rows (launch_swap_fused's instance)
    Problem P;
    P.tiles_n = tiles;
    P.nk = nk;
    return swap_split_ks_for<32, 2, 3, true>(P, dev, false) == 1;
}

bool swap_fused_preferred(const float* x, const uint16_t* W, int64_t M, int64_t N, int64_t K)
{
    // at most 32 rows: the swapped kernel with the split fused, K split over a
    // cluster when W has few tiles (W streams through 128-row MMAs; one launch)
    (void)N;
    return M <= 32 && K % 8 == 0 && aligned16(x) && aligned16(W);
}

comp_status_t launch_swap_fused(const float* x, const uint16_t* W, float* y, int64_t M, int64_t N, int64_t K,
                                const DeviceInfo& dev, cudaStream_t stream, const Epilogue& epi)
{
    if (M > 32 || K % 8 != 0 || !aligned16(x) || !aligned16(W))
        return COMP_ERR_INVALID_VALUE;
    Problem P;
    P.x = x;
    P.W = W;
    P.y = y;
    P.M = static_cast<int>(M);
    P.N = static_cast<int>(N);
    P.K = static_cast<int>(K);
    P.nk = static_cast<int>((K + BK - 1) / BK);
    P.vec_y = (N % 4 == 0) && aligned16(y);
    P.tma_y = 0;
    P.bias = epi.bias;
    P.gate = epi.gate;
    P.tiles_m = 1;
    P.tiles_n = static_cast<int>((N + swp::kTileN - 1) / swp::kTileN);
    if (static_cast<int64_t>(P.tiles_n) * P.nk > INT32_MAX / 2)
        return COMP_ERR_INVALID_VALUE;
    const uint32_t mp = M <= 16 ? 16u : 32u;
    CUtensorMap tx{}, tw{}, none{};  // FP32 x in the first map's place; the second is not read
    if (!encode_2d(&tx, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, x, K, M, BK, mp, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !encode_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, W, K, N, BK, static_cast<uint32_t>(swp::kTileN)))
        return COMP_ERR_CUDA;
    // two K blocks per stage as in the two-pass kernel; the FP32 staging makes
    // a stage larger: 4 x 48 KB (Mp 16), 3 x 64 KB (Mp 32)
    return mp == 16 ? launch_swap<16, 2, 4, true>(tx, none, tw, P, dev, stream)
                    : launch_swap<32, 2, 3, true>(tx, none, tw, P, dev, stream);
}

bool fused_pair_preferred(const float* x, const uint16_t* W, int64_t M, int64_t N, int64_t K, const DeviceInfo& dev)
{
    // CTA pairs once the output fills about one wave of 128 x 192 tiles (the
    // two-pass product's rule), TMA-legal operands
    return M > BM && M * N >= static_cast<int64_t>(dev.sm_count) * BM * 192 && K % 8 == 0 && aligned16(x) &&
           aligned16(W);
}

comp_status_t launch_fused_pair(const float* x, const uint16_t* W, float* y, int64_t M, int64_t N, int64_t K,
                                const DeviceInfo& dev, cudaStream_t stream, const Epilogue& epi)
{
    if (K % 8 != 0 || !aligned16(x) || !aligned16(W))
        return COMP_ERR_INVALID_VALUE;
    Problem P;
    P.x = x;
    P.W = W;
    P.y = y;
    P.M = static_cast<int>(M);
    P.N = static_cast<int>(N);
    P.K = static_cast<int>(K);
    P.nk = static_cast<int>((K + BK - 1) / BK);
    P.vec_y = (N % 4 == 0) && aligned16(y);
    P.tma_y = 0;
    P.bias = epi.bias;
    P.gate = epi.gate;
    // the pair product's tile width, so that both forms give identical bits
    const int bn = pick_bn_pair(M, N, dev.sm_count / 2);
    P.tiles_m = static_cast<int>((M + pair::kRows - 1) / pair::kRows);
    P.tiles_n = static_cast<int>((N + bn - 1) / bn);
    if (static_cast<int64_t>(P.tiles_m) * P.tiles_n * P.nk > INT32_MAX / 2)
        return COMP_ERR_INVALID_VALUE;
    CUtensorMap tx{}, tw{}, ty{};
    // FP32 x as two 128 x 32 boxes per K block (128 bytes of a row each)
    if (!encode_2d(&tx, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, x, K, M, 32, BM) ||
        !encode_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, W, K, N, BK, static_cast<uint32_t>(bn / 2)))
        return COMP_ERR_CUDA;
    if (P.vec_y)
        P.tma_y = encode_2d(&ty, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, y, N, M, 16, 32, CU_TENSOR_MAP_SWIZZLE_64B) ? 1 : 0;
    return bn == 224 ? launch_fpair_bn<224, 4, 2>(tx, tw, ty, P, dev, stream)
                     : launch_fpair_bn<256, 4, 2>(tx, tw, ty, P, dev, stream);
}

namespace {

// One thread waits, through the same bounded wait as the pipelines, on a
// barrier that nothing completes; the wait gives up and records the code.
__global__ void check_wait_timeout_kernel()
{
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_flag = 0;
        fence_mbar_init();
        (void)wait_bounded(&bar, 0, &abort_flag, COMP_FAULT_CHECK_TIMEOUT);
    }
}

}  // namespace

comp_status_t launch_check_wait_timeout(cudaStream_t stream)
{
    check_wait_timeout_kernel<<<1, 32, 0, stream>>>();
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

