/*
 * compfp32.h — C ABI of the GB300 (sm_103a) compensated-FP32 projection library.
 *
 * The method is the "compensated FP32" projection of laya.cpp's Vulkan backend
 * page (docs/vulkan.md):
 *   - compensated-FP32 paragraph: every FP32 activation x becomes two FP16
 *     values, both multiplied by the exactly stored FP16 weights with FP32
 *     accumulators, and the two results are combined in FP32;
 *   - split/merge paragraph: the split rounds to nearest with ties to even,
 *     keeps subnormal results, and multiplies the residual by 1024; each split
 *     and each merge is one dispatch;
 *   - true-FP32 kernels paragraph: an optional build with plain FP32 matrix
 *     kernels that never convert the FP32 operand to FP16;
 *   - fused-build paragraph: split and merge folded into the projection.
 * In formulas, with fp16_rne the IEEE 754 binary32 -> binary16 conversion
 * (round to nearest, ties to even, gradual underflow, overflow to infinity):
 *     hi = fp16_rne(x)                 lo = fp16_rne((x - hi) * 1024)
 *     acc_hi = sum_k hi[m,k] * W[n,k]  acc_lo = sum_k lo[m,k] * W[n,k]   (FP32)
 *     y = acc_hi + acc_lo * 2^-10      (binary32 multiply, then binary32 add)
 *
 * Conventions shared by every call
 *   - Binary16 values travel as uint16_t bit patterns, so this header needs no
 *     CUDA half-precision header.
 *   - Every pointer is DEVICE memory owned by the caller (for example a PyTorch
 *     tensor's data pointer) on the current CUDA device.  The library keeps no
 *     pointer after a call returns and allocates no device memory; the one
 *     device reservation it has is the static 64 MiB workspace of
 *     comp_gemm_f32x16_noalloc (see there).
 *   - Matrices are dense and row-major: x is [M, K] (K contiguous), W is [N, K]
 *     (K contiguous), y is [M, N] (N contiguous).  Any element-aligned address
 *     and any size are accepted; addresses or sizes that the fast paths cannot
 *     use (for example K not a multiple of 8) take a slower path and still
 *     return COMP_OK.
 *   - `stream` is a cudaStream_t (CUstream) of the current device; NULL is the
 *     legacy default stream.  Every call only enqueues work on `stream` and never
 *     synchronises; errors found while the kernels run are reported later (see
 *     comp_device_status).
 *   - Argument errors are detected before anything is enqueued and return
 *     COMP_ERR_INVALID_VALUE.  A device that is not compute capability 10.3
 *     returns COMP_ERR_UNSUPPORTED_DEVICE.  There is no CPU fallback (as on the
 *     laya.cpp page's backend-selection paragraph, where a missing backend is
 *     an error and nothing falls back to the CPU).
 *   - Sizes of zero are valid no-ops, except that a GEMM with K == 0 and
 *     M*N > 0 writes y = +0.
 */
#ifndef COMPFP32_H
#define COMPFP32_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Status codes.  The numeric values are part of the ABI and never change.
 * COMP_ERR_MISALIGNED is reserved: every call accepts any element-aligned
 * address and any size (a misaligned or ragged case takes a slower path and
 * still returns COMP_OK), so no call returns it today.
 */
typedef enum comp_status {
    COMP_OK = 0,
    COMP_ERR_INVALID_VALUE = 1,      /* bad pointer, size or aliasing; nothing was enqueued */
    COMP_ERR_MISALIGNED = 2,         /* reserved; never returned */
    COMP_ERR_UNSUPPORTED_DEVICE = 3, /* current device is not sm_103 (GB300), or no device */
    COMP_ERR_LAUNCH = 4,             /* the kernel launch itself failed */
    COMP_ERR_TIMEOUT = 5,            /* a kernel gave up a bounded wait (see comp_device_status) */
    COMP_ERR_CUDA = 6                /* another CUDA runtime call failed */
} comp_status_t;

/* An opaque cudaStream_t. */
typedef void* comp_stream_t;

/*
 * comp_split_f32 — the split (laya.cpp docs/vulkan.md, split/merge paragraph).
 *   x  : n binary32 values (input).
 *   hi : n binary16 values, hi[i] = fp16_rne(x[i]) (output).
 *   lo : n binary16 values, lo[i] = fp16_rne((x[i] - hi[i]) * 1024) (output).
 * The two outputs are separate planes with the same indexing as x.  For every
 * finite |x| < 65520, x - hi and its scaling are exact in binary32 and
 * |lo| <= 16384.  |x| >= 65520 gives hi = +-inf and lo = -+inf; NaN gives NaN
 * in both.  No value is flushed to zero.
 * Errors: COMP_ERR_INVALID_VALUE if n < 0, a pointer is NULL while n > 0, or an
 * output overlaps x or the other output.
 */
comp_status_t comp_split_f32(const float* x, uint16_t* hi, uint16_t* lo, int64_t n, comp_stream_t stream);

/*
 * comp_merge_f32 — the merge (laya.cpp docs/vulkan.md, compensated-FP32
 * paragraph, "combines them in FP32").
 *   acc_hi, acc_lo : n binary32 accumulators (input).
 *   y              : n binary32 values, y[i] = rn(acc_hi[i] + rn(acc_lo[i] * 2^-10))
 *                    (output; two rounded operations, never a fused multiply-add).
 * y may be exactly acc_hi or exactly acc_lo (in place); any other overlap is
 * COMP_ERR_INVALID_VALUE, as are n < 0 and a NULL pointer with n > 0.
 */
comp_status_t comp_merge_f32(const float* acc_hi, const float* acc_lo, float* y, int64_t n, comp_stream_t stream);

/*
 * comp_geglu_f32 — the GEGLU step of the FP32 feed-forward layers as one
 * dispatch (laya.cpp docs/vulkan.md, feed-forward paragraph: a fused GEGLU
 * shader, with no separate gate copy, activation or multiplication
 * dispatches):
 *   out[i] = gelu(gate[i]) * up[i],  gelu(g) = g * Phi(g),
 *   Phi(g) = erfc(-g / sqrt 2) / 2  (the exact GELU; CUDA's erfcf),
 * each operation a binary32 operation rounded to nearest even.
 *   gate, up : n binary32 values (input).   out : n binary32 values (output).
 * out may be exactly gate or exactly up (in place); any other overlap is
 * COMP_ERR_INVALID_VALUE, as are n < 0 and a NULL pointer with n > 0.
 */
comp_status_t comp_geglu_f32(const float* gate, const float* up, float* out, int64_t n, comp_stream_t stream);

/*
 * comp_gemm_f32x16 — the fused compensated projection (laya.cpp docs/vulkan.md,
 * compensated-FP32 paragraph and the fused-build paragraph):
 *   y[m,n] = acc_hi[m,n] + acc_lo[m,n] * 2^-10, with acc_hi, acc_lo the FP32
 *   tensor-core accumulations of hi(x)·W^T and lo(x)·W^T.
 *   x : [M, K] binary32 (input).   W : [N, K] binary16 (input).   y : [M, N] binary32 (output).
 * One kernel: x is split on the fly in shared memory, both products accumulate
 * in tensor memory, and the merge is the epilogue.  For at most 32 rows (K a
 * multiple of 8, x and W 16-byte aligned), the kernel swaps the operands
 * (y^T = W x^T, 128 rows of W per MMA) and splits each K block of x into
 * shared memory as it streams W; when W has few tiles of 128 rows, K is split
 * over a cluster of 2 or 4 CTAs per tile and their partial sums are added in
 * rank order (reruns give identical bits).  For more
 * than 128 rows, once the output fills about one wave of 128 x 192 tiles (same
 * operand conditions), a cluster of two CTAs computes each 256-row tile with
 * one instruction stream for both SMs' tensor cores; x arrives in FP32 and is
 * split in place in shared memory.  The accumulation order of
 * the tensor cores is not specified; results agree with an FP64 evaluation of
 * the same formula to within 4e-6 * sum_k |x[m,k]| |W[n,k]| per element.
 * Errors: COMP_ERR_INVALID_VALUE if a size is negative, M*K, N*K or M*N
 * overflows int64, a needed pointer is NULL, or y overlaps x or W.
 */
comp_status_t comp_gemm_f32x16(const float* x, const uint16_t* W, float* y, int64_t M, int64_t N, int64_t K,
                               comp_stream_t stream);

/*
 * comp_gemm_f32_simt — the true-FP32 reference product (laya.cpp docs/vulkan.md,
 * paragraph on the true FP32 matrix kernels): y = x · float(W)^T with binary32
 * fused multiply-adds on the CUDA cores; W is widened to binary32 exactly and x
 * is never converted to FP16.  Same arguments, layouts and errors as
 * comp_gemm_f32x16.
 */
comp_status_t comp_gemm_f32_simt(const float* x, const uint16_t* W, float* y, int64_t M, int64_t N, int64_t K,
                                 comp_stream_t stream);

/*
 * comp_gemm_f32x16_variant — comp_gemm_f32x16 with the kernel path chosen by
 * the caller, for testing and measurement (the paths compute the same formula):
 *   0 = automatic (what comp_gemm_f32x16 does),
 *   1 = tiled tensor-memory-accelerator loads of x and W (needs 16-byte aligned
 *       x and W and K % 8 == 0, else COMP_ERR_INVALID_VALUE),
 *   2 = plain coalesced loads (any alignment and size),
 *   3 = the swapped-operand kernel with the split fused (M <= 32, 16-byte
 *       aligned x and W, K % 8 == 0, else COMP_ERR_INVALID_VALUE),
 *   4 = CTA pairs on 256-row tiles with the split fused (16-byte aligned x
 *       and W, K % 8 == 0, else COMP_ERR_INVALID_VALUE).
 * A variant outside 0..4 is COMP_ERR_INVALID_VALUE.
 */
comp_status_t comp_gemm_f32x16_variant(const float* x, const uint16_t* W, float* y, int64_t M, int64_t N,
                                       int64_t K, int variant, comp_stream_t stream);

/*
 * comp_gemm_f16x2 — the two products and the merge, from the split planes
 * (laya.cpp docs/vulkan.md, compensated-FP32 paragraph: both FP16 components
 * multiplied by the exact FP16 weights with FP32 accumulators, combined in
 * FP32; the split/merge paragraph: the split as its own dispatch).  Together
 * with comp_split_f32 this is the two-pass form of comp_gemm_f32x16: the split
 * runs once per element instead of once per output tile.
 *   hi, lo : [M, K] binary16 planes as written by comp_split_f32 (input).
 *   W      : [N, K] binary16 (input).   y : [M, N] binary32 (output).
 *   y[m,n] = sum_k hi*W + 2^-10 * sum_k lo*W, FP32 accumulation on the tensor
 *   cores (fresh per 128 of K, those partial sums added in FP32); same
 *   tolerance as comp_gemm_f32x16.
 * hi, lo and W must be 16-byte aligned and K a multiple of 8 (the tensor
 * memory accelerator's layout rules), else COMP_ERR_INVALID_VALUE; also the
 * errors of comp_gemm_f32x16 (y may not overlap an input).
 */
comp_status_t comp_gemm_f16x2(const uint16_t* hi, const uint16_t* lo, const uint16_t* W, float* y, int64_t M,
                              int64_t N, int64_t K, comp_stream_t stream);

/*
 * comp_gemm_f16x2_variant — comp_gemm_f16x2 with the kernel chosen by the
 * caller (testing and measurement): 0 automatic, 1 one CTA per 128-row tile
 * (with K split over a cluster of 2 or 4 CTAs when the tiles are few; the
 * partial sums are added in rank order, so reruns give identical bits), 2 pairs of CTAs
 * (one cluster, both SMs' tensor cores driven by one instruction stream) per
 * 256-row tile, 3 operands swapped (y^T = W x^T with 128 rows of W per tile,
 * K split over a cluster of 2 or 4 CTAs when the tiles are few; M <= 32
 * only), 4 one tensor-core chain per product over all of K (hi and lo
 * in separate FP32 accumulators, merged once at the tile end; one CTA per
 * 128 x 128 tile).  Variant 4 exists to measure what the chunked promotion of
 * the other kernels buys (laya.cpp docs/vulkan.md, AMD accumulation
 * paragraph: separate FP32 additions of partial results against one long
 * chain); it is slower, and its error grows with K: at K = 16384 it no longer
 * meets the 100x gain over a single FP16 cast that the other variants meet.
 * Variants 0..3 give the same results within the same tolerance; a variant
 * outside 0..4, or 3 with M > 32, is COMP_ERR_INVALID_VALUE.
 */
comp_status_t comp_gemm_f16x2_variant(const uint16_t* hi, const uint16_t* lo, const uint16_t* W, float* y, int64_t M,
                                      int64_t N, int64_t K, int variant, comp_stream_t stream);

/*
 * comp_gemm_workspace_bytes — the workspace comp_gemm_f32x16_ws needs for the
 * two-pass form: 4 * M * K bytes (the hi and lo planes).  0 for a negative or
 * overflowing size.
 */
int64_t comp_gemm_workspace_bytes(int64_t M, int64_t K);

/*
 * comp_gemm_workspace_bytes_mnk — the workspace comp_gemm_f32x16_ws needs for
 * the two-pass form whatever K and the alignment of W: with
 * Kp = K rounded up to a multiple of 8, 4 * M * Kp + 2 * N * Kp bytes (hi and lo
 * planes [M, Kp] and a zero-padded copy of W [N, Kp]).  0 for a negative or
 * overflowing size.
 */
int64_t comp_gemm_workspace_bytes_mnk(int64_t M, int64_t N, int64_t K);

/*
 * comp_gemm_f32x16_ws — comp_gemm_f32x16 with a caller-provided device
 * workspace (16-byte aligned), which must not overlap x, W or y
 * (COMP_ERR_INVALID_VALUE); its contents are overwritten.  The call enqueues
 * the two-pass form: comp_split_f32 of x into the workspace, then
 * comp_gemm_f16x2.
 *   - M <= 32, K a multiple of 8, x and W 16-byte aligned: the fused
 *     swapped-operand kernel of comp_gemm_f32x16 instead (one launch; as fast
 *     as split plus product or faster); the workspace is unused.  Except with
 *     17 to 32 rows, K > 512 and W too wide for a split of K (more tiles of
 *     128 rows than clusters of 2 CTAs of that kernel the device runs at
 *     once, at most sm_count / 2), when the planes fit the workspace: the
 *     two-pass form below, whose product holds more stages in flight.
 *   - K a multiple of 8, W 16-byte aligned, workspace of at least
 *     comp_gemm_workspace_bytes(M, K): the planes [M, K] (hi, then lo) and
 *     the caller's W.
 *   - Otherwise, with at least comp_gemm_workspace_bytes_mnk(M, N, K): the
 *     planes [M, Kp] with zero columns past K and a zero-padded copy of W
 *     [N, Kp], Kp = K rounded up to 8.  The added columns contribute exact
 *     zeros.
 *   - Otherwise (no or too small a workspace) exactly comp_gemm_f32x16.
 * Same results within the same tolerance either way; x may have any alignment.
 */
comp_status_t comp_gemm_f32x16_ws(const float* x, const uint16_t* W, float* y, int64_t M, int64_t N, int64_t K,
                                  void* workspace, int64_t workspace_bytes, comp_stream_t stream);

/*
 * comp_gemm_f32x16_epilogue — the projection of comp_gemm_f32x16_ws followed
 * by the FP32 operations of a GEGLU feed-forward step (laya.cpp
 * docs/vulkan.md, feed-forward paragraph: the gate activation and
 * multiplication are fused into one dispatch, with no separate copies or
 * passes):
 *   out[m,n] = gelu(gate[m,n]) * (y[m,n] + bias[n]),
 *   gelu(g) = g * Phi(g), Phi(g) = erfc(-g / sqrt 2) / 2 (the exact GELU),
 * with y the compensated projection.  Each operation is an FP32 operation
 * rounded to nearest even; erfc is CUDA's erfcf.  The bias is added in the
 * product kernel's epilogue; the gate is applied right after on the same
 * stream by comp_geglu_f32 on y in place (on GB300 the gate's erfc work
 * stalls the tensor cores when the product kernel does it at tile ends).
 * comp_gemm_f16x2_epilogue applies both inside the product kernel; the two
 * give identical bits.
 *   bias : [N] binary32, or NULL for none (input).
 *   gate : [M, N] binary32 row-major, or NULL for a factor of 1 (input), e.g.
 *          the gate projection of the same x computed by an earlier call.
 *   out is written to y.  A GEGLU layer is then two calls: gate = x W_g^T + b_g
 *   (this call with gate NULL), then y = gelu(gate) * (x W_u^T + b_u).
 * Workspace, alignment and path rules are those of comp_gemm_f32x16_ws.
 * Errors: those of comp_gemm_f32x16_ws; COMP_ERR_INVALID_VALUE also if bias or
 * gate overlaps y.
 */
comp_status_t comp_gemm_f32x16_epilogue(const float* x, const uint16_t* W, const float* bias, const float* gate,
                                        float* y, int64_t M, int64_t N, int64_t K, void* workspace,
                                        int64_t workspace_bytes, comp_stream_t stream);

/*
 * comp_gemm_f16x2_epilogue — comp_gemm_f16x2_variant (from the split planes,
 * kernel chosen by `variant` as there) with the epilogue of
 * comp_gemm_f32x16_epilogue.  Same errors as comp_gemm_f16x2_variant, plus
 * COMP_ERR_INVALID_VALUE if bias or gate overlaps y.
 */
comp_status_t comp_gemm_f16x2_epilogue(const uint16_t* hi, const uint16_t* lo, const uint16_t* W, const float* bias,
                                       const float* gate, float* y, int64_t M, int64_t N, int64_t K, int variant,
                                       comp_stream_t stream);

/*
 * COMP_NOALLOC_MAX_WORKSPACE_BYTES — size of the static device workspace of
 * comp_gemm_f32x16_noalloc: 64 MiB, i.e. 4 * M * K <= 67108864
 * (M * K <= 16777216, e.g. a 4096 x 4096 activation).
 */
#define COMP_NOALLOC_MAX_WORKSPACE_BYTES (64LL * 1024 * 1024)

/*
 * comp_gemm_f32x16_noalloc — comp_gemm_f32x16_ws with the workspace taken from
 * a static device array of COMP_NOALLOC_MAX_WORKSPACE_BYTES inside the library,
 * so that the call allocates nothing.  The pages have no counterpart for this
 * call: it exists for callers that cannot allocate device memory per call
 * (a plain C host without a device allocator of its own; a latency-critical
 * loop that cannot pay for cudaFree's device synchronisation).
 *   Same arguments, layout, results and errors as comp_gemm_f32x16, plus
 *   COMP_ERR_INVALID_VALUE when 4 * M * K exceeds
 *   COMP_NOALLOC_MAX_WORKSPACE_BYTES (rejected, never truncated).
 *   Paths: as comp_gemm_f32x16_ws given that workspace.  With K % 8 != 0 (or
 *   W not 16-byte aligned) the two-pass form needs 4 * M * Kp + 2 * N * Kp
 *   bytes, Kp = K rounded up to a multiple of 8; when that exceeds the array
 *   the call runs the fused kernel, which needs no workspace (same results
 *   within the same tolerance).
 *   The array's device address belongs to a CUDA context.  The first call in
 *   each context on a device looks it up (cudaGetSymbolAddress, with that
 *   device current; COMP_ERR_CUDA if it fails) and caches it with the
 *   context's identifier; make that first call before any stream capture.
 *   After cudaDeviceReset, or from another context, the next call looks it
 *   up again.  The array is committed when the runtime loads this library's
 *   module that holds it into a context: at the first such call (lazy module
 *   loading, the default), or when the context is created under
 *   CUDA_MODULE_LOADING=EAGER.
 *   The array is shared by all calls in a context: calls whose executions
 *   overlap (unordered streams or threads) race on it.  Calls ordered on one
 *   stream are safe.  Nothing in it needs to start at zero.
 */
comp_status_t comp_gemm_f32x16_noalloc(const float* x, const uint16_t* W, float* y, int64_t M, int64_t N,
                                       int64_t K, comp_stream_t stream);

/*
 * comp_device_status — waits for `stream`, then reports and clears the fault
 * word that kernels of this library set when a bounded wait inside them gives
 * up (they then skip the rest of their work and exit cleanly, leaving the
 * context usable).  Returns COMP_OK, COMP_ERR_TIMEOUT, or COMP_ERR_CUDA if the
 * stream itself reported an error.  If `where` is not NULL it receives the
 * fault word (0 when clear; otherwise a code naming the wait that gave up).
 */
comp_status_t comp_device_status(comp_stream_t stream, uint32_t* where);

/*
 * comp_check_wait_timeout — diagnostic for the path above.  Enqueues one thread
 * that waits, with the library's bounded wait, on a barrier that nothing ever
 * completes.  After about a second the wait gives up, records fault code
 * COMP_FAULT_CHECK_TIMEOUT and the kernel exits.  comp_device_status then
 * returns COMP_ERR_TIMEOUT with that code, and the context stays usable.  The
 * pages have no counterpart; the call exists so that the reporting of a stuck
 * pipeline wait can be tested without faulting or hanging a GPU.  Returns
 * COMP_ERR_UNSUPPORTED_DEVICE off sm_103 and COMP_ERR_LAUNCH if the launch fails.
 */
#define COMP_FAULT_CHECK_TIMEOUT 0x0F01u
comp_status_t comp_check_wait_timeout(comp_stream_t stream);

/*
 * comp_check_stalled_pipeline — diagnostic of the same reporting inside the
 * real kernels.  Enqueues comp_gemm_f16x2_variant(hi, lo, W, y, M, N, K,
 * variant) for variant 2 (CTA pairs) or 3 (operands swapped; M <= 32),
 * except that the kernel's producer leaves out the loads of
 * its first pipeline stage.  The MMA warp's bounded wait for that stage gives
 * up after about a second and raises the abort flag; every role then leaves
 * its loop, the issued loads and MMAs are waited for (bounded) and tensor
 * memory is freed.  comp_device_status then returns COMP_ERR_TIMEOUT with one
 * of the kernel's fault codes (0x701 to 0x703 for pairs, 0x801 to 0x804 for
 * the swapped kernel), and the context stays usable.  y is left undefined.
 * The pages have no counterpart; the call exists so that the abort path of
 * the pipelined kernels can be tested without faulting or hanging a GPU.
 * Errors: those of comp_gemm_f16x2_variant, and COMP_ERR_INVALID_VALUE for
 * another variant or a shape the variant does not take.
 */
comp_status_t comp_check_stalled_pipeline(const uint16_t* hi, const uint16_t* lo, const uint16_t* W, float* y,
                                          int64_t M, int64_t N, int64_t K, int variant, comp_stream_t stream);

/* Human-readable name of a status code (a static string). */
const char* comp_status_string(comp_status_t status);

/* The library's version as major*10000 + minor*100 + patch. */
int comp_version(void);

#ifdef __cplusplus
}
#endif

#endif /* COMPFP32_H */
