// comp_gemm_f32x16_noalloc: the two-pass projection with its workspace in a
// static device array, so that the call allocates nothing.
//
// Who needs it: callers that cannot allocate device memory per call.  A plain
// C host without a device allocator of its own (no caching allocator such as
// PyTorch's) would otherwise have to pair every call with cudaMalloc/cudaFree,
// and cudaFree synchronises the device, which a latency-critical serving loop
// cannot afford.  Such a caller gets the two-pass speed here without managing
// a workspace.
//
// The scratch array below lives in this file's own device module, is
// reserved when that module loads, and is shared by every call in the
// process on that device: two calls whose executions overlap (different
// streams, or different host threads without ordering between their streams)
// race on it.  Calls ordered on one stream are safe.
//
// Nothing in the scratch has to start at zero: the split writes every hi/lo
// element that the product then reads, before it reads them (same stream).
#include <atomic>

#include "internal.h"

namespace compfp32 {
namespace {

constexpr int kMaxScratchDevices = 64;

// The static workspace: hi plane then lo plane, 4 * M * K bytes at most.
static __device__ __align__(256) unsigned char g_noalloc_scratch[COMP_NOALLOC_MAX_WORKSPACE_BYTES];

// Device address of g_noalloc_scratch per device, looked up on the first call
// made with that device current.
std::atomic<uintptr_t> g_scratch_addr[kMaxScratchDevices];

comp_status_t scratch_address(int device, void** out)
{
    if (device < 0 || device >= kMaxScratchDevices)
        return COMP_ERR_UNSUPPORTED_DEVICE;
    uintptr_t a = g_scratch_addr[device].load(std::memory_order_acquire);
    if (a == 0) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
            (void)cudaGetLastError();
            return COMP_ERR_CUDA;
        }
        a = reinterpret_cast<uintptr_t>(p);
        g_scratch_addr[device].store(a, std::memory_order_release);  // same value from any racing thread
    }
    *out = reinterpret_cast<void*>(a);
    return COMP_OK;
}

}  // namespace
}  // namespace compfp32

using namespace compfp32;

extern "C" comp_status_t comp_gemm_f32x16_noalloc(const float* x, const uint16_t* W, float* y, int64_t M,
                                                  int64_t N, int64_t K, comp_stream_t stream)
{
    if (M < 0 || N < 0 || K < 0)
        return COMP_ERR_INVALID_VALUE;
    if (M != 0 && K > COMP_NOALLOC_MAX_WORKSPACE_BYTES / 4 / M)
        return COMP_ERR_INVALID_VALUE;  // 4*M*K beyond the static workspace
    if (M == 0 || N == 0)
        return COMP_OK;
    DeviceInfo dev;
    const comp_status_t st = current_device(&dev);
    if (st != COMP_OK)
        return st;
    void* scratch = nullptr;
    const comp_status_t sa = scratch_address(dev.device, &scratch);
    if (sa != COMP_OK)
        return sa;
    return comp_gemm_f32x16_ws(x, W, y, M, N, K, scratch, COMP_NOALLOC_MAX_WORKSPACE_BYTES, stream);
}
