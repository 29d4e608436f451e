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
// The scratch array below lives in this file's own device module.  The CUDA
// runtime commits it in a context when it loads that module there: at the
// first use of the array (lazy module loading, the default), or when the
// context is created under CUDA_MODULE_LOADING=EAGER.  It is shared by every
// call in the process that runs in that context: two calls whose executions
// overlap (different streams, or different host threads without ordering
// between their streams) race on it.  Calls ordered on one stream are safe.
//
// Host code must not hand the array's name to a kernel: on the host it is a
// stand-in, not a device address.  The device address belongs to a context
// (after cudaDeviceReset the primary context is a new one and the module is
// loaded again, possibly elsewhere), so it is cached per device together with
// the identifier of the context it was looked up in, and looked up again
// (cudaGetSymbolAddress, with that device current) whenever the current
// context differs.
//
// Nothing in the scratch has to start at zero: the split writes every hi/lo
// element that the product then reads, before it reads them (same stream).
#include <cuda.h>

#include <mutex>

#include "internal.h"

namespace compfp32 {
namespace {

constexpr int kMaxScratchDevices = 64;

// The static workspace: hi plane then lo plane (and, for K % 8 != 0, a
// zero-padded copy of W), COMP_NOALLOC_MAX_WORKSPACE_BYTES at most.
static __device__ __align__(256) unsigned char g_noalloc_scratch[COMP_NOALLOC_MAX_WORKSPACE_BYTES];

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

struct DriverFns {
    CtxGetCurrentFn get_current = nullptr;
    CtxGetIdFn get_id = nullptr;
};

const DriverFns& driver_fns()
{
    static DriverFns fns;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fns.get_current = reinterpret_cast<CtxGetCurrentFn>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fns.get_id = reinterpret_cast<CtxGetIdFn>(p);
        (void)cudaGetLastError();
    });
    return fns;
}

// Identifier of the calling thread's current context (unique for the life of
// the process, never reused); false if there is none yet.
bool current_context_id(unsigned long long* id)
{
    const DriverFns& f = driver_fns();
    if (!f.get_current || !f.get_id)
        return false;
    CUcontext ctx = nullptr;
    if (f.get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr)
        return false;
    return f.get_id(ctx, id) == CUDA_SUCCESS;
}

struct ScratchEntry {
    unsigned long long ctx_id = 0;  // 0: nothing cached
    void* addr = nullptr;
};

std::mutex g_scratch_mu;
ScratchEntry g_scratch[kMaxScratchDevices];

// The device address of g_noalloc_scratch in the current context of `device`.
comp_status_t scratch_address(int device, void** out)
{
    if (device < 0 || device >= kMaxScratchDevices)
        return COMP_ERR_UNSUPPORTED_DEVICE;
    unsigned long long id = 0;
    const bool have_id = current_context_id(&id);
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    ScratchEntry& e = g_scratch[device];
    if (have_id && e.ctx_id == id && e.addr != nullptr) {
        *out = e.addr;
        return COMP_OK;
    }
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
        (void)cudaGetLastError();
        return COMP_ERR_CUDA;
    }
    // The lookup made the runtime's context current if none was; cache the
    // address under that context's identifier (or not at all if it has none).
    unsigned long long id2 = 0;
    if (current_context_id(&id2)) {
        e.ctx_id = id2;
        e.addr = p;
    } else {
        e = ScratchEntry{};
    }
    *out = p;
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
