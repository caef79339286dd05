// noalloc.cu -- kfac_precondition_noalloc: the preconditioner for callers
// that cannot allocate device memory.
//
// kfac_precondition needs scratch (the intermediate grad * A_inv, tensor
// maps, split-K partial tiles, the error word) that its caller normally
// allocates.  Some callers cannot call cudaMalloc: host frameworks that own
// all device memory through their own pool and do not let libraries allocate
// behind their back, step loops in which cudaMalloc's implicit device-wide
// synchronisation would stall the pipeline, and embedded callers whose device
// memory budget is fixed when they start.  This entry point serves them from
// a fixed scratch array in the library's own device memory (see
// NOALLOC_SCRATCH_BYTES): every GPU that loads the library holds it until the
// process exits.
#include <mutex>

#include "internal.h"

namespace kfac {
namespace {

constexpr size_t NOALLOC_SCRATCH_BYTES = 32u << 20;  // 32 MiB per device
constexpr int MAX_DEVICES = 64;

// The scratch itself.  In host code this name is only a stand-in for the
// device symbol, never a device address: the address comes from
// cudaGetSymbolAddress on each device.
static __device__ __align__(256) unsigned char g_noalloc_scratch[NOALLOC_SCRATCH_BYTES];

typedef CUresult (*CtxGetCurrentFn)(CUcontext *);

CtxGetCurrentFn ctx_get_current_fn() {
    static std::once_flag once;
    static CtxGetCurrentFn fn = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (CtxGetCurrentFn)p;
    });
    return fn;
}

struct DeviceScratch {
    void *addr = nullptr;
    CUcontext ctx = nullptr;  // the context the address belongs to
};

std::mutex g_mu;
DeviceScratch g_scratch[MAX_DEVICES];

// Device address of the scratch on the current device, looked up with that
// device current on the first call there.  The address belongs to the
// device's context: after cudaDeviceReset the runtime makes a new context
// (and loads the library's module again), so the lookup is repeated when the
// current context is not the one the cached address was found in.
kfac_status scratch_address(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) return KFAC_ERR_CUDA;
    // make sure the device's primary context exists and is current before
    // asking for it (a no-op when the runtime is already initialised)
    if (cudaFree(nullptr) != cudaSuccess) return KFAC_ERR_CUDA;
    CUcontext ctx = nullptr;
    CtxGetCurrentFn get = ctx_get_current_fn();
    if (!get || get(&ctx) != CUDA_SUCCESS || !ctx) return KFAC_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceScratch &d = g_scratch[dev];
    if (!d.addr || d.ctx != ctx) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return KFAC_ERR_CUDA;
        d.addr = p;
        d.ctx = ctx;
    }
    *out = d.addr;
    return KFAC_OK;
}

}  // namespace
}  // namespace kfac

extern "C" size_t kfac_noalloc_scratch_bytes(void) { return kfac::NOALLOC_SCRATCH_BYTES; }

extern "C" kfac_status kfac_precondition_noalloc(const kfac_precond_desc *descs, int count, int dtype,
                                                 void *stream) {
    using namespace kfac;
    if (count < 0 || (count > 0 && !descs)) return KFAC_ERR_INVALID;
    if (count == 0) return KFAC_OK;
    const size_t need = kfac_precondition_workspace_size(descs, count, dtype);
    if (need == 0) return kfac_precondition(descs, count, dtype, nullptr, 0, stream);  // reports the argument error
    if (need > NOALLOC_SCRATCH_BYTES) return KFAC_ERR_WORKSPACE;
    void *scratch = nullptr;
    kfac_status s = scratch_address(&scratch);
    if (s != KFAC_OK) return s;
    return kfac_precondition(descs, count, dtype, scratch, NOALLOC_SCRATCH_BYTES, stream);
}
