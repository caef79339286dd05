// noalloc.cu -- kfac_precondition_noalloc: the preconditioner for callers
// that cannot allocate device memory.
//
// kfac_precondition needs scratch (the intermediate grad * A_inv, tensor
// maps, split-K partial tiles) that its caller normally allocates.  Some
// callers cannot call cudaMalloc: code that runs while a CUDA graph is being
// captured (an allocation there breaks or invalidates the capture), step loops
// where cudaMalloc's implicit device synchronisation is not acceptable, and
// host frameworks that own all device memory through their own allocator.
// This entry point serves them from a fixed scratch array that lives in the
// library's own device memory (see NOALLOC_SCRATCH_BYTES): every GPU that loads
// the library holds it until the process exits.
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

std::mutex g_mu;
void *g_addr[MAX_DEVICES] = {nullptr};

// Device address of the scratch on the current device, resolved once per
// device with that device current.
kfac_status scratch_address(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) return KFAC_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return KFAC_ERR_CUDA;
        g_addr[dev] = p;
    }
    *out = g_addr[dev];
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
