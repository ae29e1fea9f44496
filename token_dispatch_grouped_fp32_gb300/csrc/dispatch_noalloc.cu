// dispatch_noalloc.cu -- moe_dispatch for callers that cannot allocate.
//
// moe_dispatch needs a small scratch buffer (per-chunk expert counts and a
// ticket counter) that its caller normally provides.  Some callers have no way to provide it:
// a plugin inside a host framework that owns all device memory and hands the
// layer only its inputs and outputs, or a service that must not call
// cudaMalloc once it has started serving (its allocations are fixed at
// start-up so latency and memory use stay predictable).  For them,
// moe_dispatch_noalloc keeps that scratch in a fixed-size array in the
// library's own device memory instead.
//
// The array is part of the library's device code, so a device holds it from
// the time that code is loaded there (with lazy module loading, the first
// use of the device) until the process exits.  The device address is looked
// up once per device and kept: a device reset after the first call is not
// supported.  Every call on a device shares it and it keeps the last call's
// contents.  The one word that must start at zero, the ticket counter, is
// cleared by every call (a 4-byte cudaMemsetAsync on the caller's stream,
// which allocates nothing) before its kernels; the counts are all written
// before they are read.  Calls whose kernels overlap on the GPU (other
// streams, other threads) race on the array and must be serialised by the
// caller.
#include <mutex>

#include "moe.h"
#include "kernels.h"

namespace {

// 1 MiB: the E x chunks int32 count matrix (E * chunks <= 262,140) and the
// 16-byte ticket after it.
constexpr size_t kNoAllocScratchInts = (size_t)1 << 18;
constexpr size_t kNoAllocScratchBytes = kNoAllocScratchInts * sizeof(int32_t);

__device__ __align__(256) int32_t g_dispatch_scratch[kNoAllocScratchInts];

constexpr int kMaxDevices = 64;
void *g_scratch_addr[kMaxDevices];  // device address of the array, per device
std::mutex g_scratch_mutex;

}  // namespace

extern "C" moe_status_t moe_dispatch_noalloc(const moe_config_t *cfg, const int32_t *topk_idx,
                                             const float *topk_w, const void *x, int32_t *counts,
                                             int32_t *offsets, int32_t *pos, int32_t *src_token,
                                             void *x_perm, void *stream) {
    const size_t need = moe_dispatch_workspace_size(cfg);
    if (need > kNoAllocScratchBytes) {
        moe::set_error_message(
            "moe_dispatch_noalloc: this call needs %zu bytes of dispatch scratch (E * chunks "
            "ints and a ticket); the static array holds %zu bytes. Use moe_dispatch with a caller "
            "buffer.",
            need, kNoAllocScratchBytes);
        return MOE_ERR_UNSUPPORTED;
    }
    void *scratch = nullptr;
    if (cfg && cfg->T > 0) {
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) {
            moe::set_error_message("moe_dispatch_noalloc: cudaGetDevice: %s",
                                   cudaGetErrorString(e));
            return MOE_ERR_CUDA;
        }
        if (dev < 0 || dev >= kMaxDevices) {
            moe::set_error_message("moe_dispatch_noalloc: device ordinal %d is beyond the %d "
                                   "devices this library keeps an address for",
                                   dev, kMaxDevices);
            return MOE_ERR_UNSUPPORTED;
        }
        std::lock_guard<std::mutex> lock(g_scratch_mutex);
        if (!g_scratch_addr[dev]) {
            // Once per device, with that device current: the array's device
            // address.  (Its host-side name is only a stand-in.)
            void *p = nullptr;
            e = cudaGetSymbolAddress(&p, g_dispatch_scratch);
            if (e != cudaSuccess || !p) {
                moe::set_error_message("moe_dispatch_noalloc: cudaGetSymbolAddress: %s",
                                       cudaGetErrorString(e));
                return MOE_ERR_CUDA;
            }
            g_scratch_addr[dev] = p;
        }
        scratch = g_scratch_addr[dev];
    }
    return moe_dispatch(cfg, topk_idx, topk_w, x, counts, offsets, pos, src_token, x_perm,
                        scratch ? scratch : x_perm, kNoAllocScratchBytes, stream);
}
