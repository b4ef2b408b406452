// moe_route_static: routing with the scratch count matrix in a file-scope
// device array instead of a caller-provided workspace, for callers that may
// not allocate device memory (see its declaration in moe_glue.h).
//
// The array is a module global: every device that loads this library holds
// MOE_ROUTE_STATIC_SCRATCH_BYTES of it until the process exits. Host code
// must not pass the array's name to a kernel (on the host it is only a
// stand-in symbol); its device address is looked up once per device with
// cudaGetSymbolAddress while that device is current, cached, and handed to
// the ordinary routing launch as its workspace pointer.
#include "moe_glue.h"

#include <cuda_runtime.h>

#include <atomic>
#include <mutex>

namespace {

static __device__ __align__(256) unsigned char g_route_scratch[MOE_ROUTE_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::atomic<void*> g_scratch_addr[kMaxDevices];
std::mutex g_setup_mutex;

// Device address of g_route_scratch on the current device; the first call
// on a device does the lookup.
cudaError_t scratch_address(void** out) {
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    void* p = g_scratch_addr[dev].load(std::memory_order_acquire);
    if (p == nullptr) {
        std::lock_guard<std::mutex> lock(g_setup_mutex);
        p = g_scratch_addr[dev].load(std::memory_order_acquire);
        if (p == nullptr) {
            err = cudaGetSymbolAddress(&p, g_route_scratch);
            if (err != cudaSuccess) return err;
            if (p == nullptr) return cudaErrorInvalidSymbol;
            g_scratch_addr[dev].store(p, std::memory_order_release);
        }
    }
    *out = p;
    return cudaSuccess;
}

}  // namespace

extern "C" moe_status_t moe_route_static(const float* logits, int64_t T, int E, int k, int renorm,
                                         int32_t* topk_ids, float* topk_weights,
                                         int32_t* expert_counts, int32_t* expert_offsets,
                                         int32_t* perm, int32_t* inv_perm, moe_stream_t stream) {
    size_t need = 0;
    const moe_status_t st = moe_route_workspace_size(T, E, k, &need);
    if (st != MOE_OK) return st;
    if (need > MOE_ROUTE_STATIC_SCRATCH_BYTES) return MOE_ERR_WORKSPACE;
    void* scratch = nullptr;
    if (need > 0 && scratch_address(&scratch) != cudaSuccess) return MOE_ERR_CUDA;
    return moe_route(logits, T, E, k, renorm, topk_ids, topk_weights, expert_counts,
                     expert_offsets, perm, inv_perm, scratch,
                     need > 0 ? size_t(MOE_ROUTE_STATIC_SCRATCH_BYTES) : 0, stream);
}
