// moe_route_static: routing with the scratch count matrix in a file-scope
// device array instead of a caller-provided workspace, for callers that may
// not allocate device memory (see its declaration in moe_glue.h).
//
// The array is a module global: every device that loads this library holds
// MOE_ROUTE_STATIC_SCRATCH_BYTES of it until the process exits. Host code
// must not pass the array's name to a kernel (on the host it is only a
// stand-in symbol); its device address is looked up with
// cudaGetSymbolAddress, while the caller's device is current, on every call
// and handed to the ordinary routing launch as its workspace pointer. The
// lookup allocates nothing. It is not cached: the address belongs to the
// CUDA context that loaded the module, and after cudaDeviceReset (or with
// another context current on the same device) the module is loaded again
// and the array may sit elsewhere, so a cached address could go stale.
#include "moe_glue.h"

#include <cuda_runtime.h>

namespace {

static __device__ __align__(256) unsigned char g_route_scratch[MOE_ROUTE_STATIC_SCRATCH_BYTES];

// Device address of g_route_scratch in the current context. The first lookup
// in a context may load the library's device code into it.
cudaError_t scratch_address(void** out) {
    void* p = nullptr;
    const cudaError_t err = cudaGetSymbolAddress(&p, g_route_scratch);
    if (err != cudaSuccess) return err;
    if (p == nullptr) return cudaErrorInvalidSymbol;
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
