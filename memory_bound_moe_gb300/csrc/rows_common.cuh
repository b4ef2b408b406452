// Host-side helpers shared by the row kernels (expand, SwiGLU, combine):
// vector-width choice and grid sizing.
#pragma once

#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <utility>

namespace moe {

// 32-byte (256-bit) accesses when every row start is 32-byte aligned, else the
// 16-byte (128-bit) form that the C-ABI validation guarantees.
inline bool can_use_32b(uint64_t row_bytes, std::initializer_list<const void*> ptrs) {
    if (row_bytes % 32 != 0) return false;
    for (const void* p : ptrs)
        if (reinterpret_cast<uintptr_t>(p) % 32 != 0) return false;
    return true;
}

// Grid for a grid-stride kernel over `items` work items, each block taking
// `per_block` items per sweep: never more blocks than the items need, and at
// most MOE_GRID_WAVES times as many as fit on the device at once (every SM
// busy). `occ` is the kernel's resident blocks per SM (resident_blocks()).
// Measured on GB300 over the row kernels: the prefill step (16384 x 14336
// SwiGLU outputs, ~12 items per thread at 4 waves) took 268.5 us at 4 waves,
// 265.3 at 8 and 264.3 at 12 and 16; the smaller workloads and the quantized
// kernels did not move, as their grids need fewer blocks than the cap. (QK
// RMSNorm, 2 resident blocks per SM, passes its own cap.)
#ifndef MOE_GRID_WAVES
#define MOE_GRID_WAVES 16
#endif
inline int grid_for(int occ, uint64_t items, uint64_t per_block, int num_sms, int waves = MOE_GRID_WAVES) {
    const uint64_t need = (items + per_block - 1) / per_block;
    const uint64_t cap = uint64_t(num_sms) * uint64_t(std::max(occ, 1)) * uint64_t(waves);
    return int(std::max<uint64_t>(1, std::min(need, cap)));
}

// Block size for a launch of `threads` threads in all: the largest of 256,
// 128, 64 and 32 that still gives every SM a block, so a small job (a decode
// batch) spreads over as many SMs as it can fill ("CuTeDSL at Perplexity",
// section "Prefill and decode specialization": fewer warps per block when
// there are fewer warps than SMs). Measured on GB300: the decode layer
// (T=16, H=7168, top-8, I=2048) in a 16-layer CUDA graph went from 10.5 to
// 9.5 us; the larger workloads keep 256-thread blocks.
inline int block_threads(uint64_t threads, int num_sms) {
    for (int nt = 256; nt > 32; nt >>= 1)
        if (threads >= uint64_t(nt) * uint64_t(num_sms)) return nt;
    return 32;
}

// Resident blocks per SM of a kernel at block size nt (no dynamic shared
// memory). The answer depends only on the kernel and the architecture, so
// callers cache it per kernel instantiation.
template <typename Kernel>
inline int resident_blocks(Kernel kernel, int nt) {
    int occ = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kernel, nt, 0) != cudaSuccess || occ < 1)
        occ = 1;
    return occ;
}

// Launch with programmatic stream serialisation (see pdl_wait_and_release):
// the kernel may be scheduled before the previous kernel on the stream ends
// and must call pdl_wait_and_release() before its first global access.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// L2 size of the current device (queried once per process).
inline uint64_t l2_bytes() {
    static const uint64_t bytes = [] {
        int dev = 0, v = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&v, cudaDevAttrL2CacheSize, dev) != cudaSuccess)
            return uint64_t(0);
        return uint64_t(v);
    }();
    return bytes;
}

// Work items per launch stay below 2^31 so 32-bit grid-stride indices never
// wrap; larger jobs are split into several launches over row ranges.
// (A build may lower it, MOE_MAX_ITEMS_PER_LAUNCH, to test the splitting on
// small inputs.)
#ifndef MOE_MAX_ITEMS_PER_LAUNCH
#define MOE_MAX_ITEMS_PER_LAUNCH (uint64_t(1) << 30)
#endif
constexpr uint64_t kMaxItemsPerLaunch = MOE_MAX_ITEMS_PER_LAUNCH;

}  // namespace moe
