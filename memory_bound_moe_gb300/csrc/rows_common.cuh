// Host-side helpers shared by the row kernels (expand, SwiGLU, combine):
// vector-width choice and grid sizing.
#pragma once

#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

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
// most as many as fit on the device at once (every SM busy, one wave).
template <typename Kernel>
inline int grid_for(Kernel kernel, int nt, uint64_t items, uint64_t per_block, int num_sms) {
    int occ = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kernel, nt, 0) != cudaSuccess || occ < 1)
        occ = 1;
    const uint64_t need = (items + per_block - 1) / per_block;
    const uint64_t cap = uint64_t(num_sms) * uint64_t(occ);
    return int(std::max<uint64_t>(1, std::min(need, cap)));
}

// Work items per launch stay below 2^31 so 32-bit grid-stride indices never
// wrap; larger jobs are split into several launches over row ranges.
constexpr uint64_t kMaxItemsPerLaunch = uint64_t(1) << 30;

}  // namespace moe
