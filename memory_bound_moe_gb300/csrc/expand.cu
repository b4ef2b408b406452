// Row expansion into expert order (expandInputRows).
//
// "CuTeDSL at Perplexity", section "Mixture of Experts (MoE) dispatch/combine",
// sub-section "Local": after routing, the tokens are copied into the buffer
// the MoE GEMM reads. "[FlashInfer] CUTLASS MoE kernel optimisation"
// (flashinfer PR #3761), section 1 "Explicit vectorization": the copy moves
// 16-byte vectors with single wide loads and stores.
//
// Scatter from the source token: each vector of x is loaded once and stored
// to the k expert-sorted rows inv_perm[t*k + j]. HBM then reads x once (2TH
// bytes) instead of k times (2SH) as a gather over expanded rows would, and
// every store is a contiguous, coalesced piece of a destination row.
//
// Work item g = (token t, chunk c of 32*U vectors of its row). A warp takes
// one item at a time: it loads the token's k row indices first (k loads in
// flight, once per item rather than once per vector), then its U vectors per
// lane (all in flight together), and stores each vector to the k rows.
//
// The kernel is launched as a programmatic dependent of the routing. x does
// not depend on the routing, so before waiting for it the first blocks issue
// bulk L2 prefetches of x (all of it when x is small next to L2, else its
// first tokens): the reads overlap the routing's last kernel, when HBM is
// nearly idle, and the copy then finds those rows in L2 and spends HBM
// bandwidth on the stores.
#include "moe_device.cuh"
#include "moe_launch.h"
#include "rows_common.cuh"

namespace moe {
namespace {

constexpr int kMaxK = 16;   // MOE_MAX_TOPK

template <int VB, int U, int NT>
__global__ void __launch_bounds__(NT) expand_kernel(const uint8_t* __restrict__ x, uint8_t* __restrict__ out,
                                                    const int32_t* __restrict__ inv_perm, int k, uint32_t S,
                                                    uint32_t items, DivU32 cpr, uint32_t nv, uint32_t row_bytes,
                                                    uint32_t pf_blocks, uint64_t x_bytes) {
    // x does not depend on the routing this kernel waits for: the first
    // pf_blocks blocks pull its first x_bytes into L2 while the routing still
    // runs.
    if (blockIdx.x < pf_blocks) {
        constexpr uint32_t kPiece = 16384;
        const uint64_t slice = (x_bytes / pf_blocks + kPiece - 1) / kPiece * kPiece;
        const uint64_t lo = uint64_t(blockIdx.x) * slice;
        const uint64_t hi = min(x_bytes, lo + slice);
        for (uint64_t off = lo + uint64_t(threadIdx.x) * kPiece; off < hi; off += uint64_t(NT) * kPiece)
            prefetch_l2(x + off, uint32_t(min(uint64_t(kPiece), hi - off)));
    }
    pdl_wait_and_release();
    constexpr int NW = NT / kWarp;
    const int lane = threadIdx.x % kWarp;
    const uint32_t W = gridDim.x * NW;
    for (uint32_t g = blockIdx.x * NW + threadIdx.x / kWarp; g < items; g += W) {
        const uint32_t t = cpr.div(g);
        const uint32_t c0 = (g - t * cpr.d) * (kWarp * U) + lane;   // this lane's first vector
        uint32_t p[kMaxK];
#pragma unroll
        for (int j = 0; j < kMaxK; ++j)
            p[j] = j < k ? uint32_t(__ldg(inv_perm + uint64_t(t) * k + j)) : 0xffffffffu;
        Bits<VB> val[U];
        const uint8_t* src = x + uint64_t(t) * row_bytes;
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (c0 + u * kWarp < nv) ld_stream(val[u], src + uint64_t(c0 + u * kWarp) * VB);
#pragma unroll
        for (int j = 0; j < kMaxK; ++j) {
            if (j >= k) break;
            if (p[j] >= S) continue;   // a slot without a row here (local routing)
            uint8_t* dst = out + uint64_t(p[j]) * row_bytes;
#pragma unroll
            for (int u = 0; u < U; ++u)
                if (c0 + u * kWarp < nv) st_global(dst + uint64_t(c0 + u * kWarp) * VB, val[u]);
        }
    }
}

// Blocks that prefetch x into L2 before waiting for the routing. At most a
// quarter of L2 is prefetched: more would evict its own first lines before
// the copy reads them, and the routing's window is over by then anyway.
constexpr uint32_t kPrefetchBlocks = 64;
// Two vectors per lane and item once the items of U = 2 still give every SM
// this many warps' worth (a few waves); fewer, smaller items otherwise, so
// that small batches spread over all SMs.
#ifndef MOE_EXPAND_U2_MIN_WARPS_PER_SM
#define MOE_EXPAND_U2_MIN_WARPS_PER_SM 32
#endif

template <int VB, int U, int NT>
cudaError_t launch_nt(const uint16_t* x, int64_t T, int H, int k, const int32_t* inv_perm, int64_t rows,
                      uint16_t* out, int num_sms, cudaStream_t stream) {
    auto kernel = expand_kernel<VB, U, NT>;
    static const int occ = resident_blocks(kernel, NT);
    const uint32_t nv = uint32_t(uint64_t(H) * 2 / VB);
    const uint32_t cpr = (nv + kWarp * U - 1) / (kWarp * U);
    const uint32_t row_bytes = uint32_t(2 * int64_t(H));
    // lanes of a launch (items * 32) stay below the per-launch item limit
    const int64_t tok_per_launch = std::max<int64_t>(1, int64_t(kMaxItemsPerLaunch / (uint64_t(cpr) * kWarp)));
    for (int64_t t0 = 0; t0 < T; t0 += tok_per_launch) {
        const int64_t nt = std::min(tok_per_launch, T - t0);
        const uint32_t items = uint32_t(nt * cpr);
        const int grid = grid_for(occ, items, uint64_t(NT / kWarp), num_sms);
        const uint64_t xb = uint64_t(nt) * row_bytes;
        // all of x when it takes at most a quarter of L2, else its first
        // quarter-L2's worth: the first blocks copy the first tokens
        const uint64_t pfb = std::min<uint64_t>(xb, l2_bytes() / 4 / 16384 * 16384);
        const uint32_t pf = pfb > 0 ? std::min<uint32_t>(kPrefetchBlocks, uint32_t(grid)) : 0;
        const cudaError_t err = launch_pdl(
            kernel, dim3(grid), dim3(NT), 0, stream, reinterpret_cast<const uint8_t*>(x + t0 * int64_t(H)),
            reinterpret_cast<uint8_t*>(out), inv_perm + t0 * k, k, uint32_t(rows), items, DivU32::make(cpr), nv,
            row_bytes, pf, pfb);
        if (err != cudaSuccess) return err;
    }
    return cudaSuccess;
}

template <int VB, int U>
cudaError_t launch_vb(const uint16_t* x, int64_t T, int H, int k, const int32_t* inv_perm, int64_t rows,
                      uint16_t* out, int num_sms, cudaStream_t stream) {
    const uint64_t nv = uint64_t(H) * 2 / VB;
    const uint64_t lanes = uint64_t(T) * ((nv + kWarp * U - 1) / (kWarp * U)) * kWarp;
    switch (block_threads(lanes, num_sms)) {
        case 256: return launch_nt<VB, U, 256>(x, T, H, k, inv_perm, rows, out, num_sms, stream);
        case 128: return launch_nt<VB, U, 128>(x, T, H, k, inv_perm, rows, out, num_sms, stream);
        case 64: return launch_nt<VB, U, 64>(x, T, H, k, inv_perm, rows, out, num_sms, stream);
        default: return launch_nt<VB, U, 32>(x, T, H, k, inv_perm, rows, out, num_sms, stream);
    }
}

template <int VB>
cudaError_t launch_u(const uint16_t* x, int64_t T, int H, int k, const int32_t* inv_perm, int64_t rows,
                     uint16_t* out, int num_sms, cudaStream_t stream) {
    const uint64_t nv = uint64_t(H) * 2 / VB;
    const uint64_t items_u2 = uint64_t(T) * ((nv + 2 * kWarp - 1) / (2 * kWarp));
    if (items_u2 >= uint64_t(num_sms) * MOE_EXPAND_U2_MIN_WARPS_PER_SM)
        return launch_vb<VB, 2>(x, T, H, k, inv_perm, rows, out, num_sms, stream);
    return launch_vb<VB, 1>(x, T, H, k, inv_perm, rows, out, num_sms, stream);
}

}  // namespace

cudaError_t launch_expand(const uint16_t* x, int64_t T, int H, int k, const int32_t* inv_perm,
                          int64_t rows, uint16_t* expanded_x, int num_sms, cudaStream_t stream) {
    if (can_use_32b(uint64_t(H) * 2, {x, expanded_x}))
        return launch_u<32>(x, T, H, k, inv_perm, rows, expanded_x, num_sms, stream);
    return launch_u<16>(x, T, H, k, inv_perm, rows, expanded_x, num_sms, stream);
}

}  // namespace moe
