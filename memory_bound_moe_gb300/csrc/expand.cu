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
// The kernel is launched as a programmatic dependent of the routing. x does
// not depend on the routing, so before waiting for it the first blocks issue
// bulk L2 prefetches of x (when x is small next to L2): the reads overlap the
// routing's last kernel, when HBM is nearly idle, and the copy then finds x in
// L2 and spends HBM bandwidth on the stores.
#include "moe_device.cuh"
#include "moe_launch.h"
#include "rows_common.cuh"

namespace moe {
namespace {

// Item v = t * nv + c is the c-th VB-byte vector of token row t.
template <int VB, int U, int NT>
__global__ void __launch_bounds__(NT) expand_kernel(const uint8_t* __restrict__ x,
                                                    uint8_t* __restrict__ out,
                                                    const int32_t* __restrict__ inv_perm, int k,
                                                    uint32_t S, uint32_t total, DivU32 nv,
                                                    uint32_t row_bytes, uint32_t pf_blocks) {
    // x does not depend on the routing this kernel waits for: the first
    // pf_blocks blocks pull all of it into L2 while the routing still runs.
    if (blockIdx.x < pf_blocks) {
        constexpr uint32_t kPiece = 16384;
        const uint64_t bytes = uint64_t(total) * VB;
        const uint64_t slice = (bytes / pf_blocks + kPiece - 1) / kPiece * kPiece;
        const uint64_t lo = uint64_t(blockIdx.x) * slice;
        const uint64_t hi = min(bytes, lo + slice);
        for (uint64_t off = lo + uint64_t(threadIdx.x) * kPiece; off < hi; off += uint64_t(NT) * kPiece)
            prefetch_l2(x + off, uint32_t(min(uint64_t(kPiece), hi - off)));
    }
    pdl_wait_and_release();
    const uint32_t stride = gridDim.x * NT * U;
    for (uint32_t base = blockIdx.x * NT * U + threadIdx.x; base < total; base += stride) {
        Bits<VB> val[U];
        uint32_t tok[U], col[U];
#pragma unroll
        for (int i = 0; i < U; ++i) {
            const uint32_t v = base + i * NT;
            if (v < total) {
                tok[i] = nv.div(v);
                col[i] = v - tok[i] * nv.d;
                ld_stream(val[i], x + uint64_t(tok[i]) * row_bytes + uint64_t(col[i]) * VB);
            }
        }
#pragma unroll
        for (int i = 0; i < U; ++i) {
            if (base + i * NT < total) {
                const int32_t* ip = inv_perm + uint64_t(tok[i]) * k;
                for (int j = 0; j < k; ++j) {
                    const uint32_t p = uint32_t(__ldg(ip + j));
                    if (p < S) st_global(out + uint64_t(p) * row_bytes + uint64_t(col[i]) * VB, val[i]);
                }
            }
        }
    }
}

#ifndef MOE_EXPAND_NT
#define MOE_EXPAND_NT 256
#endif
#ifndef MOE_EXPAND_UNROLL
#define MOE_EXPAND_UNROLL 1
#endif
constexpr int kNt = MOE_EXPAND_NT;
// Blocks that prefetch x into L2 before waiting for the routing, used when x
// takes at most a quarter of L2 (larger inputs would evict their own lines
// before the copy reads them).
constexpr uint32_t kPrefetchBlocks = 64;
constexpr int kUnroll = MOE_EXPAND_UNROLL;

template <int VB>
cudaError_t launch_vb(const uint16_t* x, int64_t T, int H, int k, const int32_t* inv_perm,
                      int64_t rows, uint16_t* out, int num_sms, cudaStream_t stream) {
    auto kernel = expand_kernel<VB, kUnroll, kNt>;
    static const int occ = resident_blocks(kernel, kNt);
    const uint32_t nv = uint32_t(uint64_t(H) * 2 / VB);
    const uint32_t S = uint32_t(rows);
    const int64_t tok_per_launch = std::max<int64_t>(1, int64_t(kMaxItemsPerLaunch / nv));
    for (int64_t t0 = 0; t0 < T; t0 += tok_per_launch) {
        const int64_t nt = std::min(tok_per_launch, T - t0);
        const uint32_t total = uint32_t(nt * nv);
        const int grid = grid_for(occ, total, uint64_t(kNt) * kUnroll, num_sms);
        const uint32_t pf = uint64_t(total) * VB <= l2_bytes() / 4 ? kPrefetchBlocks : 0;
        const cudaError_t err = launch_pdl(
            kernel, dim3(grid), dim3(kNt), 0, stream,
            reinterpret_cast<const uint8_t*>(x + t0 * int64_t(H)), reinterpret_cast<uint8_t*>(out),
            inv_perm + t0 * k, k, S, total, DivU32::make(nv), uint32_t(2 * int64_t(H)), pf);
        if (err != cudaSuccess) return err;
    }
    return cudaSuccess;
}

}  // namespace

cudaError_t launch_expand(const uint16_t* x, int64_t T, int H, int k, const int32_t* inv_perm,
                          int64_t rows, uint16_t* expanded_x, int num_sms, cudaStream_t stream) {
    if (can_use_32b(uint64_t(H) * 2, {x, expanded_x}))
        return launch_vb<32>(x, T, H, k, inv_perm, rows, expanded_x, num_sms, stream);
    return launch_vb<16>(x, T, H, k, inv_perm, rows, expanded_x, num_sms, stream);
}

}  // namespace moe
