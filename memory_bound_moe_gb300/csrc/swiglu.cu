// SwiGLU activation over the fc1 output (doActivation).
//
// "[FlashInfer] CUTLASS MoE kernel optimisation" (flashinfer PR #3761),
// section 1 "Explicit vectorization" (one wide load/store per vector instead
// of several narrow ones) and section 2 "Dynamic threads" (the fixed
// 256-thread, one-row-per-block launch idled most warps at intermediate size
// 768). Here the rows are flattened: consecutive threads take consecutive
// 16- or 32-byte vectors of act, whatever the row width, and a grid of one
// wave of resident blocks sweeps the whole [rows, I] output, so every SM stays
// busy for any I and no block shape depends on I.
//
//   act[r, i] = bf16_rn( silu(g) * u ), g = gate_up[r, i], u = gate_up[r, I + i],
//   silu(g) = g / (1 + e^-g) in float32 (swiglu2: approximate exp2 and
//   reciprocal, the rest as IEEE float32 pair operations).
#include "moe_device.cuh"
#include "moe_launch.h"
#include "rows_common.cuh"

namespace moe {
namespace {

template <int VB>
__device__ __forceinline__ void swiglu_vec(const Bits<VB>& g, const Bits<VB>& u, Bits<VB>& o) {
#pragma unroll
    for (int w = 0; w < VB / 4; ++w) {
        float lo, hi;
        f2_split(swiglu2(bf16x2_to_f2(g.w[w]), bf16x2_to_f2(u.w[w])), lo, hi);
        o.w[w] = pack_bf16x2(lo, hi);
    }
}

// Item v = r * nv + c is the c-th VB-byte vector of act row r. Each thread
// issues U items' loads before any math (2U wide loads in flight).
template <int VB, int U, int NT>
__global__ void __launch_bounds__(NT) swiglu_kernel(const uint8_t* __restrict__ gate_up,
                                                    uint8_t* __restrict__ act, uint32_t total,
                                                    DivU32 nv, uint32_t in_row_bytes,
                                                    uint32_t out_row_bytes) {
    pdl_wait_and_release();
    const uint32_t stride = gridDim.x * NT * U;
    for (uint32_t base = blockIdx.x * NT * U + threadIdx.x; base < total; base += stride) {
        Bits<VB> g[U], u[U];
        uint64_t dst[U];
#pragma unroll
        for (int i = 0; i < U; ++i) {
            const uint32_t v = base + i * NT;
            if (v < total) {
                const uint32_t r = nv.div(v);
                const uint32_t c = v - r * nv.d;
                const uint8_t* src = gate_up + uint64_t(r) * in_row_bytes + uint64_t(c) * VB;
                ld_stream(g[i], src);
                ld_stream(u[i], src + out_row_bytes);
                dst[i] = uint64_t(r) * out_row_bytes + uint64_t(c) * VB;
            }
        }
#pragma unroll
        for (int i = 0; i < U; ++i) {
            if (base + i * NT < total) {
                Bits<VB> o;
                swiglu_vec<VB>(g[i], u[i], o);
                st_global(act + dst[i], o);
            }
        }
    }
}

#ifndef MOE_SWIGLU_UNROLL
#define MOE_SWIGLU_UNROLL 1
#endif
constexpr int kUnroll = MOE_SWIGLU_UNROLL;

template <int VB, int NT>
cudaError_t launch_nt(const uint16_t* gate_up, int64_t rows, int I, uint16_t* act, int num_sms,
                      cudaStream_t stream) {
    auto kernel = swiglu_kernel<VB, kUnroll, NT>;
    static const int occ = resident_blocks(kernel, NT);
    const uint32_t nv = uint32_t(uint64_t(I) * 2 / VB);
    const int64_t rows_per_launch = std::max<int64_t>(1, int64_t(kMaxItemsPerLaunch / nv));
    for (int64_t r0 = 0; r0 < rows; r0 += rows_per_launch) {
        const int64_t nr = std::min(rows_per_launch, rows - r0);
        const uint32_t total = uint32_t(nr * nv);
        const int grid = grid_for(occ, total, uint64_t(NT) * kUnroll, num_sms);
        const cudaError_t err = launch_pdl(
            kernel, dim3(grid), dim3(NT), 0, stream,
            reinterpret_cast<const uint8_t*>(gate_up + r0 * 2 * int64_t(I)),
            reinterpret_cast<uint8_t*>(act + r0 * int64_t(I)), total, DivU32::make(nv),
            uint32_t(4 * int64_t(I)), uint32_t(2 * int64_t(I)));
        if (err != cudaSuccess) return err;
    }
    return cudaSuccess;
}

template <int VB>
cudaError_t launch_vb(const uint16_t* gate_up, int64_t rows, int I, uint16_t* act, int num_sms,
                      cudaStream_t stream) {
    const uint64_t threads = uint64_t(rows) * (uint64_t(I) * 2 / VB) / kUnroll;
    switch (block_threads(threads, num_sms)) {
        case 256: return launch_nt<VB, 256>(gate_up, rows, I, act, num_sms, stream);
        case 128: return launch_nt<VB, 128>(gate_up, rows, I, act, num_sms, stream);
        case 64: return launch_nt<VB, 64>(gate_up, rows, I, act, num_sms, stream);
        default: return launch_nt<VB, 32>(gate_up, rows, I, act, num_sms, stream);
    }
}

}  // namespace

cudaError_t launch_swiglu(const uint16_t* gate_up, int64_t rows, int I, uint16_t* act,
                          int num_sms, cudaStream_t stream) {
    if (can_use_32b(uint64_t(I) * 2, {gate_up, act}))
        return launch_vb<32>(gate_up, rows, I, act, num_sms, stream);
    return launch_vb<16>(gate_up, rows, I, act, num_sms, stream);
}

}  // namespace moe
