// Weighted top-k combine / unpermute.
//
// "CuTeDSL at Perplexity", section "Mixture of Experts (MoE) dispatch/combine",
// sub-section "Local": the combine kernel uses the token positions found by
// the routing step, accumulates in registers and writes the final token; it
// is a vectorised accumulation over the routing information and offsets.
//
//   out[t, :] = bf16_rn( sum_{j<k} w[t, j] * expert_out[inv_perm[t*k + j], :] )
//
// Item v = t * nv + c is the c-th vector of output row t. A thread loads the
// k row indices and weights of its token, issues all k wide loads of the
// gathered rows before the first multiply (k loads in flight), accumulates in
// float32 in order j = 0..k-1 and stores one rounded vector.
#include "moe_device.cuh"
#include "moe_launch.h"
#include "rows_common.cuh"

namespace moe {
namespace {

template <int VB>
__device__ __forceinline__ void fma_row(float (&acc)[VB / 2], float w, const Bits<VB>& r) {
#pragma unroll
    for (int q = 0; q < VB / 4; ++q) {
        acc[2 * q] = fmaf(w, bf16_lo(r.w[q]), acc[2 * q]);
        acc[2 * q + 1] = fmaf(w, bf16_hi(r.w[q]), acc[2 * q + 1]);
    }
}

// KC expert rows of one item: indices and weights, then all loads, then the
// multiply-adds. Out-of-range indices contribute nothing.
template <int VB, int KC>
__device__ __forceinline__ void accumulate(float (&acc)[VB / 2], const uint8_t* __restrict__ eo,
                                           const int32_t* ip, const float* wp, int kc, uint32_t S,
                                           uint64_t col_off, uint32_t row_bytes) {
    uint32_t p[KC];
    float w[KC];
    Bits<VB> r[KC];
#pragma unroll
    for (int j = 0; j < KC; ++j) {
        p[j] = j < kc ? uint32_t(__ldg(ip + j)) : 0xffffffffu;
        w[j] = j < kc ? __ldg(wp + j) : 0.0f;
    }
#pragma unroll
    for (int j = 0; j < KC; ++j) {
        if (p[j] < S) {
            ld_stream(r[j], eo + uint64_t(p[j]) * row_bytes + col_off);
        } else {
#pragma unroll
            for (int q = 0; q < VB / 4; ++q) r[j].w[q] = 0u;
        }
    }
#pragma unroll
    for (int j = 0; j < KC; ++j)
        if (j < kc) fma_row<VB>(acc, w[j], r[j]);
}

// KT > 0: k == KT known at compile time. KT == 0: any k, in chunks of 4.
template <int VB, int KT, int NT>
__global__ void __launch_bounds__(NT) combine_kernel(const uint8_t* __restrict__ eo,
                                                     uint8_t* __restrict__ out,
                                                     const float* __restrict__ w,
                                                     const int32_t* __restrict__ inv_perm, int k,
                                                     uint32_t S, uint32_t total, DivU32 nv,
                                                     uint32_t row_bytes) {
    pdl_wait_and_release();
    for (uint32_t v = blockIdx.x * NT + threadIdx.x; v < total; v += gridDim.x * NT) {
        const uint32_t t = nv.div(v);
        const uint32_t c = v - t * nv.d;
        const uint64_t col_off = uint64_t(c) * VB;
        float acc[VB / 2];
#pragma unroll
        for (int q = 0; q < VB / 2; ++q) acc[q] = 0.0f;
        const int32_t* ip = inv_perm + uint64_t(t) * k;
        const float* wp = w + uint64_t(t) * k;
        if constexpr (KT > 0) {
            accumulate<VB, KT>(acc, eo, ip, wp, KT, S, col_off, row_bytes);
        } else {
            for (int j0 = 0; j0 < k; j0 += 4)
                accumulate<VB, 4>(acc, eo, ip + j0, wp + j0, min(4, k - j0), S, col_off, row_bytes);
        }
        Bits<VB> o;
#pragma unroll
        for (int q = 0; q < VB / 4; ++q) o.w[q] = pack_bf16x2(acc[2 * q], acc[2 * q + 1]);
        st_global(out + uint64_t(t) * row_bytes + col_off, o);
    }
}

// k below this uses 32-byte vectors (k * 8 registers of loads in flight).
// Measured on GB300: 32-byte vectors win for k = 2 (prefill step 268.5 us
// against 270.5 with 16-byte ones), 16-byte vectors for k = 4 (twice the
// threads for the same bytes; skewed step 27.6 us against 29.2).
#ifndef MOE_COMBINE_WIDE_BELOW_K
#define MOE_COMBINE_WIDE_BELOW_K 3
#endif
template <int VB, int KT, int NT>
cudaError_t launch_t(const uint16_t* eo, int64_t rows, int64_t T, int H, int k, const float* w,
                     const int32_t* inv_perm, uint16_t* out, int num_sms, cudaStream_t stream) {
    auto kernel = combine_kernel<VB, KT, NT>;
    static const int occ = resident_blocks(kernel, NT);
    const uint32_t nv = uint32_t(uint64_t(H) * 2 / VB);
    const uint32_t S = uint32_t(rows);
    const int64_t tok_per_launch = std::max<int64_t>(1, int64_t(kMaxItemsPerLaunch / nv));
    for (int64_t t0 = 0; t0 < T; t0 += tok_per_launch) {
        const int64_t nt = std::min(tok_per_launch, T - t0);
        const uint32_t total = uint32_t(nt * nv);
        const int grid = grid_for(occ, total, uint64_t(NT), num_sms);
        const cudaError_t err = launch_pdl(
            kernel, dim3(grid), dim3(NT), 0, stream, reinterpret_cast<const uint8_t*>(eo),
            reinterpret_cast<uint8_t*>(out + t0 * int64_t(H)), w + t0 * k, inv_perm + t0 * k, k, S,
            total, DivU32::make(nv), uint32_t(2 * int64_t(H)));
        if (err != cudaSuccess) return err;
    }
    return cudaSuccess;
}

template <int VB, int KT>
cudaError_t launch_k(const uint16_t* eo, int64_t rows, int64_t T, int H, int k, const float* w,
                     const int32_t* inv_perm, uint16_t* out, int num_sms, cudaStream_t stream) {
    switch (block_threads(uint64_t(T) * (uint64_t(H) * 2 / VB), num_sms)) {
        case 256: return launch_t<VB, KT, 256>(eo, rows, T, H, k, w, inv_perm, out, num_sms, stream);
        case 128: return launch_t<VB, KT, 128>(eo, rows, T, H, k, w, inv_perm, out, num_sms, stream);
        case 64: return launch_t<VB, KT, 64>(eo, rows, T, H, k, w, inv_perm, out, num_sms, stream);
        default: return launch_t<VB, KT, 32>(eo, rows, T, H, k, w, inv_perm, out, num_sms, stream);
    }
}

template <int VB>
cudaError_t launch_vb(const uint16_t* eo, int64_t rows, int64_t T, int H, int k, const float* w,
                      const int32_t* inv_perm, uint16_t* out, int num_sms, cudaStream_t stream) {
    switch (k) {
        case 1: return launch_k<VB, 1>(eo, rows, T, H, k, w, inv_perm, out, num_sms, stream);
        case 2: return launch_k<VB, 2>(eo, rows, T, H, k, w, inv_perm, out, num_sms, stream);
        case 4: return launch_k<VB, 4>(eo, rows, T, H, k, w, inv_perm, out, num_sms, stream);
        case 8: return launch_k<VB, 8>(eo, rows, T, H, k, w, inv_perm, out, num_sms, stream);
        default: return launch_k<VB, 0>(eo, rows, T, H, k, w, inv_perm, out, num_sms, stream);
    }
}

}  // namespace

cudaError_t launch_combine(const uint16_t* expert_out, int64_t rows, int64_t T, int H, int k,
                           const float* topk_weights, const int32_t* inv_perm, uint16_t* out,
                           int num_sms, cudaStream_t stream) {
    // 32-byte vectors only for k <= 2; larger k keeps 16-byte vectors (still
    // k loads in flight, twice the threads).
    if (k < MOE_COMBINE_WIDE_BELOW_K && can_use_32b(uint64_t(H) * 2, {expert_out, out}))
        return launch_vb<32>(expert_out, rows, T, H, k, topk_weights, inv_perm, out, num_sms, stream);
    return launch_vb<16>(expert_out, rows, T, H, k, topk_weights, inv_perm, out, num_sms, stream);
}

}  // namespace moe
