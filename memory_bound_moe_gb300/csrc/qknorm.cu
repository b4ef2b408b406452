// QK RMSNorm: per-head RMS normalisation of q and k, in place.
//
// "CuTeDSL at Perplexity", section "QK normalization": the QK norm of recent
// Qwen attention layers is applied per head of 64, 128 or 256 elements. Unlike
// a general RMSNorm over thousands of elements it needs no cross-warp
// reduction: with 128 bits (8 bfloat16) per thread a half warp covers a
// 128-element head, the squared norm is a butterfly shuffle over those lanes,
// and several heads share a warp; the weight bias and epsilon are
// compile-time constants there (runtime arguments here), the result is
// ((w + bias) * (x * rsqrt(sum(x^2)/head_dim + eps))) stored in place.
//
// Here: head h of the flattened [T, nq + nk] list of heads is handled by
// HD/16 lanes (one 32-byte vector each; HD/8 lanes of 16-byte vectors when
// the pointers are only 16-byte aligned); q heads use q_weight, k heads
// k_weight. Each thread loads its q and k weight chunks (plus the bias) once,
// since a thread always covers the same columns, then sweeps heads
// grid-stride, U head groups per iteration with all loads issued first.
#include "moe_device.cuh"
#include "moe_launch.h"
#include "rows_common.cuh"

namespace moe {
namespace {

// 256-bit coherent load (no L1 allocation): the data is rewritten in place.
__device__ __forceinline__ void ld_coherent(Bits<32>& v, const void* p) {
    asm volatile("ld.global.L1::no_allocate.v8.u32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(v.w[0]), "=r"(v.w[1]), "=r"(v.w[2]), "=r"(v.w[3]),
                   "=r"(v.w[4]), "=r"(v.w[5]), "=r"(v.w[6]), "=r"(v.w[7])
                 : "l"(p));
}

template <int HD, int VB, int U, int NT>
__global__ void __launch_bounds__(NT) qk_norm_kernel(uint8_t* __restrict__ q, uint8_t* __restrict__ k,
                                                     int nq, int nk, uint32_t heads, DivU32 per_token,
                                                     const uint8_t* __restrict__ qw,
                                                     const uint8_t* __restrict__ kw, float bias,
                                                     float eps) {
    constexpr int EPT = VB / 2;        // elements per thread
    constexpr int TPH = HD / EPT;      // lanes per head
    constexpr int HPW = kWarp / TPH;   // heads per warp
    pdl_wait_and_release();
    const int lane = threadIdx.x % kWarp;
    const int sub = lane % TPH;        // this thread's columns: sub*EPT .. sub*EPT + EPT - 1
    float wq[EPT], wk[EPT];
    {
        Bits<VB> a, b;
        ld_stream(a, qw + sub * VB);
        ld_stream(b, kw + sub * VB);
#pragma unroll
        for (int i = 0; i < VB / 4; ++i) {
            wq[2 * i] = bf16_lo(a.w[i]) + bias;
            wq[2 * i + 1] = bf16_hi(a.w[i]) + bias;
            wk[2 * i] = bf16_lo(b.w[i]) + bias;
            wk[2 * i + 1] = bf16_hi(b.w[i]) + bias;
        }
    }
    const uint32_t warps = gridDim.x * (NT / kWarp);
    const uint32_t gwarp = blockIdx.x * (NT / kWarp) + threadIdx.x / kWarp;
    const uint32_t stride = warps * HPW * U;
    // warp-uniform loop: lanes whose head is past the end compute on zeros
    for (uint32_t base = gwarp * HPW * U; base < heads; base += stride) {
        Bits<VB> x[U];
        uint8_t* ptr[U];
        bool isq[U];
        bool valid[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const uint32_t h = base + u * HPW + lane / TPH;
            valid[u] = h < heads;
            ptr[u] = nullptr;
            isq[u] = true;
            if (valid[u]) {
                const uint32_t t = per_token.div(h);
                const int j = int(h - t * per_token.d);
                isq[u] = j < nq;
                ptr[u] = isq[u] ? q + (uint64_t(t) * nq + j) * (2 * HD) + sub * VB
                                : k + (uint64_t(t) * nk + (j - nq)) * (2 * HD) + sub * VB;
                ld_coherent(x[u], ptr[u]);
            } else {
#pragma unroll
                for (int i = 0; i < VB / 4; ++i) x[u].w[i] = 0u;
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            float v[EPT];
            float ss = 0.0f;
#pragma unroll
            for (int i = 0; i < VB / 4; ++i) {
                v[2 * i] = bf16_lo(x[u].w[i]);
                v[2 * i + 1] = bf16_hi(x[u].w[i]);
                ss = fmaf(v[2 * i], v[2 * i], ss);
                ss = fmaf(v[2 * i + 1], v[2 * i + 1], ss);
            }
#pragma unroll
            for (int o = TPH / 2; o > 0; o >>= 1) ss += __shfl_xor_sync(kFull, ss, o);
            const float rms = rsqrtf(ss / float(HD) + eps);
            if (valid[u]) {
                Bits<VB> y;
#pragma unroll
                for (int i = 0; i < VB / 4; ++i) {
                    const float w0 = isq[u] ? wq[2 * i] : wk[2 * i];
                    const float w1 = isq[u] ? wq[2 * i + 1] : wk[2 * i + 1];
                    y.w[i] = pack_bf16x2(w0 * (v[2 * i] * rms), w1 * (v[2 * i + 1] * rms));
                }
                st_global(ptr[u], y);
            }
        }
    }
}

#ifndef MOE_QKNORM_NT
#define MOE_QKNORM_NT 256
#endif
constexpr int kNt = MOE_QKNORM_NT;
// At most 4 waves of resident blocks (2 per SM at 120 registers): on GB300,
// T=8192 with 32+4 heads took 23.9 us under ncu with 1216 blocks and 26.2 us
// with the 1536 an uncapped grid needs.
constexpr int kWaves = 4;

// 32-byte vectors with 6 heads' loads in flight per thread when q, k and the
// weights allow it (measured best on GB300: 90% of the copy bandwidth, 79%
// with 16-byte vectors and 2 in flight); otherwise 16-byte vectors, 4 in
// flight.
template <int HD, int VB, int U>
cudaError_t launch_hd(uint16_t* q, uint16_t* k, int64_t T, int nq, int nk, const uint16_t* qw,
                      const uint16_t* kw, float bias, float eps, int num_sms, cudaStream_t stream) {
    auto kernel = qk_norm_kernel<HD, VB, U, kNt>;
    static const int occ = resident_blocks(kernel, kNt);
    constexpr int HPW = kWarp / (HD / (VB / 2));
    const int per = nq + nk;
    const int64_t tok_per_launch = std::max<int64_t>(1, int64_t(kMaxItemsPerLaunch / per));
    for (int64_t t0 = 0; t0 < T; t0 += tok_per_launch) {
        const int64_t nt = std::min(tok_per_launch, T - t0);
        const uint32_t heads = uint32_t(nt * per);
        const uint64_t per_block = uint64_t(kNt / kWarp) * HPW * U;
        const int grid = grid_for(occ, heads, per_block, num_sms, kWaves);
        const cudaError_t err = launch_pdl(
            kernel, dim3(grid), dim3(kNt), 0, stream, reinterpret_cast<uint8_t*>(q + t0 * nq * int64_t(HD)),
            reinterpret_cast<uint8_t*>(k + t0 * nk * int64_t(HD)), nq, nk, heads, DivU32::make(uint32_t(per)),
            reinterpret_cast<const uint8_t*>(qw), reinterpret_cast<const uint8_t*>(kw), bias, eps);
        if (err != cudaSuccess) return err;
    }
    return cudaSuccess;
}

template <int HD>
cudaError_t launch_vb(uint16_t* q, uint16_t* k, int64_t T, int nq, int nk, const uint16_t* qw,
                      const uint16_t* kw, float bias, float eps, int num_sms, cudaStream_t stream) {
    if (can_use_32b(uint64_t(2 * HD), {q, k, qw, kw}))
        return launch_hd<HD, 32, 6>(q, k, T, nq, nk, qw, kw, bias, eps, num_sms, stream);
    return launch_hd<HD, 16, 4>(q, k, T, nq, nk, qw, kw, bias, eps, num_sms, stream);
}

}  // namespace

cudaError_t launch_qk_rmsnorm(uint16_t* q, uint16_t* k, int64_t T, int nq, int nk, int head_dim,
                              const uint16_t* qw, const uint16_t* kw, float bias, float eps,
                              int num_sms, cudaStream_t stream) {
    switch (head_dim) {
        case 64: return launch_vb<64>(q, k, T, nq, nk, qw, kw, bias, eps, num_sms, stream);
        case 128: return launch_vb<128>(q, k, T, nq, nk, qw, kw, bias, eps, num_sms, stream);
        case 256: return launch_vb<256>(q, k, T, nq, nk, qw, kw, bias, eps, num_sms, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace moe
