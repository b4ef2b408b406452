// MXFP8 outputs for the next expert GEMM: SwiGLU and row expansion fused with
// block quantization (E4M3 codes, one E8M0 scale per 32 values).
//
// "CuTeDSL at Perplexity", section "Blackwell support": Blackwell has
// hardware support for MXFP8, MXFP4 and NVFP4, and the kernels were adapted
// for FP8 block-wise scaling, computing the absolute maximum over 32 (MX)
// or 16 (NVFP4) elements with sub-warp reductions. The block format follows
// the OCP Microscaling v1.0 definition of MXFP8 (E4M3): with amax the block's
// largest magnitude, X = floor(log2 amax) - 8 clamped to [-127, 127] (X =
// -127 for an all-zero block), the scale byte is X + 127 and every code is
// E4M3(v * 2^-X), rounded to nearest even and saturated to +-448 (the
// hardware cvt.rn.satfinite.e4m3x2.f32). The quantized values are the
// bfloat16 values the unquantized kernels would store, so a block's scale is
// decided on exactly those values.
//
// Layout: codes [rows, n] bytes, row-major (a row is a whole number of 32-byte
// blocks); scales [rows, n/32] bytes, row-major.
#include "moe_device.cuh"
#include "moe_launch.h"
#include "rows_common.cuh"

namespace moe {
namespace {

// Two floats -> two E4M3 bytes (the first argument in the low byte).
__device__ __forceinline__ uint16_t pack_e4m3x2(float lo, float hi) {
    uint16_t d;
    asm("{\n\t.reg .b16 t;\n\tcvt.rn.satfinite.e4m3x2.f32 t, %1, %2;\n\tmov.b16 %0, t;\n\t}"
        : "=h"(d) : "f"(hi), "f"(lo));
    return d;
}

// Shared exponent of a block from its largest magnitude (amax >= 0, a
// bfloat16 value): floor(log2 amax) is the float's exponent field minus 127
// for normal values; amax below 2^-119 (zero and subnormal included) clamps to
// X = -127.
__device__ __forceinline__ int mx_exponent(float amax) {
    const int ef = int((__float_as_uint(amax) >> 23) & 0xffu);
    if (ef == 0) return -127;
    return max(min(ef - 127 - 8, 127), -127);
}

// 2^-x for x in [-127, 126] as an exact float.
__device__ __forceinline__ float exp2_neg(int x) {
    return __uint_as_float(uint32_t(127 - x) << 23);
}

// EPT consecutive values of one row (EPT = 16 or 8) -> codes; the MX block of
// 32 spans 32/EPT consecutive lanes (aligned), reduced with xor shuffles. All
// lanes of the warp must call; `valid` lanes contribute their values.
template <int EPT>
struct MxChunk {
    uint32_t codes[EPT / 4];
    int x;
};

template <int EPT>
__device__ __forceinline__ MxChunk<EPT> quantize_chunk(const float (&v)[EPT], bool valid) {
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < EPT; ++i) amax = fmaxf(amax, fabsf(v[i]));
    if (!valid) amax = 0.0f;
#pragma unroll
    for (int o = 1; o < 32 / EPT; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, o));
    MxChunk<EPT> c;
    c.x = mx_exponent(amax);
    const float s = exp2_neg(min(c.x, 126));
#pragma unroll
    for (int q = 0; q < EPT / 4; ++q) {
        const uint32_t lo = pack_e4m3x2(v[4 * q] * s, v[4 * q + 1] * s);
        const uint32_t hi = pack_e4m3x2(v[4 * q + 2] * s, v[4 * q + 3] * s);
        c.codes[q] = lo | (hi << 16);
    }
    return c;
}

template <int EPT>
__device__ __forceinline__ void store_codes(uint8_t* p, const MxChunk<EPT>& c) {
    if constexpr (EPT == 16) {
        asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(c.codes[0]), "r"(c.codes[1]),
                     "r"(c.codes[2]), "r"(c.codes[3]) : "memory");
    } else {
        asm volatile("st.global.v2.u32 [%0], {%1,%2};" ::"l"(p), "r"(c.codes[0]), "r"(c.codes[1])
                     : "memory");
    }
}

// bfloat16 bits -> the float values, EPT of them.
template <int EPT>
__device__ __forceinline__ void unpack(const Bits<2 * EPT>& b, float (&v)[EPT]) {
#pragma unroll
    for (int q = 0; q < EPT / 2; ++q) {
        v[2 * q] = bf16_lo(b.w[q]);
        v[2 * q + 1] = bf16_hi(b.w[q]);
    }
}

__device__ __forceinline__ float silu_mul(float g, float u) {
    return __fdividef(g, 1.0f + __expf(-g)) * u;
}

// SwiGLU + MXFP8. Item v = r * nv + c covers act[r, c*EPT .. c*EPT + EPT).
template <int EPT, int NT>
__global__ void __launch_bounds__(NT) swiglu_mxfp8_kernel(const uint8_t* __restrict__ gate_up,
                                                          uint8_t* __restrict__ codes,
                                                          uint8_t* __restrict__ scales, uint32_t total,
                                                          DivU32 nv, uint32_t I) {
    constexpr int VB = 2 * EPT;   // bytes of EPT bfloat16 inputs
    pdl_wait_and_release();
    const uint32_t stride = gridDim.x * NT;
    // the loop runs the same number of times on every lane of a warp (lanes
    // past `total` compute on zeros), so the block reduction sees full warps
    const uint32_t first = blockIdx.x * NT + (threadIdx.x & ~31u);
    for (uint32_t wbase = first; wbase < total; wbase += stride) {
        const uint32_t v = wbase + (threadIdx.x & 31u);
        const bool valid = v < total;
        uint32_t r = 0, c = 0;
        float a[EPT];
        if (valid) {
            r = nv.div(v);
            c = v - r * nv.d;
            const uint8_t* src = gate_up + uint64_t(r) * (4ull * I) + uint64_t(c) * VB;
            Bits<VB> g, u;
            ld_stream(g, src);
            ld_stream(u, src + 2ull * I);
            float gf[EPT], uf[EPT];
            unpack<EPT>(g, gf);
            unpack<EPT>(u, uf);
#pragma unroll
            for (int i = 0; i < EPT; i += 2) {
                // the bfloat16 value moe_swiglu would store
                const uint32_t b = pack_bf16x2(silu_mul(gf[i], uf[i]), silu_mul(gf[i + 1], uf[i + 1]));
                a[i] = bf16_lo(b);
                a[i + 1] = bf16_hi(b);
            }
        } else {
#pragma unroll
            for (int i = 0; i < EPT; ++i) a[i] = 0.0f;
        }
        const MxChunk<EPT> q = quantize_chunk<EPT>(a, valid);
        if (valid) {
            store_codes<EPT>(codes + uint64_t(r) * I + uint64_t(c) * EPT, q);
            if (c % (32 / EPT) == 0) scales[uint64_t(r) * (I / 32) + c / (32 / EPT)] = uint8_t(q.x + 127);
        }
    }
}

// Expand + MXFP8: item v = t * nv + c covers x[t, c*EPT .. +EPT), quantized
// once and stored to the token's k rows inv_perm[t*k + j] < rows.
template <int EPT, int NT>
__global__ void __launch_bounds__(NT) expand_mxfp8_kernel(const uint8_t* __restrict__ x,
                                                          uint8_t* __restrict__ codes,
                                                          uint8_t* __restrict__ scales,
                                                          const int32_t* __restrict__ inv_perm, int k,
                                                          uint32_t rows, uint32_t total, DivU32 nv,
                                                          uint32_t H) {
    constexpr int VB = 2 * EPT;
    pdl_wait_and_release();
    const uint32_t stride = gridDim.x * NT;
    const uint32_t first = blockIdx.x * NT + (threadIdx.x & ~31u);
    for (uint32_t wbase = first; wbase < total; wbase += stride) {
        const uint32_t v = wbase + (threadIdx.x & 31u);
        const bool valid = v < total;
        uint32_t t = 0, c = 0;
        float a[EPT];
        if (valid) {
            t = nv.div(v);
            c = v - t * nv.d;
            Bits<VB> b;
            ld_stream(b, x + uint64_t(t) * (2ull * H) + uint64_t(c) * VB);
            unpack<EPT>(b, a);
        } else {
#pragma unroll
            for (int i = 0; i < EPT; ++i) a[i] = 0.0f;
        }
        const MxChunk<EPT> q = quantize_chunk<EPT>(a, valid);
        if (valid) {
            const bool scale_lane = c % (32 / EPT) == 0;
            const int32_t* ip = inv_perm + uint64_t(t) * k;
            for (int j = 0; j < k; ++j) {
                const uint32_t p = uint32_t(__ldg(ip + j));
                if (p >= rows) continue;
                store_codes<EPT>(codes + uint64_t(p) * H + uint64_t(c) * EPT, q);
                if (scale_lane) scales[uint64_t(p) * (H / 32) + c / (32 / EPT)] = uint8_t(q.x + 127);
            }
        }
    }
}

constexpr int kNt = 256;

// 16 values per thread when the bfloat16 input rows allow 32-byte loads,
// else 8 (16-byte loads).
template <int EPT>
cudaError_t launch_swiglu_q(const uint16_t* gate_up, int64_t rows, int I, uint8_t* codes,
                            uint8_t* scales, int num_sms, cudaStream_t stream) {
    auto kernel = swiglu_mxfp8_kernel<EPT, kNt>;
    static const int occ = resident_blocks(kernel, kNt);
    const uint32_t nv = uint32_t(I / EPT);
    const int64_t per_launch = std::max<int64_t>(1, int64_t(kMaxItemsPerLaunch / nv));
    for (int64_t r0 = 0; r0 < rows; r0 += per_launch) {
        const int64_t nr = std::min(per_launch, rows - r0);
        const uint32_t total = uint32_t(nr * nv);
        const int grid = grid_for(occ, total, uint64_t(kNt), num_sms);
        const cudaError_t err = launch_pdl(
            kernel, dim3(grid), dim3(kNt), 0, stream,
            reinterpret_cast<const uint8_t*>(gate_up + r0 * 2 * int64_t(I)), codes + r0 * int64_t(I),
            scales + r0 * int64_t(I / 32), total, DivU32::make(nv), uint32_t(I));
        if (err != cudaSuccess) return err;
    }
    return cudaSuccess;
}

template <int EPT>
cudaError_t launch_expand_q(const uint16_t* x, int64_t T, int H, int k, const int32_t* inv_perm,
                            int64_t rows, uint8_t* codes, uint8_t* scales, int num_sms,
                            cudaStream_t stream) {
    auto kernel = expand_mxfp8_kernel<EPT, kNt>;
    static const int occ = resident_blocks(kernel, kNt);
    const uint32_t nv = uint32_t(H / EPT);
    const int64_t per_launch = std::max<int64_t>(1, int64_t(kMaxItemsPerLaunch / nv));
    for (int64_t t0 = 0; t0 < T; t0 += per_launch) {
        const int64_t nt = std::min(per_launch, T - t0);
        const uint32_t total = uint32_t(nt * nv);
        const int grid = grid_for(occ, total, uint64_t(kNt), num_sms);
        const cudaError_t err = launch_pdl(
            kernel, dim3(grid), dim3(kNt), 0, stream, reinterpret_cast<const uint8_t*>(x + t0 * int64_t(H)),
            codes, scales, inv_perm + t0 * k, k, uint32_t(rows), total, DivU32::make(nv), uint32_t(H));
        if (err != cudaSuccess) return err;
    }
    return cudaSuccess;
}

}  // namespace

cudaError_t launch_swiglu_mxfp8(const uint16_t* gate_up, int64_t rows, int I, uint8_t* codes,
                                uint8_t* scales, int num_sms, cudaStream_t stream) {
    if (can_use_32b(uint64_t(I) * 2, {gate_up}) && reinterpret_cast<uintptr_t>(codes) % 16 == 0)
        return launch_swiglu_q<16>(gate_up, rows, I, codes, scales, num_sms, stream);
    return launch_swiglu_q<8>(gate_up, rows, I, codes, scales, num_sms, stream);
}

cudaError_t launch_expand_mxfp8(const uint16_t* x, int64_t T, int H, int k, const int32_t* inv_perm,
                                int64_t rows, uint8_t* codes, uint8_t* scales, int num_sms,
                                cudaStream_t stream) {
    if (can_use_32b(uint64_t(H) * 2, {x}) && reinterpret_cast<uintptr_t>(codes) % 16 == 0)
        return launch_expand_q<16>(x, T, H, k, inv_perm, rows, codes, scales, num_sms, stream);
    return launch_expand_q<8>(x, T, H, k, inv_perm, rows, codes, scales, num_sms, stream);
}

}  // namespace moe
