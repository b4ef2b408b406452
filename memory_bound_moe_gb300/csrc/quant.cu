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
// The same page names MXFP4 and NVFP4 with 32- and 16-value blocks; their
// element is E2M1 (OCP MX v1.0: magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6), from
// the hardware cvt.rn.satfinite.e2m1x2.f32 (nearest even, saturating, sign
// kept).
//  - MXFP4: X = floor(log2 amax) - 2 clamped to [-127, 127], scale byte
//    X + 127 (E8M0), code = E2M1(v * 2^-X).
//  - NVFP4 (NVIDIA's format) with a float32 tensor scale g: scale byte
//    E4M3(fl(fl(g * amax) / 6)) of value s, code = E2M1(fl(v * fl(g / s)))
//    (0 when s = 0), every step one float32 rounding to nearest even. The
//    division by 6 is a multiply and one corrected fused multiply-add
//    (div6), and fl(g / s) comes from a per-block table of the 128
//    possible scale values.
//
// Layout: codes [rows, n * bits / 8] bytes, row-major, two FP4 codes per byte
// with element 2i in the low nibble; scales [rows, n / block] bytes,
// row-major.
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

// Two floats -> one byte of two E2M1 codes (the first argument in the low
// nibble).
__device__ __forceinline__ uint32_t pack_e2m1x2(float lo, float hi) {
    uint16_t d;
    asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u16.u8 %0, t;\n\t}"
        : "=h"(d) : "f"(hi), "f"(lo));
    return d;
}

// The value of a non-negative E4M3 byte (4 exponent bits with bias 7, 3
// fraction bits), exactly.
__device__ __forceinline__ float e4m3_value(uint32_t b) {
    const uint32_t e = (b >> 3) & 0xfu, m = b & 7u;
    if (e == 0) return float(m) * __uint_as_float(uint32_t(127 - 9) << 23);
    return float(8u + m) * __uint_as_float((e - 10u + 127u) << 23);
}

// Shared exponent of a block from its largest magnitude (amax >= 0, a
// bfloat16 value): floor(log2 amax) is the float's exponent field minus 127
// for normal values; EMAX is the element format's largest exponent (8 for
// E4M3, 2 for E2M1); amax below 2^-119 (zero and subnormal included) clamps
// to X = -127.
template <int EMAX>
__device__ __forceinline__ int mx_exponent(float amax) {
    const int ef = int((__float_as_uint(amax) >> 23) & 0xffu);
    if (ef == 0) return -127;
    return max(min(ef - 127 - EMAX, 127), -127);
}

// 2^-x for x in [-127, 126] as an exact float.
__device__ __forceinline__ float exp2_neg(int x) {
    return __uint_as_float(uint32_t(127 - x) << 23);
}

enum Fmt { kMxfp8 = 0, kMxfp4 = 1, kNvfp4 = 2 };

template <int F>
struct FmtInfo {
    static constexpr int kBlock = F == kNvfp4 ? 16 : 32;   // values per scale
    static constexpr int kBits = F == kMxfp8 ? 8 : 4;      // bits per code
};

// EPT consecutive values of one row (EPT = 16 or 8) -> codes, and the scale
// byte of their block; a block spans kBlock / EPT consecutive lanes (aligned),
// reduced with xor shuffles. All lanes of the warp must call; `valid` lanes
// contribute their values. g: the NVFP4 tensor scale.
template <int F, int EPT>
struct QChunk {
    static constexpr int kWords = EPT * FmtInfo<F>::kBits / 32;
    uint32_t codes[kWords];
    uint32_t scale;
};

// NVFP4: the multiplier fl(g / s) of every non-negative E4M3 scale byte
// (value s; 0 for s = 0), one IEEE division each, computed once per block
// before the dependency wait. Scale bytes of absolute maxima are at most
// 0x7E (448, saturated).
constexpr int kScaleTable = 128;

__device__ __forceinline__ void fill_nvfp4_table(float* s_q, float g) {
    for (int i = threadIdx.x; i < kScaleTable; i += blockDim.x) {
        const float sv = e4m3_value(uint32_t(i));
        s_q[i] = sv > 0.0f ? __fdiv_rn(g, sv) : 0.0f;
    }
}

// fl(x / 6) for x >= 0 without a division: q0 = fl(x * fl(1/6)) corrected
// by one fused multiply-add of its residual (Markstein's method). Checked
// against the IEEE quotient for every finite float32: identical wherever the
// quotient is a normal float; below 2^-126 both lie far under half the
// smallest E4M3 step (2^-10), so the scale byte they round to is 0 either
// way. Overflowed (infinite) x passes through.
__device__ __forceinline__ float div6(float x) {
    constexpr float kSixth = 1.0f / 6.0f;
    const float q0 = __fmul_rn(x, kSixth);
    const float r = __fmaf_rn(-q0, 6.0f, x);
    return x < __int_as_float(0x7f800000) ? __fmaf_rn(r, kSixth, q0) : x;
}

template <int F, int EPT>
__device__ __forceinline__ QChunk<F, EPT> quantize_chunk(const float (&v)[EPT], bool valid, float g,
                                                         const float* s_q) {
    constexpr int kLanes = FmtInfo<F>::kBlock / EPT;
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < EPT; ++i) amax = fmaxf(amax, fabsf(v[i]));
    if (!valid) amax = 0.0f;
#pragma unroll
    for (int o = 1; o < kLanes; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, o));
    QChunk<F, EPT> c;
    float m;   // the values' multiplier before the element conversion
    if constexpr (F == kNvfp4) {
        c.scale = pack_e4m3x2(div6(__fmul_rn(g, amax)), 0.0f) & 0xffu;
        m = s_q[c.scale & (kScaleTable - 1)];
    } else {
        const int x = mx_exponent<F == kMxfp8 ? 8 : 2>(amax);
        c.scale = uint32_t(x + 127);
        m = exp2_neg(min(x, 126));   // exact: a power of two
    }
    float p[EPT];   // the values the element conversion rounds: fl(v * m), as pairs
#pragma unroll
    for (int i = 0; i < EPT; i += 2) f2_split(mul2(f2(v[i], v[i + 1]), f2(m, m)), p[i], p[i + 1]);
    if constexpr (F == kMxfp8) {
#pragma unroll
        for (int q = 0; q < EPT / 4; ++q)
            c.codes[q] = uint32_t(pack_e4m3x2(p[4 * q], p[4 * q + 1])) |
                         (uint32_t(pack_e4m3x2(p[4 * q + 2], p[4 * q + 3])) << 16);
    } else {
#pragma unroll
        for (int q = 0; q < EPT / 8; ++q)
            c.codes[q] = pack_e2m1x2(p[8 * q], p[8 * q + 1]) | (pack_e2m1x2(p[8 * q + 2], p[8 * q + 3]) << 8) |
                         (pack_e2m1x2(p[8 * q + 4], p[8 * q + 5]) << 16) |
                         (pack_e2m1x2(p[8 * q + 6], p[8 * q + 7]) << 24);
    }
    return c;
}

template <int W>
__device__ __forceinline__ void store_words(uint8_t* p, const uint32_t (&w)[W]) {
    if constexpr (W == 4) {
        asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(w[0]), "r"(w[1]), "r"(w[2]),
                     "r"(w[3]) : "memory");
    } else if constexpr (W == 2) {
        asm volatile("st.global.v2.u32 [%0], {%1,%2};" ::"l"(p), "r"(w[0]), "r"(w[1]) : "memory");
    } else {
        asm volatile("st.global.u32 [%0], %1;" ::"l"(p), "r"(w[0]) : "memory");
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

// Byte offset of value column col of a row in the code buffer.
template <int F>
__device__ __forceinline__ uint64_t code_offset(uint64_t row, uint32_t n, uint32_t col) {
    return (row * n + col) * FmtInfo<F>::kBits / 8;
}

// SwiGLU + block quantization. Item v = r * nv + c covers
// act[r, c*EPT .. c*EPT + EPT).
template <int F, int EPT, int NT>
__global__ void __launch_bounds__(NT) swiglu_q_kernel(const uint8_t* __restrict__ gate_up,
                                                      uint8_t* __restrict__ codes,
                                                      uint8_t* __restrict__ scales, uint32_t total,
                                                      DivU32 nv, uint32_t I, float g) {
    constexpr int VB = 2 * EPT;   // bytes of EPT bfloat16 inputs
    constexpr int kLanes = FmtInfo<F>::kBlock / EPT;
    __shared__ float s_q[F == kNvfp4 ? kScaleTable : 1];
    if constexpr (F == kNvfp4) {
        fill_nvfp4_table(s_q, g);
        __syncthreads();
    }
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
            Bits<VB> gb, ub;
            ld_stream(gb, src);
            ld_stream(ub, src + 2ull * I);
#pragma unroll
            for (int w = 0; w < EPT / 2; ++w) {
                // the bfloat16 value moe_swiglu would store
                float lo, hi;
                f2_split(swiglu2(bf16x2_to_f2(gb.w[w]), bf16x2_to_f2(ub.w[w])), lo, hi);
                const uint32_t b = pack_bf16x2(lo, hi);
                a[2 * w] = bf16_lo(b);
                a[2 * w + 1] = bf16_hi(b);
            }
        } else {
#pragma unroll
            for (int i = 0; i < EPT; ++i) a[i] = 0.0f;
        }
        const QChunk<F, EPT> q = quantize_chunk<F, EPT>(a, valid, g, s_q);
        if (valid) {
            store_words(codes + code_offset<F>(r, I, c * EPT), q.codes);
            if (c % kLanes == 0)
                scales[uint64_t(r) * (I / FmtInfo<F>::kBlock) + c / kLanes] = uint8_t(q.scale);
        }
    }
}

// Expand + block quantization: item v = t * nv + c covers x[t, c*EPT .. +EPT),
// quantized once and stored to the token's k rows inv_perm[t*k + j] < rows.
template <int F, int EPT, int NT>
__global__ void __launch_bounds__(NT) expand_q_kernel(const uint8_t* __restrict__ x,
                                                      uint8_t* __restrict__ codes,
                                                      uint8_t* __restrict__ scales,
                                                      const int32_t* __restrict__ inv_perm, int k,
                                                      uint32_t rows, uint32_t total, DivU32 nv,
                                                      uint32_t H, float g) {
    constexpr int VB = 2 * EPT;
    constexpr int kLanes = FmtInfo<F>::kBlock / EPT;
    __shared__ float s_q[F == kNvfp4 ? kScaleTable : 1];
    if constexpr (F == kNvfp4) {
        fill_nvfp4_table(s_q, g);
        __syncthreads();
    }
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
        const QChunk<F, EPT> q = quantize_chunk<F, EPT>(a, valid, g, s_q);
        if (valid) {
            const bool scale_lane = c % kLanes == 0;
            const int32_t* ip = inv_perm + uint64_t(t) * k;
            for (int j = 0; j < k; ++j) {
                const uint32_t p = uint32_t(__ldg(ip + j));
                if (p >= rows) continue;
                store_words(codes + code_offset<F>(p, H, c * EPT), q.codes);
                if (scale_lane) scales[uint64_t(p) * (H / FmtInfo<F>::kBlock) + c / kLanes] = uint8_t(q.scale);
            }
        }
    }
}

constexpr int kNt = 256;

template <int F, int EPT>
cudaError_t launch_swiglu_q(const uint16_t* gate_up, int64_t rows, int I, uint8_t* codes,
                            uint8_t* scales, float g, int num_sms, cudaStream_t stream) {
    auto kernel = swiglu_q_kernel<F, EPT, kNt>;
    static const int occ = resident_blocks(kernel, kNt);
    const uint32_t nv = uint32_t(I / EPT);
    const int64_t per_launch = std::max<int64_t>(1, int64_t(kMaxItemsPerLaunch / nv));
    for (int64_t r0 = 0; r0 < rows; r0 += per_launch) {
        const int64_t nr = std::min(per_launch, rows - r0);
        const uint32_t total = uint32_t(nr * nv);
        const int grid = grid_for(occ, total, uint64_t(kNt), num_sms);
        const cudaError_t err = launch_pdl(
            kernel, dim3(grid), dim3(kNt), 0, stream,
            reinterpret_cast<const uint8_t*>(gate_up + r0 * 2 * int64_t(I)),
            codes + r0 * int64_t(I) * FmtInfo<F>::kBits / 8, scales + r0 * int64_t(I / FmtInfo<F>::kBlock),
            total, DivU32::make(nv), uint32_t(I), g);
        if (err != cudaSuccess) return err;
    }
    return cudaSuccess;
}

template <int F, int EPT>
cudaError_t launch_expand_q(const uint16_t* x, int64_t T, int H, int k, const int32_t* inv_perm,
                            int64_t rows, uint8_t* codes, uint8_t* scales, float g, int num_sms,
                            cudaStream_t stream) {
    auto kernel = expand_q_kernel<F, EPT, kNt>;
    static const int occ = resident_blocks(kernel, kNt);
    const uint32_t nv = uint32_t(H / EPT);
    const int64_t per_launch = std::max<int64_t>(1, int64_t(kMaxItemsPerLaunch / nv));
    for (int64_t t0 = 0; t0 < T; t0 += per_launch) {
        const int64_t nt = std::min(per_launch, T - t0);
        const uint32_t total = uint32_t(nt * nv);
        const int grid = grid_for(occ, total, uint64_t(kNt), num_sms);
        const cudaError_t err = launch_pdl(
            kernel, dim3(grid), dim3(kNt), 0, stream, reinterpret_cast<const uint8_t*>(x + t0 * int64_t(H)),
            codes, scales, inv_perm + t0 * k, k, uint32_t(rows), total, DivU32::make(nv), uint32_t(H), g);
        if (err != cudaSuccess) return err;
    }
    return cudaSuccess;
}

// 16 values per thread when the bfloat16 input rows allow 32-byte loads and
// the code buffer the matching store, else 8 (16-byte loads).
template <int F>
cudaError_t swiglu_q(const uint16_t* gate_up, int64_t rows, int I, uint8_t* codes, uint8_t* scales, float g,
                     int num_sms, cudaStream_t stream) {
    constexpr uint32_t kStore16 = 16 * FmtInfo<F>::kBits / 8;
    if (can_use_32b(uint64_t(I) * 2, {gate_up}) && reinterpret_cast<uintptr_t>(codes) % kStore16 == 0)
        return launch_swiglu_q<F, 16>(gate_up, rows, I, codes, scales, g, num_sms, stream);
    return launch_swiglu_q<F, 8>(gate_up, rows, I, codes, scales, g, num_sms, stream);
}

template <int F>
cudaError_t expand_q(const uint16_t* x, int64_t T, int H, int k, const int32_t* inv_perm, int64_t rows,
                     uint8_t* codes, uint8_t* scales, float g, int num_sms, cudaStream_t stream) {
    constexpr uint32_t kStore16 = 16 * FmtInfo<F>::kBits / 8;
    if (can_use_32b(uint64_t(H) * 2, {x}) && reinterpret_cast<uintptr_t>(codes) % kStore16 == 0)
        return launch_expand_q<F, 16>(x, T, H, k, inv_perm, rows, codes, scales, g, num_sms, stream);
    return launch_expand_q<F, 8>(x, T, H, k, inv_perm, rows, codes, scales, g, num_sms, stream);
}

}  // namespace

cudaError_t launch_swiglu_mxfp8(const uint16_t* gate_up, int64_t rows, int I, uint8_t* codes,
                                uint8_t* scales, int num_sms, cudaStream_t stream) {
    return swiglu_q<kMxfp8>(gate_up, rows, I, codes, scales, 0.0f, num_sms, stream);
}

cudaError_t launch_expand_mxfp8(const uint16_t* x, int64_t T, int H, int k, const int32_t* inv_perm,
                                int64_t rows, uint8_t* codes, uint8_t* scales, int num_sms,
                                cudaStream_t stream) {
    return expand_q<kMxfp8>(x, T, H, k, inv_perm, rows, codes, scales, 0.0f, num_sms, stream);
}

cudaError_t launch_swiglu_fp4(const uint16_t* gate_up, int64_t rows, int I, bool nvfp4, float g,
                              uint8_t* codes, uint8_t* scales, int num_sms, cudaStream_t stream) {
    return nvfp4 ? swiglu_q<kNvfp4>(gate_up, rows, I, codes, scales, g, num_sms, stream)
                 : swiglu_q<kMxfp4>(gate_up, rows, I, codes, scales, 0.0f, num_sms, stream);
}

cudaError_t launch_expand_fp4(const uint16_t* x, int64_t T, int H, int k, const int32_t* inv_perm,
                              int64_t rows, bool nvfp4, float g, uint8_t* codes, uint8_t* scales,
                              int num_sms, cudaStream_t stream) {
    return nvfp4 ? expand_q<kNvfp4>(x, T, H, k, inv_perm, rows, codes, scales, g, num_sms, stream)
                 : expand_q<kMxfp4>(x, T, H, k, inv_perm, rows, codes, scales, 0.0f, num_sms, stream);
}

}  // namespace moe
