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

constexpr int kMaxTopK = 16;   // MOE_MAX_TOPK

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

// Codes of one lane to one row: W words (at most 16), one vector store (two
// for 64 bytes); the address is aligned to min(4 W, 32) bytes.
template <int W>
__device__ __forceinline__ void store_code_words(uint8_t* p, const uint32_t (&w)[W]) {
    if constexpr (W >= 8) {
#pragma unroll
        for (int h = 0; h < W / 8; ++h) {
            Bits<32> b;
#pragma unroll
            for (int i = 0; i < 8; ++i) b.w[i] = w[8 * h + i];
            st_global(p + 32 * h, b);
        }
    } else {
        store_words<W>(p, w);
    }
}

// N scale bytes (packed in s, the first in the low byte) to an N-aligned
// address.
template <int N>
__device__ __forceinline__ void store_scale_bytes(uint8_t* p, uint32_t s) {
    if constexpr (N == 4) {
        *reinterpret_cast<uint32_t*>(p) = s;
    } else if constexpr (N == 2) {
        *reinterpret_cast<uint16_t*>(p) = uint16_t(s);
    } else {
        *p = uint8_t(s);
    }
}

// Expand + block quantization, in the row-chunk form of moe_expand. Work
// item g = (token t, chunk c of 32 lane vectors); lane l of the warp that
// takes it holds the V = U * VB / 2 consecutive values x[t, (32 c + l) V ...),
// quantizes them once and stores their codes (one vector store) and scales
// (one store) to each of the token's k rows inv_perm[t*k + j] < rows. The
// k row indices are loaded once per item, index j by lane j, and broadcast
// by shuffles. As in moe_expand, x does not depend on the routing this
// kernel waits for: the first pf_blocks blocks prefetch its first x_bytes
// into L2 before the wait.
template <int F, int VB, int U, int NT>
__global__ void __launch_bounds__(NT) expand_q_kernel(const uint8_t* __restrict__ x,
                                                      uint8_t* __restrict__ codes,
                                                      uint8_t* __restrict__ scales,
                                                      const int32_t* __restrict__ inv_perm, int k,
                                                      uint32_t rows, uint32_t items, DivU32 cpr, uint32_t H,
                                                      float g, uint32_t pf_blocks, uint64_t x_bytes) {
    constexpr int kBlock = FmtInfo<F>::kBlock;
    constexpr int V = U * VB / 2;                 // values per lane
    constexpr int EQ = V < kBlock ? V : kBlock;   // values per quantization call
    constexpr int NQ = V / EQ;                    // calls (and scales) per lane
    constexpr int kLanes = kBlock / EQ;           // lanes that share a scale
    constexpr int QW = EQ * FmtInfo<F>::kBits / 32;
    constexpr int VPL = VB / 2;                   // values per load
    constexpr int NW = NT / kWarp;
    if (blockIdx.x < pf_blocks) {
        constexpr uint32_t kPiece = 16384;
        const uint64_t slice = (x_bytes / pf_blocks + kPiece - 1) / kPiece * kPiece;
        const uint64_t lo = uint64_t(blockIdx.x) * slice;
        const uint64_t hi = min(x_bytes, lo + slice);
        for (uint64_t off = lo + uint64_t(threadIdx.x) * kPiece; off < hi; off += uint64_t(NT) * kPiece)
            prefetch_l2(x + off, uint32_t(min(uint64_t(kPiece), hi - off)));
    }
    __shared__ float s_q[F == kNvfp4 ? kScaleTable : 1];
    if constexpr (F == kNvfp4) {
        fill_nvfp4_table(s_q, g);
        __syncthreads();
    }
    pdl_wait_and_release();
    const int lane = threadIdx.x % kWarp;
    const uint32_t W = gridDim.x * NW;
    const uint32_t sp = H / kBlock;   // scales per row
    for (uint32_t gi = blockIdx.x * NW + threadIdx.x / kWarp; gi < items; gi += W) {
        const uint32_t t = cpr.div(gi);
        const uint32_t col = ((gi - t * cpr.d) * kWarp + lane) * V;
        const bool valid = col < H;   // the row's last chunk may be partly outside it
        const uint32_t pl = lane < k ? uint32_t(__ldg(inv_perm + uint64_t(t) * k + lane)) : 0u;
        Bits<VB> b[U];
        if (valid) {
#pragma unroll
            for (int u = 0; u < U; ++u) ld_stream(b[u], x + (uint64_t(t) * H + col) * 2 + u * VB);
        } else {
#pragma unroll
            for (int u = 0; u < U; ++u)
#pragma unroll
                for (int i = 0; i < VB / 4; ++i) b[u].w[i] = 0u;
        }
        uint32_t cw[NQ * QW];
        uint32_t sc = 0;
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
            float a[EQ];
#pragma unroll
            for (int e = 0; e < EQ; e += 2) {
                const int i = q * EQ + e;
                const uint32_t w = b[i / VPL].w[(i % VPL) / 2];
                a[e] = bf16_lo(w);
                a[e + 1] = bf16_hi(w);
            }
            const QChunk<F, EQ> qc = quantize_chunk<F, EQ>(a, valid, g, s_q);
#pragma unroll
            for (int w = 0; w < QW; ++w) cw[q * QW + w] = qc.codes[w];
            sc |= (qc.scale & 0xffu) << (8 * q);
        }
#pragma unroll
        for (int j = 0; j < kMaxTopK; ++j) {
            if (j >= k) break;
            const uint32_t p = uint32_t(__shfl_sync(kFull, pl, j));
            if (!valid || p >= rows) continue;   // outside the row, or a slot without a row here
            store_code_words(codes + code_offset<F>(p, H, col), cw);
            uint8_t* sdst = scales + uint64_t(p) * sp + col / kBlock;
            if constexpr (kLanes == 1) {
                store_scale_bytes<NQ>(sdst, sc);
            } else if (lane % kLanes == 0) {
                *sdst = uint8_t(sc);
            }
        }
    }
}

constexpr int kNt = 256;
constexpr uint32_t kPrefetchBlocks = 64;   // blocks that prefetch x in the quantized expand

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

template <int F, int VB, int U, int NT>
cudaError_t launch_expand_q(const uint16_t* x, int64_t T, int H, int k, const int32_t* inv_perm,
                            int64_t rows, uint8_t* codes, uint8_t* scales, float g, int num_sms,
                            cudaStream_t stream) {
    auto kernel = expand_q_kernel<F, VB, U, NT>;
    static const int occ = resident_blocks(kernel, NT);
    constexpr uint32_t V = U * VB / 2;
    const uint32_t cpr = (uint32_t(H) + kWarp * V - 1) / (kWarp * V);
    // lanes of a launch (items * 32) stay below the per-launch item limit
    const int64_t tok_per_launch = std::max<int64_t>(1, int64_t(kMaxItemsPerLaunch / (uint64_t(cpr) * kWarp)));
    for (int64_t t0 = 0; t0 < T; t0 += tok_per_launch) {
        const int64_t nt = std::min(tok_per_launch, T - t0);
        const uint32_t items = uint32_t(nt * cpr);
        const int grid = grid_for(occ, items, uint64_t(NT / kWarp), num_sms);
        // all of x when it takes at most a quarter of L2, else its first
        // quarter-L2's worth (the rows the first blocks quantize)
        const uint64_t xb = uint64_t(nt) * 2 * uint64_t(H);
        const uint64_t pfb = std::min<uint64_t>(xb, l2_bytes() / 4 / 16384 * 16384);
        const uint32_t pf = pfb > 0 ? std::min<uint32_t>(kPrefetchBlocks, uint32_t(grid)) : 0;
        const cudaError_t err = launch_pdl(
            kernel, dim3(grid), dim3(NT), 0, stream, reinterpret_cast<const uint8_t*>(x + t0 * int64_t(H)),
            codes, scales, inv_perm + t0 * k, k, uint32_t(rows), items, DivU32::make(cpr), uint32_t(H), g, pf,
            pfb);
        if (err != cudaSuccess) return err;
    }
    return cudaSuccess;
}

template <int F, int VB, int U>
cudaError_t expand_q_u(const uint16_t* x, int64_t T, int H, int k, const int32_t* inv_perm, int64_t rows,
                       uint8_t* codes, uint8_t* scales, float g, int num_sms, cudaStream_t stream) {
    constexpr uint64_t V = U * VB / 2;
    const uint64_t lanes = uint64_t(T) * ((uint64_t(H) + kWarp * V - 1) / (kWarp * V)) * kWarp;
    switch (block_threads(lanes, num_sms)) {
        case 256: return launch_expand_q<F, VB, U, 256>(x, T, H, k, inv_perm, rows, codes, scales, g, num_sms, stream);
        case 128: return launch_expand_q<F, VB, U, 128>(x, T, H, k, inv_perm, rows, codes, scales, g, num_sms, stream);
        case 64: return launch_expand_q<F, VB, U, 64>(x, T, H, k, inv_perm, rows, codes, scales, g, num_sms, stream);
        default: return launch_expand_q<F, VB, U, 32>(x, T, H, k, inv_perm, rows, codes, scales, g, num_sms, stream);
    }
}

// Two loads per lane once the items of that width still give every SM
// this many warps' worth; fewer, smaller items otherwise, so that small
// batches spread over all SMs.
#ifndef MOE_EXPAND_Q_MIN_WARPS_PER_SM
#define MOE_EXPAND_Q_MIN_WARPS_PER_SM 32
#endif

// Whether U loads of VB bytes per lane fit: whole lane vectors in a row, the
// codes' and scales' vector stores aligned, and enough items for every SM.
template <int F, int VB>
bool expand_q_fits(int U, int64_t T, int H, const uint8_t* codes, const uint8_t* scales, int num_sms) {
    const uint64_t V = uint64_t(U) * VB / 2;
    if (uint64_t(H) % V != 0) return false;
    const uint64_t code_bytes = V * FmtInfo<F>::kBits / 8;
    if (reinterpret_cast<uintptr_t>(codes) % std::min<uint64_t>(code_bytes, 32) != 0) return false;
    if (V >= uint64_t(FmtInfo<F>::kBlock) && reinterpret_cast<uintptr_t>(scales) % (V / FmtInfo<F>::kBlock) != 0)
        return false;
    const uint64_t items = uint64_t(T) * ((uint64_t(H) + kWarp * V - 1) / (kWarp * V));
    return items >= uint64_t(num_sms) * MOE_EXPAND_Q_MIN_WARPS_PER_SM;
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

// 32-byte loads when the bfloat16 input rows allow them, else 16-byte ones;
// then two of them per lane where that fits, else one. (Four per lane left
// too few warps on mid-sized batches: 11.1 against 9.6 us for NVFP4 at
// 4096 x 2048, top-8.)
template <int F>
cudaError_t expand_q(const uint16_t* x, int64_t T, int H, int k, const int32_t* inv_perm, int64_t rows,
                     uint8_t* codes, uint8_t* scales, float g, int num_sms, cudaStream_t stream) {
    constexpr uint32_t kStore16 = 16 * FmtInfo<F>::kBits / 8;   // code bytes of 16 values
    if (can_use_32b(uint64_t(H) * 2, {x}) && reinterpret_cast<uintptr_t>(codes) % kStore16 == 0) {
        if (expand_q_fits<F, 32>(2, T, H, codes, scales, num_sms))
            return expand_q_u<F, 32, 2>(x, T, H, k, inv_perm, rows, codes, scales, g, num_sms, stream);
        return expand_q_u<F, 32, 1>(x, T, H, k, inv_perm, rows, codes, scales, g, num_sms, stream);
    }
    return expand_q_u<F, 16, 1>(x, T, H, k, inv_perm, rows, codes, scales, g, num_sms, stream);
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
