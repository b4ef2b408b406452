// Device-side building blocks shared by the glue kernels: raw-bit vectors,
// wide global loads/stores written as inline PTX, bfloat16 pack/unpack, and
// division by a loop-invariant divisor.
#pragma once

#include <cstdint>

namespace moe {

constexpr int kWarp = 32;
constexpr unsigned kFull = 0xffffffffu;

// A BYTES-wide vector of raw bits (16 = 8 bf16, 32 = 16 bf16).
template <int BYTES>
struct alignas(BYTES) Bits {
    uint32_t w[BYTES / 4];
};

// --------------------------------------------------------------------------
// Wide global accesses. Each is one instruction: a 128-bit access for 16-byte
// vectors and, on sm_100 and later, a 256-bit access for 32-byte vectors
// ("CuTeDSL at Perplexity", section "Blackwell support": Blackwell adds
// 256-bit loads; "[FlashInfer] CUTLASS MoE kernel optimisation", section 1:
// one 16-byte load instead of four 4-byte loads).
// Streaming reads of data that is read once go through the non-coherent path
// without L1 allocation; the data must stay unchanged while the kernel runs.
// --------------------------------------------------------------------------

__device__ __forceinline__ void ld_stream(Bits<16>& v, const void* p) {
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.w[0]), "=r"(v.w[1]), "=r"(v.w[2]), "=r"(v.w[3])
                 : "l"(p));
}

__device__ __forceinline__ void ld_stream(Bits<32>& v, const void* p) {
    asm volatile("ld.global.nc.L1::no_allocate.v8.u32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(v.w[0]), "=r"(v.w[1]), "=r"(v.w[2]), "=r"(v.w[3]),
                   "=r"(v.w[4]), "=r"(v.w[5]), "=r"(v.w[6]), "=r"(v.w[7])
                 : "l"(p));
}

// Coherent 128-bit load (no L1 allocation) for data the same kernel writes
// back in place, where the non-coherent path's read-only contract would not
// hold.
__device__ __forceinline__ void ld_coherent(Bits<16>& v, const void* p) {
    asm volatile("ld.global.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.w[0]), "=r"(v.w[1]), "=r"(v.w[2]), "=r"(v.w[3])
                 : "l"(p));
}

__device__ __forceinline__ void st_global(void* p, const Bits<16>& v) {
    asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};"
                 :: "l"(p), "r"(v.w[0]), "r"(v.w[1]), "r"(v.w[2]), "r"(v.w[3])
                 : "memory");
}

__device__ __forceinline__ void st_global(void* p, const Bits<32>& v) {
    asm volatile("st.global.v8.u32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};"
                 :: "l"(p), "r"(v.w[0]), "r"(v.w[1]), "r"(v.w[2]), "r"(v.w[3]),
                    "r"(v.w[4]), "r"(v.w[5]), "r"(v.w[6]), "r"(v.w[7])
                 : "memory");
}

// --------------------------------------------------------------------------
// bfloat16 <-> float32. A bfloat16 is the upper half of a float32, so the
// widening is a shift; the narrowing uses the hardware round-to-nearest-even
// conversion of two floats at once (cvt.rn.bf16x2.f32 puts its first source
// in the upper half).
// --------------------------------------------------------------------------

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t d;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}

// --------------------------------------------------------------------------
// Pairs of floats in one 64-bit register, for the packed float32 arithmetic
// of sm_100 and later (mul/add/fma .f32x2: two IEEE round-to-nearest-even
// operations in one instruction, each bit-identical to the scalar one).
// --------------------------------------------------------------------------

struct F2 {
    uint64_t v;
};

__device__ __forceinline__ F2 f2(float lo, float hi) {
    F2 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r.v) : "f"(lo), "f"(hi));
    return r;
}

__device__ __forceinline__ void f2_split(F2 a, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(a.v));
}

__device__ __forceinline__ F2 mul2(F2 a, F2 b) {
    F2 r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r.v) : "l"(a.v), "l"(b.v));
    return r;
}

__device__ __forceinline__ F2 add2(F2 a, F2 b) {
    F2 r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r.v) : "l"(a.v), "l"(b.v));
    return r;
}

// The two float32 values of a bfloat16x2 word (low half first), as a pair.
__device__ __forceinline__ F2 bf16x2_to_f2(uint32_t w) {
    return f2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

// --------------------------------------------------------------------------
// SwiGLU of two elements in float32: silu(g) * u with silu(g) = g / (1 + e^-g),
// e^-g taken as 2^(-g * log2 e) (ex2.approx) and the quotient as g times the
// approximate reciprocal (rcp.approx), both flushing subnormals to zero (an
// e^-g below 2^-126 adds nothing to 1; for g below about -87 the quotient is
// under 2^-126 and comes out as a signed zero); products and the sum are IEEE
// float32 operations done as pairs. Every kernel that stores or quantizes an
// activation uses this one formulation, so they agree bit for bit.
// --------------------------------------------------------------------------

__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float rcp_approx(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

constexpr float kNegLog2e = -1.44269504088896340736f;   // -log2(e)

__device__ __forceinline__ F2 swiglu2(F2 g, F2 u) {
    float t0, t1;
    f2_split(mul2(g, f2(kNegLog2e, kNegLog2e)), t0, t1);
    float d0, d1;
    f2_split(add2(f2(ex2_approx(t0), ex2_approx(t1)), f2(1.0f, 1.0f)), d0, d1);
    return mul2(mul2(g, f2(rcp_approx(d0), rcp_approx(d1))), u);
}

// --------------------------------------------------------------------------
// Programmatic dependent launch (sm_90 and later; "CuTeDSL at Perplexity",
// section "Grid synchronization", notes that it cuts launch overhead from
// Hopper on). Kernels launched with launch_pdl() may be scheduled while the
// previous kernel in the stream is still running: each such kernel first
// waits, before touching global memory, until that kernel has completed and
// its writes are visible, and signals right away that the next kernel may be
// scheduled. Both instructions return at once when there is no programmatic
// dependency, and the wait always ends (the previous kernel always ends).
// --------------------------------------------------------------------------

__device__ __forceinline__ void pdl_wait_and_release() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// --------------------------------------------------------------------------
// Bulk prefetch of [p, p + bytes) into L2 (no registers, no completion to
// wait for; p 16-byte aligned, bytes a multiple of 16). Reading data early
// this way is safe whoever writes it: L2 is the point of coherence, so a
// later write simply updates the prefetched lines.
// --------------------------------------------------------------------------

__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" :: "l"(p), "r"(bytes) : "memory");
}

// --------------------------------------------------------------------------
// Unsigned 32-bit division by a divisor fixed for the whole launch, as a
// multiply-high, an add and a shift (Granlund & Montgomery, "Division by
// Invariant Integers using Multiplication", PLDI 1994, the round-up variant
// with a 33-bit sum): with l = ceil(log2 d) and m = floor(2^32 (2^l - d) / d) + 1,
// n / d = (umulhi(m, n) + n) >> l for every 32-bit n.
// --------------------------------------------------------------------------

struct DivU32 {
    uint32_t d;
    uint32_t m;
    uint32_t l;

    __host__ static DivU32 make(uint32_t d_) {
        DivU32 r;
        r.d = d_;
        uint32_t l = 0;
        while ((uint64_t(1) << l) < d_) ++l;
        r.l = l;
        r.m = uint32_t(((uint64_t(1) << 32) * ((uint64_t(1) << l) - d_)) / d_ + 1);
        return r;
    }

    __device__ __forceinline__ uint32_t div(uint32_t n) const {
        return uint32_t((uint64_t(__umulhi(m, n)) + n) >> l);
    }
};

}  // namespace moe
