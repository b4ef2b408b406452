/*
 * Plain CPU oracle for the memory-bound MoE glue path:
 * routing (softmax, top-k, optional renormalisation), the expert-sorted
 * permutation (histogram, exclusive scan, stable counting sort), row
 * expansion, the SwiGLU activation and the weighted top-k combine.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may link, load or
 * call this file: only the tests, the package smoke check and the benchmark's
 * CPU-baseline leg use it. It shares no code, header, table or constant with
 * the CUDA library.
 *
 * Sources (page title, then section):
 *  - "CuTeDSL at Perplexity", section "Mixture of Experts (MoE) dispatch/combine",
 *    sub-section "Local": the local kernel counts the tokens routed to each
 *    expert, gives every token a unique index inside its expert's list, copies
 *    the tokens into a buffer for the expert GEMM, and the combine kernel uses
 *    those token positions to accumulate the expert outputs into the final
 *    token.
 *  - "[FlashInfer] CUTLASS MoE kernel optimisation" (flashinfer PR #3761
 *    analysis), section 1 "Explicit vectorization" and section 2 "Dynamic
 *    threads": expandInputRows copies rows into expert order; doActivation
 *    applies the gated activation (SwiGLU for Qwen3) to the fc1 output.
 *  The pages give no formulas for softmax, top-k, SwiGLU or combine; the
 *  plain textbook definitions are used, with these readings:
 *   - top-k selects on the logits (order-equivalent to the softmax
 *     probabilities), larger first, equal logits -> lower expert index first;
 *     -0.0 and +0.0 compare equal;
 *   - softmax runs over all E experts; renormalisation divides each selected
 *     probability by the sum of the k selected ones;
 *   - the permutation is stable in the flat slot s = t*k + j;
 *   - gate occupies columns [0, I) of the fc1 row and up occupies [I, 2I);
 *     act = silu(gate) * up with silu(g) = g / (1 + exp(-g));
 *   - combine sums w[t,j] * expert_out[inv_perm[t*k+j], :] over j.
 *
 * Precision: every real-valued quantity is computed in IEEE double and
 * rounded ONCE to the output type (float for routing weights, bfloat16 with
 * round-to-nearest-even for activations). bfloat16 values are passed as their
 * 16-bit patterns (uint16_t).
 *
 * Build: cc -std=c11 -O2 -ffp-contract=off -fPIC -shared moe_oracle.c -lm
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------------- */
/* bfloat16 <-> real                                                       */
/* ---------------------------------------------------------------------- */

/* bfloat16 is the top half of an IEEE binary32: decoding is exact. */
static double bf16_to_double(uint16_t h) {
    uint32_t bits = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* Round a real number once to bfloat16, round-to-nearest, ties to even.
 * bfloat16 has binary32's exponent range (normal exponents -126..127,
 * subnormals below) and 7 stored fraction bits, so the spacing of
 * representable values around |v| in [2^e, 2^(e+1)) is 2^(max(e,-126)-7).
 * v / spacing is exact (power-of-two scaling) and rint() rounds it half to
 * even under the default rounding mode. Results of 2^128 or more overflow. */
static uint16_t bf16_round(double v) {
    if (isnan(v)) return (uint16_t)0x7FC0u;
    uint16_t sign = signbit(v) ? (uint16_t)0x8000u : (uint16_t)0u;
    double a = fabs(v);
    if (a == 0.0) return sign;
    if (isinf(a)) return (uint16_t)(sign | 0x7F80u);
    int e2;
    (void)frexp(a, &e2); /* a = f * 2^e2, f in [0.5, 1): leading bit is 2^(e2-1) */
    int lead = e2 - 1;
    if (lead < -126) lead = -126;
    double spacing = ldexp(1.0, lead - 7);
    double r = rint(a / spacing) * spacing;
    if (r >= ldexp(1.0, 128)) return (uint16_t)(sign | 0x7F80u);
    float f = (float)r; /* exact: at most 8 significant bits, in range */
    uint32_t bits;
    memcpy(&bits, &f, sizeof bits);
    return (uint16_t)(sign | (uint16_t)(bits >> 16));
}

/* Exposed so the tests can pin the rounding against known values. */
void oracle_bf16_round(const double* in, long n, uint16_t* out) {
    for (long i = 0; i < n; ++i) out[i] = bf16_round(in[i]);
}

void oracle_bf16_decode(const uint16_t* in, long n, double* out) {
    for (long i = 0; i < n; ++i) out[i] = bf16_to_double(in[i]);
}

/* ---------------------------------------------------------------------- */
/* Routing: softmax + top-k + optional renormalisation                     */
/* ---------------------------------------------------------------------- */

/* For each token t (row of logits[T][E]):
 *   p_e = exp(l_e - max l) / sum_e' exp(l_e' - max l)          (softmax, all E)
 *   ids = the k experts with the largest logits, in descending order of
 *         logit; equal logits are taken lower index first
 *   w_j = p_{ids_j}                              (renorm == 0)
 *   w_j = p_{ids_j} / sum_{j'} p_{ids_j'}        (renorm != 0)
 * Returns 0, or -1 on bad sizes or allocation failure. */
int oracle_route_topk(const float* logits, long T, int E, int k, int renorm,
                      int32_t* topk_ids, float* topk_weights) {
    if (T < 0 || E < 1 || k < 1 || k > E) return -1;
    double* p = (double*)malloc(sizeof(double) * (size_t)E);
    unsigned char* taken = (unsigned char*)malloc((size_t)E);
    if (!p || !taken) { free(p); free(taken); return -1; }
    for (long t = 0; t < T; ++t) {
        const float* l = logits + t * (long)E;
        double m = (double)l[0];
        for (int e = 1; e < E; ++e)
            if ((double)l[e] > m) m = (double)l[e];
        double z = 0.0;
        for (int e = 0; e < E; ++e) {
            p[e] = exp((double)l[e] - m);
            z += p[e];
        }
        for (int e = 0; e < E; ++e) p[e] /= z;

        memset(taken, 0, (size_t)E);
        double sel_sum = 0.0;
        for (int j = 0; j < k; ++j) {
            int best = -1;
            for (int e = 0; e < E; ++e) {
                if (taken[e]) continue;
                /* strictly greater: on equal logits the lower index stays */
                if (best < 0 || l[e] > l[best]) best = e;
            }
            taken[best] = 1;
            topk_ids[t * k + j] = (int32_t)best;
            sel_sum += p[best];
        }
        for (int j = 0; j < k; ++j) {
            double w = p[topk_ids[t * k + j]];
            if (renorm) w /= sel_sum;
            topk_weights[t * k + j] = (float)w;
        }
    }
    free(p);
    free(taken);
    return 0;
}

/* ---------------------------------------------------------------------- */
/* Permutation: histogram, exclusive scan, stable counting sort            */
/* ---------------------------------------------------------------------- */

/* Slots s = t*k + j, S = T*k, expert e_s = topk_ids[s].
 *   counts[e]    = #{ s : e_s = e }
 *   offsets[e]   = sum_{e' < e} counts[e'],  offsets[E] = S
 *   p(s)         = offsets[e_s] + #{ s' < s : e_s' = e_s }
 *   perm[p(s)]   = s,  inv_perm[s] = p(s)
 * Returns 0, or -1 if an id lies outside [0, E). */
int oracle_route_permute(const int32_t* topk_ids, long T, int E, int k,
                         int32_t* counts, int32_t* offsets,
                         int32_t* perm, int32_t* inv_perm) {
    long S = T * (long)k;
    for (int e = 0; e < E; ++e) counts[e] = 0;
    for (long s = 0; s < S; ++s) {
        int32_t e = topk_ids[s];
        if (e < 0 || e >= E) return -1;
        counts[e] += 1;
    }
    offsets[0] = 0;
    for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
    int32_t* next = (int32_t*)malloc(sizeof(int32_t) * (size_t)E);
    if (!next) return -1;
    for (int e = 0; e < E; ++e) next[e] = offsets[e];
    for (long s = 0; s < S; ++s) {
        int32_t e = topk_ids[s];
        int32_t pos = next[e]++;
        perm[pos] = (int32_t)s;
        inv_perm[s] = pos;
    }
    free(next);
    return 0;
}

/* ---------------------------------------------------------------------- */
/* Local permutation: one expert range, padded expert segments             */
/* ---------------------------------------------------------------------- */

/* "CuTeDSL at Perplexity", section "Mixture of Experts (MoE) dispatch/combine",
 * sub-section "Single node": with tensor parallelism the inputs are
 * replicated and a rank's dispatch routes only the tokens assigned to the
 * experts it holds; its combine sums the local copies and an all-reduce adds
 * the ranks' partial results. Sub-section "Local": the tokens are copied
 * into an optionally padded buffer for the expert GEMM.
 * Reading: the top-k is over all E experts (topk_ids are global); this rank
 * holds experts [e0, e1), n = e1 - e0; every local expert's segment is
 * rounded up to a multiple of pad (pad = 1: no padding).
 *   local slots      s with e_s in [e0, e1), local expert l_s = e_s - e0
 *   counts[l]        = #{ local s : l_s = l }                         [n]
 *   offsets[0] = 0,  offsets[l+1] = offsets[l] + pad * ceil(counts[l] / pad)
 *   inv_perm[s]      = offsets[l_s] + #{ local s' < s : l_s' = l_s }, and -1
 *                      for slots whose expert is not local           [T*k]
 *   perm[p]          = s for those rows, -1 for every other row p < rows
 * rows must be at least offsets[n]. Returns -1 on bad arguments. */
int oracle_route_permute_local(const int32_t* topk_ids, long T, int E, int k, int e0, int e1,
                               int pad, long rows, int32_t* counts, int32_t* offsets,
                               int32_t* perm, int32_t* inv_perm) {
    if (e0 < 0 || e1 > E || e0 >= e1 || pad < 1) return -1;
    const int n = e1 - e0;
    const long S = T * (long)k;
    for (int l = 0; l < n; ++l) counts[l] = 0;
    for (long s = 0; s < S; ++s) {
        int32_t e = topk_ids[s];
        if (e < 0 || e >= E) return -1;
        if (e >= e0 && e < e1) counts[e - e0] += 1;
    }
    offsets[0] = 0;
    for (int l = 0; l < n; ++l)
        offsets[l + 1] = offsets[l] + (int32_t)(((long)counts[l] + pad - 1) / pad * pad);
    if ((long)offsets[n] > rows) return -1;
    for (long p = 0; p < rows; ++p) perm[p] = -1;
    int32_t* next = (int32_t*)malloc(sizeof(int32_t) * (size_t)n);
    if (!next) return -1;
    for (int l = 0; l < n; ++l) next[l] = offsets[l];
    for (long s = 0; s < S; ++s) {
        int32_t e = topk_ids[s];
        if (e >= e0 && e < e1) {
            int32_t pos = next[e - e0]++;
            perm[pos] = (int32_t)s;
            inv_perm[s] = pos;
        } else {
            inv_perm[s] = -1;
        }
    }
    free(next);
    return 0;
}

/* ---------------------------------------------------------------------- */
/* Expand: expert-sorted copy of token rows                                */
/* ---------------------------------------------------------------------- */

/* expanded_x[p, :] = x[perm[p] / k, :] for p in [0, P). Bit copy.
 * Rows with perm[p] < 0 (padding, or no local slot) are left as they are.
 * P may be smaller than T*k to produce a contiguous block of rows
 * (pass perm + p0). Returns -1 if a source token falls outside [0, T). */
int oracle_expand(const uint16_t* x, long T, int H, int k,
                  const int32_t* perm, long P, uint16_t* expanded_x) {
    for (long p = 0; p < P; ++p) {
        if (perm[p] < 0) continue;
        long t = (long)perm[p] / k;
        if (t >= T) return -1;
        memcpy(expanded_x + p * (long)H, x + t * (long)H, sizeof(uint16_t) * (size_t)H);
    }
    return 0;
}

/* ---------------------------------------------------------------------- */
/* SwiGLU                                                                  */
/* ---------------------------------------------------------------------- */

/* act[r, i] = bf16( silu(g) * u ), g = gate_up[r, i], u = gate_up[r, I + i],
 * silu(g) = g / (1 + exp(-g)); real arithmetic, one rounding. */
void oracle_swiglu(const uint16_t* gate_up, long rows, int I, uint16_t* act) {
    for (long r = 0; r < rows; ++r) {
        const uint16_t* gate = gate_up + r * 2L * I;
        const uint16_t* up = gate + I;
        for (int i = 0; i < I; ++i) {
            double g = bf16_to_double(gate[i]);
            double u = bf16_to_double(up[i]);
            double silu = g / (1.0 + exp(-g));
            act[r * (long)I + i] = bf16_round(silu * u);
        }
    }
}

/* ---------------------------------------------------------------------- */
/* MXFP8 block quantization (E4M3 elements, one E8M0 scale per 32)         */
/* ---------------------------------------------------------------------- */

/* "CuTeDSL at Perplexity", section "Blackwell support": Blackwell adds
 * hardware support for MXFP8, MXFP4 and NVFP4; the kernels were adapted for
 * FP8 block-wise scaling, computing the absolute maximum over blocks of 32
 * elements (MXFP8/MXFP4) or 16 (NVFP4). The pages give no formula; the
 * definition followed is the OCP Microscaling (MX) Formats Specification
 * v1.0 (MXFP8 E4M3): for a block of 32 values with absolute maximum amax,
 *   X       = floor(log2(amax)) - 8        (8: largest normal exponent of E4M3)
 *             clamped to [-127, 127]; amax = 0 gives X = -127
 *   scale   = 2^X, stored as the E8M0 byte X + 127
 *   code_i  = E4M3(v_i / 2^X), round to nearest even, saturating to +-448
 * The values quantized here are bfloat16 (the rows the GEMM would read), so
 * every step is exact up to the final E4M3 rounding. */

/* E4M3 (1 sign, 4 exponent bits with bias 7, 3 fraction bits; no infinity,
 * 0x7F/0xFF NaN, largest finite 448): round a real to the nearest E4M3 value,
 * ties to even, magnitudes beyond 448 saturate to 448. The spacing around
 * |v| in [2^e, 2^(e+1)) is 2^(max(e,-6)-3). */
static uint8_t e4m3_round(double v) {
    if (isnan(v)) return (uint8_t)0x7F;
    uint8_t sign = signbit(v) ? (uint8_t)0x80 : (uint8_t)0;
    double a = fabs(v);
    if (a == 0.0) return sign;
    if (a >= 448.0) return (uint8_t)(sign | 0x7E);
    int e2;
    (void)frexp(a, &e2);
    int lead = e2 - 1;
    if (lead < -6) lead = -6;
    double spacing = ldexp(1.0, lead - 3);
    double r = rint(a / spacing) * spacing;
    if (r >= 448.0) return (uint8_t)(sign | 0x7E);
    if (r == 0.0) return sign;
    /* encode r: normal if r >= 2^-6 */
    int re2;
    double f = frexp(r, &re2);          /* r = f * 2^re2, f in [0.5, 1) */
    int ex = re2 - 1;                    /* r = 1.m * 2^ex */
    if (ex < -6) {                       /* subnormal: r = m/8 * 2^-6 */
        int m = (int)(r / ldexp(1.0, -9));
        return (uint8_t)(sign | (uint8_t)m);
    }
    int m = (int)((f * 2.0 - 1.0) * 8.0);
    return (uint8_t)(sign | (uint8_t)((ex + 7) << 3) | (uint8_t)m);
}

void oracle_e4m3_round(const double* in, long n, uint8_t* out) {
    for (long i = 0; i < n; ++i) out[i] = e4m3_round(in[i]);
}

/* Shared exponent X of a block (see above). */
static int mx_exponent(double amax) {
    if (amax == 0.0) return -127;
    int e2;
    (void)frexp(amax, &e2);              /* floor(log2(amax)) = e2 - 1 */
    int x = (e2 - 1) - 8;
    if (x < -127) x = -127;
    if (x > 127) x = 127;
    return x;
}

/* MXFP8 quantization of a [rows, n] bfloat16 matrix (n a multiple of 32):
 * codes [rows, n] E4M3 bytes, scales [rows, n/32] E8M0 bytes. */
void oracle_quant_mxfp8(const uint16_t* in, long rows, int n, uint8_t* codes, uint8_t* scales) {
    for (long r = 0; r < rows; ++r) {
        for (int b = 0; b < n / 32; ++b) {
            const uint16_t* v = in + r * (long)n + b * 32;
            double amax = 0.0;
            for (int i = 0; i < 32; ++i) {
                double a = fabs(bf16_to_double(v[i]));
                if (a > amax) amax = a;
            }
            int x = mx_exponent(amax);
            scales[r * (long)(n / 32) + b] = (uint8_t)(x + 127);
            for (int i = 0; i < 32; ++i)
                codes[r * (long)n + b * 32 + i] = e4m3_round(ldexp(bf16_to_double(v[i]), -x));
        }
    }
}

/* ---------------------------------------------------------------------- */
/* FP4 block quantization: MXFP4 and NVFP4 (E2M1 elements)                 */
/* ---------------------------------------------------------------------- */

/* Same page and section as MXFP8: the pages name MXFP4 and NVFP4 and their
 * block sizes (32 and 16 values) but give no formulas. Definitions followed:
 *  - E2M1, the FP4 element of the OCP Microscaling v1.0 specification: a
 *    sign bit, 2 exponent bits with bias 1 and 1 mantissa bit, so the code
 *    c = 0..7 of a magnitude is its index in {0, 0.5, 1, 1.5, 2, 3, 4, 6};
 *    no infinity or NaN. A real converts to the nearest magnitude, ties to
 *    the even code (mantissa bit 0), saturating to 6; the sign bit (0x8) is
 *    the sign of the real, so a negative value that rounds to 0 is -0.
 *  - MXFP4 (OCP MX v1.0): 32 values share X = floor(log2 amax) - 2 (2: the
 *    largest E2M1 exponent), clamped to [-127, 127] (-127 when amax = 0),
 *    stored as the E8M0 byte X + 127; code_i = E2M1(v_i / 2^X).
 *  - NVFP4 (NVIDIA's published format): 16 values share an E4M3 scale and
 *    the tensor a float32 scale g > 0. The block scale byte is
 *    E4M3(fl(fl(g * amax) / 6)) with value s, and code_i = E2M1(fl(v_i * q))
 *    with q = fl(g / s) (q = 0 when s = 0); a code decodes as E2M1 * s / g.
 *    fl() is one float32 rounding to nearest even: these steps decide codes,
 *    so they are taken in float32 here as in the kernels.
 * Codes are packed two per byte, element 2i in the low nibble. */

static uint8_t e2m1_round(double v) {
    static const double mag[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};
    uint8_t sign = signbit(v) ? (uint8_t)0x8 : (uint8_t)0;
    double a = fabs(v);
    if (a >= 6.0) return (uint8_t)(sign | 7);
    int i = 0;
    while (i < 7 && mag[i + 1] <= a) ++i;    /* mag[i] <= a < mag[i + 1] */
    if (a == mag[i]) return (uint8_t)(sign | i);
    double d0 = a - mag[i], d1 = mag[i + 1] - a;
    int c;
    if (d0 < d1) c = i;
    else if (d1 < d0) c = i + 1;
    else c = (i % 2 == 0) ? i : i + 1;       /* tie: the even code */
    return (uint8_t)(sign | c);
}

void oracle_e2m1_round(const double* in, long n, uint8_t* out) {
    for (long i = 0; i < n; ++i) out[i] = e2m1_round(in[i]);
}

static void put_nibble(uint8_t* codes, long idx, uint8_t c) {
    if (idx % 2 == 0) codes[idx / 2] = (uint8_t)((codes[idx / 2] & 0xF0) | c);
    else codes[idx / 2] = (uint8_t)((codes[idx / 2] & 0x0F) | (c << 4));
}

/* MXFP4 of a [rows, n] bfloat16 matrix (n a multiple of 32): codes
 * [rows, n/2] bytes, scales [rows, n/32] E8M0 bytes. */
void oracle_quant_mxfp4(const uint16_t* in, long rows, int n, uint8_t* codes, uint8_t* scales) {
    for (long r = 0; r < rows; ++r) {
        for (int b = 0; b < n / 32; ++b) {
            const uint16_t* v = in + r * (long)n + b * 32;
            double amax = 0.0;
            for (int i = 0; i < 32; ++i) {
                double a = fabs(bf16_to_double(v[i]));
                if (a > amax) amax = a;
            }
            int x;
            if (amax == 0.0) {
                x = -127;
            } else {
                int e2;
                (void)frexp(amax, &e2);          /* floor(log2(amax)) = e2 - 1 */
                x = (e2 - 1) - 2;
                if (x < -127) x = -127;
                if (x > 127) x = 127;
            }
            scales[r * (long)(n / 32) + b] = (uint8_t)(x + 127);
            for (int i = 0; i < 32; ++i)
                put_nibble(codes + r * (long)(n / 2), (long)b * 32 + i,
                           e2m1_round(ldexp(bf16_to_double(v[i]), -x)));
        }
    }
}

/* NVFP4 of a [rows, n] bfloat16 matrix (n a multiple of 16) with tensor
 * scale g: codes [rows, n/2] bytes, scales [rows, n/16] E4M3 bytes. */
void oracle_quant_nvfp4(const uint16_t* in, long rows, int n, float g, uint8_t* codes, uint8_t* scales) {
    for (long r = 0; r < rows; ++r) {
        for (int b = 0; b < n / 16; ++b) {
            const uint16_t* v = in + r * (long)n + b * 16;
            float amax = 0.0f;                   /* bfloat16 values are exact in float */
            for (int i = 0; i < 16; ++i) {
                float a = (float)fabs(bf16_to_double(v[i]));
                if (a > amax) amax = a;
            }
            volatile float t = g * amax;         /* fl(g * amax) */
            volatile float u = t / 6.0f;         /* fl(t / 6) */
            uint8_t sb = e4m3_round((double)u);
            scales[r * (long)(n / 16) + b] = sb;
            /* decode the (non-negative) E4M3 scale byte */
            int e = (sb >> 3) & 0xF, m = sb & 7;
            double s = e == 0 ? ldexp((double)m, -9) : ldexp(1.0 + m / 8.0, e - 7);
            volatile float q = s > 0.0 ? g / (float)s : 0.0f;   /* fl(g / s) */
            for (int i = 0; i < 16; ++i) {
                volatile float p = (float)bf16_to_double(v[i]) * q;   /* fl(v * q) */
                put_nibble(codes + r * (long)(n / 2), (long)b * 16 + i, e2m1_round((double)p));
            }
        }
    }
}

/* ---------------------------------------------------------------------- */
/* Combine: weighted sum of each token's k expert rows                     */
/* ---------------------------------------------------------------------- */

/* out[t, :] = bf16( sum_{j<k} w[t, j] * expert_out[inv_perm[t*k + j], :] ),
 * summed in real arithmetic for j = 0..k-1 and rounded once. A negative
 * inv_perm entry (a slot whose expert another rank holds) contributes
 * nothing: the result is then this rank's partial sum.
 * S is the number of rows of expert_out (for the range check); T may be a
 * sub-range of tokens if w and inv_perm are offset to match.
 * Returns -1 if a row index is S or more. */
int oracle_combine(const uint16_t* expert_out, long S, int H, int k, long T,
                   const float* w, const int32_t* inv_perm, uint16_t* out) {
    double* acc = (double*)malloc(sizeof(double) * (size_t)H);
    if (!acc) return -1;
    for (long t = 0; t < T; ++t) {
        for (int c = 0; c < H; ++c) acc[c] = 0.0;
        for (int j = 0; j < k; ++j) {
            long p = inv_perm[t * k + j];
            if (p < 0) continue;
            if (p >= S) { free(acc); return -1; }
            double wj = (double)w[t * k + j];
            const uint16_t* row = expert_out + p * (long)H;
            for (int c = 0; c < H; ++c) acc[c] += wj * bf16_to_double(row[c]);
        }
        for (int c = 0; c < H; ++c) out[t * (long)H + c] = bf16_round(acc[c]);
    }
    free(acc);
    return 0;
}

/* ---------------------------------------------------------------------- */
/* QK RMSNorm: per-head RMS normalisation of q and k                       */
/* ---------------------------------------------------------------------- */

/* "CuTeDSL at Perplexity", section "QK normalization": the QK norm of recent
 * Qwen attention layers normalises every head of q and of k (64, 128 or 256
 * elements) with RMS normalisation and a per-head-dimension weight plus a
 * constant weight bias; its kernel computes rms = rsqrt(sum(x^2)/head_dim +
 * EPS) and stores ((w + WEIGHT_BIAS) * (x * rms)) in the element type, in
 * place. (The page's one-line formula omits the reciprocal square root that
 * its kernel applies; the kernel is followed.)
 *   y[h, i] = bf16( (w[i] + bias) * x[h, i] / sqrt(mean_i x[h, i]^2 + eps) )
 * over heads h of x [heads, head_dim] (row-major), real arithmetic, one
 * rounding. w is bfloat16 [head_dim]. Writes y (may equal x). */
void oracle_rmsnorm_heads(const uint16_t* x, long heads, int head_dim, const uint16_t* w,
                          double bias, double eps, uint16_t* y) {
    for (long h = 0; h < heads; ++h) {
        const uint16_t* xr = x + h * (long)head_dim;
        double ss = 0.0;
        for (int i = 0; i < head_dim; ++i) {
            double v = bf16_to_double(xr[i]);
            ss += v * v;
        }
        double inv = 1.0 / sqrt(ss / head_dim + eps);
        for (int i = 0; i < head_dim; ++i) {
            double v = bf16_to_double(xr[i]);
            y[h * (long)head_dim + i] = bf16_round((bf16_to_double(w[i]) + bias) * (v * inv));
        }
    }
}
