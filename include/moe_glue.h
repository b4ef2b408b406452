/*
 * moe_glue.h - C ABI of the GB300 (sm_103a) memory-bound MoE glue path.
 *
 * One MoE layer calls, in order:
 *   moe_route   router logits -> top-k experts, weights, per-expert counts and
 *               offsets, and the expert-sorted permutation
 *   moe_expand  token rows -> expert-sorted rows (input of the fc1 GEMM)
 *   moe_swiglu  fc1 output [gate | up] -> silu(gate) * up (input of fc2)
 *   moe_combine fc2 output rows -> weighted sum of each token's k rows
 * The expert GEMMs between these calls are not part of this library.
 *
 * Conventions shared by every entry point
 *   - T tokens, E experts, k experts per token, S = T*k (token, expert) slots.
 *     The flat slot index is s = t*k + j for the j-th expert of token t; the
 *     expert-sorted row index is p.
 *   - bfloat16 tensors are passed as moe_bf16_t (the 16-bit pattern), all
 *     matrices are dense row-major with no padding between rows.
 *   - Every pointer is a DEVICE pointer of the current CUDA device (or
 *     managed memory), allocated and owned by the caller. The library never
 *     allocates, frees or keeps a pointer after the call returns.
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and the call returns before it runs. MOE_OK means "validated and
 *     launched"; a device-side fault surfaces at the caller's next
 *     synchronisation.
 *   - Arguments are validated on the host before anything is launched: on any
 *     error status other than MOE_ERR_CUDA nothing has been enqueued and no
 *     output has been written. MOE_ERR_CUDA reports a failed launch; outputs
 *     are then unspecified.
 *   - Inputs are read-only. Outputs must not overlap any input or each other
 *     (checked from the address ranges; MOE_ERR_INVALID_ARG).
 *   - bfloat16 matrices and the routing workspace must be 16-byte aligned
 *     and every bfloat16 row must be a whole number of 16-byte vectors, i.e.
 *     its width a multiple of 8 elements (MOE_ERR_MISALIGNED): the 128-bit
 *     access rule of the "[FlashInfer] CUTLASS MoE kernel optimisation"
 *     analysis (flashinfer PR #3761), section 3 "Strict memory alignment
 *     validation". int32 and float32 arrays need their natural 4-byte
 *     alignment.
 *   - A zero-sized batch (T = 0 or rows = 0) is valid; pointers of empty
 *     arrays may then be NULL.
 *   - The functions are thread-safe and keep no mutable global state apart
 *     from a per-device cache of the SM count. The one exception is
 *     moe_route_static, whose calls share one static scratch array and so
 *     must not overlap on the GPU (see its comment below).
 *
 * Page citations name the page title and section; the pages themselves
 * state no formulas, so the definitions below are the plain readings
 * (softmax over all experts, top-k on logits with the lower index first on
 * ties, renormalisation over the k chosen, stable expert order, gate in the
 * first half of the fc1 row).
 */
#ifndef MOE_GLUE_H
#define MOE_GLUE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Identical to cudaStream_t; declared here so the header needs no CUDA headers. */
typedef struct CUstream_st* moe_stream_t;

/* A bfloat16 value as its IEEE bit pattern (sign, 8 exponent, 7 fraction bits). */
typedef uint16_t moe_bf16_t;

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,  /* negative size, k < 1, k > E, NULL pointer, overlapping buffers */
    MOE_ERR_MISALIGNED = 2,   /* pointer not 16-byte aligned or row not a multiple of 16 bytes */
    MOE_ERR_UNSUPPORTED = 3,  /* E > MOE_MAX_EXPERTS, k > MOE_MAX_TOPK, T*k >= 2^31 */
    MOE_ERR_WORKSPACE = 4,    /* workspace smaller than moe_route_workspace_size() */
    MOE_ERR_CUDA = 5          /* a CUDA launch failed (see cudaGetLastError semantics) */
} moe_status_t;

#define MOE_MAX_EXPERTS 1024
#define MOE_MAX_TOPK 16

/* Human-readable name of a status code. Never NULL; static storage. */
const char* moe_status_string(moe_status_t status);

/*
 * Bytes of device workspace moe_route needs for (T, E, k); 0 when the
 * single-block path applies (small T). A pure function of its arguments.
 * Errors: MOE_ERR_INVALID_ARG (bytes NULL, T < 0, E < 1, k < 1, k > E),
 * MOE_ERR_UNSUPPORTED (E > MOE_MAX_EXPERTS, k > MOE_MAX_TOPK, T*k >= 2^31).
 */
moe_status_t moe_route_workspace_size(int64_t T, int E, int k, size_t* bytes);

/*
 * Top-k routing and the expert-sorted permutation.
 * "CuTeDSL at Perplexity", section "Mixture of Experts (MoE) dispatch/combine",
 * sub-section "Local": from the routing table, count the tokens assigned to
 * each expert and give every token a unique index inside its expert's list;
 * the prefill variant counts per block and aggregates the counts of all
 * blocks in global memory to place each token.
 *
 * For each token t, with l = logits[t, 0..E-1] (float32, row-major [T, E]):
 *   softmax   p_e = exp(l_e - max l) / sum_e' exp(l_e' - max l), over all E
 *   top-k     topk_ids[t, 0..k-1] = the k experts with the largest logits in
 *             descending order; equal logits (-0.0 == +0.0) go lower index
 *             first. Selection compares the float32 logits, so it is exact.
 *   weights   topk_weights[t, j] = p_{id_j}                      (renorm == 0)
 *                                = p_{id_j} / sum_j' p_{id_j'}   (renorm != 0)
 *             computed in float32.
 * Over the S = T*k slots s = t*k + j with expert e_s = topk_ids[s]:
 *   expert_counts[e]  = #{ s : e_s = e }                            [E]
 *   expert_offsets[e] = sum_{e' < e} expert_counts[e'];
 *   expert_offsets[E] = S                                           [E + 1]
 *   inv_perm[s] = p   = expert_offsets[e_s] + #{ s' < s : e_s' = e_s }   [S]
 *   perm[p]     = s                                                      [S]
 * The permutation is deterministic (stable in s): bit-identical run to run.
 *
 * Outputs topk_ids [T, k] int32, topk_weights [T, k] float32, expert_counts,
 * expert_offsets, perm and inv_perm (int32) are written in full.
 * workspace: device scratch of at least moe_route_workspace_size(T, E, k)
 * bytes, 16-byte aligned (may be NULL when that size is 0); its contents on
 * entry are ignored and on return are unspecified. Calls that share a
 * workspace must be ordered (same stream or synchronised).
 * Logits are assumed finite; NaN logits give unspecified (but in-bounds)
 * results. T = 0 writes zero counts and offsets.
 */
moe_status_t moe_route(const float* logits, int64_t T, int E, int k, int renorm,
                       int32_t* topk_ids, float* topk_weights,
                       int32_t* expert_counts, int32_t* expert_offsets,
                       int32_t* perm, int32_t* inv_perm,
                       void* workspace, size_t workspace_bytes,
                       moe_stream_t stream);

/*
 * Routing and row expansion as one call: the same outputs as moe_route
 * followed by moe_expand (bit-identical), with the argument rules of both.
 * "CuTeDSL at Perplexity", section "Mixture of Experts (MoE) dispatch/combine",
 * sub-section "Local", and section "Grid synchronization": for decode-sized
 * batches the pages fuse routing and token copy into one launch and choose
 * between that and separate route + copy kernels on the host.
 *
 * When moe_route_workspace_size(T, E, k) is 0 (decode-sized T: at most 32
 * tokens for E > 16, 64 for E <= 16, 128 for E <= 8) this is ONE kernel
 * launch: every block routes the whole batch in shared memory (block 0
 * writes the routing outputs) and copies its share of the rows, with no
 * grid-wide synchronisation. Otherwise it launches the moe_route kernels and
 * then the moe_expand kernel on the same stream, and `workspace` must be as
 * for moe_route.
 */
moe_status_t moe_route_expand(const float* logits, int64_t T, int E, int k, int renorm,
                              const moe_bf16_t* x, int H,
                              int32_t* topk_ids, float* topk_weights,
                              int32_t* expert_counts, int32_t* expert_offsets,
                              int32_t* perm, int32_t* inv_perm, moe_bf16_t* expanded_x,
                              void* workspace, size_t workspace_bytes,
                              moe_stream_t stream);

/*
 * moe_route without a caller-provided workspace: the same computation,
 * outputs, validation and status codes as moe_route, with the routing
 * scratch held in a device array inside the library. The pages have no
 * counterpart of this entry point.
 *
 * Some callers cannot allocate device memory where they route: a runtime
 * that plans and owns all device memory at start-up and forbids allocation
 * afterwards, an allocator-free plugin or embedding host, or a call site that
 * cannot tolerate cudaMalloc's possible implicit synchronisation. moe_route
 * would need such a caller to find a workspace for it; this entry point needs
 * none and calls no allocating routine.
 *
 *   - The scratch is one static device array of MOE_ROUTE_STATIC_SCRATCH_BYTES
 *     (128 KiB); every device that loads the library reserves it until the
 *     process exits. Sizes whose workspace (moe_route_workspace_size) exceeds
 *     it are rejected with MOE_ERR_WORKSPACE before anything is launched; no
 *     size accepted by moe_route currently needs more than 128 KiB.
 *   - Every call looks up the array's device address in the current CUDA
 *     context (cudaGetSymbolAddress, which allocates nothing), so the
 *     address stays right after cudaDeviceReset or with another context
 *     current. The first call in a context may load the library's device
 *     code into it: make that first call before any stream capture on that
 *     device.
 *   - All calls share the one array and it keeps whatever the last call left
 *     there. Nothing in it has to start at zero: each call writes every entry
 *     it later reads. Calls that can overlap on the GPU (different streams
 *     without ordering between them, or several host threads) race on the
 *     array and give wrong results; order them.
 */
#define MOE_ROUTE_STATIC_SCRATCH_BYTES (128u * 1024u)

moe_status_t moe_route_static(const float* logits, int64_t T, int E, int k, int renorm,
                              int32_t* topk_ids, float* topk_weights,
                              int32_t* expert_counts, int32_t* expert_offsets,
                              int32_t* perm, int32_t* inv_perm,
                              moe_stream_t stream);

/*
 * Local routing for one tensor-parallel rank: experts [e0, e1) only, with
 * every local expert's segment padded to a multiple of pad.
 * "CuTeDSL at Perplexity", section "Mixture of Experts (MoE) dispatch/combine",
 * sub-section "Single node": with tensor parallelism the routing information
 * and the tokens are replicated; a rank's dispatch routes only the tokens
 * assigned to the experts it holds (the local kernel reused with a small
 * change), its combine sums the local copies and an all-reduce across ranks
 * adds the partial results. Sub-section "Local": the tokens go to an
 * optionally padded buffer for the MoE GEMM.
 *
 * The top-k runs over all E experts, so topk_ids/topk_weights are exactly
 * those of moe_route. With n = e1 - e0 and local slots s (e_s in [e0, e1)):
 *   expert_counts[l]  = #{ local s : e_s = e0 + l }                    [n]
 *   expert_offsets[0] = 0, expert_offsets[l+1] = expert_offsets[l] +
 *                       pad * ceil(expert_counts[l] / pad)               [n + 1]
 *   inv_perm[s]       = expert_offsets[e_s - e0] + #{ local s' < s with
 *                       the same expert }, or -1 if e_s is not local    [T*k]
 *   perm[p]           = s for those rows and -1 for every other row     [rows]
 * where rows = moe_route_local_rows(T, k, e0, e1, pad) = T*k + n*(pad-1),
 * the most rows a padded local buffer can need. With e0 = 0, e1 = E, pad = 1
 * every output equals moe_route's. workspace: at least
 * moe_route_local_workspace_size(T, E, k, e0, e1) bytes (0: may be NULL).
 * Use moe_expand_rows / moe_combine_rows with `rows` rows; the combine then
 * yields this rank's partial sum (slots with inv_perm -1 contribute nothing).
 * Errors: as moe_route, plus MOE_ERR_INVALID_ARG unless 0 <= e0 < e1 <= E
 * and pad >= 1, MOE_ERR_UNSUPPORTED if rows >= 2^31.
 */
moe_status_t moe_route_local_rows(int64_t T, int k, int e0, int e1, int pad, int64_t* rows);
moe_status_t moe_route_local_workspace_size(int64_t T, int E, int k, int e0, int e1,
                                            size_t* bytes);
moe_status_t moe_route_local(const float* logits, int64_t T, int E, int k, int renorm,
                             int e0, int e1, int pad,
                             int32_t* topk_ids, float* topk_weights,
                             int32_t* expert_counts, int32_t* expert_offsets,
                             int32_t* perm, int32_t* inv_perm,
                             void* workspace, size_t workspace_bytes,
                             moe_stream_t stream);

/*
 * Row expansion into expert order (expandInputRows).
 * "CuTeDSL at Perplexity", section "Mixture of Experts (MoE) dispatch/combine",
 * sub-section "Local" (tokens are copied to the buffer the MoE GEMM reads),
 * and "[FlashInfer] CUTLASS MoE kernel optimisation", section 1 "Explicit
 * vectorization" (expandInputRowsKernel, 128-bit loads and stores).
 *
 *   expanded_x[inv_perm[t*k + j], :] = x[t, :]   for all t < T, j < k
 * i.e. expanded_x[p, :] = x[perm[p] / k, :]: a bit copy of bfloat16 rows.
 * x [T, H], inv_perm [T*k] (a permutation of 0..S-1, as moe_route writes
 * it), expanded_x [S, H]. H must be a multiple of 8. Entries of inv_perm
 * outside [0, S) are skipped (their rows are not written); if inv_perm is not
 * a permutation some rows stay unwritten.
 */
moe_status_t moe_expand(const moe_bf16_t* x, int64_t T, int H, int k,
                        const int32_t* inv_perm, moe_bf16_t* expanded_x,
                        moe_stream_t stream);

/*
 * moe_expand into a buffer of `rows` rows (a padded local buffer): entries of
 * inv_perm outside [0, rows), such as the -1 of slots another rank holds, are
 * skipped, and rows no slot maps to (padding) are left as they are.
 */
moe_status_t moe_expand_rows(const moe_bf16_t* x, int64_t T, int H, int k,
                             const int32_t* inv_perm, int64_t rows, moe_bf16_t* expanded_x,
                             moe_stream_t stream);

/*
 * Gated SwiGLU activation (doActivation).
 * "[FlashInfer] CUTLASS MoE kernel optimisation", section 1 "Explicit
 * vectorization" and section 2 "Dynamic threads" (doActivationKernel over the
 * fc1 output, block size chosen from the intermediate size).
 *
 *   act[r, i] = bf16_rn( silu(g) * u ),  g = gate_up[r, i], u = gate_up[r, I + i],
 *   silu(g) = g / (1 + exp(-g)),  computed in float32, rounded once to
 *   bfloat16 (nearest, ties to even).
 * gate_up [rows, 2I] (gate = first I columns, up = last I), act [rows, I].
 * I must be a multiple of 8.
 */
moe_status_t moe_swiglu(const moe_bf16_t* gate_up, int64_t rows, int I,
                        moe_bf16_t* act, moe_stream_t stream);

/*
 * Weighted top-k combine / unpermute.
 * "CuTeDSL at Perplexity", section "Mixture of Experts (MoE) dispatch/combine",
 * sub-section "Local" (the combine kernel uses the token positions from the
 * routing step, accumulates in registers and writes the final token) and the
 * same section's note that combine is a vectorised accumulation.
 *
 *   out[t, :] = bf16_rn( sum_{j=0}^{k-1} topk_weights[t, j] *
 *                        expert_out[inv_perm[t*k + j], :] )
 * accumulated in float32 in order j = 0..k-1, rounded once.
 * expert_out [S, H], topk_weights [T, k] float32, inv_perm [T*k], out [T, H].
 * H must be a multiple of 8. Entries of inv_perm outside [0, S) contribute
 * nothing.
 */
moe_status_t moe_combine(const moe_bf16_t* expert_out, int64_t T, int H, int k,
                         const float* topk_weights, const int32_t* inv_perm,
                         moe_bf16_t* out, moe_stream_t stream);

/*
 * moe_combine over an expert_out of `rows` rows (a padded local buffer):
 * entries of inv_perm outside [0, rows), such as -1, contribute nothing, so
 * after moe_route_local the result is this rank's partial sum, to be added
 * across ranks (the all-reduce is not part of this library).
 */
moe_status_t moe_combine_rows(const moe_bf16_t* expert_out, int64_t rows, int64_t T, int H, int k,
                              const float* topk_weights, const int32_t* inv_perm,
                              moe_bf16_t* out, moe_stream_t stream);

/*
 * MXFP8 outputs for the next expert GEMM.
 * "CuTeDSL at Perplexity", section "Blackwell support": Blackwell supports
 * MXFP8 / MXFP4 / NVFP4 in hardware and the kernels were adapted for FP8
 * block-wise scaling, with absolute maxima over 32-element (MX) blocks.
 * Block format (OCP Microscaling v1.0, MXFP8 E4M3): for every 32 consecutive
 * values of a row with largest magnitude amax,
 *   X = floor(log2 amax) - 8, clamped to [-127, 127] (-127 if amax = 0)
 *   scale byte (E8M0) = X + 127;  code = E4M3(v * 2^-X), round to nearest
 *   even, saturated to +-448.  Dequantized value: E4M3(code) * 2^X.
 * codes [rows, n] bytes (16-byte aligned), scales [rows, n/32] bytes, both
 * row-major; n (I or H) must be a multiple of 32 (MOE_ERR_MISALIGNED).
 * The values quantized are the bfloat16 values moe_swiglu / moe_expand would
 * store. Inputs are assumed finite.
 *
 * moe_swiglu_mxfp8: act = silu(gate) * up as moe_swiglu, then quantized.
 * moe_expand_mxfp8: token rows quantized once and written to the k rows
 *   inv_perm[t*k + j] < rows of the code and scale buffers (rows as for
 *   moe_expand_rows: T*k, or a padded local capacity).
 */
moe_status_t moe_swiglu_mxfp8(const moe_bf16_t* gate_up, int64_t rows, int I,
                              uint8_t* act_codes, uint8_t* act_scales, moe_stream_t stream);
moe_status_t moe_expand_mxfp8(const moe_bf16_t* x, int64_t T, int H, int k,
                              const int32_t* inv_perm, int64_t rows,
                              uint8_t* codes, uint8_t* scales, moe_stream_t stream);

/*
 * FP4 outputs for the next expert GEMM, fused into SwiGLU and row expansion.
 * "CuTeDSL at Perplexity", section "Blackwell support": besides MXFP8,
 * Blackwell supports MXFP4 and NVFP4 in hardware, and the kernels compute
 * the absolute maximum over 32 (MXFP4) or 16 (NVFP4) values with sub-warp
 * reductions. Element: E2M1 (OCP Microscaling v1.0; magnitudes 0, 0.5, 1,
 * 1.5, 2, 3, 4, 6), a real rounded to nearest, ties to the even code,
 * saturating to +-6, sign kept (a negative value rounding to 0 is code 0x8).
 *
 *   MOE_FP4_MXFP4 (OCP MX v1.0): per 32 values with largest magnitude amax,
 *     X = floor(log2 amax) - 2 clamped to [-127, 127] (-127 if amax = 0);
 *     scale byte (E8M0) = X + 127; code = E2M1(v * 2^-X); value = E2M1 * 2^X.
 *     global_scale is ignored.
 *   MOE_FP4_NVFP4 (NVIDIA's format): per 16 values, with the float32 tensor
 *     scale g = global_scale (finite, > 0; e.g. 448 * 6 / the tensor's amax),
 *     scale byte (E4M3) = E4M3(fl(fl(g * amax) / 6)) of value s, round to
 *     nearest even, saturating to 448; code = E2M1(fl(v * fl(g / s))), 0 if
 *     s = 0; fl() is one float32 rounding. value = E2M1 * s / g.
 *
 * codes [rows, n/2] bytes, two codes per byte, element 2i in the LOW nibble
 * (16-byte aligned); scales [rows, n/32] (MXFP4) or [rows, n/16] (NVFP4)
 * bytes; both row-major. n (I or H) must be a multiple of the block
 * (MOE_ERR_MISALIGNED); an unknown format or a bad NVFP4 scale is
 * MOE_ERR_INVALID_ARG. The values quantized are the bfloat16 values
 * moe_swiglu / moe_expand would store. Inputs are assumed finite.
 *
 * moe_swiglu_fp4: act = silu(gate) * up as moe_swiglu, then quantized.
 * moe_expand_fp4: token rows quantized once and written to the k rows
 *   inv_perm[t*k + j] < rows (rows as for moe_expand_rows).
 */
#define MOE_FP4_NVFP4 0
#define MOE_FP4_MXFP4 1
moe_status_t moe_swiglu_fp4(const moe_bf16_t* gate_up, int64_t rows, int I, int format,
                            float global_scale, uint8_t* act_codes, uint8_t* act_scales,
                            moe_stream_t stream);
moe_status_t moe_expand_fp4(const moe_bf16_t* x, int64_t T, int H, int k,
                            const int32_t* inv_perm, int64_t rows, int format,
                            float global_scale, uint8_t* codes, uint8_t* scales,
                            moe_stream_t stream);

/*
 * QK RMSNorm, in place, for the attention layer of the same models.
 * "CuTeDSL at Perplexity", section "QK normalization": recent Qwen models
 * normalise every head of q and of k (64, 128 or 256 elements) with RMS
 * normalisation, a per-dimension weight and a constant weight bias; the
 * page's kernel stores ((w + bias) * (x * rsqrt(sum(x^2)/head_dim + eps))).
 *
 *   q[t, h, :] = bf16_rn( (q_weight + weight_bias) * q[t, h, :] * r ),
 *   r = 1 / sqrt(mean(q[t, h, :]^2) + eps)   (float32), likewise k with k_weight.
 * q [T, num_q_heads, head_dim], k [T, num_k_heads, head_dim] (bfloat16,
 * row-major, 16-byte aligned; either head count may be 0 and its pointer
 * then NULL), q_weight / k_weight [head_dim]. head_dim must be 64, 128 or 256
 * (MOE_ERR_UNSUPPORTED). q and k must not overlap the weights.
 */
moe_status_t moe_qk_rmsnorm(moe_bf16_t* q, moe_bf16_t* k, int64_t T, int num_q_heads,
                            int num_k_heads, int head_dim, const moe_bf16_t* q_weight,
                            const moe_bf16_t* k_weight, float weight_bias, float eps,
                            moe_stream_t stream);

#ifdef __cplusplus
}  /* extern "C" */
#endif

#endif  /* MOE_GLUE_H */
