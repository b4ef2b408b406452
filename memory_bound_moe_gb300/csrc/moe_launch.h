// Host-side interface between the C-ABI layer (api.cu) and the kernel
// translation units. Not installed; not part of the public ABI.
#pragma once

#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

namespace moe {

// Launch geometry of the routing step, a pure function of (T, E, k).
struct RoutePlan {
    int gs = 32;        // lanes that cooperate on one token (8, 16 or 32)
    int epl = 1;        // experts held per lane: E <= gs * epl
    bool fused = false; // one block does everything (small T)
    int nt = 512;       // threads per block
    int G = 1;          // blocks of the two-kernel path
    int tpc = 0;        // tokens per block
    int tpw = 0;        // tokens per warp (contiguous run inside the block)
    int Ep = 0;         // E rounded up to a multiple of 4 (row stride of the count matrix)
    size_t ws_bytes = 0;
    size_t smem_topk = 0;
    size_t smem_scatter = 0;
};

// nloc: number of counted experts (0 = all E); it sets the count-matrix width.
RoutePlan plan_route(int64_t T, int E, int k, int nloc = 0);

// A local routing: experts [e0, e0 + n) are counted, their segments padded
// to a multiple of pad, perm has `rows` entries.
struct LocalRange {
    int e0, n, pad, rows;
};

cudaError_t launch_route(const RoutePlan& plan, const float* logits, int T, int E, int k,
                         int renorm, int32_t* topk_ids, float* topk_weights,
                         int32_t* expert_counts, int32_t* expert_offsets, int32_t* perm,
                         int32_t* inv_perm, void* workspace, cudaStream_t stream,
                         const LocalRange* local = nullptr);

// One-launch route + expand for decode-sized batches (route_expand.cu).
bool route_expand_fits(const RoutePlan& plan);
cudaError_t launch_route_expand(const RoutePlan& plan, const float* logits, int T, int E, int k,
                                int renorm, int32_t* topk_ids, float* topk_weights,
                                int32_t* expert_counts, int32_t* expert_offsets, int32_t* perm,
                                int32_t* inv_perm, const uint16_t* x, int H, uint16_t* expanded_x,
                                int num_sms, cudaStream_t stream);

// rows: rows of expanded_x (T*k, or a padded local capacity); inv_perm
// entries outside [0, rows) are skipped.
cudaError_t launch_expand(const uint16_t* x, int64_t T, int H, int k, const int32_t* inv_perm,
                          int64_t rows, uint16_t* expanded_x, int num_sms, cudaStream_t stream);

cudaError_t launch_swiglu(const uint16_t* gate_up, int64_t rows, int I, uint16_t* act,
                          int num_sms, cudaStream_t stream);

// rows: rows of expert_out; inv_perm entries outside [0, rows) contribute nothing.
cudaError_t launch_combine(const uint16_t* expert_out, int64_t rows, int64_t T, int H, int k,
                           const float* topk_weights, const int32_t* inv_perm, uint16_t* out,
                           int num_sms, cudaStream_t stream);

// SwiGLU / expand with MXFP8 outputs (quant.cu): codes [rows, n] E4M3 bytes,
// scales [rows, n/32] E8M0 bytes; n (I or H) a multiple of 32.
cudaError_t launch_swiglu_mxfp8(const uint16_t* gate_up, int64_t rows, int I, uint8_t* codes,
                                uint8_t* scales, int num_sms, cudaStream_t stream);
cudaError_t launch_expand_mxfp8(const uint16_t* x, int64_t T, int H, int k, const int32_t* inv_perm,
                                int64_t rows, uint8_t* codes, uint8_t* scales, int num_sms,
                                cudaStream_t stream);
// FP4 outputs: NVFP4 (nvfp4, tensor scale g) or MXFP4.
cudaError_t launch_swiglu_fp4(const uint16_t* gate_up, int64_t rows, int I, bool nvfp4, float g,
                              uint8_t* codes, uint8_t* scales, int num_sms, cudaStream_t stream);
cudaError_t launch_expand_fp4(const uint16_t* x, int64_t T, int H, int k, const int32_t* inv_perm,
                              int64_t rows, bool nvfp4, float g, uint8_t* codes, uint8_t* scales,
                              int num_sms, cudaStream_t stream);

// Per-head RMSNorm of q [T, nq, head_dim] and k [T, nk, head_dim] in place
// (qknorm.cu); head_dim 64, 128 or 256.
cudaError_t launch_qk_rmsnorm(uint16_t* q, uint16_t* k, int64_t T, int nq, int nk, int head_dim,
                              const uint16_t* qw, const uint16_t* kw, float bias, float eps,
                              int num_sms, cudaStream_t stream);

}  // namespace moe
