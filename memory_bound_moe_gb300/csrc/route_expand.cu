// Decode-sized routing and row expansion in ONE launch.
//
// "CuTeDSL at Perplexity", section "Mixture of Experts (MoE) dispatch/combine",
// sub-section "Local", and section "Grid synchronization": for few tokens the
// dispatch routes in one block, signals the rest of the grid through a grid
// barrier and lets every block copy a chunk of tokens, all in one launch; a
// host-side check picks this decode kernel when the copy needs fewer blocks
// than there are SMs and the separate route + copy kernels otherwise.
//
// Here the grid barrier is replaced by redundancy: the routing of a decode
// batch (T <= 32 tokens for E > 16) reads at most a few tens of KB of logits
// from L2, so EVERY block routes the whole batch in its own shared memory and
// only block 0 writes the routing outputs. Nothing waits on another block, so
// there is no spin, no cooperative launch and no co-residency requirement.
// Each block first loads the x vectors it will copy, so those loads overlap
// the routing, then stores each one to its token's k expert-sorted rows.
// The results are bit-identical to moe_route followed by moe_expand.
#include "moe_device.cuh"
#include "moe_launch.h"
#include "route_device.cuh"
#include "rows_common.cuh"

namespace moe {
namespace {

constexpr int kNt = 512;

template <int GS, int EPL, int VB>
__global__ void __launch_bounds__(kNt) route_expand_kernel(RouteArgs a, const uint8_t* __restrict__ x,
                                                           uint8_t* __restrict__ out, uint32_t items,
                                                           uint32_t per_block, DivU32 nv,
                                                           uint32_t row_bytes) {
    constexpr int NW = kNt / kWarp;
    extern __shared__ int32_t smem[];
    int32_t* s_cnt = smem;                      // [NW][E]
    int32_t* s_tot = s_cnt + (size_t)NW * a.nloc;  // [Ep] totals, then offsets
    int32_t* s_warp = s_tot + a.Ep;             // [32]
    int32_t* s_inv = s_warp + 32;               // [T*k] sorted row of every slot
    pdl_wait_and_release();

    // This block's first copy item per thread, loaded before the routing.
    const uint32_t i0 = blockIdx.x * per_block;
    const uint32_t i1 = min(items, i0 + per_block);
    const uint32_t v = i0 + threadIdx.x;
    const bool have = v < i1;
    Bits<VB> val;
    uint32_t tok = 0, col = 0;
    if (have) {
        tok = nv.div(v);
        col = v - tok * nv.d;
        ld_stream(val, x + uint64_t(tok) * row_bytes + uint64_t(col) * VB);
    }

    RouteArgs la = a;
    la.write_out = blockIdx.x == 0;
    zero_warp_counters(s_cnt, a.nloc);
    int re[kRegRounds], rr[kRegRounds];
    topk_rank_range<GS, EPL, kNt>(la, 0, a.T, s_cnt, re, rr);
    __syncthreads();
    scan_over_warps<kNt>(s_cnt, s_tot, a.nloc);
    __syncthreads();
    if (la.write_out)
        for (int e = threadIdx.x; e < a.E; e += kNt) a.expert_counts[e] = s_tot[e];
    block_exclusive_scan<kNt>(s_tot, s_tot, a.E, s_warp);
    if (la.write_out) {
        for (int e = threadIdx.x; e < a.E; e += kNt) a.expert_offsets[e] = s_tot[e];
        if (threadIdx.x == 0) a.expert_offsets[a.E] = a.T * a.k;
    }
    finish_ranks<GS, kNt, true>(la, 0, a.T, s_cnt, s_tot, re, rr, s_inv);
    __syncthreads();

    const uint32_t S = uint32_t(a.T * a.k);
    if (have) {
        for (int j = 0; j < a.k; ++j) {
            const uint32_t p = uint32_t(s_inv[tok * a.k + j]);
            if (p < S) st_global(out + uint64_t(p) * row_bytes + uint64_t(col) * VB, val);
        }
    }
    for (uint32_t w = v + kNt; w < i1; w += kNt) {   // more than one item per thread
        const uint32_t t = nv.div(w);
        const uint32_t c = w - t * nv.d;
        Bits<VB> u;
        ld_stream(u, x + uint64_t(t) * row_bytes + uint64_t(c) * VB);
        for (int j = 0; j < a.k; ++j) {
            const uint32_t p = uint32_t(s_inv[t * a.k + j]);
            if (p < S) st_global(out + uint64_t(p) * row_bytes + uint64_t(c) * VB, u);
        }
    }
}

template <int GS, int EPL, int VB>
cudaError_t launch_t(const RouteArgs& a, const uint16_t* x, int H, uint16_t* out, int num_sms,
                     cudaStream_t stream) {
    auto kernel = route_expand_kernel<GS, EPL, VB>;
    const uint32_t nv = uint32_t(uint64_t(H) * 2 / VB);
    const uint32_t items = uint32_t(a.T) * nv;
    const uint32_t blocks = std::max<uint32_t>(1, std::min<uint32_t>(uint32_t(num_sms), items));
    const uint32_t per_block = (items + blocks - 1) / blocks;
    const size_t smem = sizeof(int32_t) * (size_t(kNt / kWarp) * a.E + a.Ep + 32 + size_t(a.T) * a.k);
    if (smem > 48 * 1024) {
        const cudaError_t err =
            cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
        if (err != cudaSuccess) return err;
    }
    return launch_pdl(kernel, dim3(blocks), dim3(kNt), smem, stream, a,
                      reinterpret_cast<const uint8_t*>(x), reinterpret_cast<uint8_t*>(out), items,
                      per_block, DivU32::make(nv), uint32_t(2 * int64_t(H)));
}

template <int GS, int EPL>
cudaError_t launch_gs(const RouteArgs& a, const uint16_t* x, int H, uint16_t* out, int num_sms,
                      cudaStream_t stream) {
    if (can_use_32b(uint64_t(H) * 2, {x, out}))
        return launch_t<GS, EPL, 32>(a, x, H, out, num_sms, stream);
    return launch_t<GS, EPL, 16>(a, x, H, out, num_sms, stream);
}

}  // namespace

bool route_expand_fits(const RoutePlan& plan) {
    // one-block routing plan with every warp's tokens in register rounds
    return plan.fused && plan.nt == kNt &&
           plan.tpw / (kWarp / plan.gs) <= kRegRounds;
}

cudaError_t launch_route_expand(const RoutePlan& plan, const float* logits, int T, int E, int k,
                                int renorm, int32_t* topk_ids, float* topk_weights,
                                int32_t* expert_counts, int32_t* expert_offsets, int32_t* perm,
                                int32_t* inv_perm, const uint16_t* x, int H, uint16_t* expanded_x,
                                int num_sms, cudaStream_t stream) {
    if (!route_expand_fits(plan)) return cudaErrorNotSupported;
    RouteArgs a;
    a.logits = logits;
    a.T = T; a.E = E; a.k = k; a.renorm = renorm;
    a.e0 = 0; a.nloc = E; a.pad = 1; a.rows = T * k;
    a.Ep = plan.Ep; a.tpc = plan.tpc; a.tpw = plan.tpw; a.G = 1;
    a.topk_ids = topk_ids; a.topk_weights = topk_weights;
    a.expert_counts = expert_counts; a.expert_offsets = expert_offsets;
    a.perm = perm; a.inv_perm = inv_perm;
    a.ws_counts = nullptr;
    a.write_out = true;
    a.vec4 = E % 4 == 0 && reinterpret_cast<uintptr_t>(logits) % 16 == 0;
    switch (plan.gs * 100 + plan.epl) {
        case 801: return launch_gs<8, 1>(a, x, H, expanded_x, num_sms, stream);
        case 1601: return launch_gs<16, 1>(a, x, H, expanded_x, num_sms, stream);
        case 3201: return launch_gs<32, 1>(a, x, H, expanded_x, num_sms, stream);
        case 3202: return launch_gs<32, 2>(a, x, H, expanded_x, num_sms, stream);
        case 3204: return launch_gs<32, 4>(a, x, H, expanded_x, num_sms, stream);
        case 3208: return launch_gs<32, 8>(a, x, H, expanded_x, num_sms, stream);
        case 3216: return launch_gs<32, 16>(a, x, H, expanded_x, num_sms, stream);
        case 3232: return launch_gs<32, 32>(a, x, H, expanded_x, num_sms, stream);
        default: return cudaErrorInvalidConfiguration;
    }
}

}  // namespace moe
