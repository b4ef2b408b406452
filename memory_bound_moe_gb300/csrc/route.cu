// Routing: softmax + top-k per token, per-expert histogram, exclusive scan and
// the stable expert-sorted permutation.
//
// "CuTeDSL at Perplexity", section "Mixture of Experts (MoE) dispatch/combine",
// sub-section "Local": the routing step counts the tokens of every expert and
// gives each token a unique index inside its expert's list. For many tokens
// the pages count per block in shared memory and aggregate the block counts in
// global memory; for few tokens one block routes everything. Both shapes are
// kept here, with one change: the pages hand out indices with shared-memory
// atomics, whose order is not reproducible, while these kernels rank slots in
// flat slot order (s = t*k + j) so the permutation is deterministic.
//
//   two-kernel path  route_rank_kernel    G blocks, each a contiguous token
//                                         range: top-k and weights, the rank of
//                                         every slot among the block's slots of
//                                         the same expert (kept in inv_perm),
//                                         and the block's histogram (row b of
//                                         the count matrix in the workspace)
//                    route_place_kernel   G blocks: reduce the count matrix
//                                         (totals; prefix of earlier blocks),
//                                         scan the totals into offsets, place
//                                         each slot at offset + prefix + rank
//   one-block path   route_fused_kernel   both in one block (small T)
//
// Ranking inside a block: warp w owns a contiguous run of the block's tokens
// and keeps per-expert counters cnt[w][e] in shared memory. In every round a
// warp finishes the top-k of one token per lane group; lanes holding a pick
// are in slot order, so __match_any_sync on the expert gives each pick its
// rank among same-expert picks of the round (the popcount of lower peers),
// added to cnt[w][e]. After all rounds an exclusive scan over warps turns the
// counters into per-warp starts, added to every slot's rank.
#include "moe_device.cuh"
#include "moe_launch.h"
#include "route_device.cuh"
#include "rows_common.cuh"

#include <algorithm>

namespace moe {
namespace {

template <int GS, int EPL, int NT, bool LOCAL, int N>
__global__ void __launch_bounds__(NT) route_rank_kernel(RouteArgs a) {
    constexpr int NW = NT / kWarp;
    extern __shared__ int32_t smem[];
    int32_t* s_cnt = smem;                         // [NW][nloc]
    int32_t* s_tot = s_cnt + (size_t)NW * a.nloc;  // [Ep]
    // this block's tokens (64-bit products: b * tpc may pass 2^31 for huge T)
    const int t0 = int(min(int64_t(a.T), int64_t(blockIdx.x) * a.tpc));
    const int t1 = int(min(int64_t(a.T), int64_t(t0) + a.tpc));
    // Warm L2 with this block's logit rows before waiting for the kernel
    // that produced them (a prefetch carries no data into the kernel).
    if (a.vec4 && t1 > t0) {
        constexpr uint64_t kPiece = 16384;
        const uint8_t* base = reinterpret_cast<const uint8_t*>(a.logits + (size_t)t0 * a.E);
        const uint64_t bytes = uint64_t(t1 - t0) * a.E * sizeof(float);
        for (uint64_t off = uint64_t(threadIdx.x) * kPiece; off < bytes; off += uint64_t(NT) * kPiece)
            prefetch_l2(base + off, uint32_t(min(kPiece, bytes - off)));
    }
    pdl_wait_and_release();
    zero_warp_counters(s_cnt, a.nloc);
    // rounds held in registers: the wide blocks give every warp one token
    constexpr int R = NT > 512 ? 1 : kRegRounds;
    int re[R], rr[R];
    topk_rank_range<GS, EPL, NT, LOCAL, N, R>(a, t0, t1, s_cnt, re, rr);
    __syncthreads();
    scan_over_warps<NT>(s_cnt, s_tot, a.nloc);
    for (int e = a.nloc + threadIdx.x; e < a.Ep; e += NT) s_tot[e] = 0;
    __syncthreads();
    int32_t* row = a.ws_counts + (size_t)blockIdx.x * a.Ep;
    for (int e = threadIdx.x; e < a.Ep; e += NT) row[e] = s_tot[e];
    finish_ranks<GS, NT, false, LOCAL, R>(a, t0, t1, s_cnt, nullptr, re, rr);
}

// The place kernel's split of the count matrix: column groups of 4 experts
// (int4), padded to a power of two below a warp so that the lanes of a warp
// sharing a column group are a shuffle butterfly apart; row groups (one per
// thread and column group); and the partial rows left after the in-warp sum.
struct PlaceSplit {
    int CG, CGp, R, LPW, Rp;
};
__host__ __device__ inline PlaceSplit place_split(int Ep, int nt) {
    PlaceSplit q;
    q.CG = Ep / 4;
    q.CGp = q.CG;
    if (q.CG < kWarp) {
        q.CGp = 1;
        while (q.CGp < q.CG) q.CGp <<= 1;
    }
    q.R = q.CGp >= nt ? 1 : nt / q.CGp;
    q.LPW = q.CGp < kWarp ? kWarp / q.CGp : 1;
    q.Rp = q.R / q.LPW;
    return q;
}

// Offsets from the block's expert totals s_tot[0..nloc): the exclusive scan
// of the counts, each rounded up to a multiple of pad for a local routing.
// Writes s_off[0..nloc] (s_off[nloc] = total rows used) and, when `out`,
// expert_counts and expert_offsets. Block-wide; returns the total.
template <int NT, bool LOCAL>
__device__ __forceinline__ int compute_offsets(const RouteArgs& a, const int32_t* s_tot, int32_t* s_off,
                                              int32_t* s_warp, bool out) {
    for (int e = threadIdx.x; e < a.nloc; e += NT) {
        const int c = s_tot[e];
        if (out) a.expert_counts[e] = c;
        s_off[e] = LOCAL ? (c + a.pad - 1) / a.pad * a.pad : c;
    }
    __syncthreads();
    const int total = block_exclusive_scan<NT>(s_off, s_off, a.nloc, s_warp);
    if (threadIdx.x == 0) s_off[a.nloc] = total;
    for (int e = threadIdx.x; e < a.nloc; e += NT)
        if (out) a.expert_offsets[e] = s_off[e];
    if (out && threadIdx.x == 0) a.expert_offsets[a.nloc] = total;
    __syncthreads();
    return total;
}

// Offsets by one warp (lane l scans a contiguous run of experts) from the
// expert totals s_tot[0..nloc): the exclusive scan of the counts, each rounded
// up to a multiple of pad for a local routing. Writes s_off[0..nloc]
// (s_off[nloc] = total rows used), adds the offsets to s_base and, when `out`,
// writes expert_counts and expert_offsets.
template <bool LOCAL>
__device__ __forceinline__ void warp_offsets(const RouteArgs& a, const int32_t* s_tot, int32_t* s_off,
                                             int32_t* s_base, bool out) {
    const int lane = threadIdx.x % kWarp;
    const int per = (a.nloc + kWarp - 1) / kWarp;
    const int e0 = lane * per;
    const int e1 = min(a.nloc, e0 + per);
    auto rows_of = [&](int c) { return LOCAL ? (c + a.pad - 1) / a.pad * a.pad : c; };
    int local = 0;
    for (int e = e0; e < e1; ++e) local += rows_of(s_tot[e]);
    int x = local;
#pragma unroll
    for (int o = 1; o < kWarp; o <<= 1) {
        const int y = __shfl_up_sync(kFull, x, o);
        if (lane >= o) x += y;
    }
    const int total = __shfl_sync(kFull, x, kWarp - 1);
    int run = x - local;
    for (int e = e0; e < e1; ++e) {
        const int c = s_tot[e];
        s_off[e] = run;
        s_base[e] += run;
        if (out) {
            a.expert_counts[e] = c;
            a.expert_offsets[e] = run;
        }
        run += rows_of(c);
    }
    if (lane == 0) {
        s_off[a.nloc] = total;
        if (out) a.expert_offsets[a.nloc] = total;
    }
}

// perm = -1 on the padding rows of local experts l = l0, l0 + dl, ... and on
// the rows [total + r0, rows) in steps of dr (block-strided by the caller).
template <int NT>
__device__ __forceinline__ void fill_padding(const RouteArgs& a, const int32_t* s_tot, const int32_t* s_off,
                                             int l0, int dl, int r0, int dr) {
    for (int l = l0; l < a.nloc; l += dl)
        for (int q = s_off[l] + s_tot[l] + threadIdx.x; q < s_off[l + 1]; q += NT) a.perm[q] = -1;
    for (int q = s_off[a.nloc] + r0 + threadIdx.x; q < a.rows; q += dr) a.perm[q] = -1;
}

template <int NT, bool LOCAL>
__global__ void __launch_bounds__(NT) route_place_kernel(RouteArgs a) {
    extern __shared__ int32_t smem[];
    const int Ep = a.Ep;
    const PlaceSplit q = place_split(Ep, NT);
    int32_t* s_ptot = smem;                 // [Rp][Ep]
    int32_t* s_ppre = s_ptot + q.Rp * Ep;   // [Rp][Ep]
    int32_t* s_tot = s_ppre + q.Rp * Ep;    // [Ep]
    int32_t* s_base = s_tot + Ep;           // [Ep]
    int32_t* s_off = s_base + Ep;           // [Ep + 4]
    const int b = blockIdx.x;
    pdl_wait_and_release();

    // This thread's first slot, read before the count matrix so that both
    // loads are in flight together.
    const int s0 = int(min(int64_t(a.T), int64_t(b) * a.tpc)) * a.k;
    const int s1 = int(min(int64_t(a.T), int64_t(b + 1) * a.tpc)) * a.k;
    const int sf = s0 + threadIdx.x;
    int ef = 0, rf = 0;
    if (sf < s1) {
        ef = __ldcg(a.topk_ids + sf);
        rf = __ldcg(a.inv_perm + sf);
    }

    // Column sums of the count matrix over all blocks (totals) and over the
    // blocks before this one (prefix). Thread (r, cg) sums rows r, r + R, ...
    // of column group cg, read as int4 (contiguous across the lanes of one
    // row); lanes of a warp holding the same column group then add up by
    // shuffles, leaving Rp partial rows.
    const int4* mat = reinterpret_cast<const int4*>(a.ws_counts);
    for (int idx = threadIdx.x; idx < q.R * q.CGp; idx += NT) {
        const int r = idx / q.CGp;
        const int cg = idx % q.CGp;
        int4 tot = make_int4(0, 0, 0, 0), pre = make_int4(0, 0, 0, 0);
        if (cg < q.CG) {
            for (int rb0 = r; rb0 < a.G; rb0 += 8 * q.R) {
                int4 v[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {   // 8 independent loads in flight
                    const int rb = rb0 + u * q.R;
                    v[u] = rb < a.G ? __ldcg(mat + (size_t)rb * q.CG + cg) : make_int4(0, 0, 0, 0);
                }
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    tot.x += v[u].x; tot.y += v[u].y; tot.z += v[u].z; tot.w += v[u].w;
                    if (rb0 + u * q.R < b) { pre.x += v[u].x; pre.y += v[u].y; pre.z += v[u].z; pre.w += v[u].w; }
                }
            }
        }
        // q.LPW > 1 only when q.R * q.CGp == NT: every lane is here
        for (int o = q.CGp; o < kWarp; o <<= 1) {
            tot.x += __shfl_xor_sync(kFull, tot.x, o); tot.y += __shfl_xor_sync(kFull, tot.y, o);
            tot.z += __shfl_xor_sync(kFull, tot.z, o); tot.w += __shfl_xor_sync(kFull, tot.w, o);
            pre.x += __shfl_xor_sync(kFull, pre.x, o); pre.y += __shfl_xor_sync(kFull, pre.y, o);
            pre.z += __shfl_xor_sync(kFull, pre.z, o); pre.w += __shfl_xor_sync(kFull, pre.w, o);
        }
        if (r % q.LPW == 0 && cg < q.CG) {
            reinterpret_cast<int4*>(s_ptot + (r / q.LPW) * Ep)[cg] = tot;
            reinterpret_cast<int4*>(s_ppre + (r / q.LPW) * Ep)[cg] = pre;
        }
    }
    __syncthreads();
    for (int c = threadIdx.x; c < Ep; c += NT) {
        int tot = 0, pre = 0;
#pragma unroll 8
        for (int r = 0; r < q.Rp; ++r) { tot += s_ptot[r * Ep + c]; pre += s_ppre[r * Ep + c]; }
        s_tot[c] = tot;
        s_base[c] = pre;
    }
    __syncthreads();
    if (threadIdx.x < kWarp) warp_offsets<LOCAL>(a, s_tot, s_off, s_base, b == 0);
    __syncthreads();

    auto place = [&](int s, int e, int rank) {
        if constexpr (LOCAL) {
            e -= a.e0;
            if (e < 0 || e >= a.nloc) return;   // inv_perm already -1
        }
        const int p = s_base[e] + rank;
        a.perm[p] = s;
        a.inv_perm[s] = p;
    };
    if (sf < s1) place(sf, ef, rf);
    for (int s = sf + NT; s < s1; s += NT) place(s, __ldcg(a.topk_ids + s), __ldcg(a.inv_perm + s));
    if constexpr (LOCAL) fill_padding<NT>(a, s_tot, s_off, b, a.G, b * NT, a.G * NT);
}

template <int GS, int EPL, int NT, bool LOCAL>
__global__ void __launch_bounds__(NT) route_fused_kernel(RouteArgs a) {
    constexpr int NW = NT / kWarp;
    extern __shared__ int32_t smem[];
    int32_t* s_cnt = smem;                         // [NW][nloc]
    int32_t* s_tot = s_cnt + (size_t)NW * a.nloc;  // [Ep] totals
    int32_t* s_off = s_tot + a.Ep;                 // [Ep + 4] offsets
    int32_t* s_warp = s_off + a.Ep + 4;            // [32]
    pdl_wait_and_release();
    zero_warp_counters(s_cnt, a.nloc);
    int re[kRegRounds], rr[kRegRounds];
    topk_rank_range<GS, EPL, NT, LOCAL>(a, 0, a.T, s_cnt, re, rr);
    __syncthreads();
    scan_over_warps<NT>(s_cnt, s_tot, a.nloc);
    __syncthreads();
    compute_offsets<NT, LOCAL>(a, s_tot, s_off, s_warp, true);
    finish_ranks<GS, NT, true, LOCAL>(a, 0, a.T, s_cnt, s_off, re, rr);
    if constexpr (LOCAL) fill_padding<NT>(a, s_tot, s_off, 0, 1, 0, NT);
}

#ifndef MOE_ROUTE_NT
#define MOE_ROUTE_NT 512
#endif
// Wide blocks of the two-kernel path: for 32-lane groups with 2 to 8 keys
// per lane, when blocks of MOE_ROUTE_NT threads would give each warp two
// tokens, blocks of this many give each warp one (every token of a block in
// flight at once). 0 turns them off.
#ifndef MOE_ROUTE_WIDE_NT
#define MOE_ROUTE_WIDE_NT 1024
#endif
#ifndef MOE_ROUTE_FUSED_NT
#define MOE_ROUTE_FUSED_NT 512
#endif
#ifndef MOE_ROUTE_GMAX
#define MOE_ROUTE_GMAX 128
#endif
#ifndef MOE_ROUTE_PAIR
#define MOE_ROUTE_PAIR 1
#endif
constexpr int kNtSplit = MOE_ROUTE_NT;
constexpr int kNtFused = MOE_ROUTE_FUSED_NT;
constexpr int kNtWide = MOE_ROUTE_WIDE_NT;
constexpr bool wide_eligible(int gs, int epl) { return kNtWide > kNtSplit && gs == 32 && epl >= 2 && epl <= 8; }

template <typename K>
cudaError_t allow_smem(K kernel, size_t bytes) {
    if (bytes <= 48 * 1024) return cudaSuccess;
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(bytes));
}

// The two-kernel path with blocks of NT threads.
template <int GS, int EPL, bool LOCAL, int NT>
cudaError_t launch_split(const RoutePlan& p, const RouteArgs& a, cudaStream_t stream) {
    cudaError_t err;
    // two tokens per step where a warp owns two or more (32-lane groups, at
    // most 8 keys per lane: the pair's keys stay in registers; 512-thread
    // blocks, whose register budget holds them)
    constexpr bool kCanPair = MOE_ROUTE_PAIR && GS == 32 && EPL <= 8 && NT <= 512;
    auto k1 = (kCanPair && p.tpw >= 2) ? route_rank_kernel<GS, EPL, NT, LOCAL, kCanPair ? 2 : 1>
                                       : route_rank_kernel<GS, EPL, NT, LOCAL, 1>;
    if ((err = allow_smem(k1, p.smem_topk)) != cudaSuccess) return err;
    if ((err = launch_pdl(k1, dim3(p.G), dim3(NT), p.smem_topk, stream, a)) != cudaSuccess) return err;
    auto k2 = route_place_kernel<NT, LOCAL>;
    if ((err = allow_smem(k2, p.smem_scatter)) != cudaSuccess) return err;
    return launch_pdl(k2, dim3(p.G), dim3(NT), p.smem_scatter, stream, a);
}

template <int GS, int EPL, bool LOCAL>
cudaError_t launch_route_t(const RoutePlan& p, const RouteArgs& a, cudaStream_t stream) {
    cudaError_t err;
    if (p.fused) {
        auto kf = route_fused_kernel<GS, EPL, kNtFused, LOCAL>;
        if ((err = allow_smem(kf, p.smem_topk)) != cudaSuccess) return err;
        return launch_pdl(kf, dim3(1), dim3(kNtFused), p.smem_topk, stream, a);
    }
    if constexpr (wide_eligible(GS, EPL)) {
        if (p.nt == kNtWide) return launch_split<GS, EPL, LOCAL, (kNtWide > kNtSplit ? kNtWide : kNtSplit)>(p, a, stream);
    }
    return launch_split<GS, EPL, LOCAL, kNtSplit>(p, a, stream);
}

template <bool LOCAL>
cudaError_t launch_route_local(const RoutePlan& plan, const RouteArgs& a, cudaStream_t stream) {
    switch (plan.gs * 100 + plan.epl) {
        case 801: return launch_route_t<8, 1, LOCAL>(plan, a, stream);
        case 1601: return launch_route_t<16, 1, LOCAL>(plan, a, stream);
        case 3201: return launch_route_t<32, 1, LOCAL>(plan, a, stream);
        case 3202: return launch_route_t<32, 2, LOCAL>(plan, a, stream);
        case 3204: return launch_route_t<32, 4, LOCAL>(plan, a, stream);
        case 3208: return launch_route_t<32, 8, LOCAL>(plan, a, stream);
        case 3216: return launch_route_t<32, 16, LOCAL>(plan, a, stream);
        case 3232: return launch_route_t<32, 32, LOCAL>(plan, a, stream);
        default: return cudaErrorInvalidConfiguration;
    }
}

}  // namespace

RoutePlan plan_route(int64_t T, int E, int k, int nloc) {
    (void)k;
    if (nloc <= 0) nloc = E;
    RoutePlan p;
    if (E <= 8) { p.gs = 8; p.epl = 1; }
    else if (E <= 16) { p.gs = 16; p.epl = 1; }
    else { p.gs = 32; p.epl = (E + 31) / 32; }
    if (p.epl > 2) p.epl = p.epl <= 4 ? 4 : p.epl <= 8 ? 8 : p.epl <= 16 ? 16 : 32;
    p.Ep = (nloc + 3) / 4 * 4;
    const int gpw = kWarp / p.gs;
    const int fused_groups = (kNtFused / kWarp) * gpw;
    p.fused = T <= 2 * fused_groups;
    if (p.fused) {
        const int nw = kNtFused / kWarp;
        p.nt = kNtFused;
        p.G = 1;
        p.tpc = int(T);
        p.tpw = int(((T + nw - 1) / nw + gpw - 1) / gpw * gpw);
        p.ws_bytes = 0;
        p.smem_topk = sizeof(int32_t) * (size_t(nw) * nloc + 2 * size_t(p.Ep) + 4 + 32);
        return p;
    }
    const int gmax = std::max(1, std::min(MOE_ROUTE_GMAX, 32768 / p.Ep));
    const int64_t tpc_min = (T + gmax - 1) / gmax;   // tokens per block at the most blocks
    // NT threads per block: at least one lane group per warp of tokens
    p.nt = kNtSplit;
    if (wide_eligible(p.gs, p.epl) && tpc_min > kNtSplit / kWarp && tpc_min <= kNtWide / kWarp) p.nt = kNtWide;
    const int nw = p.nt / kWarp;
    const int groups = nw * gpw;
    const int64_t tpc = std::max<int64_t>(groups, tpc_min);
    p.tpc = int(tpc);
    p.tpw = int(((tpc + nw - 1) / nw + gpw - 1) / gpw * gpw);
    p.G = int((T + tpc - 1) / tpc);
    p.ws_bytes = sizeof(int32_t) * size_t(p.G) * size_t(p.Ep);
    p.smem_topk = sizeof(int32_t) * (size_t(nw) * nloc + p.Ep);
    const PlaceSplit q = place_split(p.Ep, p.nt);
    p.smem_scatter = sizeof(int32_t) * (size_t(2) * q.Rp * p.Ep + 3 * size_t(p.Ep) + 4);
    return p;
}

cudaError_t launch_route(const RoutePlan& plan, const float* logits, int T, int E, int k,
                         int renorm, int32_t* topk_ids, float* topk_weights,
                         int32_t* expert_counts, int32_t* expert_offsets, int32_t* perm,
                         int32_t* inv_perm, void* workspace, cudaStream_t stream,
                         const LocalRange* local) {
    RouteArgs a;
    a.logits = logits;
    a.T = T; a.E = E; a.k = k; a.renorm = renorm;
    a.e0 = local ? local->e0 : 0;
    a.nloc = local ? local->n : E;
    a.pad = local ? local->pad : 1;
    a.rows = local ? local->rows : T * k;
    a.Ep = plan.Ep; a.tpc = plan.tpc; a.tpw = plan.tpw; a.G = plan.G;
    a.topk_ids = topk_ids; a.topk_weights = topk_weights;
    a.expert_counts = expert_counts; a.expert_offsets = expert_offsets;
    a.perm = perm; a.inv_perm = inv_perm;
    a.ws_counts = static_cast<int32_t*>(workspace);
    a.write_out = true;
    a.vec4 = E % 4 == 0 && reinterpret_cast<uintptr_t>(logits) % 16 == 0;
    return local ? launch_route_local<true>(plan, a, stream) : launch_route_local<false>(plan, a, stream);
}

}  // namespace moe
