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
#include "rows_common.cuh"

#include <algorithm>

namespace moe {
namespace {

struct RouteArgs {
    const float* logits;
    int T, E, k, renorm;
    int Ep;    // count-matrix row stride (E rounded up to 4)
    int tpc;   // tokens per block
    int tpw;   // tokens per warp (a multiple of the token groups per warp)
    int G;     // blocks
    int32_t* topk_ids;
    float* topk_weights;
    int32_t* expert_counts;
    int32_t* expert_offsets;
    int32_t* perm;
    int32_t* inv_perm;
    int32_t* ws_counts;  // [G][Ep]
};

// Order-preserving map of a float onto uint32 (larger float -> larger key).
// -0.0 is first folded onto +0.0 so that the two compare equal. Key 0 marks
// "empty / already taken"; every real logit maps to 1 or more (only one NaN
// bit pattern would map to 0, and it is lifted to 1), so a pick is always a
// valid expert.
__device__ __forceinline__ uint32_t order_key(float v) {
    v = (v == 0.0f) ? 0.0f : v;
    const uint32_t b = __float_as_uint(v);
    return max((b & 0x80000000u) ? ~b : (b | 0x80000000u), 1u);
}

__device__ __forceinline__ float key_value(uint32_t key) {
    uint32_t b = (key & 0x80000000u) ? (key & 0x7fffffffu) : ~key;
    return __uint_as_float(b);
}

// Reductions over aligned groups of GS lanes; every lane of the warp calls.
template <int GS>
__device__ __forceinline__ uint32_t group_max(uint32_t v) {
    if constexpr (GS == 32) {
        return __reduce_max_sync(kFull, v);
    } else {
#pragma unroll
        for (int o = GS / 2; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(kFull, v, o));
        return v;
    }
}

template <int GS>
__device__ __forceinline__ uint32_t group_min(uint32_t v) {
    if constexpr (GS == 32) {
        return __reduce_min_sync(kFull, v);
    } else {
#pragma unroll
        for (int o = GS / 2; o > 0; o >>= 1) v = min(v, __shfl_xor_sync(kFull, v, o));
        return v;
    }
}

template <int GS>
__device__ __forceinline__ float group_sum(float v) {
#pragma unroll
    for (int o = GS / 2; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
    return v;
}

// Keys of token t for lane gl of a GS-lane group: experts gl, gl + GS, ...
// (a coalesced row read) as order-preserving keys; 0 outside the row.
template <int GS, int EPL>
__device__ __forceinline__ void load_keys(const RouteArgs& a, int t, bool valid, int gl,
                                          uint32_t (&key)[EPL]) {
    const float* row = a.logits + (size_t)t * a.E;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
        const int e = gl + GS * i;
        key[i] = (valid && e < a.E) ? order_key(__ldg(row + e)) : 0u;
    }
}

// Top-k of one token by a group of GS lanes from its keys (the float is
// recovered exactly from its key). Each of the k rounds takes the group
// maximum of the keys and, among lanes holding it, the lowest expert index;
// the owner then drops that expert. Lane j < k keeps the j-th pick, writes it
// and its weight, and returns the expert (-1 for lanes without a pick). Every
// lane of the warp must call (valid may differ between groups of one warp;
// invalid groups compute on empty keys and write nothing).
template <int GS, int EPL>
__device__ __forceinline__ int topk_select(const RouteArgs& a, int t, bool valid, int gl,
                                           uint32_t (&key)[EPL]) {
    // Softmax denominator over all E experts (only without renormalisation),
    // taken before the picks remove keys.
    float z = 0.0f;
    if (!a.renorm) {
        uint32_t lmax = key[0];
#pragma unroll
        for (int i = 1; i < EPL; ++i) lmax = max(lmax, key[i]);
        const float vmax = key_value(group_max<GS>(lmax));
#pragma unroll
        for (int i = 0; i < EPL; ++i)
            if (key[i] != 0u) z += expf(key_value(key[i]) - vmax);
        z = group_sum<GS>(z);
    }

    int my_id = 0;
    float my_val = 0.0f;
    float vmax = 0.0f;
    for (int j = 0; j < a.k; ++j) {
        uint32_t bk = key[0];
        int bi = 0;
#pragma unroll
        for (int i = 1; i < EPL; ++i) {
            if (key[i] > bk) { bk = key[i]; bi = i; }
        }
        const uint32_t gk = group_max<GS>(bk);
        const uint32_t cand = (bk == gk) ? uint32_t(gl + GS * bi) : 0xffffffffu;
        const uint32_t ge = group_min<GS>(cand);
        if (int(ge % GS) == gl) {
            const int wi = int(ge / GS);
#pragma unroll
            for (int i = 0; i < EPL; ++i) if (i == wi) key[i] = 0u;
        }
        const float gv = key_value(gk);
        if (j == 0) vmax = gv;
        if (gl == j) { my_id = int(ge); my_val = gv; }
    }

    // Weights in float32. The largest logit is the first pick.
    const bool mine = gl < a.k;
    const float ej = mine ? expf(my_val - vmax) : 0.0f;
    const float denom = a.renorm ? group_sum<GS>(ej)   // sum over the k picks
                                 : z;                  // sum over all E experts
    if (valid && mine) {
        a.topk_ids[(size_t)t * a.k + gl] = my_id;
        a.topk_weights[(size_t)t * a.k + gl] = ej / denom;
        return my_id;
    }
    return -1;
}

// Rounds whose (expert, rank) per lane stay in registers until the ranks are
// finished; later rounds (only for very long token runs) go through inv_perm.
constexpr int kRegRounds = 4;

// Top-k of the tokens [t0, t1) and the rank of every slot among this warp's
// slots of the same expert; s_cnt is [NW][E] and counts each warp's picks per
// expert. Warp w owns tokens [t0 + w*tpw, t0 + (w+1)*tpw); each round takes
// GPW consecutive tokens, one per lane group, so lane order within a round
// is slot order. The first kRegRounds rounds return each lane's expert and
// rank in re/rr (expert -1: no slot); the rank of later rounds is written to
// inv_perm[s]. The next round's logits are loaded before the current round's
// selection.
template <int GS, int EPL, int NT>
__device__ __forceinline__ void topk_rank_range(const RouteArgs& a, int t0, int t1, int32_t* s_cnt,
                                                int (&re)[kRegRounds], int (&rr)[kRegRounds]) {
    constexpr int GPW = kWarp / GS;
    const int lane = threadIdx.x % kWarp;
    const int warp = threadIdx.x / kWarp;
    const int grp = lane / GS;
    const int gl = lane % GS;
    const unsigned lower = (1u << lane) - 1u;
    int32_t* cnt = s_cnt + (size_t)warp * a.E;
    const int w0 = t0 + warp * a.tpw;
    const int w1 = min(t1, w0 + a.tpw);

    uint32_t key[EPL], next[EPL];
    load_keys<GS, EPL>(a, w0 + grp, w0 + grp < w1, gl, key);
#pragma unroll
    for (int r = 0; r < kRegRounds; ++r) {
        re[r] = -1;
        rr[r] = 0;
        const int tb = w0 + r * GPW;
        if (tb < w1) {
            const int tn = tb + GPW + grp;
            load_keys<GS, EPL>(a, tn, tn < w1, gl, next);
            const int t = tb + grp;
            const int e = topk_select<GS, EPL>(a, t, t < w1, gl, key);
            const unsigned peers = __match_any_sync(kFull, e);
            re[r] = e;
            rr[r] = (e >= 0) ? cnt[e] + __popc(peers & lower) : 0;
            __syncwarp();
            if (e >= 0 && lane == __ffs(peers) - 1) cnt[e] += __popc(peers);
            __syncwarp();
#pragma unroll
            for (int i = 0; i < EPL; ++i) key[i] = next[i];
        }
    }
    for (int tb = w0 + kRegRounds * GPW; tb < w1; tb += GPW) {
        const int t = tb + grp;
        const int e = topk_select<GS, EPL>(a, t, t < w1, gl, key);
        const int tn = tb + GPW + grp;
        load_keys<GS, EPL>(a, tn, tn < w1, gl, key);
        const unsigned peers = __match_any_sync(kFull, e);
        if (e >= 0) a.inv_perm[(size_t)t * a.k + gl] = cnt[e] + __popc(peers & lower);
        __syncwarp();
        if (e >= 0 && lane == __ffs(peers) - 1) cnt[e] += __popc(peers);
        __syncwarp();
    }
}

// Exclusive scan over warps of s_cnt[w][e] for every expert; s_tot[e] gets
// the block total.
template <int NT>
__device__ __forceinline__ void scan_over_warps(int32_t* s_cnt, int32_t* s_tot, int E) {
    constexpr int NW = NT / kWarp;
    for (int e = threadIdx.x; e < E; e += NT) {
        int run = 0;
#pragma unroll 4
        for (int w = 0; w < NW; ++w) {
            const int v = s_cnt[(size_t)w * E + e];
            s_cnt[(size_t)w * E + e] = run;
            run += v;
        }
        s_tot[e] = run;
    }
}

// Exclusive scan of in[0..n) into out[0..n) (may alias) by a block of NT
// threads, n <= MOE_MAX_EXPERTS. Uses s_warp[32].
template <int NT>
__device__ void block_exclusive_scan(const int32_t* in, int32_t* out, int n, int32_t* s_warp) {
    constexpr int ITEMS = (1024 + NT - 1) / NT;
    constexpr int NW = NT / kWarp;
    const int lane = threadIdx.x % kWarp;
    const int warp = threadIdx.x / kWarp;
    const int base = threadIdx.x * ITEMS;
    int v[ITEMS];
    int local = 0;
#pragma unroll
    for (int i = 0; i < ITEMS; ++i) {
        v[i] = (base + i < n) ? in[base + i] : 0;
        local += v[i];
    }
    int x = local;
#pragma unroll
    for (int o = 1; o < kWarp; o <<= 1) {
        const int y = __shfl_up_sync(kFull, x, o);
        if (lane >= o) x += y;
    }
    if (lane == kWarp - 1) s_warp[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = lane < NW ? s_warp[lane] : 0;
#pragma unroll
        for (int o = 1; o < kWarp; o <<= 1) {
            const int y = __shfl_up_sync(kFull, w, o);
            if (lane >= o) w += y;
        }
        s_warp[lane] = w;
    }
    __syncthreads();
    int run = (warp > 0 ? s_warp[warp - 1] : 0) + x - local;
#pragma unroll
    for (int i = 0; i < ITEMS; ++i) {
        if (base + i < n) out[base + i] = run;
        run += v[i];
    }
    __syncthreads();
}

// Add each slot's per-warp start to its within-warp rank (s_cnt now holds
// the exclusive scan over warps). With PLACE (one-block path) the expert's
// offset is added too, the result is final and perm is written.
template <int GS, int NT, bool PLACE>
__device__ __forceinline__ void finish_ranks(const RouteArgs& a, int t0, int t1, const int32_t* s_cnt,
                                             const int32_t* s_off, const int (&re)[kRegRounds],
                                             const int (&rr)[kRegRounds]) {
    constexpr int GPW = kWarp / GS;
    const int lane = threadIdx.x % kWarp;
    const int warp = threadIdx.x / kWarp;
    const int grp = lane / GS;
    const int gl = lane % GS;
    const int32_t* start = s_cnt + (size_t)warp * a.E;
    const int w0 = t0 + warp * a.tpw;
    const int w1 = min(t1, w0 + a.tpw);
#pragma unroll
    for (int r = 0; r < kRegRounds; ++r) {
        if (re[r] >= 0) {
            const int s = (w0 + r * GPW + grp) * a.k + gl;
            int p = rr[r] + start[re[r]];
            if constexpr (PLACE) {
                p += s_off[re[r]];
                a.perm[p] = s;
            }
            a.inv_perm[s] = p;
        }
    }
    // slots of rounds past kRegRounds: the rank was kept in inv_perm
    const int s_lo = (w0 + kRegRounds * GPW) * a.k;
    for (int s = s_lo + lane; s < w1 * a.k; s += kWarp) {
        const int e = __ldcg(a.topk_ids + s);
        int p = __ldcg(a.inv_perm + s) + start[e];
        if constexpr (PLACE) {
            p += s_off[e];
            a.perm[p] = s;
        }
        a.inv_perm[s] = p;
    }
}

template <int GS, int EPL, int NT>
__global__ void __launch_bounds__(NT) route_rank_kernel(RouteArgs a) {
    constexpr int NW = NT / kWarp;
    extern __shared__ int32_t smem[];
    int32_t* s_cnt = smem;                      // [NW][E]
    int32_t* s_tot = s_cnt + (size_t)NW * a.E;  // [Ep]
    pdl_wait_and_release();
    for (int i = threadIdx.x; i < NW * a.E; i += NT) s_cnt[i] = 0;
    for (int e = threadIdx.x; e < a.Ep; e += NT) s_tot[e] = 0;
    __syncthreads();
    const int t0 = blockIdx.x * a.tpc;
    const int t1 = min(a.T, t0 + a.tpc);
    int re[kRegRounds], rr[kRegRounds];
    topk_rank_range<GS, EPL, NT>(a, t0, t1, s_cnt, re, rr);
    __syncthreads();
    scan_over_warps<NT>(s_cnt, s_tot, a.E);
    __syncthreads();
    int32_t* row = a.ws_counts + (size_t)blockIdx.x * a.Ep;
    for (int e = threadIdx.x; e < a.Ep; e += NT) row[e] = s_tot[e];
    finish_ranks<GS, NT, false>(a, t0, t1, s_cnt, nullptr, re, rr);
}

// Number of row groups the place kernel splits the count matrix into.
__host__ __device__ inline int place_rowgroups(int Ep, int nt) {
    const int cg = Ep / 4;
    return cg >= nt ? 1 : nt / cg;
}

template <int NT>
__global__ void __launch_bounds__(NT) route_place_kernel(RouteArgs a) {
    extern __shared__ int32_t smem[];
    const int Ep = a.Ep;
    const int CG = Ep / 4;
    const int R = place_rowgroups(Ep, NT);
    int32_t* s_ptot = smem;                 // [R][Ep]
    int32_t* s_ppre = s_ptot + R * Ep;      // [R][Ep]
    int32_t* s_tot = s_ppre + R * Ep;       // [Ep]
    int32_t* s_base = s_tot + Ep;           // [Ep]
    int32_t* s_warp = s_base + Ep;          // [32]
    const int b = blockIdx.x;
    pdl_wait_and_release();

    // Column sums of the count matrix over all blocks (totals) and over the
    // blocks before this one (prefix). Rows are interleaved over R row
    // groups; columns are read as int4, contiguous across a warp.
    for (int idx = threadIdx.x; idx < R * CG; idx += NT) {
        const int r = idx / CG;
        const int cg = idx % CG;
        int4 tot = make_int4(0, 0, 0, 0), pre = make_int4(0, 0, 0, 0);
        const int4* col = reinterpret_cast<const int4*>(a.ws_counts) + cg;
        const int q = Ep / 4;   // int4 per row
        for (int rb0 = r; rb0 < a.G; rb0 += 8 * R) {
            int4 v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {   // 8 independent loads in flight
                const int rb = rb0 + u * R;
                v[u] = rb < a.G ? __ldcg(col + (size_t)rb * q) : make_int4(0, 0, 0, 0);
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                tot.x += v[u].x; tot.y += v[u].y; tot.z += v[u].z; tot.w += v[u].w;
                if (rb0 + u * R < b) { pre.x += v[u].x; pre.y += v[u].y; pre.z += v[u].z; pre.w += v[u].w; }
            }
        }
        reinterpret_cast<int4*>(s_ptot + r * Ep)[cg] = tot;
        reinterpret_cast<int4*>(s_ppre + r * Ep)[cg] = pre;
    }
    __syncthreads();
    for (int c = threadIdx.x; c < Ep; c += NT) {
        int tot = 0, pre = 0;
        for (int r = 0; r < R; ++r) { tot += s_ptot[r * Ep + c]; pre += s_ppre[r * Ep + c]; }
        s_tot[c] = tot;
        s_base[c] = pre;
    }
    __syncthreads();
    if (b == 0) {
        for (int e = threadIdx.x; e < a.E; e += NT) a.expert_counts[e] = s_tot[e];
    }
    block_exclusive_scan<NT>(s_tot, s_tot, a.E, s_warp);   // s_tot := offsets
    for (int e = threadIdx.x; e < a.E; e += NT) {
        if (b == 0) a.expert_offsets[e] = s_tot[e];
        s_base[e] += s_tot[e];
    }
    if (b == 0 && threadIdx.x == 0) a.expert_offsets[a.E] = a.T * a.k;
    __syncthreads();

    const int s0 = b * a.tpc * a.k;
    const int s1 = min(a.T, (b + 1) * a.tpc) * a.k;
    for (int s = s0 + threadIdx.x; s < s1; s += NT) {
        const int e = __ldcg(a.topk_ids + s);
        const int p = s_base[e] + __ldcg(a.inv_perm + s);
        a.perm[p] = s;
        a.inv_perm[s] = p;
    }
}

template <int GS, int EPL, int NT>
__global__ void __launch_bounds__(NT) route_fused_kernel(RouteArgs a) {
    constexpr int NW = NT / kWarp;
    extern __shared__ int32_t smem[];
    int32_t* s_cnt = smem;                      // [NW][E]
    int32_t* s_tot = s_cnt + (size_t)NW * a.E;  // [Ep] totals, then offsets
    int32_t* s_warp = s_tot + a.Ep;             // [32]
    pdl_wait_and_release();
    for (int i = threadIdx.x; i < NW * a.E; i += NT) s_cnt[i] = 0;
    __syncthreads();
    int re[kRegRounds], rr[kRegRounds];
    topk_rank_range<GS, EPL, NT>(a, 0, a.T, s_cnt, re, rr);
    __syncthreads();
    scan_over_warps<NT>(s_cnt, s_tot, a.E);
    __syncthreads();
    for (int e = threadIdx.x; e < a.E; e += NT) a.expert_counts[e] = s_tot[e];
    block_exclusive_scan<NT>(s_tot, s_tot, a.E, s_warp);
    for (int e = threadIdx.x; e < a.E; e += NT) a.expert_offsets[e] = s_tot[e];
    if (threadIdx.x == 0) a.expert_offsets[a.E] = a.T * a.k;
    finish_ranks<GS, NT, true>(a, 0, a.T, s_cnt, s_tot, re, rr);
}

#ifndef MOE_ROUTE_NT
#define MOE_ROUTE_NT 512
#endif
#ifndef MOE_ROUTE_FUSED_NT
#define MOE_ROUTE_FUSED_NT 512
#endif
#ifndef MOE_ROUTE_GMAX
#define MOE_ROUTE_GMAX 128
#endif
constexpr int kNtSplit = MOE_ROUTE_NT;
constexpr int kNtFused = MOE_ROUTE_FUSED_NT;

template <typename K>
cudaError_t allow_smem(K kernel, size_t bytes) {
    if (bytes <= 48 * 1024) return cudaSuccess;
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(bytes));
}

template <int GS, int EPL>
cudaError_t launch_route_t(const RoutePlan& p, const RouteArgs& a, cudaStream_t stream) {
    cudaError_t err;
    if (p.fused) {
        auto kf = route_fused_kernel<GS, EPL, kNtFused>;
        if ((err = allow_smem(kf, p.smem_topk)) != cudaSuccess) return err;
        return launch_pdl(kf, dim3(1), dim3(kNtFused), p.smem_topk, stream, a);
    }
    auto k1 = route_rank_kernel<GS, EPL, kNtSplit>;
    auto k2 = route_place_kernel<kNtSplit>;
    if ((err = allow_smem(k1, p.smem_topk)) != cudaSuccess) return err;
    if ((err = allow_smem(k2, p.smem_scatter)) != cudaSuccess) return err;
    if ((err = launch_pdl(k1, dim3(p.G), dim3(kNtSplit), p.smem_topk, stream, a)) != cudaSuccess)
        return err;
    return launch_pdl(k2, dim3(p.G), dim3(kNtSplit), p.smem_scatter, stream, a);
}

}  // namespace

RoutePlan plan_route(int64_t T, int E, int k) {
    (void)k;
    RoutePlan p;
    if (E <= 8) { p.gs = 8; p.epl = 1; }
    else if (E <= 16) { p.gs = 16; p.epl = 1; }
    else { p.gs = 32; p.epl = (E + 31) / 32; }
    if (p.epl > 2) p.epl = p.epl <= 4 ? 4 : p.epl <= 8 ? 8 : p.epl <= 16 ? 16 : 32;
    p.Ep = (E + 3) / 4 * 4;
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
        p.smem_topk = sizeof(int32_t) * (size_t(nw) * E + p.Ep + 32);
        return p;
    }
    const int nw = kNtSplit / kWarp;
    p.nt = kNtSplit;
    const int groups = nw * gpw;
    const int gmax = std::max(1, std::min(MOE_ROUTE_GMAX, 32768 / p.Ep));
    const int64_t tpc = std::max<int64_t>(groups, (T + gmax - 1) / gmax);
    p.tpc = int(tpc);
    p.tpw = int(((tpc + nw - 1) / nw + gpw - 1) / gpw * gpw);
    p.G = int((T + tpc - 1) / tpc);
    p.ws_bytes = sizeof(int32_t) * size_t(p.G) * size_t(p.Ep);
    p.smem_topk = sizeof(int32_t) * (size_t(nw) * E + p.Ep);
    const int R = place_rowgroups(p.Ep, kNtSplit);
    p.smem_scatter = sizeof(int32_t) * (size_t(2) * R * p.Ep + 2 * size_t(p.Ep) + 32);
    return p;
}

cudaError_t launch_route(const RoutePlan& plan, const float* logits, int T, int E, int k,
                         int renorm, int32_t* topk_ids, float* topk_weights,
                         int32_t* expert_counts, int32_t* expert_offsets, int32_t* perm,
                         int32_t* inv_perm, void* workspace, cudaStream_t stream) {
    RouteArgs a;
    a.logits = logits;
    a.T = T; a.E = E; a.k = k; a.renorm = renorm;
    a.Ep = plan.Ep; a.tpc = plan.tpc; a.tpw = plan.tpw; a.G = plan.G;
    a.topk_ids = topk_ids; a.topk_weights = topk_weights;
    a.expert_counts = expert_counts; a.expert_offsets = expert_offsets;
    a.perm = perm; a.inv_perm = inv_perm;
    a.ws_counts = static_cast<int32_t*>(workspace);
    switch (plan.gs * 100 + plan.epl) {
        case 801: return launch_route_t<8, 1>(plan, a, stream);
        case 1601: return launch_route_t<16, 1>(plan, a, stream);
        case 3201: return launch_route_t<32, 1>(plan, a, stream);
        case 3202: return launch_route_t<32, 2>(plan, a, stream);
        case 3204: return launch_route_t<32, 4>(plan, a, stream);
        case 3208: return launch_route_t<32, 8>(plan, a, stream);
        case 3216: return launch_route_t<32, 16>(plan, a, stream);
        case 3232: return launch_route_t<32, 32>(plan, a, stream);
        default: return cudaErrorInvalidConfiguration;
    }
}

}  // namespace moe
