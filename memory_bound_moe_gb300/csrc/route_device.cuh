// Device-side building blocks of the routing step, shared by the routing
// kernels (route.cu) and the one-launch decode route-and-expand kernel
// (route_expand.cu): order-preserving keys, lane-group top-k with softmax
// weights, in-block stable ranking and scans. See route.cu for the scheme.
#pragma once

#include "moe_device.cuh"

#include <cstdint>

namespace moe {

struct RouteArgs {
    const float* logits;
    int T, E, k, renorm;
    int e0, nloc;  // counted experts: [e0, e0 + nloc) (all E unless a local routing)
    int pad;       // expert segments rounded up to a multiple of pad (local routing)
    int rows;      // entries of perm (T*k, or the padded capacity of a local routing)
    int Ep;    // count-matrix row stride (nloc rounded up to 4)
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
    bool write_out;      // write topk_ids/weights, perm, inv_perm (false: block-private results)
    bool vec4;           // logits rows may be read as 16-byte vectors (E % 4 == 0, 16-byte base)
};

// Largest k the selection loop unrolls for (the public MOE_MAX_TOPK).
constexpr int kMaxTopk = 16;

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

// Keys of token t for lane gl of a GS-lane group: the EPL consecutive experts
// gl*EPL .. gl*EPL + EPL - 1, so that lane order is expert order, as
// order-preserving keys; 0 outside the row. Whole 16-byte vectors when the
// row layout allows it.
template <int GS, int EPL>
__device__ __forceinline__ void load_keys(const RouteArgs& a, int t, bool valid, int gl,
                                          uint32_t (&key)[EPL]) {
    const int e0 = gl * EPL;
    const float* row = a.logits + (size_t)t * a.E + e0;
    if constexpr (EPL % 4 == 0) {
        if (a.vec4 && valid && e0 + EPL <= a.E) {
#pragma unroll
            for (int q = 0; q < EPL / 4; ++q) {
                const float4 v = __ldg(reinterpret_cast<const float4*>(row) + q);
                key[4 * q] = order_key(v.x);
                key[4 * q + 1] = order_key(v.y);
                key[4 * q + 2] = order_key(v.z);
                key[4 * q + 3] = order_key(v.w);
            }
            return;
        }
    }
#pragma unroll
    for (int i = 0; i < EPL; ++i)
        key[i] = (valid && e0 + i < a.E) ? order_key(__ldg(row + i)) : 0u;
}

// Top-k of N tokens at once, each by the same group of GS lanes holding its
// keys in expert order (the float is recovered exactly from its key). With
// N > 1 the tokens' selections are independent dependency chains written as
// one interleaved instruction stream, so each one's reduction latencies hide
// behind the other's.
// Pick j is the largest key left and, among equal keys, the lowest expert.
// Each lane offers its best key (the lowest of its experts among equal keys);
// the pick is the group maximum of the offers, taken from the lowest lane
// offering it, which holds the lowest such expert since lanes hold
// consecutive experts. One group maximum and one ballot per pick.
//   EPL <= 8: a lane first sorts its keys in descending order by swapping
//   neighbours only when the later key is strictly larger, so equal keys keep
//   their expert order; its offer is then the head of the list, and the
//   owner of a pick shifts its list by one. The expert of every sorted
//   position is packed into one register, LB bits each.
//   EPL > 8: a lane takes the arg-max of its keys every round and the owner
//   zeroes the picked key.
// Lane j < k keeps the j-th pick of every token, writes it and its weight,
// and returns the expert in out[n] (-1 for lanes without a pick or invalid
// tokens). Every lane of the warp must call (valid may differ between groups
// of one warp and between the N tokens; invalid tokens compute on empty keys
// and write nothing).
template <int GS, int EPL, int N>
__device__ __forceinline__ void topk_select_n(const RouteArgs& a, const int (&t)[N], const bool (&valid)[N],
                                              int gl, uint32_t (&key)[N][EPL], int (&out)[N]) {
    constexpr bool kSorted = EPL <= 8;
    constexpr int LB = EPL <= 2 ? 1 : EPL <= 4 ? 2 : 3;
    constexpr uint32_t kIdxMask = (1u << LB) - 1u;
    const int lane = threadIdx.x % kWarp;
    const unsigned gmask = GS == 32 ? kFull : (((1u << GS) - 1u) << (lane & ~(GS - 1)));

    uint32_t pidx[N];   // sorted: expert index (within the lane) of position q at bits q*LB
#pragma unroll
    for (int n = 0; n < N; ++n) pidx[n] = 0;
    if constexpr (kSorted) {
        uint32_t ix[N][EPL];
#pragma unroll
        for (int n = 0; n < N; ++n)
#pragma unroll
            for (int i = 0; i < EPL; ++i) ix[n][i] = uint32_t(i);
#pragma unroll
        for (int p = 0; p < EPL; ++p) {
#pragma unroll
            for (int i = p & 1; i + 1 < EPL; i += 2) {
#pragma unroll
                for (int n = 0; n < N; ++n) {
                    const bool sw = key[n][i + 1] > key[n][i];
                    const uint32_t k0 = sw ? key[n][i + 1] : key[n][i], k1 = sw ? key[n][i] : key[n][i + 1];
                    const uint32_t i0 = sw ? ix[n][i + 1] : ix[n][i], i1 = sw ? ix[n][i] : ix[n][i + 1];
                    key[n][i] = k0; key[n][i + 1] = k1; ix[n][i] = i0; ix[n][i + 1] = i1;
                }
            }
        }
#pragma unroll
        for (int n = 0; n < N; ++n)
#pragma unroll
            for (int i = 0; i < EPL; ++i) pidx[n] |= ix[n][i] << (i * LB);
    }
    // this lane's offer for token n: best key and its expert index within the lane
    uint32_t bk[N];
    int bi[N];
    auto offer = [&](int n) {
        if constexpr (kSorted) {
            bk[n] = key[n][0];
            bi[n] = int(pidx[n] & kIdxMask);
        } else {
            bk[n] = key[n][0];
            bi[n] = 0;
#pragma unroll
            for (int i = 1; i < EPL; ++i)
                if (key[n][i] > bk[n]) { bk[n] = key[n][i]; bi[n] = i; }
        }
    };

    uint32_t top[N];
    float vmax[N], z[N];
#pragma unroll
    for (int n = 0; n < N; ++n) offer(n);
#pragma unroll
    for (int n = 0; n < N; ++n) top[n] = group_max<GS>(bk[n]);   // the first pick's key
#pragma unroll
    for (int n = 0; n < N; ++n) {
        vmax[n] = key_value(top[n]);
        z[n] = 0.0f;
    }
    // Softmax denominator over all E experts (only without renormalisation),
    // taken before the picks remove keys.
    if (!a.renorm) {
#pragma unroll
        for (int n = 0; n < N; ++n)
#pragma unroll
            for (int i = 0; i < EPL; ++i)
                if (key[n][i] != 0u) z[n] += expf(key_value(key[n][i]) - vmax[n]);
#pragma unroll
        for (int n = 0; n < N; ++n) z[n] = group_sum<GS>(z[n]);
    }

    uint32_t my_key[N];
    int my_id[N];
#pragma unroll
    for (int n = 0; n < N; ++n) { my_key[n] = 0; my_id[n] = 0; }
#pragma unroll
    for (int j = 0; j < kMaxTopk; ++j) {
        if (j >= a.k) break;
        uint32_t gk[N];
        unsigned bal[N];
        int ol[N], id[N];
        if (j > 0) {
#pragma unroll
            for (int n = 0; n < N; ++n) offer(n);
#pragma unroll
            for (int n = 0; n < N; ++n) gk[n] = group_max<GS>(bk[n]);
        } else {
#pragma unroll
            for (int n = 0; n < N; ++n) gk[n] = top[n];
        }
#pragma unroll
        for (int n = 0; n < N; ++n) bal[n] = __ballot_sync(kFull, bk[n] == gk[n]) & gmask;
#pragma unroll
        for (int n = 0; n < N; ++n) ol[n] = __ffs(bal[n]) - 1;   // owner: a lane of this group
#pragma unroll
        for (int n = 0; n < N; ++n) id[n] = __shfl_sync(kFull, gl * EPL + bi[n], ol[n]);
#pragma unroll
        for (int n = 0; n < N; ++n) {
            const bool own = ol[n] == lane;
            if constexpr (kSorted) {
#pragma unroll
                for (int i = 0; i + 1 < EPL; ++i) key[n][i] = own ? key[n][i + 1] : key[n][i];
                key[n][EPL - 1] = own ? 0u : key[n][EPL - 1];
                pidx[n] = own ? pidx[n] >> LB : pidx[n];
            } else {
#pragma unroll
                for (int i = 0; i < EPL; ++i) key[n][i] = (own && i == bi[n]) ? 0u : key[n][i];
            }
            if (gl == j) { my_key[n] = gk[n]; my_id[n] = id[n]; }
        }
    }

    // Weights in float32. The largest logit is the first pick.
    const bool mine = gl < a.k;
    float ej[N], denom[N];
#pragma unroll
    for (int n = 0; n < N; ++n) {
        ej[n] = mine ? expf(key_value(my_key[n]) - vmax[n]) : 0.0f;
        denom[n] = a.renorm ? ej[n] : z[n];   // sum over the k picks (lanes 0..k-1), or over all E
    }
    if (a.renorm) {
        for (int o = 1; o < a.k; o <<= 1) {
#pragma unroll
            for (int n = 0; n < N; ++n) denom[n] += __shfl_xor_sync(kFull, denom[n], o);
        }
    }
#pragma unroll
    for (int n = 0; n < N; ++n) {
        out[n] = -1;
        if (valid[n] && mine) {
            if (a.write_out) {
                a.topk_ids[(size_t)t[n] * a.k + gl] = my_id[n];
                a.topk_weights[(size_t)t[n] * a.k + gl] = ej[n] / denom[n];
            }
            out[n] = my_id[n];
        }
    }
}

// One token per lane group (see topk_select_n).
template <int GS, int EPL>
__device__ __forceinline__ int topk_select(const RouteArgs& a, int t, bool valid, int gl, uint32_t (&key)[EPL]) {
    const int tt[1] = {t};
    const bool vv[1] = {valid};
    uint32_t kk[1][EPL];
#pragma unroll
    for (int i = 0; i < EPL; ++i) kk[0][i] = key[i];
    int out[1];
    topk_select_n<GS, EPL, 1>(a, tt, vv, gl, kk, out);
#pragma unroll
    for (int i = 0; i < EPL; ++i) key[i] = kk[0][i];
    return out[0];
}

// Rounds whose (expert, rank) per lane stay in registers until the ranks are
// finished; later rounds (only for very long token runs) go through inv_perm.
constexpr int kRegRounds = 4;

// The same for 32-lane groups (one token per round), two tokens per step:
// a warp selects tokens w0 + r and w0 + r + 1 together (topk_select_n with
// N = 2), keeping rounds r and r + 1 in re/rr. Ranks follow slot order, so
// the first token's slots rank before the second's. A token's k experts are
// distinct, so within one token every pick of an expert is its only one: the
// rank of a pick is the warp's counter of its expert, read after the first
// token's picks have been counted.
template <int EPL, bool LOCAL>
__device__ __forceinline__ void topk_rank_range_pairs(const RouteArgs& a, int t0, int t1, int32_t* s_cnt,
                                                      int (&re)[kRegRounds], int (&rr)[kRegRounds]) {
    constexpr int GS = 32;
    static_assert(kRegRounds % 2 == 0, "rounds in pairs");
    const int lane = threadIdx.x % kWarp;
    const int warp = threadIdx.x / kWarp;
    const int gl = lane;
    int32_t* cnt = s_cnt + (size_t)warp * a.nloc;
    const int w0 = t0 + warp * a.tpw;
    const int w1 = min(t1, w0 + a.tpw);
    auto counted = [&](int e) {
        if constexpr (LOCAL) return (e < 0) ? -1 : (e >= a.e0 && e < a.e0 + a.nloc) ? e - a.e0 : -2;
        else return e;
    };
    // ranks of the two tokens' picks (eA, eB counted indices), in slot order
    auto rank2 = [&](int eA, int eB, int& rA, int& rB) {
        rA = eA >= 0 ? cnt[eA] : 0;
        __syncwarp();
        if (eA >= 0) cnt[eA] = rA + 1;
        __syncwarp();
        rB = eB >= 0 ? cnt[eB] : 0;
        __syncwarp();
        if (eB >= 0) cnt[eB] = rB + 1;
        __syncwarp();
    };

    uint32_t key[2][EPL], next[2][EPL];
    load_keys<GS, EPL>(a, w0, w0 < w1, gl, key[0]);
    load_keys<GS, EPL>(a, w0 + 1, w0 + 1 < w1, gl, key[1]);
#pragma unroll
    for (int r = 0; r < kRegRounds; r += 2) {
        re[r] = re[r + 1] = -1;
        rr[r] = rr[r + 1] = 0;
        const int tA = w0 + r;
        if (tA < w1) {
            load_keys<GS, EPL>(a, tA + 2, tA + 2 < w1, gl, next[0]);
            load_keys<GS, EPL>(a, tA + 3, tA + 3 < w1, gl, next[1]);
            const int tt[2] = {tA, tA + 1};
            const bool vv[2] = {true, tA + 1 < w1};
            int e2[2];
            topk_select_n<GS, EPL, 2>(a, tt, vv, gl, key, e2);
            const int eA = counted(e2[0]), eB = counted(e2[1]);
            int rA, rB;
            rank2(eA, eB, rA, rB);
            re[r] = eA; rr[r] = rA;
            re[r + 1] = eB; rr[r + 1] = rB;
#pragma unroll
            for (int n = 0; n < 2; ++n)
#pragma unroll
                for (int i = 0; i < EPL; ++i) key[n][i] = next[n][i];
        }
    }
    for (int tA = w0 + kRegRounds; tA < w1; tA += 2) {
        const int tt[2] = {tA, tA + 1};
        const bool vv[2] = {true, tA + 1 < w1};
        int e2[2];
        topk_select_n<GS, EPL, 2>(a, tt, vv, gl, key, e2);
        load_keys<GS, EPL>(a, tA + 2, tA + 2 < w1, gl, key[0]);
        load_keys<GS, EPL>(a, tA + 3, tA + 3 < w1, gl, key[1]);
        const int eA = counted(e2[0]), eB = counted(e2[1]);
        int rA, rB;
        rank2(eA, eB, rA, rB);
        if (eA >= 0) a.inv_perm[(size_t)tA * a.k + gl] = rA;
        if (eA == -2) a.inv_perm[(size_t)tA * a.k + gl] = -1;
        if (eB >= 0) a.inv_perm[(size_t)(tA + 1) * a.k + gl] = rB;
        if (eB == -2) a.inv_perm[(size_t)(tA + 1) * a.k + gl] = -1;
    }
}

// Top-k of the tokens [t0, t1) and the rank of every slot among this warp's
// slots of the same expert; s_cnt is [NW][nloc] and counts each warp's picks
// per counted expert. Warp w owns tokens [t0 + w*tpw, t0 + (w+1)*tpw); each
// round takes GPW consecutive tokens, one per lane group, so lane order
// within a round is slot order. The first R rounds return each
// lane's counted expert and rank in re/rr (re: -1 no slot, -2 a slot whose
// expert is not counted); the rank of later rounds is written to inv_perm[s]
// (-1 for uncounted slots). The next round's logits are loaded before the
// current round's selection. LOCAL counts only experts [e0, e0 + nloc).
template <int GS, int EPL, int NT, bool LOCAL = false, int N = 1, int R = kRegRounds>
__device__ __forceinline__ void topk_rank_range(const RouteArgs& a, int t0, int t1, int32_t* s_cnt,
                                                int (&re)[R], int (&rr)[R]) {
    if constexpr (N == 2) {
        static_assert(R == kRegRounds, "pairs keep kRegRounds rounds in registers");
        topk_rank_range_pairs<EPL, LOCAL>(a, t0, t1, s_cnt, re, rr);
        return;
    }
    constexpr int GPW = kWarp / GS;
    const int lane = threadIdx.x % kWarp;
    const int warp = threadIdx.x / kWarp;
    const int grp = lane / GS;
    const int gl = lane % GS;
    const unsigned lower = (1u << lane) - 1u;
    int32_t* cnt = s_cnt + (size_t)warp * a.nloc;
    const int w0 = t0 + warp * a.tpw;
    const int w1 = min(t1, w0 + a.tpw);
    auto counted = [&](int e) {
        if constexpr (LOCAL) return (e < 0) ? -1 : (e >= a.e0 && e < a.e0 + a.nloc) ? e - a.e0 : -2;
        else return e;
    };

    uint32_t key[EPL], next[EPL];
    load_keys<GS, EPL>(a, w0 + grp, w0 + grp < w1, gl, key);
#pragma unroll
    for (int r = 0; r < R; ++r) {
        re[r] = -1;
        rr[r] = 0;
        const int tb = w0 + r * GPW;
        if (tb < w1) {
            const int tn = tb + GPW + grp;
            load_keys<GS, EPL>(a, tn, tn < w1, gl, next);
            const int t = tb + grp;
            const int e = counted(topk_select<GS, EPL>(a, t, t < w1, gl, key));
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
    for (int tb = w0 + R * GPW; tb < w1; tb += GPW) {
        const int t = tb + grp;
        const int e = counted(topk_select<GS, EPL>(a, t, t < w1, gl, key));
        const int tn = tb + GPW + grp;
        load_keys<GS, EPL>(a, tn, tn < w1, gl, key);
        const unsigned peers = __match_any_sync(kFull, e);
        if (e >= 0) a.inv_perm[(size_t)t * a.k + gl] = cnt[e] + __popc(peers & lower);
        if (e == -2) a.inv_perm[(size_t)t * a.k + gl] = -1;
        __syncwarp();
        if (e >= 0 && lane == __ffs(peers) - 1) cnt[e] += __popc(peers);
        __syncwarp();
    }
}

// Zero this warp's row of the per-warp counters s_cnt[NW][nloc]; only the
// warp itself touches the row until the scan over warps, so a warp barrier is
// enough.
__device__ __forceinline__ void zero_warp_counters(int32_t* s_cnt, int nloc) {
    int32_t* c = s_cnt + (size_t)(threadIdx.x / kWarp) * nloc;
    for (int i = threadIdx.x % kWarp; i < nloc; i += kWarp) c[i] = 0;
    __syncwarp();
}

// Exclusive scan over warps of s_cnt[w][e] for every expert; s_tot[e] gets
// the block total.
template <int NT>
__device__ __forceinline__ void scan_over_warps(int32_t* s_cnt, int32_t* s_tot, int E) {
    constexpr int NW = NT / kWarp;
    for (int e = threadIdx.x; e < E; e += NT) {
        int v[NW];   // all loads first: one shared-memory round trip, not NW
#pragma unroll
        for (int w = 0; w < NW; ++w) v[w] = s_cnt[(size_t)w * E + e];
        int run = 0;
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            s_cnt[(size_t)w * E + e] = run;
            run += v[w];
        }
        s_tot[e] = run;
    }
}

// Exclusive scan of in[0..n) into out[0..n) (may alias) by a block of NT
// threads, n <= MOE_MAX_EXPERTS; returns the total. Uses s_warp[32].
template <int NT>
__device__ int block_exclusive_scan(const int32_t* in, int32_t* out, int n, int32_t* s_warp) {
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
    const int total = s_warp[NW - 1];
    __syncthreads();
    return total;
}

// Add each slot's per-warp start to its within-warp rank (s_cnt now holds
// the exclusive scan over warps). With PLACE (one-block paths) the expert's
// offset is added too and the result is final: it goes to perm/inv_perm when
// a.write_out and, if s_inv is given, to s_inv[s] (shared memory). Slots of
// uncounted experts (LOCAL) get inv_perm -1.
template <int GS, int NT, bool PLACE, bool LOCAL = false, int R = kRegRounds>
__device__ __forceinline__ void finish_ranks(const RouteArgs& a, int t0, int t1, const int32_t* s_cnt,
                                             const int32_t* s_off, const int (&re)[R],
                                             const int (&rr)[R], int32_t* s_inv = nullptr) {
    constexpr int GPW = kWarp / GS;
    const int lane = threadIdx.x % kWarp;
    const int warp = threadIdx.x / kWarp;
    const int grp = lane / GS;
    const int gl = lane % GS;
    const int32_t* start = s_cnt + (size_t)warp * a.nloc;
    const int w0 = t0 + warp * a.tpw;
    const int w1 = min(t1, w0 + a.tpw);
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const int s = (w0 + r * GPW + grp) * a.k + gl;
        if (re[r] >= 0) {
            int p = rr[r] + start[re[r]];
            if constexpr (PLACE) {
                p += s_off[re[r]];
                if (a.write_out) a.perm[p] = s;
                if (s_inv != nullptr) s_inv[s] = p;
            }
            if (a.write_out) a.inv_perm[s] = p;
        } else if (LOCAL && re[r] == -2) {
            if (a.write_out) a.inv_perm[s] = -1;
            if (PLACE && s_inv != nullptr) s_inv[s] = -1;
        }
    }
    // slots of rounds past R (the two-kernel path only, where
    // write_out holds): the rank was kept in inv_perm
    const int s_lo = (w0 + R * GPW) * a.k;
    for (int s = s_lo + lane; s < w1 * a.k; s += kWarp) {
        int e = __ldcg(a.topk_ids + s);
        if constexpr (LOCAL) {
            e -= a.e0;
            if (e < 0 || e >= a.nloc) continue;   // inv_perm already -1
        }
        int p = __ldcg(a.inv_perm + s) + start[e];
        if constexpr (PLACE) {
            p += s_off[e];
            a.perm[p] = s;
            if (s_inv != nullptr) s_inv[s] = p;
        }
        a.inv_perm[s] = p;
    }
}

}  // namespace moe
