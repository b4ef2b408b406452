// C-ABI entry points (declared in include/moe_glue.h): argument validation on
// the host, then one launch sequence on the caller's stream. No allocation,
// no synchronisation, no host copies, no fallback path.
#include "moe_glue.h"
#include "moe_launch.h"

#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

namespace {

using moe::RoutePlan;

constexpr int kMaxDevices = 64;
std::atomic<int> g_sm_count[kMaxDevices];

// SM count of the current device (cached per device; racing first calls all
// store the same value).
cudaError_t current_sm_count(int* out) {
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev >= 0 && dev < kMaxDevices) {
        const int cached = g_sm_count[dev].load(std::memory_order_relaxed);
        if (cached > 0) { *out = cached; return cudaSuccess; }
    }
    int sms = 0;
    err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (err != cudaSuccess) return err;
    if (dev >= 0 && dev < kMaxDevices) g_sm_count[dev].store(sms, std::memory_order_relaxed);
    *out = sms;
    return cudaSuccess;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

struct Range {
    const void* p;
    uint64_t bytes;
};

bool overlap(Range a, Range b) {
    if (a.bytes == 0 || b.bytes == 0) return false;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a.p), b0 = reinterpret_cast<uintptr_t>(b.p);
    return a0 < b0 + b.bytes && b0 < a0 + a.bytes;
}

bool any_overlap(std::initializer_list<Range> outs, std::initializer_list<Range> ins) {
    for (auto o = outs.begin(); o != outs.end(); ++o) {
        for (const Range& i : ins)
            if (overlap(*o, i)) return true;
        for (auto o2 = o + 1; o2 != outs.end(); ++o2)
            if (overlap(*o, *o2)) return true;
    }
    return false;
}

moe_status_t check_route_sizes(int64_t T, int E, int k) {
    if (T < 0 || E < 1 || k < 1 || k > E) return MOE_ERR_INVALID_ARG;
    if (E > MOE_MAX_EXPERTS || k > MOE_MAX_TOPK) return MOE_ERR_UNSUPPORTED;
    if (T * int64_t(k) >= (int64_t(1) << 31)) return MOE_ERR_UNSUPPORTED;
    return MOE_OK;
}

// Rows of bfloat16 vectors: width a multiple of 8 elements (16 bytes).
moe_status_t check_rows(int64_t rows, int width, int64_t slots_mult) {
    if (rows < 0 || width < 1) return MOE_ERR_INVALID_ARG;
    if (width % 8 != 0) return MOE_ERR_MISALIGNED;
    if (rows * slots_mult >= (int64_t(1) << 31)) return MOE_ERR_UNSUPPORTED;
    return MOE_OK;
}

moe_status_t from_cuda(cudaError_t err) { return err == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

// Local routing arguments: 0 <= e0 < e1 <= E, pad >= 1, padded capacity < 2^31.
moe_status_t check_local(int64_t T, int E, int k, int e0, int e1, int pad, int64_t* rows) {
    moe_status_t st = check_route_sizes(T, E, k);
    if (st != MOE_OK) return st;
    if (e0 < 0 || e1 > E || e0 >= e1 || pad < 1) return MOE_ERR_INVALID_ARG;
    const int64_t r = T * int64_t(k) + int64_t(e1 - e0) * int64_t(pad - 1);
    if (r >= (int64_t(1) << 31)) return MOE_ERR_UNSUPPORTED;
    if (rows) *rows = r;
    return MOE_OK;
}

}  // namespace

extern "C" {

const char* moe_status_string(moe_status_t status) {
    switch (status) {
        case MOE_OK: return "MOE_OK";
        case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
        case MOE_ERR_MISALIGNED: return "MOE_ERR_MISALIGNED";
        case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
        case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE";
        case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
    }
    return "MOE_ERR_UNKNOWN";
}

moe_status_t moe_route_workspace_size(int64_t T, int E, int k, size_t* bytes) {
    if (bytes == nullptr) return MOE_ERR_INVALID_ARG;
    const moe_status_t st = check_route_sizes(T, E, k);
    if (st != MOE_OK) return st;
    *bytes = T == 0 ? 0 : moe::plan_route(T, E, k).ws_bytes;
    return MOE_OK;
}

moe_status_t moe_route(const float* logits, int64_t T, int E, int k, int renorm,
                       int32_t* topk_ids, float* topk_weights, int32_t* expert_counts,
                       int32_t* expert_offsets, int32_t* perm, int32_t* inv_perm,
                       void* workspace, size_t workspace_bytes, moe_stream_t stream) {
    moe_status_t st = check_route_sizes(T, E, k);
    if (st != MOE_OK) return st;
    if (expert_counts == nullptr || expert_offsets == nullptr) return MOE_ERR_INVALID_ARG;
    if (!aligned4(expert_counts) || !aligned4(expert_offsets)) return MOE_ERR_MISALIGNED;
    const uint64_t S = uint64_t(T) * uint64_t(k);
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (T == 0) {
        if (any_overlap({{expert_counts, 4ull * E}, {expert_offsets, 4ull * (E + 1)}}, {}))
            return MOE_ERR_INVALID_ARG;
        cudaError_t err = cudaMemsetAsync(expert_counts, 0, sizeof(int32_t) * E, s);
        if (err == cudaSuccess) err = cudaMemsetAsync(expert_offsets, 0, sizeof(int32_t) * (E + 1), s);
        return from_cuda(err);
    }
    if (logits == nullptr || topk_ids == nullptr || topk_weights == nullptr || perm == nullptr ||
        inv_perm == nullptr)
        return MOE_ERR_INVALID_ARG;
    if (!aligned4(logits) || !aligned4(topk_ids) || !aligned4(topk_weights) || !aligned4(perm) ||
        !aligned4(inv_perm))
        return MOE_ERR_MISALIGNED;
    const RoutePlan plan = moe::plan_route(T, E, k);
    if (plan.ws_bytes > 0) {
        if (workspace == nullptr || workspace_bytes < plan.ws_bytes) return MOE_ERR_WORKSPACE;
        if (!aligned16(workspace)) return MOE_ERR_MISALIGNED;
    }
    const uint64_t ws = plan.ws_bytes;
    if (any_overlap({{topk_ids, 4 * S}, {topk_weights, 4 * S}, {expert_counts, 4ull * E},
                     {expert_offsets, 4ull * (E + 1)}, {perm, 4 * S}, {inv_perm, 4 * S},
                     {workspace, ws}},
                    {{logits, 4ull * uint64_t(T) * E}}))
        return MOE_ERR_INVALID_ARG;
    return from_cuda(moe::launch_route(plan, logits, int(T), E, k, renorm ? 1 : 0, topk_ids,
                                       topk_weights, expert_counts, expert_offsets, perm, inv_perm,
                                       workspace, s));
}

moe_status_t moe_route_expand(const float* logits, int64_t T, int E, int k, int renorm,
                              const moe_bf16_t* x, int H, int32_t* topk_ids, float* topk_weights,
                              int32_t* expert_counts, int32_t* expert_offsets, int32_t* perm,
                              int32_t* inv_perm, moe_bf16_t* expanded_x, void* workspace,
                              size_t workspace_bytes, moe_stream_t stream) {
    moe_status_t st = check_route_sizes(T, E, k);
    if (st != MOE_OK) return st;
    if ((st = check_rows(T, H, k)) != MOE_OK) return st;
    if (T > 0) {
        if (x == nullptr || expanded_x == nullptr) return MOE_ERR_INVALID_ARG;
        if (!aligned16(x) || !aligned16(expanded_x)) return MOE_ERR_MISALIGNED;
        const uint64_t S = uint64_t(T) * uint64_t(k);
        const uint64_t ws = moe::plan_route(T, E, k).ws_bytes;
        // expanded_x against every other buffer of the call
        if (any_overlap({{expanded_x, 2 * S * uint64_t(H)}},
                        {{x, 2 * uint64_t(T) * uint64_t(H)}, {logits, 4ull * uint64_t(T) * E},
                         {topk_ids, 4 * S}, {topk_weights, 4 * S}, {expert_counts, 4ull * E},
                         {expert_offsets, 4ull * (E + 1)}, {perm, 4 * S}, {inv_perm, 4 * S},
                         {workspace, ws}}))
            return MOE_ERR_INVALID_ARG;
        // x is an input of the expansion: no routing output may overlap it
        if (any_overlap({{x, 2 * uint64_t(T) * uint64_t(H)}},
                        {{topk_ids, 4 * S}, {topk_weights, 4 * S}, {expert_counts, 4ull * E},
                         {expert_offsets, 4ull * (E + 1)}, {perm, 4 * S}, {inv_perm, 4 * S},
                         {workspace, ws}}))
            return MOE_ERR_INVALID_ARG;
    }
    const moe::RoutePlan plan = moe::plan_route(T, E, k);
    if (T > 0 && moe::route_expand_fits(plan)) {
        // validate the routing arguments exactly as moe_route does
        if (expert_counts == nullptr || expert_offsets == nullptr || logits == nullptr ||
            topk_ids == nullptr || topk_weights == nullptr || perm == nullptr || inv_perm == nullptr)
            return MOE_ERR_INVALID_ARG;
        if (!aligned4(expert_counts) || !aligned4(expert_offsets) || !aligned4(logits) ||
            !aligned4(topk_ids) || !aligned4(topk_weights) || !aligned4(perm) || !aligned4(inv_perm))
            return MOE_ERR_MISALIGNED;
        const uint64_t S = uint64_t(T) * uint64_t(k);
        if (any_overlap({{topk_ids, 4 * S}, {topk_weights, 4 * S}, {expert_counts, 4ull * E},
                         {expert_offsets, 4ull * (E + 1)}, {perm, 4 * S}, {inv_perm, 4 * S}},
                        {{logits, 4ull * uint64_t(T) * E}}))
            return MOE_ERR_INVALID_ARG;
        int sms = 0;
        if (current_sm_count(&sms) != cudaSuccess) return MOE_ERR_CUDA;
        return from_cuda(moe::launch_route_expand(
            plan, logits, int(T), E, k, renorm ? 1 : 0, topk_ids, topk_weights, expert_counts,
            expert_offsets, perm, inv_perm, x, H, expanded_x, sms, reinterpret_cast<cudaStream_t>(stream)));
    }
    st = moe_route(logits, T, E, k, renorm, topk_ids, topk_weights, expert_counts, expert_offsets,
                   perm, inv_perm, workspace, workspace_bytes, stream);
    if (st != MOE_OK || T == 0) return st;
    return moe_expand(x, T, H, k, inv_perm, expanded_x, stream);
}

moe_status_t moe_route_local_rows(int64_t T, int k, int e0, int e1, int pad, int64_t* rows) {
    if (rows == nullptr || T < 0 || k < 1 || e0 < 0 || e0 >= e1 || pad < 1) return MOE_ERR_INVALID_ARG;
    const int64_t r = T * int64_t(k) + int64_t(e1 - e0) * int64_t(pad - 1);
    if (r >= (int64_t(1) << 31)) return MOE_ERR_UNSUPPORTED;
    *rows = r;
    return MOE_OK;
}

moe_status_t moe_route_local_workspace_size(int64_t T, int E, int k, int e0, int e1, size_t* bytes) {
    if (bytes == nullptr) return MOE_ERR_INVALID_ARG;
    const moe_status_t st = check_local(T, E, k, e0, e1, 1, nullptr);
    if (st != MOE_OK) return st;
    *bytes = T == 0 ? 0 : moe::plan_route(T, E, k, e1 - e0).ws_bytes;
    return MOE_OK;
}

moe_status_t moe_route_local(const float* logits, int64_t T, int E, int k, int renorm, int e0,
                             int e1, int pad, int32_t* topk_ids, float* topk_weights,
                             int32_t* expert_counts, int32_t* expert_offsets, int32_t* perm,
                             int32_t* inv_perm, void* workspace, size_t workspace_bytes,
                             moe_stream_t stream) {
    int64_t rows = 0;
    moe_status_t st = check_local(T, E, k, e0, e1, pad, &rows);
    if (st != MOE_OK) return st;
    const int n = e1 - e0;
    if (expert_counts == nullptr || expert_offsets == nullptr) return MOE_ERR_INVALID_ARG;
    if (!aligned4(expert_counts) || !aligned4(expert_offsets)) return MOE_ERR_MISALIGNED;
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (T == 0) {
        if (any_overlap({{expert_counts, 4ull * n}, {expert_offsets, 4ull * (n + 1)}, {perm, 4ull * rows}}, {}))
            return MOE_ERR_INVALID_ARG;
        cudaError_t err = cudaMemsetAsync(expert_counts, 0, sizeof(int32_t) * n, s);
        if (err == cudaSuccess) err = cudaMemsetAsync(expert_offsets, 0, sizeof(int32_t) * (n + 1), s);
        if (err == cudaSuccess && rows > 0) {
            if (perm == nullptr) return MOE_ERR_INVALID_ARG;
            err = cudaMemsetAsync(perm, 0xff, sizeof(int32_t) * rows, s);   // all -1
        }
        return from_cuda(err);
    }
    if (logits == nullptr || topk_ids == nullptr || topk_weights == nullptr || perm == nullptr ||
        inv_perm == nullptr)
        return MOE_ERR_INVALID_ARG;
    if (!aligned4(logits) || !aligned4(topk_ids) || !aligned4(topk_weights) || !aligned4(perm) ||
        !aligned4(inv_perm))
        return MOE_ERR_MISALIGNED;
    const moe::RoutePlan plan = moe::plan_route(T, E, k, n);
    if (plan.ws_bytes > 0) {
        if (workspace == nullptr || workspace_bytes < plan.ws_bytes) return MOE_ERR_WORKSPACE;
        if (!aligned16(workspace)) return MOE_ERR_MISALIGNED;
    }
    const uint64_t S = uint64_t(T) * uint64_t(k);
    if (any_overlap({{topk_ids, 4 * S}, {topk_weights, 4 * S}, {expert_counts, 4ull * n},
                     {expert_offsets, 4ull * (n + 1)}, {perm, 4ull * rows}, {inv_perm, 4 * S},
                     {workspace, plan.ws_bytes}},
                    {{logits, 4ull * uint64_t(T) * E}}))
        return MOE_ERR_INVALID_ARG;
    const moe::LocalRange local{e0, n, pad, int(rows)};
    return from_cuda(moe::launch_route(plan, logits, int(T), E, k, renorm ? 1 : 0, topk_ids,
                                       topk_weights, expert_counts, expert_offsets, perm, inv_perm,
                                       workspace, s, &local));
}

moe_status_t moe_expand_rows(const moe_bf16_t* x, int64_t T, int H, int k, const int32_t* inv_perm,
                             int64_t rows, moe_bf16_t* expanded_x, moe_stream_t stream) {
    if (k < 1) return MOE_ERR_INVALID_ARG;
    if (k > MOE_MAX_TOPK) return MOE_ERR_UNSUPPORTED;
    moe_status_t st = check_rows(T, H, k);
    if (st != MOE_OK) return st;
    if (rows < 0) return MOE_ERR_INVALID_ARG;
    if (rows >= (int64_t(1) << 31)) return MOE_ERR_UNSUPPORTED;
    if (T == 0 || rows == 0) return MOE_OK;
    if (x == nullptr || inv_perm == nullptr || expanded_x == nullptr) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(expanded_x) || !aligned4(inv_perm)) return MOE_ERR_MISALIGNED;
    const uint64_t S = uint64_t(T) * uint64_t(k);
    if (any_overlap({{expanded_x, 2 * uint64_t(rows) * uint64_t(H)}},
                    {{x, 2 * uint64_t(T) * uint64_t(H)}, {inv_perm, 4 * S}}))
        return MOE_ERR_INVALID_ARG;
    int sms = 0;
    if (current_sm_count(&sms) != cudaSuccess) return MOE_ERR_CUDA;
    return from_cuda(moe::launch_expand(x, T, H, k, inv_perm, rows, expanded_x, sms,
                                        reinterpret_cast<cudaStream_t>(stream)));
}

moe_status_t moe_combine_rows(const moe_bf16_t* expert_out, int64_t rows, int64_t T, int H, int k,
                              const float* topk_weights, const int32_t* inv_perm, moe_bf16_t* out,
                              moe_stream_t stream) {
    if (k < 1) return MOE_ERR_INVALID_ARG;
    if (k > MOE_MAX_TOPK) return MOE_ERR_UNSUPPORTED;
    moe_status_t st = check_rows(T, H, k);
    if (st != MOE_OK) return st;
    if (rows < 0) return MOE_ERR_INVALID_ARG;
    if (rows >= (int64_t(1) << 31)) return MOE_ERR_UNSUPPORTED;
    if (T == 0) return MOE_OK;
    if (topk_weights == nullptr || inv_perm == nullptr || out == nullptr ||
        (rows > 0 && expert_out == nullptr))
        return MOE_ERR_INVALID_ARG;
    if ((rows > 0 && !aligned16(expert_out)) || !aligned16(out) || !aligned4(topk_weights) ||
        !aligned4(inv_perm))
        return MOE_ERR_MISALIGNED;
    const uint64_t S = uint64_t(T) * uint64_t(k);
    if (any_overlap({{out, 2 * uint64_t(T) * uint64_t(H)}},
                    {{expert_out, 2 * uint64_t(rows) * uint64_t(H)}, {topk_weights, 4 * S},
                     {inv_perm, 4 * S}}))
        return MOE_ERR_INVALID_ARG;
    int sms = 0;
    if (current_sm_count(&sms) != cudaSuccess) return MOE_ERR_CUDA;
    return from_cuda(moe::launch_combine(expert_out, rows, T, H, k, topk_weights, inv_perm, out, sms,
                                         reinterpret_cast<cudaStream_t>(stream)));
}

moe_status_t moe_expand(const moe_bf16_t* x, int64_t T, int H, int k, const int32_t* inv_perm,
                        moe_bf16_t* expanded_x, moe_stream_t stream) {
    if (k < 1) return MOE_ERR_INVALID_ARG;
    if (k > MOE_MAX_TOPK) return MOE_ERR_UNSUPPORTED;
    moe_status_t st = check_rows(T, H, k);
    if (st != MOE_OK) return st;
    if (T == 0) return MOE_OK;
    if (x == nullptr || inv_perm == nullptr || expanded_x == nullptr) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(expanded_x) || !aligned4(inv_perm)) return MOE_ERR_MISALIGNED;
    const uint64_t S = uint64_t(T) * uint64_t(k);
    if (any_overlap({{expanded_x, 2 * S * uint64_t(H)}},
                    {{x, 2 * uint64_t(T) * uint64_t(H)}, {inv_perm, 4 * S}}))
        return MOE_ERR_INVALID_ARG;
    int sms = 0;
    cudaError_t err = current_sm_count(&sms);
    if (err != cudaSuccess) return MOE_ERR_CUDA;
    return from_cuda(moe::launch_expand(x, T, H, k, inv_perm, T * k, expanded_x, sms,
                                        reinterpret_cast<cudaStream_t>(stream)));
}

moe_status_t moe_swiglu(const moe_bf16_t* gate_up, int64_t rows, int I, moe_bf16_t* act,
                        moe_stream_t stream) {
    moe_status_t st = check_rows(rows, I, 1);
    if (st != MOE_OK) return st;
    if (rows == 0) return MOE_OK;
    if (gate_up == nullptr || act == nullptr) return MOE_ERR_INVALID_ARG;
    if (!aligned16(gate_up) || !aligned16(act)) return MOE_ERR_MISALIGNED;
    if (any_overlap({{act, 2 * uint64_t(rows) * uint64_t(I)}},
                    {{gate_up, 4 * uint64_t(rows) * uint64_t(I)}}))
        return MOE_ERR_INVALID_ARG;
    int sms = 0;
    cudaError_t err = current_sm_count(&sms);
    if (err != cudaSuccess) return MOE_ERR_CUDA;
    return from_cuda(moe::launch_swiglu(gate_up, rows, I, act, sms,
                                        reinterpret_cast<cudaStream_t>(stream)));
}

moe_status_t moe_combine(const moe_bf16_t* expert_out, int64_t T, int H, int k,
                         const float* topk_weights, const int32_t* inv_perm, moe_bf16_t* out,
                         moe_stream_t stream) {
    if (k < 1) return MOE_ERR_INVALID_ARG;
    if (k > MOE_MAX_TOPK) return MOE_ERR_UNSUPPORTED;
    moe_status_t st = check_rows(T, H, k);
    if (st != MOE_OK) return st;
    if (T == 0) return MOE_OK;
    if (expert_out == nullptr || topk_weights == nullptr || inv_perm == nullptr || out == nullptr)
        return MOE_ERR_INVALID_ARG;
    if (!aligned16(expert_out) || !aligned16(out) || !aligned4(topk_weights) ||
        !aligned4(inv_perm))
        return MOE_ERR_MISALIGNED;
    const uint64_t S = uint64_t(T) * uint64_t(k);
    if (any_overlap({{out, 2 * uint64_t(T) * uint64_t(H)}},
                    {{expert_out, 2 * S * uint64_t(H)}, {topk_weights, 4 * S}, {inv_perm, 4 * S}}))
        return MOE_ERR_INVALID_ARG;
    int sms = 0;
    cudaError_t err = current_sm_count(&sms);
    if (err != cudaSuccess) return MOE_ERR_CUDA;
    return from_cuda(moe::launch_combine(expert_out, T * k, T, H, k, topk_weights, inv_perm, out, sms,
                                         reinterpret_cast<cudaStream_t>(stream)));
}

moe_status_t moe_swiglu_mxfp8(const moe_bf16_t* gate_up, int64_t rows, int I, uint8_t* act_codes,
                              uint8_t* act_scales, moe_stream_t stream) {
    moe_status_t st = check_rows(rows, I, 1);
    if (st != MOE_OK) return st;
    if (I % 32 != 0) return MOE_ERR_MISALIGNED;
    if (rows == 0) return MOE_OK;
    if (gate_up == nullptr || act_codes == nullptr || act_scales == nullptr) return MOE_ERR_INVALID_ARG;
    if (!aligned16(gate_up) || !aligned16(act_codes)) return MOE_ERR_MISALIGNED;
    const uint64_t n = uint64_t(rows) * uint64_t(I);
    if (any_overlap({{act_codes, n}, {act_scales, n / 32}}, {{gate_up, 4 * n}}))
        return MOE_ERR_INVALID_ARG;
    int sms = 0;
    if (current_sm_count(&sms) != cudaSuccess) return MOE_ERR_CUDA;
    return from_cuda(moe::launch_swiglu_mxfp8(gate_up, rows, I, act_codes, act_scales, sms,
                                              reinterpret_cast<cudaStream_t>(stream)));
}

moe_status_t moe_expand_mxfp8(const moe_bf16_t* x, int64_t T, int H, int k, const int32_t* inv_perm,
                              int64_t rows, uint8_t* codes, uint8_t* scales, moe_stream_t stream) {
    if (k < 1) return MOE_ERR_INVALID_ARG;
    if (k > MOE_MAX_TOPK) return MOE_ERR_UNSUPPORTED;
    moe_status_t st = check_rows(T, H, k);
    if (st != MOE_OK) return st;
    if (H % 32 != 0) return MOE_ERR_MISALIGNED;
    if (rows < 0) return MOE_ERR_INVALID_ARG;
    if (rows >= (int64_t(1) << 31)) return MOE_ERR_UNSUPPORTED;
    if (T == 0 || rows == 0) return MOE_OK;
    if (x == nullptr || inv_perm == nullptr || codes == nullptr || scales == nullptr)
        return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(codes) || !aligned4(inv_perm)) return MOE_ERR_MISALIGNED;
    const uint64_t S = uint64_t(T) * uint64_t(k);
    const uint64_t n = uint64_t(rows) * uint64_t(H);
    if (any_overlap({{codes, n}, {scales, n / 32}},
                    {{x, 2 * uint64_t(T) * uint64_t(H)}, {inv_perm, 4 * S}}))
        return MOE_ERR_INVALID_ARG;
    int sms = 0;
    if (current_sm_count(&sms) != cudaSuccess) return MOE_ERR_CUDA;
    return from_cuda(moe::launch_expand_mxfp8(x, T, H, k, inv_perm, rows, codes, scales, sms,
                                              reinterpret_cast<cudaStream_t>(stream)));
}

namespace {

// The FP4 format arguments: a known format, n a multiple of its block, and
// for NVFP4 a finite positive tensor scale.
moe_status_t check_fp4(int format, int n, float global_scale) {
    if (format != MOE_FP4_NVFP4 && format != MOE_FP4_MXFP4) return MOE_ERR_INVALID_ARG;
    if (format == MOE_FP4_NVFP4 && !(global_scale > 0.0f && global_scale <= 3.4028234663852886e38f))
        return MOE_ERR_INVALID_ARG;
    if (n % (format == MOE_FP4_NVFP4 ? 16 : 32) != 0) return MOE_ERR_MISALIGNED;
    return MOE_OK;
}

}  // namespace

moe_status_t moe_swiglu_fp4(const moe_bf16_t* gate_up, int64_t rows, int I, int format,
                            float global_scale, uint8_t* act_codes, uint8_t* act_scales,
                            moe_stream_t stream) {
    moe_status_t st = check_rows(rows, I, 1);
    if (st != MOE_OK) return st;
    if ((st = check_fp4(format, I, global_scale)) != MOE_OK) return st;
    if (rows == 0) return MOE_OK;
    if (gate_up == nullptr || act_codes == nullptr || act_scales == nullptr) return MOE_ERR_INVALID_ARG;
    if (!aligned16(gate_up) || !aligned16(act_codes)) return MOE_ERR_MISALIGNED;
    const uint64_t n = uint64_t(rows) * uint64_t(I);
    const uint64_t block = format == MOE_FP4_NVFP4 ? 16 : 32;
    if (any_overlap({{act_codes, n / 2}, {act_scales, n / block}}, {{gate_up, 4 * n}}))
        return MOE_ERR_INVALID_ARG;
    int sms = 0;
    if (current_sm_count(&sms) != cudaSuccess) return MOE_ERR_CUDA;
    return from_cuda(moe::launch_swiglu_fp4(gate_up, rows, I, format == MOE_FP4_NVFP4, global_scale, act_codes,
                                            act_scales, sms, reinterpret_cast<cudaStream_t>(stream)));
}

moe_status_t moe_expand_fp4(const moe_bf16_t* x, int64_t T, int H, int k, const int32_t* inv_perm,
                            int64_t rows, int format, float global_scale, uint8_t* codes,
                            uint8_t* scales, moe_stream_t stream) {
    if (k < 1) return MOE_ERR_INVALID_ARG;
    if (k > MOE_MAX_TOPK) return MOE_ERR_UNSUPPORTED;
    moe_status_t st = check_rows(T, H, k);
    if (st != MOE_OK) return st;
    if ((st = check_fp4(format, H, global_scale)) != MOE_OK) return st;
    if (rows < 0) return MOE_ERR_INVALID_ARG;
    if (rows >= (int64_t(1) << 31)) return MOE_ERR_UNSUPPORTED;
    if (T == 0 || rows == 0) return MOE_OK;
    if (x == nullptr || inv_perm == nullptr || codes == nullptr || scales == nullptr)
        return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(codes) || !aligned4(inv_perm)) return MOE_ERR_MISALIGNED;
    const uint64_t S = uint64_t(T) * uint64_t(k);
    const uint64_t n = uint64_t(rows) * uint64_t(H);
    const uint64_t block = format == MOE_FP4_NVFP4 ? 16 : 32;
    if (any_overlap({{codes, n / 2}, {scales, n / block}},
                    {{x, 2 * uint64_t(T) * uint64_t(H)}, {inv_perm, 4 * S}}))
        return MOE_ERR_INVALID_ARG;
    int sms = 0;
    if (current_sm_count(&sms) != cudaSuccess) return MOE_ERR_CUDA;
    return from_cuda(moe::launch_expand_fp4(x, T, H, k, inv_perm, rows, format == MOE_FP4_NVFP4, global_scale,
                                            codes, scales, sms, reinterpret_cast<cudaStream_t>(stream)));
}

moe_status_t moe_qk_rmsnorm(moe_bf16_t* q, moe_bf16_t* k, int64_t T, int num_q_heads,
                            int num_k_heads, int head_dim, const moe_bf16_t* q_weight,
                            const moe_bf16_t* k_weight, float weight_bias, float eps,
                            moe_stream_t stream) {
    if (T < 0 || num_q_heads < 0 || num_k_heads < 0 || num_q_heads + num_k_heads < 1)
        return MOE_ERR_INVALID_ARG;
    if (head_dim != 64 && head_dim != 128 && head_dim != 256) return MOE_ERR_UNSUPPORTED;
    if (T * int64_t(num_q_heads + num_k_heads) >= (int64_t(1) << 31)) return MOE_ERR_UNSUPPORTED;
    if (T == 0) return MOE_OK;
    if ((num_q_heads > 0 && q == nullptr) || (num_k_heads > 0 && k == nullptr) ||
        q_weight == nullptr || k_weight == nullptr)
        return MOE_ERR_INVALID_ARG;
    if ((num_q_heads > 0 && !aligned16(q)) || (num_k_heads > 0 && !aligned16(k)) ||
        !aligned16(q_weight) || !aligned16(k_weight))
        return MOE_ERR_MISALIGNED;
    const uint64_t qb = 2 * uint64_t(T) * uint64_t(num_q_heads) * uint64_t(head_dim);
    const uint64_t kb = 2 * uint64_t(T) * uint64_t(num_k_heads) * uint64_t(head_dim);
    if (any_overlap({{q, qb}, {k, kb}}, {{q_weight, 2ull * head_dim}, {k_weight, 2ull * head_dim}}))
        return MOE_ERR_INVALID_ARG;
    int sms = 0;
    if (current_sm_count(&sms) != cudaSuccess) return MOE_ERR_CUDA;
    return from_cuda(moe::launch_qk_rmsnorm(q, k, T, num_q_heads, num_k_heads, head_dim, q_weight,
                                            k_weight, weight_bias, eps, sms,
                                            reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"
