// abi.cu -- the extern "C" entry points declared in include/moe.h: host-side
// argument checks, workspace carving, then kernel launches on the caller's
// stream.  No allocation, no stream synchronisation.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "../../include/moe.h"
#include "kernels.h"

namespace moe {

int sm_count() {
    int dev = 0, n = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    return n > 0 ? n : 1;
}

cudaError_t ensure_dynamic_smem(const void* func, int bytes) {
    constexpr int kSlots = 256;
    static std::mutex mu;
    static const void* seen_func[kSlots];
    static int seen_dev[kSlots];
    static int nseen = 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < nseen; ++i)
        if (seen_func[i] == func && seen_dev[i] == dev) return cudaSuccess;
    e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && nseen < kSlots) {  // a full table only means the call repeats
        seen_func[nseen] = func;
        seen_dev[nseen] = dev;
        ++nseen;
    }
    return e;
}

cudaError_t max_active_clusters(const void* func, int cluster_size, int threads, int smem_bytes, int* clusters) {
    constexpr int kSlots = 64;
    static std::mutex mu;
    static const void* seen_func[kSlots];
    static int seen_dev[kSlots], seen_n[kSlots];
    static int nseen = 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < nseen; ++i)
        if (seen_func[i] == func && seen_dev[i] == dev) {
            *clusters = seen_n[i];
            return cudaSuccess;
        }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(cluster_size);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = (size_t)smem_bytes;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = cluster_size;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, func, &cfg);
    if (e != cudaSuccess) return e;
    if (n < 1) return cudaErrorInvalidConfiguration;
    if (nseen < kSlots) {
        seen_func[nseen] = func;
        seen_dev[nseen] = dev;
        seen_n[nseen] = n;
        ++nseen;
    }
    *clusters = n;
    return cudaSuccess;
}

namespace {

constexpr size_t kAlign = 256;
inline size_t align_up(size_t v) { return (v + kAlign - 1) & ~(kAlign - 1); }

bool aligned16(const void* p) { return p && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_dims(const moe_dims* d) {
    if (!d) return MOE_ERR_INVALID_ARG;
    if (d->T < 1 || d->E < 1 || d->E > 1024 || d->k < 1 || d->k > 32 || d->k > d->E) return MOE_ERR_INVALID_ARG;
    if (d->e0 < 0 || d->e1 <= d->e0 || d->e1 > d->E) return MOE_ERR_INVALID_ARG;
    if ((long long)d->T * d->k >= (1ll << 31)) return MOE_ERR_INVALID_ARG;
    if (d->H < 64 || d->I < 64 || d->H > 16384 || d->I > 16384 || d->H % 64 || d->I % 64) return MOE_ERR_INVALID_ARG;
    // weight rows of all local experts must be addressable by a TMA coordinate
    if ((long long)(d->e1 - d->e0) * (d->H > d->I ? d->H : d->I) >= (1ll << 31)) return MOE_ERR_UNSUPPORTED;
    return MOE_OK;
}

int check_device() {
    int dev = 0, major = 0, minor = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
        return MOE_ERR_CUDA;
    return (major == 10 && minor == 3) ? MOE_OK : MOE_ERR_UNSUPPORTED;
}

int launched(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

size_t pairs_of(const moe_dims* d) { return (size_t)d->T * (size_t)d->k; }

// moe_layer workspace carving (all pieces 256-byte aligned)
struct LayerWs {
    int32_t* topk_idx;
    float* topk_w;
    int32_t* counts;
    int32_t* offsets;
    int32_t* row_pair;
    int32_t* pair_row;
    uint16_t* x_perm;
    float* y_perm;
    void* dispatch_ws;
    void* ffn_ws;
    unsigned* sync;
    size_t dispatch_bytes, ffn_bytes, total;
};

LayerWs carve(const moe_dims* d, void* base) {
    LayerWs w{};
    const size_t P = pairs_of(d), n = (size_t)(d->e1 - d->e0);
    uint8_t* p = static_cast<uint8_t*>(base);
    size_t off = 0;
    auto take = [&](size_t bytes) {
        uint8_t* r = p ? p + off : nullptr;
        off += align_up(bytes);
        return r;
    };
    w.topk_idx = reinterpret_cast<int32_t*>(take(P * 4));
    w.topk_w = reinterpret_cast<float*>(take(P * 4));
    w.counts = reinterpret_cast<int32_t*>(take(n * 4));
    w.offsets = reinterpret_cast<int32_t*>(take((n + 1) * 4));
    w.row_pair = reinterpret_cast<int32_t*>(take(P * 4));
    w.pair_row = reinterpret_cast<int32_t*>(take(P * 4));
    w.x_perm = reinterpret_cast<uint16_t*>(take(P * (size_t)d->H * 2));
    w.y_perm = reinterpret_cast<float*>(take(P * (size_t)d->H * 4));
    w.dispatch_bytes = align_up(dispatch_scratch_bytes((long long)d->T, (int)n));
    w.dispatch_ws = take(w.dispatch_bytes);
    w.ffn_bytes = align_up(ffn_scratch_bytes((long long)P, d->I));
    w.ffn_ws = take(w.ffn_bytes);
    w.sync = reinterpret_cast<unsigned*>(take(64));
    w.total = off;
    return w;
}

// moe_layer_mxfp8 workspace: the routing and dispatch buffers, x and x_perm in
// MXFP8, the MX FFN scratch (h codes and scales) and y_perm
struct MxLayerWs {
    int32_t* topk_idx;
    float* topk_w;
    int32_t* counts;
    int32_t* offsets;
    int32_t* row_pair;
    int32_t* pair_row;
    void* dispatch_ws;
    uint8_t *xpq, *xps;
    void* ffn_ws;
    float* y_perm;
    unsigned* sync;  // grid-barrier words of the fused launch
    size_t dispatch_bytes, total;
};

MxLayerWs carve_mx(const moe_dims* d, void* base) {
    MxLayerWs w{};
    const size_t P = pairs_of(d), n = (size_t)(d->e1 - d->e0), H = (size_t)d->H;
    uint8_t* p = static_cast<uint8_t*>(base);
    size_t off = 0;
    auto take = [&](size_t bytes) {
        uint8_t* r = p ? p + off : nullptr;
        off += align_up(bytes);
        return r;
    };
    w.topk_idx = reinterpret_cast<int32_t*>(take(P * 4));
    w.topk_w = reinterpret_cast<float*>(take(P * 4));
    w.counts = reinterpret_cast<int32_t*>(take(n * 4));
    w.offsets = reinterpret_cast<int32_t*>(take((n + 1) * 4));
    w.row_pair = reinterpret_cast<int32_t*>(take(P * 4));
    w.pair_row = reinterpret_cast<int32_t*>(take(P * 4));
    w.dispatch_bytes = align_up(dispatch_scratch_bytes((long long)d->T, (int)n));
    w.dispatch_ws = take(w.dispatch_bytes);
    w.xpq = take(P * H);
    w.xps = take(P * H / 32);
    w.ffn_ws = take(mx_ffn_scratch_bytes((long long)P, d->I));
    w.y_perm = reinterpret_cast<float*>(take(P * H * 4));
    w.sync = reinterpret_cast<unsigned*>(take(64));
    w.total = off;
    return w;
}

// MXFP8 entries: k-blocks of 128 elements along H and I
int check_mx_dims(const moe_dims* d) {
    const int st = check_dims(d);
    if (st) return st;
    return (d->H % 128 || d->I % 128) ? MOE_ERR_UNSUPPORTED : MOE_OK;
}

bool ws_ok(const void* ws, size_t have, size_t need) {
    if (need == 0) return true;
    return ws && (reinterpret_cast<uintptr_t>(ws) % kAlign) == 0 && have >= need;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

const char* moe_status_string(int s) {
    switch (s) {
        case MOE_OK: return "ok";
        case MOE_ERR_INVALID_ARG: return "invalid argument";
        case MOE_ERR_UNSUPPORTED: return "unsupported device or size";
        case MOE_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
        case MOE_ERR_CUDA: return "CUDA error";
        case MOE_ERR_NONFINITE: return "non-finite router logit";
        case MOE_ERR_TIMEOUT: return "internal wait timed out";
        default: return "unknown status";
    }
}

size_t moe_dispatch_workspace_size(const moe_dims* d) {
    if (check_dims(d) != MOE_OK) return 0;
    return align_up(dispatch_scratch_bytes((long long)d->T, d->e1 - d->e0));
}

size_t moe_expert_ffn_workspace_size(const moe_dims* d) {
    if (check_dims(d) != MOE_OK) return 0;
    return align_up(ffn_scratch_bytes((long long)pairs_of(d), d->I));
}

size_t moe_workspace_size(const moe_dims* d) {
    if (check_dims(d) != MOE_OK) return 0;
    return carve(d, nullptr).total;
}

int moe_route(const moe_dims* d, const float* logits, int32_t* topk_idx, float* topk_w, int32_t* status_dev,
              void* stream) {
    int st = check_dims(d);
    if (st) return st;
    if (!aligned16(logits) || !aligned16(topk_idx) || !aligned16(topk_w)) return MOE_ERR_INVALID_ARG;
    if ((st = check_device())) return st;
    return launched(launch_route(logits, d->T, d->E, d->k, topk_idx, topk_w, status_dev, (cudaStream_t)stream));
}

int moe_dispatch(const moe_dims* d, const uint16_t* x, const int32_t* topk_idx, int32_t* counts, int32_t* offsets,
                 int32_t* row_pair, int32_t* pair_row, uint16_t* x_perm, void* ws, size_t ws_bytes, void* stream) {
    int st = check_dims(d);
    if (st) return st;
    if (!aligned16(x) || !aligned16(topk_idx) || !aligned16(counts) || !aligned16(offsets) || !aligned16(row_pair) ||
        !aligned16(pair_row) || !aligned16(x_perm))
        return MOE_ERR_INVALID_ARG;
    if (!ws_ok(ws, ws_bytes, moe_dispatch_workspace_size(d))) return MOE_ERR_WORKSPACE;
    if ((st = check_device())) return st;
    return launched(launch_dispatch(x, topk_idx, d->T, d->H, d->k, d->e0, d->e1, counts, offsets, row_pair, pair_row,
                                    x_perm, ws, (cudaStream_t)stream));
}

int moe_dispatch_noalloc(const moe_dims* d, const uint16_t* x, const int32_t* topk_idx, int32_t* counts,
                         int32_t* offsets, int32_t* row_pair, int32_t* pair_row, uint16_t* x_perm, void* stream) {
    int st = check_dims(d);
    if (st) return st;
    if (!aligned16(x) || !aligned16(topk_idx) || !aligned16(counts) || !aligned16(offsets) || !aligned16(row_pair) ||
        !aligned16(pair_row) || !aligned16(x_perm))
        return MOE_ERR_INVALID_ARG;
    if (!dispatch_noalloc_fits((long long)pairs_of(d), d->e1 - d->e0)) return MOE_ERR_UNSUPPORTED;
    if ((st = check_device())) return st;
    return launched(launch_dispatch_noalloc(x, topk_idx, d->T, d->H, d->k, d->e0, d->e1, counts, offsets, row_pair,
                                            pair_row, x_perm, (cudaStream_t)stream));
}

int moe_expert_ffn(const moe_dims* d, const uint16_t* x_perm, const int32_t* offsets, const uint16_t* w_gate,
                   const uint16_t* w_up, const uint16_t* w_down, float* y_perm, void* ws, size_t ws_bytes,
                   int32_t* status_dev, void* stream) {
    int st = check_dims(d);
    if (st) return st;
    if (!aligned16(x_perm) || !aligned16(offsets) || !aligned16(w_gate) || !aligned16(w_up) || !aligned16(w_down) ||
        !aligned16(y_perm))
        return MOE_ERR_INVALID_ARG;
    if (!ws_ok(ws, ws_bytes, moe_expert_ffn_workspace_size(d))) return MOE_ERR_WORKSPACE;
    if ((st = check_device())) return st;
    return launched(launch_expert_ffn(x_perm, offsets, w_gate, w_up, w_down, y_perm, (long long)pairs_of(d), d->H,
                                      d->I, d->e1 - d->e0, ws, status_dev, (cudaStream_t)stream));
}

static int gate_up_impl(const moe_dims* d, const uint16_t* x_perm, const int32_t* offsets, const uint16_t* w_gate,
                        const uint16_t* w_up, uint16_t* h, int32_t* status_dev, void* stream, int stall) {
    int st = check_dims(d);
    if (st) return st;
    if (!aligned16(x_perm) || !aligned16(offsets) || !aligned16(w_gate) || !aligned16(w_up) || !aligned16(h))
        return MOE_ERR_INVALID_ARG;
    if ((st = check_device())) return st;
    return launched(launch_gate_up(x_perm, offsets, w_gate, w_up, h, (long long)pairs_of(d), d->H, d->I,
                                   d->e1 - d->e0, status_dev, (cudaStream_t)stream, stall));
}

int moe_expert_gate_up(const moe_dims* d, const uint16_t* x_perm, const int32_t* offsets, const uint16_t* w_gate,
                       const uint16_t* w_up, uint16_t* h, int32_t* status_dev, void* stream) {
    return gate_up_impl(d, x_perm, offsets, w_gate, w_up, h, status_dev, stream, 0);
}

int moe_testing_expert_gate_up_stalled(const moe_dims* d, const uint16_t* x_perm, const int32_t* offsets,
                                       const uint16_t* w_gate, const uint16_t* w_up, uint16_t* h,
                                       int32_t* status_dev, void* stream) {
    return gate_up_impl(d, x_perm, offsets, w_gate, w_up, h, status_dev, stream, 1);
}

int moe_expert_down(const moe_dims* d, const uint16_t* h, const int32_t* offsets, const uint16_t* w_down,
                    float* y_perm, int32_t* status_dev, void* stream) {
    int st = check_dims(d);
    if (st) return st;
    if (!aligned16(h) || !aligned16(offsets) || !aligned16(w_down) || !aligned16(y_perm)) return MOE_ERR_INVALID_ARG;
    if ((st = check_device())) return st;
    return launched(launch_down(h, offsets, w_down, y_perm, (long long)pairs_of(d), d->H, d->I, d->e1 - d->e0,
                                status_dev, (cudaStream_t)stream));
}

int moe_combine(const moe_dims* d, const float* y_perm, const int32_t* pair_row, const float* topk_w, float* out,
                void* stream) {
    int st = check_dims(d);
    if (st) return st;
    if (!aligned16(y_perm) || !aligned16(pair_row) || !aligned16(topk_w) || !aligned16(out)) return MOE_ERR_INVALID_ARG;
    if ((st = check_device())) return st;
    return launched(launch_combine(y_perm, pair_row, topk_w, d->T, d->H, d->k, out, (cudaStream_t)stream));
}

int moe_combine_accumulate(const moe_dims* d, const float* y_perm, const int32_t* pair_row, const float* topk_w,
                           float* out, void* stream) {
    int st = check_dims(d);
    if (st) return st;
    if (!aligned16(y_perm) || !aligned16(pair_row) || !aligned16(topk_w) || !aligned16(out)) return MOE_ERR_INVALID_ARG;
    if ((st = check_device())) return st;
    return launched(launch_combine(y_perm, pair_row, topk_w, d->T, d->H, d->k, out, (cudaStream_t)stream, true));
}

static int layer_impl(const moe_dims* d, const uint16_t* x, const float* logits, const uint16_t* w_gate,
                      const uint16_t* w_up, const uint16_t* w_down, float* out, int32_t* topk_idx_opt,
                      float* topk_w_opt, void* ws, size_t ws_bytes, int32_t* status_dev, void* stream, int stall,
                      int gather = 0) {
    int st = check_dims(d);
    if (st) return st;
    if (!aligned16(x) || !aligned16(logits) || !aligned16(w_gate) || !aligned16(w_up) || !aligned16(w_down) ||
        !aligned16(out))
        return MOE_ERR_INVALID_ARG;
    if ((topk_idx_opt && !aligned16(topk_idx_opt)) || (topk_w_opt && !aligned16(topk_w_opt)))
        return MOE_ERR_INVALID_ARG;
    const bool fused = (long long)pairs_of(d) <= MOE_FUSED_MAX_PAIRS;
    if (stall && !fused) return MOE_ERR_INVALID_ARG;
    if (gather && !fused) return MOE_ERR_UNSUPPORTED;
    const LayerWs need = carve(d, nullptr);
    if (!ws_ok(ws, ws_bytes, need.total)) return MOE_ERR_WORKSPACE;
    if ((st = check_device())) return st;
    LayerWs w = carve(d, ws);
    int32_t* idx = topk_idx_opt ? topk_idx_opt : w.topk_idx;
    float* wt = topk_w_opt ? topk_w_opt : w.topk_w;
    cudaStream_t s = (cudaStream_t)stream;
    if (fused)
        return launched(launch_layer_fused(x, logits, w_gate, w_up, w_down, out, idx, wt, w.counts, w.offsets,
                                           w.row_pair, w.pair_row, w.x_perm, static_cast<uint16_t*>(w.ffn_ws),
                                           w.y_perm, w.sync, d->T, d->H, d->I, d->E, d->k, d->e0, d->e1,
                                           status_dev, stall, s, gather));
    // route also accumulates the dispatch chunk histograms; place then needs no counting pass
    int32_t* hist = static_cast<int32_t*>(w.dispatch_ws);
    if (cudaMemsetAsync(hist, 0, w.dispatch_bytes, s) != cudaSuccess) return MOE_ERR_CUDA;
    if (launch_route_hist(logits, d->T, d->E, d->k, idx, wt, status_dev, hist, dispatch_chunk_tokens(d->T), d->e0,
                          d->e1 - d->e0, s) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (launch_dispatch_place(x, idx, hist, d->T, d->H, d->k, d->e0, d->e1, w.counts, w.offsets, w.row_pair,
                              w.pair_row, w.x_perm, s) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (launch_expert_ffn(w.x_perm, w.offsets, w_gate, w_up, w_down, w.y_perm, (long long)pairs_of(d), d->H, d->I,
                          d->e1 - d->e0, w.ffn_ws, status_dev, s) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (launch_combine(w.y_perm, w.pair_row, wt, d->T, d->H, d->k, out, s) != cudaSuccess) return MOE_ERR_CUDA;
    return MOE_OK;
}

int moe_layer(const moe_dims* d, const uint16_t* x, const float* logits, const uint16_t* w_gate, const uint16_t* w_up,
              const uint16_t* w_down, float* out, int32_t* topk_idx_opt, float* topk_w_opt, void* ws, size_t ws_bytes,
              int32_t* status_dev, void* stream) {
    return layer_impl(d, x, logits, w_gate, w_up, w_down, out, topk_idx_opt, topk_w_opt, ws, ws_bytes, status_dev,
                      stream, 0);
}

int moe_layer_gather(const moe_dims* d, const uint16_t* x, const float* logits, const uint16_t* w_gate,
                     const uint16_t* w_up, const uint16_t* w_down, float* out, int32_t* topk_idx_opt,
                     float* topk_w_opt, void* ws, size_t ws_bytes, int32_t* status_dev, void* stream) {
    return layer_impl(d, x, logits, w_gate, w_up, w_down, out, topk_idx_opt, topk_w_opt, ws, ws_bytes, status_dev,
                      stream, 0, 1);
}

int moe_testing_layer_stalled_barrier(const moe_dims* d, const uint16_t* x, const float* logits,
                                      const uint16_t* w_gate, const uint16_t* w_up, const uint16_t* w_down,
                                      float* out, void* ws, size_t ws_bytes, int32_t* status_dev, void* stream) {
    return layer_impl(d, x, logits, w_gate, w_up, w_down, out, nullptr, nullptr, ws, ws_bytes, status_dev, stream, 1);
}

// ------------------------------------------------------------------ MXFP8

int moe_quantize_mxfp8(const uint16_t* src, int64_t rows, int32_t K, uint8_t* q, uint8_t* s, void* stream) {
    if (rows < 0 || K < 32 || K % 32 || rows * (int64_t)K >= (1ll << 40)) return MOE_ERR_INVALID_ARG;
    if (rows == 0) return MOE_OK;
    if (!aligned16(src) || !aligned16(q) || !s) return MOE_ERR_INVALID_ARG;
    int st = check_device();
    if (st) return st;
    return launched(launch_mx_quantize(src, rows, K, q, s, (cudaStream_t)stream));
}

size_t moe_expert_ffn_mxfp8_workspace_size(const moe_dims* d) {
    if (check_mx_dims(d) != MOE_OK) return 0;
    return align_up(mx_ffn_scratch_bytes((long long)pairs_of(d), d->I));
}

static int ffn_mxfp8_impl(const moe_dims* d, const uint8_t* x_perm_q, const uint8_t* x_perm_s,
                          const int32_t* offsets, const uint8_t* w_gate_q, const uint8_t* w_gate_s,
                          const uint8_t* w_up_q, const uint8_t* w_up_s, const uint8_t* w_down_q,
                          const uint8_t* w_down_s, float* y_perm, void* ws, size_t ws_bytes, int32_t* status_dev,
                          void* stream, int stall) {
    int st = check_mx_dims(d);
    if (st) return st;
    const void* ptrs[] = {x_perm_q, x_perm_s, offsets, w_gate_q, w_gate_s, w_up_q, w_up_s, w_down_q, w_down_s, y_perm};
    for (const void* p : ptrs)
        if (!aligned16(p)) return MOE_ERR_INVALID_ARG;
    if (!ws_ok(ws, ws_bytes, moe_expert_ffn_mxfp8_workspace_size(d))) return MOE_ERR_WORKSPACE;
    if ((st = check_device())) return st;
    return launched(launch_mx_expert_ffn(x_perm_q, x_perm_s, offsets, w_gate_q, w_gate_s, w_up_q, w_up_s, w_down_q,
                                         w_down_s, y_perm, (long long)pairs_of(d), d->H, d->I, d->e1 - d->e0, ws,
                                         status_dev, (cudaStream_t)stream, stall));
}

int moe_expert_ffn_mxfp8(const moe_dims* d, const uint8_t* x_perm_q, const uint8_t* x_perm_s, const int32_t* offsets,
                         const uint8_t* w_gate_q, const uint8_t* w_gate_s, const uint8_t* w_up_q,
                         const uint8_t* w_up_s, const uint8_t* w_down_q, const uint8_t* w_down_s, float* y_perm,
                         void* ws, size_t ws_bytes, int32_t* status_dev, void* stream) {
    return ffn_mxfp8_impl(d, x_perm_q, x_perm_s, offsets, w_gate_q, w_gate_s, w_up_q, w_up_s, w_down_q, w_down_s,
                          y_perm, ws, ws_bytes, status_dev, stream, 0);
}

int moe_testing_expert_ffn_mxfp8_stalled(const moe_dims* d, const uint8_t* x_perm_q, const uint8_t* x_perm_s,
                                         const int32_t* offsets, const uint8_t* w_gate_q, const uint8_t* w_gate_s,
                                         const uint8_t* w_up_q, const uint8_t* w_up_s, const uint8_t* w_down_q,
                                         const uint8_t* w_down_s, float* y_perm, void* ws, size_t ws_bytes,
                                         int32_t* status_dev, void* stream) {
    return ffn_mxfp8_impl(d, x_perm_q, x_perm_s, offsets, w_gate_q, w_gate_s, w_up_q, w_up_s, w_down_q, w_down_s,
                          y_perm, ws, ws_bytes, status_dev, stream, 1);
}

size_t moe_layer_mxfp8_workspace_size(const moe_dims* d) {
    if (check_mx_dims(d) != MOE_OK) return 0;
    return carve_mx(d, nullptr).total;
}

int moe_layer_mxfp8(const moe_dims* d, const uint16_t* x, const float* logits, const uint8_t* w_gate_q,
                    const uint8_t* w_gate_s, const uint8_t* w_up_q, const uint8_t* w_up_s, const uint8_t* w_down_q,
                    const uint8_t* w_down_s, float* out, int32_t* topk_idx_opt, float* topk_w_opt, void* ws,
                    size_t ws_bytes, int32_t* status_dev, void* stream) {
    int st = check_mx_dims(d);
    if (st) return st;
    const void* ptrs[] = {x, logits, w_gate_q, w_gate_s, w_up_q, w_up_s, w_down_q, w_down_s, out};
    for (const void* p : ptrs)
        if (!aligned16(p)) return MOE_ERR_INVALID_ARG;
    if ((topk_idx_opt && !aligned16(topk_idx_opt)) || (topk_w_opt && !aligned16(topk_w_opt)))
        return MOE_ERR_INVALID_ARG;
    if (!ws_ok(ws, ws_bytes, carve_mx(d, nullptr).total)) return MOE_ERR_WORKSPACE;
    if ((st = check_device())) return st;
    MxLayerWs w = carve_mx(d, ws);
    int32_t* idx = topk_idx_opt ? topk_idx_opt : w.topk_idx;
    float* wt = topk_w_opt ? topk_w_opt : w.topk_w;
    cudaStream_t s = (cudaStream_t)stream;
    const int n = d->e1 - d->e0;
    if ((long long)pairs_of(d) <= MOE_FUSED_MAX_PAIRS) {  // decode sizes: one cooperative launch
        uint8_t* hq = static_cast<uint8_t*>(w.ffn_ws);
        uint8_t* hs = hq + align_up(pairs_of(d) * (size_t)d->I);
        return launched(launch_layer_mx_fused(x, logits, w_gate_q, w_gate_s, w_up_q, w_up_s, w_down_q, w_down_s, out,
                                              idx, wt, w.counts, w.offsets, w.row_pair, w.pair_row, w.xpq, w.xps, hq,
                                              hs, w.y_perm, w.sync, d->T, d->H, d->I, d->E, d->k, d->e0, d->e1,
                                              status_dev, s));
    }
    int32_t* hist = static_cast<int32_t*>(w.dispatch_ws);
    if (cudaMemsetAsync(hist, 0, w.dispatch_bytes, s) != cudaSuccess) return MOE_ERR_CUDA;
    if (launch_route_hist(logits, d->T, d->E, d->k, idx, wt, status_dev, hist, dispatch_chunk_tokens(d->T), d->e0, n,
                          s) != cudaSuccess ||
        launch_dispatch_place(x, idx, hist, d->T, d->H, d->k, d->e0, d->e1, w.counts, w.offsets, w.row_pair,
                              w.pair_row, nullptr, s) != cudaSuccess ||
        launch_mx_dispatch_quantize(x, d->T, d->H, d->k, w.pair_row, w.xpq, w.xps, s) != cudaSuccess ||
        launch_mx_expert_ffn(w.xpq, w.xps, w.offsets, w_gate_q, w_gate_s, w_up_q, w_up_s, w_down_q, w_down_s,
                             w.y_perm, (long long)pairs_of(d), d->H, d->I, n, w.ffn_ws, status_dev, s) != cudaSuccess ||
        launch_combine(w.y_perm, w.pair_row, wt, d->T, d->H, d->k, out, s) != cudaSuccess)
        return MOE_ERR_CUDA;
    return MOE_OK;
}

}  // extern "C"
