// dispatch.cu -- K2: select the pairs routed to the local experts and group them
// into per-expert GEMM buffers.
//
// "Hosting Qwen on Blackwell", section "Expert Parallel": the inputs are the
// same on every rank, so dispatch only picks the tokens routed to this rank's
// experts, gathers the routing information and stages those tokens in the
// buffers the grouped MoE GEMM reads.
//
// The order is fixed (a stable counting sort): rows of local expert e are
// offsets[e] .. offsets[e+1]-1 and hold their pairs p = t*k + j in ascending p.
//
// Main path over chunks of consecutive tokens (no host round trip):
//   count : per-chunk histogram of local experts (moe_layer's router produces
//           the same histogram itself, see route.cu)
//   place : every CTA derives the offsets and its chunk's first row per expert
//           from all chunk histograms (a redundant prefix, no scan launch), then
//           ranks its pairs in order (match_any + popc) -> row_pair, pair_row
//   gather: one CTA per token copies its x row into x_perm with 16-byte vectors,
//           reading each token's row once however many local slots it has
// The variant without a workspace (moe_dispatch_noalloc, bottom of the file)
// runs the original four kernels: count / scan / scatter / gather over chunks of
// 2048 pairs, with its histograms in a fixed device array.
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

constexpr int kWarps = 8;
constexpr int kPairsPerWarp = 256;
constexpr int kChunk = kWarps * kPairsPerWarp;  // pairs per CTA
constexpr int kMaxLocal = 1024;

__global__ void __launch_bounds__(256) dispatch_count_kernel(const int32_t* __restrict__ topk_idx, long long P,
                                                             int e0, int n, int32_t* __restrict__ chunk_hist) {
    __shared__ int hist[kMaxLocal];
    for (int e = threadIdx.x; e < n; e += blockDim.x) hist[e] = 0;
    __syncthreads();
    long long base = (long long)blockIdx.x * kChunk;
    for (int i = threadIdx.x; i < kChunk; i += blockDim.x) {
        long long p = base + i;
        if (p < P) {
            int e = __ldg(topk_idx + p) - e0;
            if (e >= 0 && e < n) atomicAdd(&hist[e], 1);
        }
    }
    __syncthreads();
    for (int e = threadIdx.x; e < n; e += blockDim.x) chunk_hist[(size_t)blockIdx.x * n + e] = hist[e];
}

// one CTA of 1024 threads.  Pass 1: warp w scans the chunk column of experts w,
// w + 32, ... (exclusive within the expert, in place, 32 chunks per step) and
// records the expert's total; then a block scan of the totals gives the offsets;
// pass 2 adds each expert's offset to its column.  Work per thread is at most
// n * nchunks / 1024 entries.
__global__ void __launch_bounds__(1024) dispatch_scan_kernel(int32_t* __restrict__ chunk_hist, int nchunks, int n,
                                                             int32_t* __restrict__ counts,
                                                             int32_t* __restrict__ offsets) {
    __shared__ int tot[kMaxLocal];
    __shared__ int warp_tot[32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int e = warp; e < n; e += 32) {
        int carry = 0;
        for (int c0 = 0; c0 < nchunks; c0 += 32) {
            const int c = c0 + lane;
            const int v = c < nchunks ? chunk_hist[(size_t)c * n + e] : 0;
            int incl = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            if (c < nchunks) chunk_hist[(size_t)c * n + e] = carry + incl - v;  // exclusive within the expert
            carry += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (lane == 0) tot[e] = carry;
    }
    __syncthreads();
    // block exclusive scan of the totals over e (thread e)
    const int e = threadIdx.x;
    const int total = e < n ? tot[e] : 0;
    int incl = total;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int v = warp_tot[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int y = __shfl_up_sync(0xffffffffu, v, o);
            if (lane >= o) v += y;
        }
        warp_tot[lane] = v;  // inclusive over warps
    }
    __syncthreads();
    const int excl = incl - total + (warp > 0 ? warp_tot[warp - 1] : 0);
    if (e < n) {
        counts[e] = total;
        offsets[e] = excl;
        if (e == n - 1) offsets[n] = excl + total;
        tot[e] = excl;
    }
    __syncthreads();
    for (int e2 = warp; e2 < n; e2 += 32) {
        const int base = tot[e2];
        for (int c = lane; c < nchunks; c += 32) chunk_hist[(size_t)c * n + e2] += base;
    }
}

__global__ void __launch_bounds__(256) dispatch_scatter_kernel(const int32_t* __restrict__ topk_idx, long long P,
                                                               int e0, int n,
                                                               const int32_t* __restrict__ chunk_base,
                                                               int32_t* __restrict__ row_pair,
                                                               int32_t* __restrict__ pair_row) {
    __shared__ int cur[kWarps][kMaxLocal];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int i = threadIdx.x; i < kWarps * n; i += blockDim.x) cur[i / n][i % n] = 0;
    __syncthreads();
    const long long wbase = (long long)blockIdx.x * kChunk + (long long)warp * kPairsPerWarp;
    const unsigned lt = (1u << lane) - 1u;
    // pass 1: per-warp counts
    for (int s = 0; s < kPairsPerWarp; s += 32) {
        long long p = wbase + s + lane;
        int e = (p < P) ? __ldg(topk_idx + p) - e0 : -1;
        bool local = (e >= 0 && e < n);
        unsigned peers = __match_any_sync(0xffffffffu, local ? e : -1);
        if (local && (peers & lt) == 0) cur[warp][e] += __popc(peers);
        __syncwarp();
    }
    __syncthreads();
    // per-warp starting rows: chunk base + counts of the earlier warps
    for (int e = threadIdx.x; e < n; e += blockDim.x) {
        int run = chunk_base[(size_t)blockIdx.x * n + e];
        for (int w = 0; w < kWarps; ++w) {
            int c = cur[w][e];
            cur[w][e] = run;
            run += c;
        }
    }
    __syncthreads();
    // pass 2: ranks in pair order
    for (int s = 0; s < kPairsPerWarp; s += 32) {
        long long p = wbase + s + lane;
        bool valid = p < P;
        int e = valid ? __ldg(topk_idx + p) - e0 : -1;
        bool local = valid && e >= 0 && e < n;
        unsigned peers = __match_any_sync(0xffffffffu, local ? e : -1);
        int b = local ? cur[warp][e] : 0;
        __syncwarp();
        if (local) {
            int row = b + __popc(peers & lt);
            if ((peers & lt) == 0) cur[warp][e] = b + __popc(peers);
            row_pair[row] = (int32_t)p;
            pair_row[p] = row;
        } else if (valid) {
            pair_row[p] = -1;
        }
        __syncwarp();
    }
}

// one CTA per token: read x[t] once, write it to each of its local rows
__global__ void __launch_bounds__(128) dispatch_gather_kernel(const uint4* __restrict__ x, int T, int H8, int k,
                                                              const int32_t* __restrict__ pair_row,
                                                              uint4* __restrict__ x_perm) {
    __shared__ int rows[32];
    __shared__ int nrows;
    const int t = blockIdx.x;
    if (threadIdx.x < 32) {
        int r = (threadIdx.x < k) ? __ldg(pair_row + (size_t)t * k + threadIdx.x) : -1;
        unsigned m = __ballot_sync(0xffffffffu, r >= 0);
        if (r >= 0) rows[__popc(m & ((1u << threadIdx.x) - 1u))] = r;
        if (threadIdx.x == 0) nrows = __popc(m);
    }
    __syncthreads();
    const int nr = nrows;
    if (nr == 0) return;
    const uint4* src = x + (size_t)t * H8;
    // four independent 16-byte loads in flight per thread, then the stores
    for (int v0 = threadIdx.x; v0 < H8; v0 += 4 * blockDim.x) {
        uint4 val[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int v = v0 + u * blockDim.x;
            if (v < H8) val[u] = __ldg(src + v);
        }
        for (int i = 0; i < nr; ++i) {
            uint4* dst = x_perm + (size_t)rows[i] * H8;
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int v = v0 + u * blockDim.x;
                if (v < H8) dst[v] = val[u];
            }
        }
    }
}

// ---------------------------------------------------------------- token chunks
constexpr int kPlaceThreads = 256;
constexpr int kPlaceWarps = kPlaceThreads / 32;

// per-chunk histogram: chunk c = tokens [c*chunk_t, (c+1)*chunk_t)
__global__ void __launch_bounds__(kPlaceThreads) dispatch_count_tokens_kernel(const int32_t* __restrict__ topk_idx,
                                                                              int T, int k, int chunk_t, int e0,
                                                                              int n, int32_t* __restrict__ hist) {
    __shared__ int h[kMaxLocal];
    for (int e = threadIdx.x; e < n; e += kPlaceThreads) h[e] = 0;
    __syncthreads();
    const long long p0 = (long long)blockIdx.x * chunk_t * k;
    const long long p1 = (long long)min(T, (int)(blockIdx.x + 1) * chunk_t) * k;
    for (long long p = p0 + threadIdx.x; p < p1; p += kPlaceThreads) {
        const int e = __ldg(topk_idx + p) - e0;
        if (e >= 0 && e < n) atomicAdd(&h[e], 1);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < n; e += kPlaceThreads) hist[(size_t)blockIdx.x * n + e] = h[e];
}

__global__ void __launch_bounds__(kPlaceThreads) dispatch_place_kernel(
    const int32_t* __restrict__ topk_idx, const int32_t* __restrict__ hist, int nchunks, int chunk_t, int T, int k,
    int e0, int n, int32_t* __restrict__ counts, int32_t* __restrict__ offsets, int32_t* __restrict__ row_pair,
    int32_t* __restrict__ pair_row) {
    __shared__ int tot[kMaxLocal];                // pairs of each expert, all chunks
    __shared__ int base[kMaxLocal];               // first row of each expert for this chunk
    __shared__ int cur[kPlaceWarps][kMaxLocal];   // per-warp counts, then per-warp cursors
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int c = blockIdx.x;
    for (int e = tid; e < n; e += kPlaceThreads) {
        tot[e] = 0;
        base[e] = 0;
    }
    for (int i = tid; i < kPlaceWarps * n; i += kPlaceThreads) cur[i / n][i % n] = 0;
    __syncthreads();
    // 1. totals and this chunk's prefix per expert; G threads share an expert's chunk list
    {
        const int G = n >= kPlaceThreads ? 1 : kPlaceThreads / n;
        for (int i = tid; i < n * G; i += kPlaceThreads) {
            const int e = i % n, g = i / n;
            int t = 0, pre = 0;
            // eight independent loads in flight per pass (a dependent chain of L2
            // loads made this loop the kernel's critical path)
            for (int cb = g; cb < nchunks; cb += 8 * G) {
                int v[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int cc = cb + u * G;
                    v[u] = cc < nchunks ? __ldg(hist + (size_t)cc * n + e) : 0;
                }
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    t += v[u];
                    pre += (cb + u * G < c) ? v[u] : 0;
                }
            }
            if (t) atomicAdd(&tot[e], t);
            if (pre) atomicAdd(&base[e], pre);
        }
    }
    __syncthreads();
    // 2. exclusive scan of the totals over experts (warp 0), base += offset
    if (warp == 0) {
        int carry = 0;
        for (int b0 = 0; b0 < n; b0 += 32) {
            const int e = b0 + lane;
            const int v0 = (e < n) ? tot[e] : 0;
            int v = v0;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, v, o);
                if (lane >= o) v += y;
            }
            if (e < n) {
                const int off = carry + v - v0;
                base[e] += off;
                if (c == 0) {
                    counts[e] = v0;
                    offsets[e] = off;
                }
            }
            carry += __shfl_sync(0xffffffffu, v, 31);
        }
        if (c == 0 && lane == 0) offsets[n] = carry;
    }
    // 3. this chunk's pairs, split into contiguous warp slices; per-warp counts
    const int t0 = c * chunk_t, t1 = min(T, t0 + chunk_t);
    const long long p0 = (long long)t0 * k, np = (long long)(t1 - t0) * k;
    const long long per_warp = (np + kPlaceWarps - 1) / kPlaceWarps;
    const long long wb = p0 + (long long)warp * per_warp, we = min(p0 + np, wb + per_warp);
    const unsigned lt = (1u << lane) - 1u;
    for (long long b = wb; b < we; b += 32) {
        const long long p = b + lane;
        const int e = (p < we) ? __ldg(topk_idx + p) - e0 : -1;
        const bool local = e >= 0 && e < n;
        const unsigned peers = __match_any_sync(0xffffffffu, local ? e : -1);
        if (local && (peers & lt) == 0) cur[warp][e] += __popc(peers);
        __syncwarp();
    }
    __syncthreads();
    for (int e = tid; e < n; e += kPlaceThreads) {  // per-warp starting rows
        int run = base[e];
        for (int w = 0; w < kPlaceWarps; ++w) {
            const int cnt = cur[w][e];
            cur[w][e] = run;
            run += cnt;
        }
    }
    __syncthreads();
    // 4. ranks in pair order
    for (long long b = wb; b < we; b += 32) {
        const long long p = b + lane;
        const bool valid = p < we;
        const int e = valid ? __ldg(topk_idx + p) - e0 : -1;
        const bool local = valid && e >= 0 && e < n;
        const unsigned peers = __match_any_sync(0xffffffffu, local ? e : -1);
        const int bse = local ? cur[warp][e] : 0;
        __syncwarp();
        if (local) {
            const int row = bse + __popc(peers & lt);
            if ((peers & lt) == 0) cur[warp][e] = bse + __popc(peers);
            row_pair[row] = (int32_t)p;
            pair_row[p] = row;
        } else if (valid) {
            pair_row[p] = -1;
        }
        __syncwarp();
    }
}

}  // namespace

// Chunks of at least 32 tokens, about 304 of them (two per SM of a GB300) for
// large T.  Independent of the device, so workspace sizes are too; the result
// does not depend on the chunking (the stable order is unique).
int dispatch_chunk_tokens(int T) {
    const int target = 304;
    const int c = (T + target - 1) / target;
    return c < 32 ? 32 : c;
}

size_t dispatch_scratch_bytes(long long T, int n) {
    const long long chunk = dispatch_chunk_tokens((int)T);
    const long long nchunks = (T + chunk - 1) / chunk;
    return (size_t)(nchunks * n * (long long)sizeof(int32_t));
}

cudaError_t launch_dispatch_place(const uint16_t* x, const int32_t* topk_idx, const int32_t* hist, int T, int H,
                                  int k, int e0, int e1, int32_t* counts, int32_t* offsets, int32_t* row_pair,
                                  int32_t* pair_row, uint16_t* x_perm, cudaStream_t s) {
    const int chunk = dispatch_chunk_tokens(T);
    const int nchunks = (T + chunk - 1) / chunk;
    dispatch_place_kernel<<<nchunks, kPlaceThreads, 0, s>>>(topk_idx, hist, nchunks, chunk, T, k, e0, e1 - e0, counts,
                                                            offsets, row_pair, pair_row);
    // the row copy wants far more CTAs than there are chunks: one CTA per token
    // (x_perm NULL: the caller copies the rows itself, e.g. in another format).
    // Folding the copy into the place kernel's ~200-600 CTAs was measured slower.
    if (x_perm)
        dispatch_gather_kernel<<<T, 128, 0, s>>>(reinterpret_cast<const uint4*>(x), T, H / 8, k, pair_row,
                                                 reinterpret_cast<uint4*>(x_perm));
    return cudaGetLastError();
}

cudaError_t launch_dispatch(const uint16_t* x, const int32_t* topk_idx, int T, int H, int k, int e0, int e1,
                            int32_t* counts, int32_t* offsets, int32_t* row_pair, int32_t* pair_row,
                            uint16_t* x_perm, void* scratch, cudaStream_t s) {
    const int chunk = dispatch_chunk_tokens(T);
    const int nchunks = (T + chunk - 1) / chunk;
    int32_t* hist = static_cast<int32_t*>(scratch);
    dispatch_count_tokens_kernel<<<nchunks, kPlaceThreads, 0, s>>>(topk_idx, T, k, chunk, e0, e1 - e0, hist);
    return launch_dispatch_place(x, topk_idx, hist, T, H, k, e0, e1, counts, offsets, row_pair, pair_row, x_perm, s);
}

// ---------------------------------------------------------------------------
// Variant for callers that cannot allocate device memory.  The per-chunk
// histograms live in this fixed array, which belongs to the library's device
// module: every GPU that loads the library keeps these bytes until the process
// exits.  All calls share it, so calls that overlap on the GPU race on it.
// Nothing in it needs clearing: the count kernel writes every entry that the
// scan and scatter kernels later read.
static __device__ __align__(256) int32_t g_noalloc_chunk_hist[kNoAllocScratchInts];

namespace {

constexpr int kMaxDevices = 64;

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

// Unique id of the calling thread's current context (0 if there is none or the
// driver cannot tell).  Ids are never reused within a process, so a context
// rebuilt after cudaDeviceReset gets a new one.
unsigned long long current_context_id() {
    static CtxGetCurrentFn get_current = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            p = nullptr;
        return reinterpret_cast<CtxGetCurrentFn>(p);
    }();
    static CtxGetIdFn get_id = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            p = nullptr;
        return reinterpret_cast<CtxGetIdFn>(p);
    }();
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

// Device address of g_noalloc_chunk_hist on the current device.  Host code
// cannot use the symbol's host-side shadow as a pointer, so the address is looked
// up with cudaGetSymbolAddress once per device and context: a context rebuilt
// after cudaDeviceReset (a new context id) gets a fresh lookup instead of a stale
// address.
cudaError_t noalloc_scratch(int32_t** out) {
    static std::mutex mu;
    static int32_t* addr[kMaxDevices] = {};
    static unsigned long long ctx_of_addr[kMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    const unsigned long long ctx = current_context_id();
    if (!addr[dev] || ctx == 0 || ctx != ctx_of_addr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_chunk_hist);
        if (e != cudaSuccess) return e;
        addr[dev] = static_cast<int32_t*>(p);
        ctx_of_addr[dev] = current_context_id();  // the lookup made the device's context current
    }
    *out = addr[dev];
    return cudaSuccess;
}

}  // namespace

bool dispatch_noalloc_fits(long long pairs, int n) {
    long long nchunks = (pairs + kChunk - 1) / kChunk;
    return nchunks * (long long)n <= (long long)kNoAllocScratchInts;
}

cudaError_t launch_dispatch_noalloc(const uint16_t* x, const int32_t* topk_idx, int T, int H, int k, int e0, int e1,
                                    int32_t* counts, int32_t* offsets, int32_t* row_pair, int32_t* pair_row,
                                    uint16_t* x_perm, cudaStream_t s) {
    int32_t* chunk_hist = nullptr;
    cudaError_t e = noalloc_scratch(&chunk_hist);
    if (e != cudaSuccess) return e;
    const long long P = (long long)T * k;
    const int n = e1 - e0;
    const int nchunks = (int)((P + kChunk - 1) / kChunk);
    dispatch_count_kernel<<<nchunks, 256, 0, s>>>(topk_idx, P, e0, n, chunk_hist);
    dispatch_scan_kernel<<<1, 1024, 0, s>>>(chunk_hist, nchunks, n, counts, offsets);
    dispatch_scatter_kernel<<<nchunks, 256, 0, s>>>(topk_idx, P, e0, n, chunk_hist, row_pair, pair_row);
    dispatch_gather_kernel<<<T, 128, 0, s>>>(reinterpret_cast<const uint4*>(x), T, H / 8, k, pair_row,
                                             reinterpret_cast<uint4*>(x_perm));
    return cudaGetLastError();
}

}  // namespace moe
