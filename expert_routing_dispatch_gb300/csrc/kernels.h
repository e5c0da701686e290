// kernels.h -- internal launchers of the libmoe kernels (called by abi.cu after
// the host-side argument checks).  Every launcher only enqueues work on `s`.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace moe {

// route.cu
cudaError_t launch_route(const float* logits, int T, int E, int k, int32_t* topk_idx, float* topk_w,
                         int32_t* status, cudaStream_t s);

cudaError_t launch_route_hist(const float* logits, int T, int E, int k, int32_t* topk_idx, float* topk_w,
                              int32_t* status, int32_t* hist, int chunk_t, int e0, int n, cudaStream_t s);

// dispatch.cu
int dispatch_chunk_tokens(int T);             // tokens per dispatch chunk
size_t dispatch_scratch_bytes(long long T, int n);  // per-chunk histograms
cudaError_t launch_dispatch_place(const uint16_t* x, const int32_t* topk_idx, const int32_t* hist, int T, int H,
                                  int k, int e0, int e1, int32_t* counts, int32_t* offsets, int32_t* row_pair,
                                  int32_t* pair_row, uint16_t* x_perm, cudaStream_t s);
cudaError_t launch_dispatch(const uint16_t* x, const int32_t* topk_idx, int T, int H, int k, int e0, int e1,
                            int32_t* counts, int32_t* offsets, int32_t* row_pair, int32_t* pair_row,
                            uint16_t* x_perm, void* scratch, cudaStream_t s);

// size of the fixed scratch array used by moe_dispatch_noalloc (int32 entries, 1 MiB)
constexpr int kNoAllocScratchInts = 1 << 18;
bool dispatch_noalloc_fits(long long pairs, int n);
cudaError_t launch_dispatch_noalloc(const uint16_t* x, const int32_t* topk_idx, int T, int H, int k, int e0, int e1,
                                    int32_t* counts, int32_t* offsets, int32_t* row_pair, int32_t* pair_row,
                                    uint16_t* x_perm, cudaStream_t s);

// combine.cu
cudaError_t launch_combine(const float* y_perm, const int32_t* pair_row, const float* topk_w, int T, int H, int k,
                           float* out, cudaStream_t s, bool accumulate = false);

// grouped_ffn.cu
size_t ffn_scratch_bytes(long long rows, int I);
cudaError_t launch_expert_ffn(const uint16_t* x_perm, const int32_t* offsets, const uint16_t* w_gate,
                              const uint16_t* w_up, const uint16_t* w_down, float* y_perm, long long rows, int H,
                              int I, int n, void* scratch, int32_t* status, cudaStream_t s);

// stall > 0: testing hook, the GEMM's first ring stage never completes (bounded
// waits run out, the status word gets MOE_ERR_TIMEOUT)
cudaError_t launch_gate_up(const uint16_t* x_perm, const int32_t* offsets, const uint16_t* w_gate,
                           const uint16_t* w_up, uint16_t* h, long long rows, int H, int I, int n, int32_t* status,
                           cudaStream_t s, int stall = 0);
cudaError_t launch_down(const uint16_t* h, const int32_t* offsets, const uint16_t* w_down, float* y_perm,
                        long long rows, int H, int I, int n, int32_t* status, cudaStream_t s);

// TMA descriptor of a bf16 row-major [rows, cols] matrix: boxes of 64 columns
// (128 B, 128-byte swizzle) x box_rows rows
bool make_tmap_bf16(CUtensorMap* m, const void* ptr, long long rows, int cols, int box_rows);

// Weight maps of one grouped GEMM (grouped_gemm.cuh): boxes of `rows`, rows / 2 and
// rows / 4 weight rows over W0 (and W1, or W0 again when w1 is NULL)
namespace gemm {
struct WMaps;
}
bool make_wmaps(gemm::WMaps* m, const void* w0, const void* w1, long long total_rows, int cols, int rows);

// decode_fused.cu: the whole layer in one persistent cooperative launch
cudaError_t launch_layer_fused(const uint16_t* x, const float* logits, const uint16_t* w_gate, const uint16_t* w_up,
                               const uint16_t* w_down, float* out, int32_t* topk_idx, float* topk_w,
                               int32_t* counts, int32_t* offsets, int32_t* row_pair, int32_t* pair_row,
                               uint16_t* x_perm, uint16_t* h, float* y_perm, unsigned* sync, int T, int H, int I,
                               int E, int k, int e0, int e1, int32_t* status, int stall_first_barrier,
                               cudaStream_t s, int gather = 0);

// mxfp8.cu: the MXFP8 expert FFN (E4M3 codes, UE8M0 scales per 32 elements along K)
cudaError_t launch_mx_quantize(const uint16_t* src, long long rows, int K, uint8_t* q, uint8_t* s, cudaStream_t st);
// the x rows of the tokens with local slots, quantised once per token, into the grouped rows
cudaError_t launch_mx_dispatch_quantize(const uint16_t* x, int T, int H, int k, const int32_t* pair_row,
                                       uint8_t* xpq, uint8_t* xps, cudaStream_t s);
size_t mx_ffn_scratch_bytes(long long rows, int I);  // h codes + h scales
cudaError_t launch_mx_expert_ffn(const uint8_t* xq, const uint8_t* xs, const int32_t* offsets, const uint8_t* wgq,
                                 const uint8_t* wgs, const uint8_t* wuq, const uint8_t* wus, const uint8_t* wdq,
                                 const uint8_t* wds, float* y_perm, long long rows, int H, int I, int n,
                                 void* scratch, int32_t* status, cudaStream_t s, int stall_gate_up = 0);

// mxfp8.cu: the MXFP8 layer in one persistent cooperative launch (decode sizes);
// sync[0..1] are cleared on the stream by the launcher
cudaError_t launch_layer_mx_fused(const uint16_t* x, const float* logits, const uint8_t* wgq, const uint8_t* wgs,
                                  const uint8_t* wuq, const uint8_t* wus, const uint8_t* wdq, const uint8_t* wds,
                                  float* out, int32_t* topk_idx, float* topk_w, int32_t* counts, int32_t* offsets,
                                  int32_t* row_pair, int32_t* pair_row, uint8_t* xpq, uint8_t* xps, uint8_t* hq,
                                  uint8_t* hs, float* y_perm, unsigned* sync, int T, int H, int I, int E, int k,
                                  int e0, int e1, int32_t* status, cudaStream_t s);

// device query shared by the launchers
int sm_count();

// cudaFuncSetAttribute(func, MaxDynamicSharedMemorySize, bytes) on the current
// device, once per (kernel, device): the attribute belongs to the device's copy
// of the kernel, so a process that drives several GPUs sets it on each of them.
cudaError_t ensure_dynamic_smem(const void* func, int bytes);

// Largest number of clusters of `cluster_size` CTAs of `func` (threads, dynamic
// shared memory as given) resident on the current device at once; queried once
// per (kernel, device).
cudaError_t max_active_clusters(const void* func, int cluster_size, int threads, int smem_bytes, int* clusters);

}  // namespace moe
