// Launchers of the device kernels (internal; called by forward.cu).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace rimuru {

constexpr int kChunkAssign = 512;  // assignments per routing chunk (= align CTA size)
constexpr int kTileM = 128;        // rows (assignments) per GEMM tile
constexpr int kMaxExperts = 512;
constexpr int kMaxTopK = 32;

struct LaunchOpts {
  cudaStream_t stream = nullptr;
  bool pdl = false;  // programmatic dependent launch on the previous kernel
  int sm_count = 148;
};

// a1: softmax top-k routing.  One warp per token; chunk c covers tokens
// [c * tpc, (c + 1) * tpc) and writes its expert histogram to chunk_hist[c].
cudaError_t launch_route(const float* logits, int T, int E, int k, int renorm, int tpc,
                         int32_t* ids, float* w, int32_t* chunk_hist, int* err,
                         const LaunchOpts& o);

// a2: offsets, stable expert-sorted permutation, its inverse and the 128-row
// tile table.  One CTA per routing chunk.
cudaError_t launch_align(const int32_t* ids, const int32_t* chunk_hist, int chunks, int A, int E,
                         int chunk, int32_t* offsets, int32_t* sorted, int32_t* inv,
                         int32_t* tiles, int32_t* num_tiles, int* err, const LaunchOpts& o);

// x rows in expert-sorted order: x_sorted[r] = x[sorted[r] / k].
cudaError_t launch_gather(const __nv_bfloat16* x, const int32_t* sorted, int A, int k, int H,
                          __nv_bfloat16* x_sorted, const LaunchOpts& o);

struct GemmArgs {
  const int32_t* page_table;  // [E][3] of the layer
  const int32_t* tiles;       // [max_tiles][2]
  const int32_t* num_tiles;
  const int32_t* offsets;     // [E + 1]
  __nv_bfloat16* out;         // [A][ldo]
  int ldo;
  int n_blocks;               // output column blocks per row block
  int num_k_blocks;           // K / 64
  int num_pages;              // pages of the expert view
  int max_tiles;              // upper bound of num_tiles (grid sizing)
  int weights_evict_first;    // 1: weights are streamed once (decode-sized batches)
  int* err;
};

// a3: h = silu(x_sorted w1_e) * (x_sorted w3_e); w1/w3 read in place from pages.
cudaError_t launch_gemm1_swiglu(const CUtensorMap& tm_x, const CUtensorMap& tm_w13,
                                const GemmArgs& a, const LaunchOpts& o);
// a4: y = h w2_e; w2 read in place from its page.
cudaError_t launch_gemm2(const CUtensorMap& tm_h, const CUtensorMap& tm_w2, const GemmArgs& a,
                         const LaunchOpts& o);

// a5: out[t] = sum_j w[t*k+j] * y[inv[t*k+j]], j ascending, fp32 then bf16.
cudaError_t launch_combine(const __nv_bfloat16* y, const int32_t* inv, const float* w, int T,
                           int k, int H, __nv_bfloat16* out, const LaunchOpts& o);

}  // namespace rimuru
