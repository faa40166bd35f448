// Launchers of the device kernels (internal; called by forward.cu).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "../../include/rimuru.h"

namespace rimuru {

constexpr int kChunkAssign = 1024;  // most assignments in one routing chunk (= align CTA size)
constexpr int kRouteWarps = 32;     // tokens per routing chunk: one warp per token
constexpr int kTileM = 128;         // rows (assignments) per GEMM tile
constexpr int kMaxExperts = 512;
constexpr int kMaxTopK = 32;
// k blocks of weights (32 KiB each) a GEMM CTA prefetches into L2 ahead of its first tile.
constexpr int kPrefetchKBlocks = 16;

// Split-K for layers with few tiles: the K range of a tile is cut into S
// parts computed by different CTAs (fp32 partials in the workspace, summed
// in split order by the last CTA to finish the tile).  S is chosen from an
// upper bound of the tile count so the workspace size does not depend on
// the device: about kSplitTarget work units (two waves of a 152-SM GPU),
// only when the tiles fill less than half a wave, and at least
// kMinSplitBlocks k blocks per split (shorter splits cost more in the
// pipeline fill and the reduction than they save).
constexpr int kSplitTarget = 304;
// Work-unit counters after the split-K tile counters (zeroed with them by the
// kernel that writes the tile tables): [0] feeds the 256-row GEMM 1's dynamic
// unit scheduler.
constexpr int kSchedCounters = 2;
constexpr int kMinSplitBlocks = 8;
inline int split_count(long long tiles_ub, int nkb) {
  if (tiles_ub <= 0 || tiles_ub * 4 > kSplitTarget) return 1;
  long long s = kSplitTarget / tiles_ub;
  if (s > nkb / kMinSplitBlocks) s = nkb / kMinSplitBlocks;
  return s < 1 ? 1 : static_cast<int>(s);
}

// Tokens routed by one CTA (one warp each); their k assignments form one chunk.
inline int tokens_per_chunk(int k) {
  return kRouteWarps * k <= kChunkAssign ? kRouteWarps : kChunkAssign / k;
}

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
// Also writes the table of 256-row pairs of blocks (ptiles) and zeroes the
// split-K tile counters (cnt_len ints at tile_cnt).
cudaError_t launch_align(const int32_t* ids, const int32_t* chunk_hist, int chunks, int A, int E,
                         int chunk, int32_t* offsets, int32_t* sorted, int32_t* inv,
                         int32_t* tiles, int32_t* num_tiles, int32_t* ptiles,
                         int32_t* num_ptiles, int32_t* tile_cnt, int cnt_len, int* err,
                         const LaunchOpts& o);

// a1 + a2 + gather in one launch for batches whose A = T * k assignments fit
// one CTA (A <= kChunkAssign): every CTA routes and groups all assignments in
// shared memory, CTA 0 writes the tables, each CTA gathers its share of rows
// (about kFusedRowsPerCta of them).
constexpr int kFusedRowsPerCta = 8;
cudaError_t launch_route_align_gather(const float* logits, const __nv_bfloat16* x, int T, int E,
                                      int k, int renorm, int H, int32_t* ids, float* w,
                                      int32_t* offsets, int32_t* sorted, int32_t* inv,
                                      int32_t* tiles, int32_t* num_tiles, int32_t* ptiles,
                                      int32_t* num_ptiles, int32_t* tile_cnt, int cnt_len,
                                      __nv_bfloat16* x_sorted, int* err, const LaunchOpts& o);


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
  int splits;                 // split-K parts per tile (1: no split)
  int part_rows;              // rows of one partial slab (>= rows of any tile)
  float* part;                // [tiles * splits][part_rows][256] fp32 partials
  int32_t* tile_cnt;          // [tiles] finished splits per tile (zeroed by align)
  // GEMM 1 with gathered A: row r of the sorted order is row sorted[r] / top_k of x
  const __nv_bfloat16* x;     // [T][ldx]
  const int32_t* sorted;      // [A]
  int top_k;
  int ldx;
  // Weight prefetch before the grid dependency wait: the CTA guesses its first
  // tile's expert as if every expert had prefetch_bpe row blocks (0: reads it
  // from the tile table, which must then come from a kernel that finished
  // before the one this launch follows started) and prefetches the first
  // prefetch_kb k blocks of that tile's weights into L2 (prefetch_kb 0: off).
  int prefetch_kb;
  int prefetch_bpe;
  int num_experts;
  // Dynamic scheduling (256-row GEMM 1): units after the first gridDim.x are
  // taken from this counter, zero when the kernel starts.
  int32_t* sched;
};

// a3: h = silu(x_sorted w1_e) * (x_sorted w3_e); w1/w3 read in place from pages.
// A is staged by TMA from x_sorted, which the fused small-batch kernel writes
// (batches of at most kChunkAssign assignments).
cudaError_t launch_gemm1_swiglu(const CUtensorMap& tm_x, const CUtensorMap& tm_w13,
                                const GemmArgs& a, const LaunchOpts& o);
// Use the CTA-pair GEMM 2 when the assignments average at least this many
// 128-row blocks per expert (most experts then have pairs of blocks).
constexpr int kPairMinBlocksPerExpert = 2;

// a3 with the gather fused in: four loader warps copy each A stage straight
// from x (cp.async) using `sorted`, so x_sorted is neither written nor read.
cudaError_t launch_gemm1_swiglu_gather(const CUtensorMap& tm_w13, const GemmArgs& a,
                                       const LaunchOpts& o);

// a3 for large batches (the same condition as the CTA-pair GEMM 2): 256-row
// tiles of the pair table (tiles/num_tiles in `a` name it) on one SM, two
// M = 128 MMAs per k step sharing the staged weights, A rows gathered from x
// like launch_gemm1_swiglu_gather.  No split-K.
// tm_h maps a.out (h) in 32-row x 64-column boxes for the epilogue's TMA stores.
cudaError_t launch_gemm1_wide(const CUtensorMap& tm_w13, const CUtensorMap& tm_h,
                              const GemmArgs& a, const LaunchOpts& o);

// a4 for large batches on CTA pairs (tcgen05 cta_group::2): a tile is one
// entry of the pair table (tiles/num_tiles in `a` name it) times one column
// block; each CTA stages half of every weight tile.  tm_y maps a.out (y) in
// 32-row x 64-column boxes for the epilogue's TMA stores.
cudaError_t launch_gemm2_pair(const CUtensorMap& tm_h, const CUtensorMap& tm_w2,
                              const CUtensorMap& tm_y, const GemmArgs& a, const LaunchOpts& o);

// a4: y = h w2_e; w2 read in place from its page.
cudaError_t launch_gemm2(const CUtensorMap& tm_h, const CUtensorMap& tm_w2, const GemmArgs& a,
                         const LaunchOpts& o);

// a5: out[t] = sum_j w[t*k+j] * y[inv[t*k+j]], j ascending, fp32 then bf16.
cudaError_t launch_combine(const __nv_bfloat16* y, const int32_t* inv, const float* w, int T,
                           int k, int H, __nv_bfloat16* out, const LaunchOpts& o);

// ------------------------------------------------ decode-sized batches
// Batches of at most kDecodeMaxT tokens and kDecodeMaxA assignments (and whose
// x rows and h fit the kernels' shared memory, decode_path_fits) may run as
// three kernels: decode_gemm1 (routing in every CTA, W1/W3 streamed in
// balanced k-block units with fp32 partials, W2 pages prefetched into L2),
// decode_reduce (h from the partials) and decode_gemm2 (y from L2-resident W2
// and the combine).
constexpr int kDecodeMaxT = 4;
constexpr int kDecodeMaxA = 64;
constexpr int kDecodeGridMax = 160;     // decode_gemm1 CTAs at most (sizes the partials)
constexpr int kDecodeStagesMax = 12;    // ring stages of 16 KiB
constexpr int kDecodeMaxHBytes = 98304;  // h of the batch in decode_gemm2's shared memory
constexpr int kDecodePlanInts = 1 + 3 * kDecodeMaxA;

struct DecodeArgs {
  const float* logits;          // [T][E]
  const __nv_bfloat16* x;       // [T][H]
  int T, E, k, renorm, H, I;
  const int32_t* page_table;    // [E][3] of the layer
  int num_pages;
  const uint8_t* pool;          // pool base: W2 pages are read (and prefetched) by address
  uint64_t page_bytes;
  int32_t *ids, *sorted, *inv, *offsets, *tiles, *num_tiles, *ptiles, *num_ptiles, *plan;
  float* w;
  float* part;                  // fp32 partials, [groups + grid1 slots][T][128]
  __nv_bfloat16 *h, *y, *out;   // h [A][I], y [A][H] in sorted order; out [T][H]
  int* err;
  int grid1;                    // CTAs of decode_gemm1
  int stages;                   // set by the launcher
  int prefetch_w2;              // 1: decode_gemm1 prefetches the routed W2 pages into L2
};

bool decode_path_fits(int T, int k, int H, int I);
int decode_grid1(int sm_count);
uint64_t decode_part_bytes(int T, int k, int E, int I);
cudaError_t launch_decode_gemm1(const CUtensorMap& tm_w13, DecodeArgs a, const LaunchOpts& o);
cudaError_t launch_decode_reduce(DecodeArgs a, const LaunchOpts& o);
cudaError_t launch_decode_gemm2(DecodeArgs a, const LaunchOpts& o);

// bf16 TMA descriptor with 128-byte swizzle (dims and box innermost first,
// strides in bytes for dims 1..rank-1).  Returns a rimuru status.
int make_bf16_map(CUtensorMap* m, void* base, int rank, const cuuint64_t* dims,
                  const cuuint64_t* strides, const cuuint32_t* box);
// The expert view as two 3-D maps over the whole pool: [pages][H][I] (w1, w3)
// and [pages][I][H] (w2), 64 x 64 boxes.
int make_weight_maps(void* pool_base, uint64_t page_bytes, int64_t n_pages, int hidden, int inter,
                     CUtensorMap* tm_w13, CUtensorMap* tm_w2);

// Everything one forward needs; filled by the entry points.
struct LayerLaunch {
  const void* x = nullptr;          // bf16 [T][H]
  const float* logits = nullptr;    // fp32 [T][E]
  void* out = nullptr;              // bf16 [T][H]
  int T = 0, E = 0, k = 0, H = 0, I = 0, renorm = 1, num_pages = 0;
  uint8_t* ws = nullptr;            // workspace base
  rimuru_ws_layout layout{};        // region offsets inside ws
  const int32_t* table = nullptr;   // this layer's page table [E][3] (device)
  int* err = nullptr;               // device error word
  const CUtensorMap* tm_w13 = nullptr;
  const CUtensorMap* tm_w2 = nullptr;
  cudaStream_t stream = nullptr;
  int sm_count = 0;
  bool pdl = true;
  uint8_t* pool = nullptr;          // pool base (the decode path reads W2 pages by address)
  uint64_t page_bytes = 0;
  int decode_max_tokens = 0;        // batches of at most this many tokens take the decode path
  cudaEvent_t* ev = nullptr;        // 2 * RIMURU_K_COUNT events, or null
  unsigned ev_mask = 0;             // kernels bracketed by their event pair
  unsigned* hits = nullptr;         // bit k set when kernel k was launched between its events
};

// Launch the six kernels of one layer.  Returns a rimuru status.
int launch_layer(const LayerLaunch& a);
// The same in two halves: routing (route, align) and the expert part (GEMM 1,
// GEMM 2, combine).  Host-side work may sit between the two; after_route =
// false when it does (GEMM 1 then follows it in plain stream order).
int launch_layer_route(const LayerLaunch& a);
// gathered = true when x_sorted is already written (the small-batch kernel).
int launch_layer_experts(const LayerLaunch& a, bool after_route, bool gathered = false);

}  // namespace rimuru
