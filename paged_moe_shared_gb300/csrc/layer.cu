// The launch sequence of one paged fused-MoE layer, shared by every forward
// entry point: route -> align -> gather -> GEMM 1 + SwiGLU -> GEMM 2 ->
// combine, all on one stream.  Every kernel after the first is launched with
// programmatic dependent launch, so its launch and prologue overlap the tail
// of the kernel before it; each kernel waits (griddepcontrol.wait) before it
// touches what its predecessor wrote.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>
#include <string>

#include "internal.h"
#include "kernels.h"

namespace rimuru {

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

std::string cuda_msg(const char* what, cudaError_t e) {
  return std::string(what) + ": " + cudaGetErrorName(e) + " (" + cudaGetErrorString(e) + ")";
}

}  // namespace

int make_bf16_map(CUtensorMap* m, void* base, int rank, const cuuint64_t* dims,
                  const cuuint64_t* strides, const cuuint32_t* box) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return fail(RIMURU_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, static_cast<cuuint32_t>(rank), base, dims,
                  strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(RIMURU_ERR_CUDA, "cuTensorMapEncodeTiled failed with CUresult " + std::to_string(r));
  return RIMURU_OK;
}

int make_weight_maps(void* pool_base, uint64_t page_bytes, int64_t n_pages, int hidden, int inter,
                     CUtensorMap* tm_w13, CUtensorMap* tm_w2) {
  const uint64_t H = hidden, I = inter, P = static_cast<uint64_t>(n_pages);
  cuuint64_t dims13[3] = {I, H, P};
  cuuint64_t str13[2] = {I * 2, page_bytes};
  cuuint64_t dims2[3] = {H, I, P};
  cuuint64_t str2[2] = {H * 2, page_bytes};
  cuuint32_t box[3] = {64, 64, 1};
  int st = make_bf16_map(tm_w13, pool_base, 3, dims13, str13, box);
  if (st == RIMURU_OK) st = make_bf16_map(tm_w2, pool_base, 3, dims2, str2, box);
  return st;
}

namespace {

struct LayerPtrs {
  int32_t *ids, *chunk_hist, *offsets, *sorted, *inv, *tiles, *num_tiles, *ptiles, *num_ptiles,
      *tile_cnt;
  float *w, *part;
  __nv_bfloat16 *xs, *h, *y;
};

LayerPtrs pointers_of(const LayerLaunch& a) {
  const rimuru_ws_layout& L = a.layout;
  uint8_t* ws = a.ws;
  LayerPtrs q;
  q.ids = reinterpret_cast<int32_t*>(ws + L.ids);
  q.w = reinterpret_cast<float*>(ws + L.weights);
  q.chunk_hist = reinterpret_cast<int32_t*>(ws + L.chunk_hist);
  q.offsets = reinterpret_cast<int32_t*>(ws + L.offsets);
  q.sorted = reinterpret_cast<int32_t*>(ws + L.sorted);
  q.inv = reinterpret_cast<int32_t*>(ws + L.inv);
  q.tiles = reinterpret_cast<int32_t*>(ws + L.tiles);
  q.num_tiles = reinterpret_cast<int32_t*>(ws + L.num_tiles);
  q.xs = reinterpret_cast<__nv_bfloat16*>(ws + L.x_sorted);
  q.h = reinterpret_cast<__nv_bfloat16*>(ws + L.h);
  q.y = reinterpret_cast<__nv_bfloat16*>(ws + L.y);
  q.ptiles = reinterpret_cast<int32_t*>(ws + L.ptiles);
  q.num_ptiles = reinterpret_cast<int32_t*>(ws + L.num_ptiles);
  q.tile_cnt = reinterpret_cast<int32_t*>(ws + L.tile_cnt);
  q.part = reinterpret_cast<float*>(ws + L.part);
  return q;
}

// Tile-count upper bounds and split-K parts of the two GEMMs (as in the layout).
struct Splits {
  long long t1, t2;
  int s1, s2;
};
Splits splits_of(const LayerLaunch& a) {
  Splits s;
  s.t1 = static_cast<long long>(a.layout.max_tiles) * (a.I / 128);
  s.t2 = static_cast<long long>(a.layout.max_tiles) * (a.H / 256);
  s.s1 = split_count(s.t1, a.H / 64);
  s.s2 = split_count(s.t2, a.I / 64);
  return s;
}

}  // namespace

int launch_layer_route(const LayerLaunch& a) {
  const LayerPtrs q = pointers_of(a);
  LaunchOpts first;
  first.stream = a.stream;
  first.sm_count = a.sm_count;
  // The first kernel may be scheduled while the caller's last kernel drains:
  // it runs griddepcontrol.wait before touching any data, which waits for that
  // kernel's completion and memory flush (and is a no-op behind non-kernel work).
  first.pdl = a.pdl;
  LaunchOpts next = first;
  next.pdl = a.pdl;
  cudaError_t e = cudaSuccess;
  auto mark = [&](int kidx, int which) {
    if (a.ev && (a.ev_mask >> kidx & 1u) && e == cudaSuccess) {
      e = cudaEventRecord(a.ev[kidx * 2 + which], a.stream);
      if (which == 1 && a.hits) *a.hits |= 1u << kidx;
    }
  };
  const int tpc = tokens_per_chunk(a.k);
  mark(RIMURU_K_ROUTE, 0);
  if (e == cudaSuccess)
    e = launch_route(a.logits, a.T, a.E, a.k, a.renorm, tpc, q.ids, q.w, q.chunk_hist, a.err, first);
  mark(RIMURU_K_ROUTE, 1);
  mark(RIMURU_K_ALIGN, 0);
  if (e == cudaSuccess)
    e = launch_align(q.ids, q.chunk_hist, a.layout.chunks, a.T * a.k, a.E, tpc * a.k, q.offsets,
                     q.sorted, q.inv, q.tiles, q.num_tiles, q.ptiles, q.num_ptiles, q.tile_cnt,
                     static_cast<int>(2 * std::max(splits_of(a).t1, splits_of(a).t2) + kSchedCounters), a.err, next);
  mark(RIMURU_K_ALIGN, 1);
  if (e != cudaSuccess) return fail(RIMURU_ERR_CUDA, cuda_msg("kernel launch", e));
  return RIMURU_OK;
}

int launch_layer_experts(const LayerLaunch& a, bool after_route, bool gathered) {
  const rimuru_ws_layout& L = a.layout;
  const LayerPtrs q = pointers_of(a);
  const int T = a.T, E = a.E, k = a.k, H = a.H, I = a.I;
  const int A = T * k;
  CUtensorMap tm_x{}, tm_h, tm_h_st{}, tm_y{};
  // Large batches (at least two 128-row blocks per expert on average) run
  // GEMM 1 as 256-row tiles and GEMM 2 on CTA pairs over the table of 256-row
  // pairs of blocks; their epilogues store 32-row boxes of h and y by TMA.
  const bool pairs = static_cast<long long>(A) >=
                     static_cast<long long>(kPairMinBlocksPerExpert) * kTileM * E;
  if (gathered) {  // x_sorted exists (and is read by GEMM 1) only behind the small-batch kernel
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(A)};
    cuuint64_t str[1] = {static_cast<cuuint64_t>(H) * 2};
    cuuint32_t box[2] = {64, 128};
    int st = make_bf16_map(&tm_x, q.xs, 2, dims, str, box);
    if (st != RIMURU_OK) return st;
  }
  {
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(I), static_cast<cuuint64_t>(A)};
    cuuint64_t str[1] = {static_cast<cuuint64_t>(I) * 2};
    cuuint32_t box[2] = {64, 128};
    int st = make_bf16_map(&tm_h, q.h, 2, dims, str, box);
    if (st != RIMURU_OK) return st;
    cuuint32_t box_st[2] = {64, 32};
    if (pairs) st = make_bf16_map(&tm_h_st, q.h, 2, dims, str, box_st);
    if (st != RIMURU_OK) return st;
  }
  if (pairs) {
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(A)};
    cuuint64_t str[1] = {static_cast<cuuint64_t>(H) * 2};
    cuuint32_t box[2] = {64, 32};
    int st = make_bf16_map(&tm_y, q.y, 2, dims, str, box);
    if (st != RIMURU_OK) return st;
  }
  GemmArgs g1{};
  g1.page_table = a.table;
  g1.tiles = q.tiles;
  g1.num_tiles = q.num_tiles;
  g1.offsets = q.offsets;
  g1.num_pages = a.num_pages;
  g1.max_tiles = L.max_tiles;
  g1.weights_evict_first = (A <= E * kTileM / 4) ? 1 : 0;
  g1.err = a.err;
  const Splits sp = splits_of(a);
  g1.part_rows = A < kTileM ? A : kTileM;
  g1.part = q.part;
  GemmArgs g2 = g1;
  g1.splits = sp.s1;
  g1.tile_cnt = q.tile_cnt;
  g1.x = static_cast<const __nv_bfloat16*>(a.x);
  g1.sorted = q.sorted;
  g1.top_k = k;
  g1.ldx = H;
  g2.splits = sp.s2;
  g2.tile_cnt = q.tile_cnt + std::max(sp.t1, sp.t2);
  g1.sched = q.tile_cnt + 2 * std::max(sp.t1, sp.t2);
  g1.out = q.h;
  g1.ldo = I;
  g1.n_blocks = I / 128;
  g1.num_k_blocks = H / 64;
  g2.out = q.y;
  g2.ldo = H;
  g2.n_blocks = H / 256;
  g2.num_k_blocks = I / 64;
  // Weight-bound batches prefetch their first weight tile into L2 while the
  // kernel before them finishes.  The guess (tile i's expert = i / n_blocks)
  // holds when nearly every expert is touched (at least two assignments per
  // expert on average: about 86 % of the experts or more) and none has a second
  // row block (at most half a block per expert on average); larger batches
  // reuse weights from L2, smaller ones would prefetch the wrong experts.
  if (A >= 2 * E && 2LL * A <= static_cast<long long>(E) * kTileM) {
    g1.prefetch_kb = kPrefetchKBlocks;
    g1.prefetch_bpe = 1;
  }
  // GEMM 2 follows GEMM 1, which follows the kernel that wrote the tile table:
  // it reads its first tile's expert from the table instead of guessing.
  if (2LL * A <= static_cast<long long>(E) * kTileM) {
    g2.prefetch_kb = kPrefetchKBlocks;
    g2.prefetch_bpe = 0;
  }
  g1.num_experts = g2.num_experts = E;

  LaunchOpts o;
  o.stream = a.stream;
  o.sm_count = a.sm_count;
  o.pdl = a.pdl;
  cudaError_t e = cudaSuccess;
  auto mark = [&](int kidx, int which) {
    if (a.ev && (a.ev_mask >> kidx & 1u) && e == cudaSuccess) {
      e = cudaEventRecord(a.ev[kidx * 2 + which], a.stream);
      if (which == 1 && a.hits) *a.hits |= 1u << kidx;
    }
  };
  mark(RIMURU_K_GEMM1, 0);
  GemmArgs p2 = g2;
  p2.tiles = q.ptiles;
  p2.num_tiles = q.num_ptiles;
  // GEMM 1 gathers its rows from x, except behind the small-batch kernel,
  // which has written x_sorted already.
  if (e == cudaSuccess) {
    LaunchOpts o1 = o;
    o1.pdl = after_route && a.pdl;  // behind align or the small-batch kernel; not behind host work
    if (gathered) {
      e = launch_gemm1_swiglu(tm_x, *a.tm_w13, g1, o1);
    } else if (pairs && sp.s1 == 1) {
      GemmArgs w1 = g1;  // 256-row tiles from the pair table
      w1.tiles = q.ptiles;
      w1.num_tiles = q.num_ptiles;
      e = launch_gemm1_wide(*a.tm_w13, tm_h_st, w1, o1);
    } else {
      e = launch_gemm1_swiglu_gather(*a.tm_w13, g1, o1);
    }
  }
  mark(RIMURU_K_GEMM1, 1);
  mark(RIMURU_K_GEMM2, 0);
  if (e == cudaSuccess) {
    if (pairs && sp.s2 == 1)
      e = launch_gemm2_pair(tm_h, *a.tm_w2, tm_y, p2, o);
    else
      e = launch_gemm2(tm_h, *a.tm_w2, g2, o);
  }
  mark(RIMURU_K_GEMM2, 1);
  mark(RIMURU_K_COMBINE, 0);
  if (e == cudaSuccess)
    e = launch_combine(q.y, q.inv, q.w, T, k, H, static_cast<__nv_bfloat16*>(a.out), o);
  mark(RIMURU_K_COMBINE, 1);
  if (e != cudaSuccess) return fail(RIMURU_ERR_CUDA, cuda_msg("kernel launch", e));
  return RIMURU_OK;
}

// Decode-sized batches: decode_gemm1 -> decode_reduce -> decode_gemm2.
int launch_layer_decode(const LayerLaunch& a) {
  const rimuru_ws_layout& L = a.layout;
  const LayerPtrs q = pointers_of(a);
  DecodeArgs d{};
  d.logits = a.logits;
  d.x = static_cast<const __nv_bfloat16*>(a.x);
  d.T = a.T;
  d.E = a.E;
  d.k = a.k;
  d.renorm = a.renorm;
  d.H = a.H;
  d.I = a.I;
  d.page_table = a.table;
  d.num_pages = a.num_pages;
  d.pool = a.pool;
  d.page_bytes = a.page_bytes;
  d.ids = q.ids;
  d.w = q.w;
  d.sorted = q.sorted;
  d.inv = q.inv;
  d.offsets = q.offsets;
  d.tiles = q.tiles;
  d.num_tiles = q.num_tiles;
  d.ptiles = q.ptiles;
  d.num_ptiles = q.num_ptiles;
  d.plan = reinterpret_cast<int32_t*>(a.ws + L.plan);
  d.part = q.part;
  d.h = q.h;
  d.y = q.y;
  d.out = static_cast<__nv_bfloat16*>(a.out);
  d.err = a.err;
  d.grid1 = decode_grid1(a.sm_count);
  d.prefetch_w2 = 1;
  LaunchOpts o;
  o.stream = a.stream;
  o.sm_count = a.sm_count;
  o.pdl = a.pdl;
  cudaError_t e = cudaSuccess;
  auto mark = [&](int kidx, int which) {
    if (a.ev && (a.ev_mask >> kidx & 1u) && e == cudaSuccess) {
      e = cudaEventRecord(a.ev[kidx * 2 + which], a.stream);
      if (which == 1 && a.hits) *a.hits |= 1u << kidx;
    }
  };
  mark(RIMURU_K_DECODE_GEMM1, 0);
  if (e == cudaSuccess) e = launch_decode_gemm1(*a.tm_w13, d, o);
  mark(RIMURU_K_DECODE_GEMM1, 1);
  mark(RIMURU_K_DECODE_REDUCE, 0);
  if (e == cudaSuccess) e = launch_decode_reduce(d, o);
  mark(RIMURU_K_DECODE_REDUCE, 1);
  mark(RIMURU_K_DECODE_GEMM2, 0);
  if (e == cudaSuccess) e = launch_decode_gemm2(d, o);
  mark(RIMURU_K_DECODE_GEMM2, 1);
  if (e != cudaSuccess) return fail(RIMURU_ERR_CUDA, cuda_msg("kernel launch", e));
  return RIMURU_OK;
}

int launch_layer(const LayerLaunch& a) {
  if (a.T <= a.decode_max_tokens && a.pool && decode_path_fits(a.T, a.k, a.H, a.I))
    return launch_layer_decode(a);
  if (static_cast<long long>(a.T) * a.k > kChunkAssign) {
    int st = launch_layer_route(a);
    if (st != RIMURU_OK) return st;
    return launch_layer_experts(a, /*after_route=*/true, /*gathered=*/false);
  }
  // small batch: route, align and gather in one kernel
  const LayerPtrs q = pointers_of(a);
  LaunchOpts first;
  first.stream = a.stream;
  first.sm_count = a.sm_count;
  // The first kernel may be scheduled while the caller's last kernel drains:
  // it runs griddepcontrol.wait before touching any data, which waits for that
  // kernel's completion and memory flush (and is a no-op behind non-kernel work).
  first.pdl = a.pdl;
  cudaError_t e = cudaSuccess;
  const int kidx = RIMURU_K_ROUTE_ALIGN_GATHER;
  const bool prof = a.ev && (a.ev_mask >> kidx & 1u);
  if (prof) e = cudaEventRecord(a.ev[kidx * 2], a.stream);
  if (e == cudaSuccess)
    e = launch_route_align_gather(
        a.logits, static_cast<const __nv_bfloat16*>(a.x), a.T, a.E, a.k, a.renorm, a.H, q.ids, q.w,
        q.offsets, q.sorted, q.inv, q.tiles, q.num_tiles, q.ptiles, q.num_ptiles, q.tile_cnt,
        static_cast<int>(2 * std::max(splits_of(a).t1, splits_of(a).t2) + kSchedCounters), q.xs, a.err, first);
  if (prof && e == cudaSuccess) {
    e = cudaEventRecord(a.ev[kidx * 2 + 1], a.stream);
    if (a.hits) *a.hits |= 1u << kidx;
  }
  if (e != cudaSuccess) return fail(RIMURU_ERR_CUDA, cuda_msg("kernel launch", e));
  return launch_layer_experts(a, /*after_route=*/true, /*gathered=*/true);
}

}  // namespace rimuru
