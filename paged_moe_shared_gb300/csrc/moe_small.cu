// Routing, grouping, row gather and combine kernels of the paged fused MoE
// layer (Rimuru, arXiv 2610.40305: the fused MoE layer around the
// page-table-aware expert GEMMs; the pages name the layer but not these
// steps, which follow the standard top-k MoE definition).
#include <cfloat>
#include <climits>

#include "device.cuh"
#include "kernels.h"
#include "route.cuh"

namespace rimuru {
namespace {

using dev::grid_dep_launch;
using dev::grid_dep_wait;
using dev::set_error;
using dev::cluster_addr;
using dev::cluster_id_x;
using dev::cluster_rank;
using dev::cluster_sync;
using dev::ld_cluster_u32;
using dev::route_token;

constexpr unsigned kFull = 0xffffffffu;

// Launch helper: optional programmatic dependent launch.
template <typename... KArgs, typename... Args>
cudaError_t launch(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                   const LaunchOpts& o, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = o.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = o.pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// The same with thread-block clusters of `cluster` CTAs along x.
template <typename... KArgs, typename... Args>
cudaError_t launch_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block, int cluster,
                           const LaunchOpts& o, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = 0;
  cfg.stream = o.stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = o.pdl ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// One warp per token over the chunk's tokens; the chunk's expert histogram
// goes to chunk_hist[blockIdx.x].
template <int EPL>
__global__ void __launch_bounds__(1024) moe_route_kernel(const float* __restrict__ logits, int T,
                                                         int E, int k, int renorm, int tpc,
                                                         int32_t* __restrict__ ids,
                                                         float* __restrict__ w,
                                                         int32_t* __restrict__ chunk_hist,
                                                         int* err) {
  extern __shared__ int s_hist[];  // [E]
  grid_dep_wait();
  grid_dep_launch();
  for (int e = threadIdx.x; e < E; e += blockDim.x) s_hist[e] = 0;
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nwarps = blockDim.x >> 5;
  const int t_begin = blockIdx.x * tpc;
  const int t_end = min(t_begin + tpc, T);
  for (int t = t_begin + warp; t < t_end; t += nwarps) {
    int my_id;
    float my_w;
    route_token<EPL>(logits + static_cast<size_t>(t) * E, E, k, renorm, lane, err, my_id, my_w);
    if (lane < k) {
      ids[static_cast<size_t>(t) * k + lane] = my_id;
      w[static_cast<size_t>(t) * k + lane] = my_w;
      atomicAdd(&s_hist[my_id], 1);
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    chunk_hist[static_cast<size_t>(blockIdx.x) * E + e] = s_hist[e];
}

// Exclusive prefix sums over the block of three per-thread counts at once
// (blockDim <= 1024): one scan of a packed 64-bit value, a in bits 0-25, b in
// 26-44 and c in 45-63, so the block's sums must stay below 2^26, 2^19 and
// 2^19.  Here a counts assignments (at most 2^25) and b, c the 128-row blocks
// and pairs of blocks (at most 2^18 + E).  The barriers inside also order the
// callers' earlier shared-memory writes before their later reads.
struct Scan3 {
  int a, b, c;
};
__device__ Scan3 block_exclusive_scan3(int a, int b, int c, unsigned long long* s_warp) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nwarps = blockDim.x >> 5;
  const unsigned long long v = static_cast<unsigned long long>(a) |
                               (static_cast<unsigned long long>(b) << 26) |
                               (static_cast<unsigned long long>(c) << 45);
  unsigned long long x = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const unsigned long long y = __shfl_up_sync(kFull, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) s_warp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    unsigned long long t = lane < nwarps ? s_warp[lane] : 0ull;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const unsigned long long y = __shfl_up_sync(kFull, t, off);
      if (lane >= off) t += y;
    }
    if (lane < nwarps) s_warp[lane] = t;  // inclusive warp totals
  }
  __syncthreads();
  const unsigned long long before = warp > 0 ? s_warp[warp - 1] : 0ull;
  __syncthreads();  // s_warp may be reused by the caller
  const unsigned long long ex = before + x - v;
  return {static_cast<int>(ex & ((1ull << 26) - 1)), static_cast<int>((ex >> 26) & ((1ull << 19) - 1)),
          static_cast<int>(ex >> 45)};
}

// Offsets, the 128-row tile table, the table of 256-row pairs of blocks and the
// zeroed split-K counters, from each expert's count `tot`, its 128-row blocks
// `nb` and pairs of blocks `np` (the last one possibly alone), and their
// exclusive prefixes `off`, `first` and `pfirst` (held by thread e of the CTA
// for e < E).  Every thread of the CTA calls it.
__device__ void write_tables(int E, int tot, int off, int nb, int first, int np, int pfirst,
                             int32_t* __restrict__ offsets, int32_t* __restrict__ tiles,
                             int32_t* __restrict__ num_tiles, int32_t* __restrict__ ptiles,
                             int32_t* __restrict__ num_ptiles, int32_t* __restrict__ tile_cnt,
                             int cnt_len) {
  const int tid = threadIdx.x;
  for (int i = tid; i < cnt_len; i += blockDim.x) tile_cnt[i] = 0;
  if (tid < E) offsets[tid] = off;
  if (tid == E - 1) offsets[E] = off + tot;
  for (int b = 0; b < nb; ++b) {
    tiles[2 * (first + b)] = tid;
    tiles[2 * (first + b) + 1] = off + b * kTileM;
  }
  if (tid == E - 1) *num_tiles = first + nb;
  for (int b = 0; b < np; ++b) {
    ptiles[2 * (pfirst + b)] = tid;
    ptiles[2 * (pfirst + b) + 1] = off + b * 2 * kTileM;
  }
  if (tid == E - 1) *num_ptiles = pfirst + np;
}

// ----------------------------------------------------------------- align
// One CTA per routing chunk (kChunkAssign threads).  Every CTA sums the chunk
// histograms (all chunks -> totals, earlier chunks -> this chunk's base per
// expert), with parts = blockDim / E threads per expert column, each issuing
// its loads in batches; CTA 0 also writes the offsets and the tile tables.
// Inside the chunk an assignment's rank among same-expert assignments is the
// number of earlier ones: inside a warp by __match_any_sync, across warps by a
// prefix over per-warp counts, which keeps the order stable.
constexpr int kHistBatch = 8;  // chunk histogram loads in flight per thread

__global__ void __launch_bounds__(kChunkAssign, 2) moe_align_kernel(
    const int32_t* __restrict__ ids, const int32_t* __restrict__ chunk_hist, int chunks, int A,
    int E, int chunk, int32_t* __restrict__ offsets, int32_t* __restrict__ sorted,
    int32_t* __restrict__ inv, int32_t* __restrict__ tiles, int32_t* __restrict__ num_tiles,
    int32_t* __restrict__ ptiles, int32_t* __restrict__ num_ptiles, int32_t* __restrict__ tile_cnt,
    int cnt_len, int* err) {
  __shared__ int s_part_tot[kChunkAssign];
  __shared__ int s_part_bef[kChunkAssign];
  __shared__ int s_base[kMaxExperts];
  __shared__ uint16_t s_wh[kChunkAssign / 32][kMaxExperts];  // per-warp counts, then their prefix
  __shared__ unsigned long long s_warp[32];
  grid_dep_wait();
  grid_dep_launch();
  const int c = blockIdx.x;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int f0 = c * chunk;
  const int n = min(chunk, A - f0);
  const int groups = (n + 31) / 32;
  for (int i = tid; i < groups * E; i += blockDim.x) s_wh[i / E][i % E] = 0;
  const int parts = blockDim.x / E;  // >= 2 since E <= kMaxExperts = blockDim / 2
  {
    const int e = tid % E, part = tid / E;
    int tot = 0, bef = 0;
    if (part < parts) {
      int cc = part;
      for (; cc + (kHistBatch - 1) * parts < chunks; cc += kHistBatch * parts) {
        int v[kHistBatch];
#pragma unroll
        for (int u = 0; u < kHistBatch; ++u)
          v[u] = __ldg(chunk_hist + static_cast<size_t>(cc + u * parts) * E + e);
#pragma unroll
        for (int u = 0; u < kHistBatch; ++u) {
          tot += v[u];
          if (cc + u * parts < c) bef += v[u];
        }
      }
      for (; cc < chunks; cc += parts) {
        const int v = __ldg(chunk_hist + static_cast<size_t>(cc) * E + e);
        tot += v;
        if (cc < c) bef += v;
      }
    }
    s_part_tot[tid] = tot;
    s_part_bef[tid] = bef;
  }
  // this thread's assignment f0 + tid: its expert and its rank in the warp
  int my = -1, rank_in = 0, in_warp = 0;
  const unsigned valid = __ballot_sync(kFull, tid < n);
  if (tid < n) {
    my = ids[f0 + tid];
    if (my < 0 || my >= E) {
      set_error(err, RIMURU_DEV_BAD_SHAPE);
      my = -1;  // grouped apart, never scattered
    }
    const unsigned peers = __match_any_sync(valid, my);
    rank_in = __popc(peers & ((1u << lane) - 1u));
    in_warp = __popc(peers);
  }
  __syncthreads();  // s_wh zeroed, s_part_* written
  if (my >= 0 && rank_in == 0) s_wh[warp][my] = static_cast<uint16_t>(in_warp);
  int tot = 0, before = 0;
  if (tid < E) {
    for (int p = 0; p < parts; ++p) {
      tot += s_part_tot[p * E + tid];
      before += s_part_bef[p * E + tid];
    }
  }
  const int nb = tid < E ? (tot + kTileM - 1) / kTileM : 0;
  const int np = (nb + 1) / 2;
  const Scan3 sc = block_exclusive_scan3(tot, nb, np, s_warp);  // also orders the s_wh counts
  const int off = sc.a;
  if (tid < E) {
    s_base[tid] = off + before;
    int acc = 0;  // earlier warps' assignments of expert tid inside this chunk
    for (int g = 0; g < groups; ++g) {
      const int v = s_wh[g][tid];
      s_wh[g][tid] = static_cast<uint16_t>(acc);
      acc += v;
    }
  }
  if (c == 0)
    write_tables(E, tot, off, nb, sc.b, np, sc.c, offsets, tiles, num_tiles, ptiles, num_ptiles,
                 tile_cnt, cnt_len);
  __syncthreads();
  if (my >= 0) {
    const int pos = s_base[my] + s_wh[warp][my] + rank_in;
    sorted[pos] = f0 + tid;
    inv[f0 + tid] = pos;
  }
}

// ----------------------------------------------------- small batches, one launch
// Route, align and gather in one kernel when all A = T * k assignments fit one
// CTA (A <= kChunkAssign, decode-sized batches).  CTAs come in clusters of
// kFusedCluster: the CTA of rank r routes the tokens t = r (mod kFusedCluster)
// and, after a cluster barrier, every CTA copies the others' expert ids out of
// their shared memory, so each cluster holds the whole routing without a
// grid-wide step and each SM routes an eighth of the tokens.  Every CTA then
// groups the assignments in shared memory: a few microseconds of repeated work
// per CTA instead of two kernel boundaries and the global round trip of the
// routing tables.  Cluster 0 writes ids and weights (each CTA its own
// tokens), CTA 0 offsets, sorted, inv and the tile tables; every CTA copies its
// share of the rows into x_sorted.
// Grouping: assignment f = 32 g + lane belongs to warp g; within the warp its
// rank among equal experts comes from __match_any_sync, across warps from a
// prefix over per-warp counts, so the order is f ascending inside each expert.
constexpr int kFusedWarps = kChunkAssign / 32;
constexpr int kFusedCluster = 8;

template <int EPL>
__global__ void __launch_bounds__(kChunkAssign) moe_route_align_gather_kernel(
    const float* __restrict__ logits, const uint4* __restrict__ x, int T, int E, int k,
    int renorm, int H8, int32_t* __restrict__ ids, float* __restrict__ w,
    int32_t* __restrict__ offsets, int32_t* __restrict__ sorted, int32_t* __restrict__ inv,
    int32_t* __restrict__ tiles, int32_t* __restrict__ num_tiles, int32_t* __restrict__ ptiles,
    int32_t* __restrict__ num_ptiles, int32_t* __restrict__ tile_cnt, int cnt_len,
    uint4* __restrict__ xs, int* err) {
  __shared__ int s_ids[kChunkAssign];                     // expert of assignment f
  __shared__ int s_sorted[kChunkAssign];                  // assignment held by sorted row r
  __shared__ uint16_t s_wh[kFusedWarps][kMaxExperts];     // per-warp counts, then their prefix
  __shared__ int s_off[kMaxExperts];
  __shared__ unsigned long long s_warp[32];
  grid_dep_wait();
  grid_dep_launch();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int A = T * k;
  const int groups = (A + 31) / 32;
  const bool lead = blockIdx.x == 0;
  const uint32_t crank = cluster_rank();
  const bool lead_cluster = cluster_id_x() == 0;
  for (int i = tid; i < groups * kMaxExperts; i += blockDim.x) (&s_wh[0][0])[i] = 0;
  for (int t = static_cast<int>(crank) + kFusedCluster * warp; t < T;
       t += kFusedCluster * kFusedWarps) {
    int my_id;
    float my_w;
    route_token<EPL>(logits + static_cast<size_t>(t) * E, E, k, renorm, lane, err, my_id, my_w);
    if (lane < k) {
      s_ids[t * k + lane] = my_id;
      if (lead_cluster) {
        ids[t * k + lane] = my_id;
        w[t * k + lane] = my_w;
      }
    }
  }
  cluster_sync();  // every CTA's routed ids are in its shared memory
  if (tid < A) {
    const uint32_t owner = static_cast<uint32_t>((tid / k) % kFusedCluster);
    if (owner != crank) s_ids[tid] = static_cast<int>(ld_cluster_u32(cluster_addr(&s_ids[tid], owner)));
  }
  cluster_sync();  // no CTA leaves or moves on while a peer still reads its ids
  const int f = warp * 32 + lane;
  const unsigned valid = __ballot_sync(kFull, f < A);
  int my_e = 0, rank_in = 0;
  if (f < A) {
    my_e = s_ids[f];
    const unsigned peers = __match_any_sync(valid, my_e);
    rank_in = __popc(peers & ((1u << lane) - 1u));
    if (rank_in == 0) s_wh[warp][my_e] = static_cast<uint16_t>(__popc(peers));
  }
  __syncthreads();
  int tot = 0;
  if (tid < E) {
    for (int g = 0; g < groups; ++g) {
      const int v = s_wh[g][tid];
      s_wh[g][tid] = static_cast<uint16_t>(tot);
      tot += v;
    }
  }
  const int nb = tid < E ? (tot + kTileM - 1) / kTileM : 0;
  const int np = (nb + 1) / 2;
  const Scan3 sc = block_exclusive_scan3(tot, nb, np, s_warp);
  const int off = sc.a;
  if (tid < E) s_off[tid] = off;
  if (lead)
    write_tables(E, tot, off, nb, sc.b, np, sc.c, offsets, tiles, num_tiles, ptiles, num_ptiles,
                 tile_cnt, cnt_len);
  __syncthreads();
  if (f < A) {
    const int pos = s_off[my_e] + s_wh[warp][my_e] + rank_in;
    s_sorted[pos] = f;
    if (lead) {
      sorted[pos] = f;
      inv[f] = pos;
    }
  }
  __syncthreads();
  // this CTA's rows of x_sorted, four 16-byte loads in flight per thread
  const int per = (A + gridDim.x - 1) / gridDim.x;
  const int r0 = min(A, blockIdx.x * per), r1 = min(A, r0 + per);
  const int n = (r1 - r0) * H8;
  for (int i0 = tid; i0 < n; i0 += 4 * blockDim.x) {
    uint4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = i0 + u * blockDim.x;
      if (i < n) {
        const int r = r0 + i / H8, c = i % H8;
        v[u] = x[static_cast<size_t>(s_sorted[r] / k) * H8 + c];
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = i0 + u * blockDim.x;
      if (i < n) xs[static_cast<size_t>(r0) * H8 + i] = v[u];
    }
  }
}

// ----------------------------------------------------------------- combine
// out[t] = sum_j w[t*k+j] * y[inv[t*k+j]], j ascending, fp32, bf16 result.
// Each thread owns one 16-byte column slice of a token and issues the loads of
// up to eight slots before it accumulates them in slot order.
__global__ void __launch_bounds__(256, 4) moe_combine_kernel(const uint4* __restrict__ y,
                                                          const int32_t* __restrict__ inv,
                                                          const float* __restrict__ w, int T,
                                                          int k, int H8, uint4* __restrict__ out) {
  grid_dep_wait();
  grid_dep_launch();
  for (int t = blockIdx.x; t < T; t += gridDim.x) {
    for (int c = threadIdx.x; c < H8; c += blockDim.x) {
      float acc[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = 0.f;
      for (int j0 = 0; j0 < k; j0 += 8) {
        uint4 v[8];
        float wj[8];
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
          const int j = j0 + jj;
          if (j < k) {
            const int f = t * k + j;
            wj[jj] = w[f];
            v[jj] = __ldcs(&y[static_cast<size_t>(inv[f]) * H8 + c]);
          }
        }
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
          if (j0 + jj < k) {
            const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&v[jj]);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const float2 f2 = __bfloat1622float2(p[i]);
              acc[2 * i] = fmaf(wj[jj], f2.x, acc[2 * i]);
              acc[2 * i + 1] = fmaf(wj[jj], f2.y, acc[2 * i + 1]);
            }
          }
        }
      }
      uint4 o;
      o.x = dev::pack_bf16x2(acc[0], acc[1]);
      o.y = dev::pack_bf16x2(acc[2], acc[3]);
      o.z = dev::pack_bf16x2(acc[4], acc[5]);
      o.w = dev::pack_bf16x2(acc[6], acc[7]);
      out[static_cast<size_t>(t) * H8 + c] = o;
    }
  }
}

}  // namespace

cudaError_t launch_route(const float* logits, int T, int E, int k, int renorm, int tpc,
                         int32_t* ids, float* w, int32_t* chunk_hist, int* err,
                         const LaunchOpts& o) {
  const int chunks = (T + tpc - 1) / tpc;
  const size_t smem = static_cast<size_t>(E) * sizeof(int);
  const dim3 grid(chunks), block(32 * tpc < 1024 ? 32 * tpc : 1024);
  if (E <= 32)
    return launch(moe_route_kernel<1>, grid, block, smem, o, logits, T, E, k, renorm, tpc, ids, w,
                  chunk_hist, err);
  if (E <= 128)
    return launch(moe_route_kernel<4>, grid, block, smem, o, logits, T, E, k, renorm, tpc, ids, w,
                  chunk_hist, err);
  if (E <= 256)
    return launch(moe_route_kernel<8>, grid, block, smem, o, logits, T, E, k, renorm, tpc, ids, w,
                  chunk_hist, err);
  return launch(moe_route_kernel<16>, grid, block, smem, o, logits, T, E, k, renorm, tpc, ids, w,
                chunk_hist, err);
}

cudaError_t launch_align(const int32_t* ids, const int32_t* chunk_hist, int chunks, int A, int E,
                         int chunk, int32_t* offsets, int32_t* sorted, int32_t* inv,
                         int32_t* tiles, int32_t* num_tiles, int32_t* ptiles,
                         int32_t* num_ptiles, int32_t* tile_cnt, int cnt_len, int* err,
                         const LaunchOpts& o) {
  return launch(moe_align_kernel, dim3(chunks), dim3(kChunkAssign), 0, o, ids, chunk_hist, chunks,
                A, E, chunk, offsets, sorted, inv, tiles, num_tiles, ptiles, num_ptiles, tile_cnt,
                cnt_len, err);
}

cudaError_t launch_route_align_gather(const float* logits, const __nv_bfloat16* x, int T, int E,
                                      int k, int renorm, int H, int32_t* ids, float* w,
                                      int32_t* offsets, int32_t* sorted, int32_t* inv,
                                      int32_t* tiles, int32_t* num_tiles, int32_t* ptiles,
                                      int32_t* num_ptiles, int32_t* tile_cnt, int cnt_len,
                                      __nv_bfloat16* x_sorted, int* err, const LaunchOpts& o) {
  const int A = T * k;
  int grid = max(1, min((A + kFusedRowsPerCta - 1) / kFusedRowsPerCta, o.sm_count));
  grid = (grid + kFusedCluster - 1) / kFusedCluster * kFusedCluster;  // whole clusters
  const uint4* xv = reinterpret_cast<const uint4*>(x);
  uint4* xsv = reinterpret_cast<uint4*>(x_sorted);
  const dim3 g(grid), b(kChunkAssign);
  if (E <= 32)
    return launch_cluster(moe_route_align_gather_kernel<1>, g, b, kFusedCluster, o, logits, xv, T,
                          E, k, renorm, H / 8, ids, w, offsets, sorted, inv, tiles, num_tiles,
                          ptiles, num_ptiles, tile_cnt, cnt_len, xsv, err);
  if (E <= 128)
    return launch_cluster(moe_route_align_gather_kernel<4>, g, b, kFusedCluster, o, logits, xv, T,
                          E, k, renorm, H / 8, ids, w, offsets, sorted, inv, tiles, num_tiles,
                          ptiles, num_ptiles, tile_cnt, cnt_len, xsv, err);
  if (E <= 256)
    return launch_cluster(moe_route_align_gather_kernel<8>, g, b, kFusedCluster, o, logits, xv, T,
                          E, k, renorm, H / 8, ids, w, offsets, sorted, inv, tiles, num_tiles,
                          ptiles, num_ptiles, tile_cnt, cnt_len, xsv, err);
  return launch_cluster(moe_route_align_gather_kernel<16>, g, b, kFusedCluster, o, logits, xv, T,
                        E, k, renorm, H / 8, ids, w, offsets, sorted, inv, tiles, num_tiles,
                        ptiles, num_ptiles, tile_cnt, cnt_len, xsv, err);
}

cudaError_t launch_combine(const __nv_bfloat16* y, const int32_t* inv, const float* w, int T,
                           int k, int H, __nv_bfloat16* out, const LaunchOpts& o) {
  const int grid = min(T, o.sm_count * 8);
  return launch(moe_combine_kernel, dim3(grid), dim3(256), 0, o, reinterpret_cast<const uint4*>(y),
                inv, w, T, k, H / 8, reinterpret_cast<uint4*>(out));
}

}  // namespace rimuru
