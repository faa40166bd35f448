// Routing, grouping, row gather and combine kernels of the paged fused MoE
// layer (Rimuru, arXiv 2610.40305: the fused MoE layer around the
// page-table-aware expert GEMMs; the pages name the layer but not these
// steps, which follow the standard top-k MoE definition).
#include <cfloat>
#include <climits>

#include "device.cuh"
#include "kernels.h"

namespace rimuru {
namespace {

using dev::grid_dep_launch;
using dev::grid_dep_wait;
using dev::set_error;

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

// ----------------------------------------------------------------- route
// Experts per lane: lane l holds experts l, l + 32, l + 64, ...
template <int EPL>
__global__ void __launch_bounds__(512) moe_route_kernel(const float* __restrict__ logits, int T,
                                                        int E, int k, int renorm, int tpc,
                                                        int32_t* __restrict__ ids,
                                                        float* __restrict__ w,
                                                        int32_t* __restrict__ chunk_hist,
                                                        int* err) {
  extern __shared__ int s_hist[];  // [E]
  grid_dep_wait();
  for (int e = threadIdx.x; e < E; e += blockDim.x) s_hist[e] = 0;
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nwarps = blockDim.x >> 5;
  const int t_begin = blockIdx.x * tpc;
  const int t_end = min(t_begin + tpc, T);
  for (int t = t_begin + warp; t < t_end; t += nwarps) {
    const float* row = logits + static_cast<size_t>(t) * E;
    float v[EPL];
    bool bad = false;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      int e = lane + 32 * i;
      float x = -INFINITY;
      if (e < E) {
        x = row[e];
        if (!isfinite(x)) {
          bad = true;
          x = -INFINITY;  // invalid input: rank it last, keep ids valid
        }
      }
      v[i] = x;
    }
    if (__any_sync(kFull, bad) && lane == 0) set_error(err, RIMURU_DEV_NONFINITE);
    uint32_t taken = 0;
    float m = 0.f, psum = 0.f, my_p = 0.f;
    int my_id = 0;
    for (int j = 0; j < k; ++j) {
      // best untaken expert of this lane: larger logit, then lower index
      float bv = -INFINITY;
      int be = INT_MAX;
#pragma unroll
      for (int i = 0; i < EPL; ++i) {
        int e = lane + 32 * i;
        if (e < E && !((taken >> i) & 1u) && (v[i] > bv || (v[i] == bv && e < be))) {
          bv = v[i];
          be = e;
        }
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        float ov = __shfl_xor_sync(kFull, bv, off);
        int oe = __shfl_xor_sync(kFull, be, off);
        if (ov > bv || (ov == bv && oe < be)) {
          bv = ov;
          be = oe;
        }
      }
      if (j == 0) m = (bv == -INFINITY) ? 0.f : bv;  // largest logit of the token
      if ((be & 31) == lane) taken |= 1u << (be >> 5);
      float p = expf(bv - m);
      psum += p;
      if (lane == j) {
        my_id = be;
        my_p = p;
      }
    }
    float denom = psum;
    if (!renorm) {
      float s = 0.f;
#pragma unroll
      for (int i = 0; i < EPL; ++i)
        if (lane + 32 * i < E) s += expf(v[i] - m);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(kFull, s, off);
      denom = s;
    }
    if (lane < k) {
      ids[static_cast<size_t>(t) * k + lane] = my_id;
      w[static_cast<size_t>(t) * k + lane] = my_p / denom;
      atomicAdd(&s_hist[my_id], 1);
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    chunk_hist[static_cast<size_t>(blockIdx.x) * E + e] = s_hist[e];
  grid_dep_launch();
}

// Exclusive prefix sum over the block (one value per thread, blockDim <= 1024).
__device__ int block_exclusive_scan(int v, int* s_warp) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nwarps = blockDim.x >> 5;
  int x = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    int y = __shfl_up_sync(kFull, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) s_warp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int s = lane < nwarps ? s_warp[lane] : 0;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      int y = __shfl_up_sync(kFull, s, off);
      if (lane >= off) s += y;
    }
    if (lane < nwarps) s_warp[lane] = s;  // inclusive warp totals
  }
  __syncthreads();
  int before = warp > 0 ? s_warp[warp - 1] : 0;
  __syncthreads();  // s_warp may be reused by the caller
  return before + x - v;
}

// ----------------------------------------------------------------- align
__global__ void __launch_bounds__(kChunkAssign) moe_align_kernel(
    const int32_t* __restrict__ ids, const int32_t* __restrict__ chunk_hist, int chunks, int A,
    int E, int chunk, int32_t* __restrict__ offsets, int32_t* __restrict__ sorted,
    int32_t* __restrict__ inv, int32_t* __restrict__ tiles, int32_t* __restrict__ num_tiles,
    int* err) {
  __shared__ int s_base[kMaxExperts];
  __shared__ int s_ids[kChunkAssign];
  __shared__ int s_warp[32];
  grid_dep_wait();
  const int c = blockIdx.x;
  const int e = threadIdx.x;  // blockDim == kChunkAssign >= E
  int tot = 0, before = 0;
  if (e < E) {
    for (int cc = 0; cc < chunks; ++cc) {
      int n = chunk_hist[static_cast<size_t>(cc) * E + e];
      tot += n;
      if (cc < c) before += n;
    }
  }
  const int off = block_exclusive_scan(tot, s_warp);
  if (e < E) s_base[e] = off + before;
  if (c == 0) {
    if (e < E) offsets[e] = off;
    if (e == E - 1) offsets[E] = off + tot;
    const int nb = (tot + kTileM - 1) / kTileM;
    const int first = block_exclusive_scan(nb, s_warp);
    if (e < E) {
      for (int b = 0; b < nb; ++b) {
        tiles[2 * (first + b)] = e;
        tiles[2 * (first + b) + 1] = off + b * kTileM;
      }
    }
    if (e == E - 1) *num_tiles = first + nb;
  }
  const int f0 = c * chunk;
  const int n = min(chunk, A - f0);
  if (static_cast<int>(threadIdx.x) < n) s_ids[threadIdx.x] = ids[f0 + threadIdx.x];
  __syncthreads();
  if (static_cast<int>(threadIdx.x) < n) {
    const int my = s_ids[threadIdx.x];
    if (my < 0 || my >= E) {
      set_error(err, RIMURU_DEV_BAD_SHAPE);
    } else {
      int rank = 0;  // earlier assignments of the same expert inside this chunk
      for (int j = 0; j < static_cast<int>(threadIdx.x); ++j) rank += (s_ids[j] == my);
      const int pos = s_base[my] + rank;
      sorted[pos] = f0 + threadIdx.x;
      inv[f0 + threadIdx.x] = pos;
    }
  }
  grid_dep_launch();
}

// ----------------------------------------------------------------- gather
__global__ void __launch_bounds__(256) moe_gather_kernel(const uint4* __restrict__ x,
                                                         const int32_t* __restrict__ sorted, int A,
                                                         int k, int H8, uint4* __restrict__ xs) {
  grid_dep_wait();
  for (int r = blockIdx.x; r < A; r += gridDim.x) {
    const int t = sorted[r] / k;
    const uint4* src = x + static_cast<size_t>(t) * H8;
    uint4* dst = xs + static_cast<size_t>(r) * H8;
    for (int c = threadIdx.x; c < H8; c += blockDim.x) dst[c] = src[c];
  }
  grid_dep_launch();
}

// ----------------------------------------------------------------- combine
__global__ void __launch_bounds__(256) moe_combine_kernel(const uint4* __restrict__ y,
                                                          const int32_t* __restrict__ inv,
                                                          const float* __restrict__ w, int T,
                                                          int k, int H8, uint4* __restrict__ out) {
  grid_dep_wait();
  for (int t = blockIdx.x; t < T; t += gridDim.x) {
    for (int c = threadIdx.x; c < H8; c += blockDim.x) {
      float acc[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = 0.f;
      for (int j = 0; j < k; ++j) {
        const int f = t * k + j;
        const float wj = w[f];
        uint4 v = y[static_cast<size_t>(inv[f]) * H8 + c];
        const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          float2 f2 = __bfloat1622float2(p[i]);
          acc[2 * i] = fmaf(wj, f2.x, acc[2 * i]);
          acc[2 * i + 1] = fmaf(wj, f2.y, acc[2 * i + 1]);
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
  grid_dep_launch();
}

}  // namespace

cudaError_t launch_route(const float* logits, int T, int E, int k, int renorm, int tpc,
                         int32_t* ids, float* w, int32_t* chunk_hist, int* err,
                         const LaunchOpts& o) {
  const int chunks = (T + tpc - 1) / tpc;
  const size_t smem = static_cast<size_t>(E) * sizeof(int);
  const dim3 grid(chunks), block(512);
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
                         int32_t* tiles, int32_t* num_tiles, int* err, const LaunchOpts& o) {
  return launch(moe_align_kernel, dim3(chunks), dim3(kChunkAssign), 0, o, ids, chunk_hist, chunks,
                A, E, chunk, offsets, sorted, inv, tiles, num_tiles, err);
}

cudaError_t launch_gather(const __nv_bfloat16* x, const int32_t* sorted, int A, int k, int H,
                          __nv_bfloat16* x_sorted, const LaunchOpts& o) {
  const int grid = min(A, o.sm_count * 8);
  return launch(moe_gather_kernel, dim3(grid), dim3(256), 0, o, reinterpret_cast<const uint4*>(x),
                sorted, A, k, H / 8, reinterpret_cast<uint4*>(x_sorted));
}

cudaError_t launch_combine(const __nv_bfloat16* y, const int32_t* inv, const float* w, int T,
                           int k, int H, __nv_bfloat16* out, const LaunchOpts& o) {
  const int grid = min(T, o.sm_count * 8);
  return launch(moe_combine_kernel, dim3(grid), dim3(256), 0, o, reinterpret_cast<const uint4*>(y),
                inv, w, T, k, H / 8, reinterpret_cast<uint4*>(out));
}

}  // namespace rimuru
