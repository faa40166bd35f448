// The paged fused MoE layer for decode-sized batches (a few tokens): three
// kernels instead of the five of the general launch sequence.
//
// What the layer computes is unchanged (Rimuru, arXiv 2610.40305, abstract and
// the explainer page's paragraph on the fused MoE kernel: expert weights read
// in place from their pool pages through the expert view's page table).  What
// changes is how the few rows of a decode step meet the weights.  With one to
// a few tokens each routed expert has one to a few rows, so the layer is bound
// by the bytes of the routed experts' pages (three 2-3 MiB pages each) and by
// latency, not by arithmetic: the general path spends most of a one-token step
// in launch chains, pipeline fills and split-K bookkeeping.  Here:
//
//   decode_gemm1  every CTA routes the whole batch itself (a warp per token),
//                 so the first weight copy is issued about a microsecond after
//                 the logits are readable, with no routing kernel in front.
//                 The W1/W3 weights of the routed experts are cut into
//                 (expert, 64-column block, 64-deep k block) units spread
//                 evenly over the grid; each CTA streams its contiguous run of
//                 units through a TMA ring and multiplies them on the CUDA
//                 cores with the expert's rows (tensor-core tiles would be
//                 almost all padding).  A CTA writes one fp32 partial of gate
//                 and up per (expert, column block) it touched.  Each CTA also
//                 prefetches its share of the routed experts' W2 pages into L2,
//                 so the second GEMM reads them from L2.
//   decode_reduce one CTA per (expert, column block): sums the partials in CTA
//                 order (deterministic) and writes h = silu(gate) * up in bf16.
//   decode_gemm2  one CTA per 8 output columns: y = h W2_e for every routed
//                 row (a warp per expert, W2 read from L2), rounded to bf16 as
//                 in the general path, then the weighted combine of each
//                 token's k rows in slot order, written as bf16 out.
//
// All three run with programmatic dependent launch and wait (griddepcontrol)
// before touching their predecessor's output; every CTA executes that wait, so
// a kernel's completion implies its predecessor's.
#include <atomic>

#include "device.cuh"
#include "kernels.h"
#include "route.cuh"

namespace rimuru {
namespace {

using namespace dev;

constexpr int kBox = 64;                            // 64 x 64 bf16 boxes of the w1/w3 pages
constexpr int kBoxBytes = kBox * kBox * 2;          // 8 KiB
constexpr int kUnitBytes = 2 * kBoxBytes;           // one unit: the w1 box and the w3 box
constexpr int kConsumerWarps = 8;                   // 2 matrices x 4 quarters of the k block
constexpr int kThreads1 = 32 * (kConsumerWarps + 1);  // + the TMA producer warp
constexpr int kThreadsR = 128;
constexpr int kThreads2 = 256;
constexpr int kCols2 = 8;                           // output columns per decode_gemm2 CTA
constexpr int kSmemLimit = 232448;                  // opt-in shared memory per block

// Plan written by CTA 0 of decode_gemm1 for the two kernels after it:
// [0] = U (routed experts), then per routed expert u (ascending expert id):
// expert id, first sorted row, row count.
constexpr int kPlanExp = 1;
constexpr int kPlanOff = 1 + kDecodeMaxA;
constexpr int kPlanCnt = 1 + 2 * kDecodeMaxA;

struct Shared1 {
  uint64_t full[kDecodeStagesMax];   // the unit's two boxes have landed
  uint64_t empty[kDecodeStagesMax];  // the eight consumer warps are done with the stage
  int ids[kDecodeMaxA];
  float w[kDecodeMaxA];
  int sorted[kDecodeMaxA];
  int first[kDecodeMaxA];
  int uexp[kDecodeMaxA], uoff[kDecodeMaxA], ucnt[kDecodeMaxA];
  int U;
  int abort;
};

__device__ __forceinline__ void consumer_bar() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

// Range of work units of CTA c out of G: [c W / G, (c + 1) W / G).
__device__ __forceinline__ long long unit_lo(long long c, long long W, long long G) {
  return c * W / G;
}

// This CTA's share of the routed experts' W2 pages, as L2 prefetches: the
// pages' bytes are split evenly over the grid in 16-byte-aligned pieces.
__device__ void prefetch_w2_share(const DecodeArgs& p, const Shared1* sh, int U) {
  const uint64_t P2 = static_cast<uint64_t>(p.I) * p.H * 2;
  const uint64_t total = static_cast<uint64_t>(U) * P2;
  const uint64_t G = gridDim.x, c = blockIdx.x;
  uint64_t b0 = (c * total / G) & ~15ull;
  const uint64_t b1 = ((c + 1) * total / G) & ~15ull;
  while (b0 < b1) {
    const int u = static_cast<int>(b0 / P2);
    const uint64_t off = b0 % P2;
    uint64_t n = b1 - b0;
    if (n > P2 - off) n = P2 - off;
    if (n > 32768) n = 32768;
    const int pg = p.page_table[3 * sh->uexp[u] + RIMURU_PROJ_W2];
    if (pg >= 0 && pg < p.num_pages)
      bulk_prefetch_l2(p.pool + static_cast<uint64_t>(pg) * p.page_bytes + off,
                       static_cast<uint32_t>(n));
    b0 += n;
  }
}

// One unit's multiply-accumulate for R rows of the expert (R known at compile
// time, so a one-token step does one row's work): warp (m, hq) covers k rows
// 16 hq .. 16 hq + 15 of the box of matrix m; lane l columns 2l, 2l + 1.
template <int R>
__device__ __forceinline__ void mac_unit(const uint8_t* __restrict__ box,
                                         const __nv_bfloat16* __restrict__ xs,
                                         const int (&tok)[kDecodeMaxT], int H, int hoff, int hq,
                                         int lane, float (&acc)[kDecodeMaxT][2]) {
  // 16-byte chunk c of box row h sits at chunk c ^ (h % 8) (128-byte swizzle)
  const int c16 = (lane * 4) >> 4, in16 = (lane * 4) & 15;
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    // eight x values of each row for these k rows (the same for every lane: broadcast)
    float xv[R][8];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const uint4 a =
          *reinterpret_cast<const uint4*>(xs + tok[r] * H + hoff + hq * 16 + half * 8);
      const __nv_bfloat162* pa = reinterpret_cast<const __nv_bfloat162*>(&a);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 f = __bfloat1622float2(pa[i]);
        xv[r][2 * i] = f.x;
        xv[r][2 * i + 1] = f.y;
      }
    }
#pragma unroll
    for (int hh = 0; hh < 8; ++hh) {
      const int h = hq * 16 + half * 8 + hh;
      const uint32_t wbits =
          *reinterpret_cast<const uint32_t*>(box + h * 128 + ((c16 ^ (h & 7)) << 4) + in16);
      const float2 wf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wbits));
#pragma unroll
      for (int r = 0; r < R; ++r) {
        acc[r][0] = fmaf(xv[r][hh], wf.x, acc[r][0]);
        acc[r][1] = fmaf(xv[r][hh], wf.y, acc[r][1]);
      }
    }
  }
}

template <int EPL>
__global__ void __launch_bounds__(kThreads1, 1)
    decode_gemm1_kernel(const __grid_constant__ CUtensorMap tm_w, const DecodeArgs p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int S = p.stages;
  const int T = p.T, H = p.H, I = p.I, k = p.k, E = p.E;
  const int A = T * k;
  uint8_t* ring = smem;                                               // [S][w1 box | w3 box]
  __nv_bfloat16* xs = reinterpret_cast<__nv_bfloat16*>(smem + S * kUnitBytes);  // [T][H]
  float* red = reinterpret_cast<float*>(smem + S * kUnitBytes + T * H * 2);     // [2][4][T][64]
  Shared1* sh = reinterpret_cast<Shared1*>(red + 2 * 4 * T * 64);
  volatile int* abort = &sh->abort;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool lead = blockIdx.x == 0;

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&sh->full[s], 1);
      mbar_init(&sh->empty[s], kConsumerWarps);
    }
    sh->abort = 0;
    fence_barrier_init();
    prefetch_tmap(&tm_w);
  }
  __syncthreads();
  grid_dep_wait();    // x and logits may come from the kernel before this one
  grid_dep_launch();  // the next kernel may be scheduled; it waits for our completion

  {  // the batch's x rows into shared memory
    const uint4* src = reinterpret_cast<const uint4*>(p.x);
    uint4* dst = reinterpret_cast<uint4*>(xs);
    const int n = T * H / 8;
    for (int i = tid; i < n; i += blockDim.x) dst[i] = src[i];
  }
  // routing, every CTA for itself: warp w routes token w
  for (int t = warp; t < T; t += blockDim.x / 32) {
    int id;
    float wt;
    route_token<EPL>(p.logits + static_cast<size_t>(t) * E, E, k, p.renorm, lane, p.err, id, wt);
    if (lane < k) {
      sh->ids[t * k + lane] = id;
      sh->w[t * k + lane] = wt;
      if (lead) {
        p.ids[t * k + lane] = id;
        p.w[t * k + lane] = wt;
      }
    }
  }
  __syncthreads();
  // grouping: assignment f goes to sorted row (#assignments of smaller experts)
  // + (#earlier assignments of its own expert), i.e. stable by f within an expert
  int my_e = 0, before = 0, same = 0;
  if (tid < A) {
    my_e = sh->ids[tid];
    int same_before = 0;
    for (int f = 0; f < A; ++f) {
      const int e = sh->ids[f];
      before += e < my_e;
      same += e == my_e;
      same_before += (e == my_e) && (f < tid);
    }
    const int pos = before + same_before;
    sh->sorted[pos] = tid;
    sh->first[tid] = same_before == 0;
    if (lead) {
      p.sorted[pos] = tid;
      p.inv[tid] = pos;
    }
  }
  __syncthreads();
  if (tid < A && sh->first[tid]) {  // one thread per routed expert: its rank among them
    int u = 0;
    for (int f = 0; f < A; ++f) u += sh->first[f] && sh->ids[f] < my_e;
    sh->uexp[u] = my_e;
    sh->uoff[u] = before;
    sh->ucnt[u] = same;
  }
  if (tid == 0) {
    int U = 0;
    for (int f = 0; f < A; ++f) U += sh->first[f];
    sh->U = U;
  }
  __syncthreads();
  const int U = sh->U;
  if (lead) {  // the tables of the general path (one 128-row block per routed expert) and the plan
    for (int e = tid; e <= E; e += blockDim.x) {
      int c = 0;
      for (int f = 0; f < A; ++f) c += sh->ids[f] < e;
      p.offsets[e] = c;
    }
    for (int u = tid; u < U; u += blockDim.x) {
      p.tiles[2 * u] = p.ptiles[2 * u] = sh->uexp[u];
      p.tiles[2 * u + 1] = p.ptiles[2 * u + 1] = sh->uoff[u];
      p.plan[kPlanExp + u] = sh->uexp[u];
      p.plan[kPlanOff + u] = sh->uoff[u];
      p.plan[kPlanCnt + u] = sh->ucnt[u];
    }
    if (tid == 0) {
      *p.num_tiles = U;
      *p.num_ptiles = U;
      p.plan[0] = U;
    }
  }

  // work units q = (group g = (routed expert u, column block nb), k block kb)
  const int NB = I / kBox, KB = H / kBox;
  const long long W = static_cast<long long>(U) * NB * KB;
  const long long lo = unit_lo(blockIdx.x, W, gridDim.x);
  const long long hi = unit_lo(blockIdx.x + 1, W, gridDim.x);

  if (warp == kConsumerWarps) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer
      const uint64_t pol = policy_evict_first();  // each weight byte is read once
      uint32_t s = 0, ph = 0;
      int issued = 0;
      bool ok = true, prefetched = p.prefetch_w2 == 0;
      // (group, k block) of unit lo, then advanced one unit at a time
      int g = static_cast<int>(lo / KB), kb = static_cast<int>(lo % KB);
      for (long long q = lo; q < hi; ++q) {
        const int u = g / NB, nb = g - u * NB;
        const int e = sh->uexp[u];
        int pg1 = p.page_table[3 * e + RIMURU_PROJ_W1];
        int pg3 = p.page_table[3 * e + RIMURU_PROJ_W3];
        if (pg1 < 0 || pg1 >= p.num_pages || pg3 < 0 || pg3 >= p.num_pages) {
          set_error(p.err, RIMURU_DEV_BAD_PAGE);  // host checks make this unreachable
          pg1 = pg3 = 0;
        }
        if (!mbar_wait(&sh->empty[s], ph ^ 1u, abort)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&sh->full[s], kUnitBytes);
        uint8_t* st = ring + s * kUnitBytes;
        tma_load_3d(st, &tm_w, &sh->full[s], nb * kBox, kb * kBox, pg1, pol);
        tma_load_3d(st + kBoxBytes, &tm_w, &sh->full[s], nb * kBox, kb * kBox, pg3, pol);
        ++issued;
        if (++kb == KB) {
          kb = 0;
          ++g;
        }
        if (++s == static_cast<uint32_t>(S)) {
          s = 0;
          ph ^= 1u;
        }
        // the W2 prefetches go out once the ring's first fill is on its way
        if (!prefetched && issued == S) {
          prefetch_w2_share(p, sh, U);
          prefetched = true;
        }
      }
      if (!prefetched) prefetch_w2_share(p, sh, U);
      if (!ok) {
        set_error(p.err, RIMURU_DEV_TIMEOUT);
        sh->abort = 1;
      }
      // every copy this thread issued must have landed before the CTA exits
      volatile int never = 0;
      for (int j = issued > S ? issued - S : 0; j < issued; ++j)
        mbar_wait(&sh->full[j % S], static_cast<uint32_t>(j / S) & 1u, &never);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  // Warp w multiplies matrix m = w / 4 (0: w1 -> gate, 1: w3 -> up) over rows
  // 16 (w % 4) .. + 15 of each 64-deep k block; lane l owns output columns
  // 2l, 2l + 1 of the block, for every row of the unit's expert.
  const int m = warp >> 2, hq = warp & 3;
  float acc[kDecodeMaxT][2];
  int tok[kDecodeMaxT];
  int cur_g = -1, rows = 0;
  uint32_t s = 0, ph = 0;
  bool ok = true;

  // Sum the four k quarters of the finished group through shared memory and
  // write its fp32 partial (64 gate then 64 up columns per row) to slot g + c.
  auto flush = [&](int g) {
    consumer_bar();  // the previous flush has read `red`
    float* rb = red + ((m * 4 + hq) * T) * 64;
#pragma unroll
    for (int r = 0; r < kDecodeMaxT; ++r) {
      if (r < rows) {
        rb[r * 64 + 2 * lane] = acc[r][0];
        rb[r * 64 + 2 * lane + 1] = acc[r][1];
      }
    }
    consumer_bar();
    float* dst = p.part + (static_cast<size_t>(g) + blockIdx.x) * T * 128;
    for (int idx = tid; idx < 2 * rows * 64; idx += 32 * kConsumerWarps) {
      const int mm = idx / (rows * 64), rem = idx - mm * rows * 64;
      const int r = rem >> 6, c = rem & 63;
      float v = 0.f;
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) v += red[((mm * 4 + q4) * T + r) * 64 + c];
      dst[r * 128 + mm * 64 + c] = v;
    }
  };

  int g = static_cast<int>(lo / KB), kb = static_cast<int>(lo % KB);
  for (long long q = lo; q < hi; ++q) {
    if (g != cur_g) {
      if (cur_g >= 0) flush(cur_g);
      cur_g = g;
      const int u = g / NB;
      rows = sh->ucnt[u];
#pragma unroll
      for (int r = 0; r < kDecodeMaxT; ++r) {
        tok[r] = r < rows ? sh->sorted[sh->uoff[u] + r] / k : 0;
        acc[r][0] = acc[r][1] = 0.f;
      }
    }
    if (ok) {
      // every lane observes the stage's completion itself (the TMA bytes are then
      // visible to it)
      const bool got = __all_sync(0xffffffffu, mbar_wait(&sh->full[s], ph, abort));
      if (!got) {
        ok = false;
        if (lane == 0) {
          set_error(p.err, RIMURU_DEV_TIMEOUT);
          sh->abort = 1;
        }
      }
    }
    if (ok) {
      const uint8_t* box = ring + s * kUnitBytes + m * kBoxBytes;
      const int hoff = kb * kBox;
      switch (rows) {
        case 1: mac_unit<1>(box, xs, tok, H, hoff, hq, lane, acc); break;
        case 2: mac_unit<2>(box, xs, tok, H, hoff, hq, lane, acc); break;
        case 3: mac_unit<3>(box, xs, tok, H, hoff, hq, lane, acc); break;
        default: mac_unit<4>(box, xs, tok, H, hoff, hq, lane, acc); break;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh->empty[s]);
    }
    if (++s == static_cast<uint32_t>(S)) {
      s = 0;
      ph ^= 1u;
    }
    if (++kb == KB) {
      kb = 0;
      ++g;
    }
  }
  if (cur_g >= 0) flush(cur_g);
}

// One CTA per (routed expert, 64-column block of h).
__global__ void __launch_bounds__(kThreadsR) decode_reduce_kernel(const DecodeArgs p) {
  grid_dep_wait();
  grid_dep_launch();
  const int U = __ldcg(p.plan);
  const int NB = p.I / kBox, KB = p.H / kBox;
  const int NG = U * NB, g = blockIdx.x;
  if (g >= NG) return;
  const int u = g / NB, nb = g % NB;
  const int rows = __ldcg(p.plan + kPlanCnt + u), uoff = __ldcg(p.plan + kPlanOff + u);
  const long long W = static_cast<long long>(NG) * KB, G = p.grid1;
  // CTAs of decode_gemm1 whose unit range meets units [g KB, (g + 1) KB): from
  // the last one starting at or before the group's first unit to the last one
  // starting at or before its last unit (empty ranges wrote nothing)
  const long long x0 = static_cast<long long>(g) * KB, x1 = x0 + KB - 1;
  const int c0 = static_cast<int>(((x0 + 1) * G + W - 1) / W) - 1;
  const int c1 = static_cast<int>(((x1 + 1) * G + W - 1) / W) - 1;
  for (int idx = threadIdx.x; idx < rows * 64; idx += blockDim.x) {
    const int r = idx >> 6, c = idx & 63;
    float gs = 0.f, us = 0.f;
    for (int cc = c0; cc <= c1; ++cc) {
      if (unit_lo(cc, W, G) == unit_lo(cc + 1, W, G)) continue;
      const float* pr = p.part + ((static_cast<size_t>(g) + cc) * p.T + r) * 128;
      gs += __ldcg(pr + c);
      us += __ldcg(pr + 64 + c);
    }
    p.h[static_cast<size_t>(uoff + r) * p.I + nb * kBox + c] = __float2bfloat16_rn(silu_mul(gs, us));
  }
}

// y rows uoff .. uoff + R - 1 (one expert) for this CTA's kCols2 columns, by one
// warp: lane l takes w2 rows i = l, l + 32, ... (two to eight 16-byte loads in
// flight, fewer as R grows),
// the warp sums over i with shuffles; lane 0 writes y (bf16) and keeps the
// rounded values for the combine.
template <int R>
__device__ __forceinline__ void y_rows(const __nv_bfloat16* __restrict__ w2,
                                       const __nv_bfloat16* __restrict__ hs, int uoff, int I,
                                       int H, int c0, int lane, __nv_bfloat16* __restrict__ y,
                                       float (*s_y)[kCols2]) {
  float acc[R][kCols2];
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int c = 0; c < kCols2; ++c) acc[r][c] = 0.f;
  constexpr int kInFlight = R <= 2 ? 8 : (R <= 4 ? 4 : 2);  // registers: acc grows with R
  for (int i0 = lane; i0 < I; i0 += 32 * kInFlight) {
    uint4 wv[kInFlight];
#pragma unroll
    for (int j = 0; j < kInFlight; ++j) {
      const int i = i0 + 32 * j;
      if (i < I) wv[j] = ld_nc_na_v4(w2 + static_cast<size_t>(i) * H + c0);
    }
#pragma unroll
    for (int j = 0; j < kInFlight; ++j) {
      const int i = i0 + 32 * j;
      if (i < I) {
        const __nv_bfloat162* wp = reinterpret_cast<const __nv_bfloat162*>(&wv[j]);
        float wf[kCols2];
#pragma unroll
        for (int c = 0; c < kCols2 / 2; ++c) {
          const float2 f2 = __bfloat1622float2(wp[c]);
          wf[2 * c] = f2.x;
          wf[2 * c + 1] = f2.y;
        }
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const float hv = __bfloat162float(hs[(uoff + r) * I + i]);
#pragma unroll
          for (int c = 0; c < kCols2; ++c) acc[r][c] = fmaf(hv, wf[c], acc[r][c]);
        }
      }
    }
  }
#pragma unroll
  for (int r = 0; r < R; ++r) {
#pragma unroll
    for (int c = 0; c < kCols2; ++c) {
      float v = acc[r][c];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
      acc[r][c] = v;
    }
    if (lane == 0) {
      uint4 o;
      o.x = pack_bf16x2(acc[r][0], acc[r][1]);
      o.y = pack_bf16x2(acc[r][2], acc[r][3]);
      o.z = pack_bf16x2(acc[r][4], acc[r][5]);
      o.w = pack_bf16x2(acc[r][6], acc[r][7]);
      *reinterpret_cast<uint4*>(y + static_cast<size_t>(uoff + r) * H + c0) = o;
      const __nv_bfloat162* ob = reinterpret_cast<const __nv_bfloat162*>(&o);
#pragma unroll
      for (int c = 0; c < kCols2 / 2; ++c) {
        const float2 f2 = __bfloat1622float2(ob[c]);
        s_y[uoff + r][2 * c] = f2.x;
        s_y[uoff + r][2 * c + 1] = f2.y;
      }
    }
  }
}

// One CTA per kCols2 output columns: y for every routed row, then the combine.
// RMAX bounds the rows of one expert (<= T): a one-token step runs the lean
// RMAX = 1 instance, which fits several CTAs per SM.
template <int RMAX>
__global__ void __launch_bounds__(kThreads2, RMAX <= 2 ? 2 : 1) decode_gemm2_kernel(const DecodeArgs p) {
  extern __shared__ uint8_t smem2[];
  __nv_bfloat16* hs = reinterpret_cast<__nv_bfloat16*>(smem2);  // [A][I]
  __shared__ int s_uexp[kDecodeMaxA], s_uoff[kDecodeMaxA], s_ucnt[kDecodeMaxA];
  __shared__ int s_inv[kDecodeMaxA];
  __shared__ float s_w[kDecodeMaxA];
  __shared__ float s_y[kDecodeMaxA][kCols2];
  grid_dep_wait();
  grid_dep_launch();
  const int T = p.T, k = p.k, H = p.H, I = p.I;
  const int A = T * k;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int U = __ldcg(p.plan);
  for (int i = tid; i < U; i += blockDim.x) {
    s_uexp[i] = __ldcg(p.plan + kPlanExp + i);
    s_uoff[i] = __ldcg(p.plan + kPlanOff + i);
    s_ucnt[i] = __ldcg(p.plan + kPlanCnt + i);
  }
  for (int f = tid; f < A; f += blockDim.x) {
    s_inv[f] = __ldcg(p.inv + f);
    s_w[f] = __ldcg(p.w + f);
  }
  {
    const uint4* src = reinterpret_cast<const uint4*>(p.h);
    uint4* dst = reinterpret_cast<uint4*>(hs);
    for (int i = tid; i < A * I / 8; i += blockDim.x) dst[i] = __ldcg(src + i);
  }
  __syncthreads();
  const int c0 = blockIdx.x * kCols2;
  for (int u = warp; u < U; u += kThreads2 / 32) {
    const int e = s_uexp[u], rows = s_ucnt[u], uoff = s_uoff[u];
    int pg = p.page_table[3 * e + RIMURU_PROJ_W2];
    if (pg < 0 || pg >= p.num_pages) {
      set_error(p.err, RIMURU_DEV_BAD_PAGE);  // host checks make this unreachable
      pg = 0;
    }
    const __nv_bfloat16* w2 =
        reinterpret_cast<const __nv_bfloat16*>(p.pool + static_cast<uint64_t>(pg) * p.page_bytes);
    if (RMAX == 1 || rows == 1) {
      y_rows<1>(w2, hs, uoff, I, H, c0, lane, p.y, s_y);
    } else if (RMAX == 2 || rows == 2) {
      y_rows<(RMAX >= 2 ? 2 : 1)>(w2, hs, uoff, I, H, c0, lane, p.y, s_y);
    } else if (rows == 3) {
      y_rows<(RMAX >= 3 ? 3 : 1)>(w2, hs, uoff, I, H, c0, lane, p.y, s_y);
    } else {
      y_rows<(RMAX >= 4 ? 4 : 1)>(w2, hs, uoff, I, H, c0, lane, p.y, s_y);
    }
  }
  __syncthreads();
  // combine: out[t] = sum_j w[t, j] * y[t * k + j] over the bf16 y rows, j ascending, fp32
  for (int idx = tid; idx < T * kCols2; idx += blockDim.x) {
    const int t = idx / kCols2, c = idx % kCols2;
    float o = 0.f;
    for (int j = 0; j < k; ++j) {
      const int f = t * k + j;
      o = fmaf(s_w[f], s_y[s_inv[f]][c], o);
    }
    p.out[static_cast<size_t>(t) * H + c0 + c] = __float2bfloat16_rn(o);
  }
}

// The dynamic shared-memory opt-in is a per-device function attribute: set it
// once per device and kernel, to the most the kernel can ask for.
template <typename Kern>
cudaError_t set_smem_once(Kern kernel, int bytes, std::atomic<bool>* configured) {
  int dev = 0;
  cudaError_t st = cudaGetDevice(&dev);
  if (st != cudaSuccess) return st;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!configured[dev].load(std::memory_order_acquire)) {
    st = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (st != cudaSuccess) return st;
    configured[dev].store(true, std::memory_order_release);
  }
  return cudaSuccess;
}

cudaError_t launch_pdl(const void* fn, dim3 grid, dim3 block, size_t smem, const LaunchOpts& o,
                       void** args) {
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
  return cudaLaunchKernelExC(&cfg, fn, args);
}

// Shared memory of decode_gemm1 with `stages` ring stages.
int smem1_bytes(int T, int H, int stages) {
  return 1024 + stages * kUnitBytes + T * H * 2 + 2 * 4 * T * 64 * 4 +
         static_cast<int>(sizeof(Shared1));
}

}  // namespace

bool decode_path_fits(int T, int k, int H, int I) {
  const long long A = static_cast<long long>(T) * k;
  return T >= 1 && T <= kDecodeMaxT && A <= kDecodeMaxA && H % kBox == 0 && I % kBox == 0 &&
         T * H * 2 <= 32768 && A * I * 2 <= kDecodeMaxHBytes && smem1_bytes(T, H, 4) <= kSmemLimit;
}

int decode_grid1(int sm_count) { return sm_count < kDecodeGridMax ? sm_count : kDecodeGridMax; }

uint64_t decode_part_bytes(int T, int k, int E, int I) {
  const long long A = static_cast<long long>(T) * k;
  const long long groups = (A < E ? A : E) * (I / kBox);
  return static_cast<uint64_t>(groups + kDecodeGridMax) * T * 128 * sizeof(float);
}

template <int EPL>
cudaError_t launch_gemm1_epl(const CUtensorMap& tm_w13, DecodeArgs& a, int smem,
                             const LaunchOpts& o) {
  static std::atomic<bool> configured[64];
  cudaError_t st = set_smem_once(decode_gemm1_kernel<EPL>, kSmemLimit, configured);
  if (st != cudaSuccess) return st;
  CUtensorMap tm = tm_w13;
  void* args[] = {&tm, &a};
  return launch_pdl(reinterpret_cast<const void*>(decode_gemm1_kernel<EPL>), dim3(a.grid1),
                    dim3(kThreads1), smem, o, args);
}

cudaError_t launch_decode_gemm1(const CUtensorMap& tm_w13, DecodeArgs a, const LaunchOpts& o) {
  int stages = kDecodeStagesMax;
  while (stages > 2 && smem1_bytes(a.T, a.H, stages) > kSmemLimit) --stages;
  a.stages = stages;
  const int smem = smem1_bytes(a.T, a.H, stages);
  if (a.E <= 32) return launch_gemm1_epl<1>(tm_w13, a, smem, o);
  if (a.E <= 128) return launch_gemm1_epl<4>(tm_w13, a, smem, o);
  if (a.E <= 256) return launch_gemm1_epl<8>(tm_w13, a, smem, o);
  return launch_gemm1_epl<16>(tm_w13, a, smem, o);
}

cudaError_t launch_decode_reduce(DecodeArgs a, const LaunchOpts& o) {
  const long long A = static_cast<long long>(a.T) * a.k;
  const int grid = static_cast<int>((A < a.E ? A : a.E) * (a.I / kBox));
  void* args[] = {&a};
  return launch_pdl(reinterpret_cast<const void*>(decode_reduce_kernel), dim3(grid),
                    dim3(kThreadsR), 0, o, args);
}

template <int RMAX>
cudaError_t launch_gemm2_rmax(DecodeArgs& a, const LaunchOpts& o) {
  static std::atomic<bool> configured[64];
  const int smem = a.T * a.k * a.I * 2;
  cudaError_t st = set_smem_once(decode_gemm2_kernel<RMAX>, kDecodeMaxHBytes, configured);
  if (st != cudaSuccess) return st;
  void* args[] = {&a};
  return launch_pdl(reinterpret_cast<const void*>(decode_gemm2_kernel<RMAX>), dim3(a.H / kCols2),
                    dim3(kThreads2), smem, o, args);
}

cudaError_t launch_decode_gemm2(DecodeArgs a, const LaunchOpts& o) {
  // an expert's rows are at most T (each token picks an expert once)
  if (a.T <= 1) return launch_gemm2_rmax<1>(a, o);
  if (a.T <= 2) return launch_gemm2_rmax<2>(a, o);
  return launch_gemm2_rmax<4>(a, o);  // T <= kDecodeMaxT = 4
}

}  // namespace rimuru
