// GEMM 1 + SwiGLU for large batches: one CTA takes two 128-row blocks of the
// same expert and shares each weight tile between them.
//
// Same computation as paged_gemm_kernel<true> (moe_gemm.cu): h = silu(x w1) *
// (x w3) with w1 and w3 read in place from their pool pages through the 3-D
// tensor map (page coordinate = page table entry).  The difference is the
// amount of operand traffic per MMA: a 64-deep k block stages rows
// row0 .. row0 + 255 of the sorted activations (two 16 KiB boxes) and one
// 32 KiB weight tile (128 columns of w1 and the same columns of w3), and
// issues the MMAs of both row blocks against that one weight tile: 64 KiB per
// two blocks of MMAs instead of 96 KiB.  Prefill at 8192 tokens is limited by
// operand delivery, not by the tensor pipe, so this is what moves it.
//
// Costs: the two 256-column accumulators fill all 512 TMEM columns, so the
// epilogue of a tile is not overlapped with the next tile's MMAs (the
// producer keeps loading meanwhile); stages are 64 KiB, so three fit.  An
// expert's last block runs alone when its block count is odd.
//
// Warps: 0 = TMA producer, 1 = TMEM owner + MMA issuer, 2-5 = epilogue of the
// first row block, 6-9 = epilogue of the second (warp w reads TMEM lanes
// 32 * (w % 4) of its accumulator).
#include "device.cuh"
#include "kernels.h"

namespace rimuru {
namespace {

using namespace dev;

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int BN = 256;                          // MMA N: 128 gate + 128 up columns
constexpr int kStages = 3;
constexpr int kABytes = BM * BK * 2;             // 16 KiB per row block
constexpr int kBChunk = BK * 64 * 2;             // 8 KiB: [64 k rows][64 cols]
constexpr int kBBytes = 4 * kBChunk;             // 32 KiB
constexpr int kStageBytes = 2 * kABytes + kBBytes;
constexpr int kThreads = 320;
constexpr int kTmemCols = 2 * BN;
constexpr int kSmemBytes = kStages * kStageBytes + 1024 /*align slack*/ + 256 /*barriers*/;

struct Shared {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t tfull;
  uint64_t tempty;
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

__global__ void __launch_bounds__(kThreads, 1)
    paired_gemm1_kernel(const __grid_constant__ CUtensorMap tm_x,
                        const __grid_constant__ CUtensorMap tm_w, const GemmArgs p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  Shared* sh = reinterpret_cast<Shared*>(smem + kStages * kStageBytes);
  volatile int* abort = &sh->abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sh->full[s], 1);
      mbar_init(&sh->empty[s], 1);
    }
    mbar_init(&sh->tfull, 1);
    mbar_init(&sh->tempty, 256);
    mbar_init(&sh->drain, 1);
    sh->abort = 0;
    fence_barrier_init();
    prefetch_tmap(&tm_x);
    prefetch_tmap(&tm_w);
  }
  if (warp == 1) {
    tmem_alloc(&sh->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = sh->tmem_base;

  grid_dep_wait();
  grid_dep_launch();
  const int n_tiles = *p.num_tiles * p.n_blocks;  // (pair of row blocks, column block)
  const int nkb = p.num_k_blocks;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer
      const uint64_t pol = policy_evict_last();
      uint32_t it = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < n_tiles; tile += gridDim.x) {
        const int pt = tile / p.n_blocks, nb = tile % p.n_blocks;
        const int e = p.tiles[2 * pt], row0 = p.tiles[2 * pt + 1];
        const bool pair = p.offsets[e + 1] - row0 > BM;
        int pg0 = p.page_table[3 * e + RIMURU_PROJ_W1];
        int pg1 = p.page_table[3 * e + RIMURU_PROJ_W3];
        const int n0 = nb * (BN / 2);
        if (pg0 < 0 || pg0 >= p.num_pages || pg1 < 0 || pg1 >= p.num_pages) {
          set_error(p.err, RIMURU_DEV_BAD_PAGE);  // host checks make this unreachable
          pg0 = pg1 = 0;
        }
        for (int kb = 0; kb < nkb; ++kb, ++it) {
          const uint32_t s = it % kStages, ph = (it / kStages) & 1u;
          if (!mbar_wait(&sh->empty[s], ph ^ 1u, abort)) {
            ok = false;
            break;
          }
          uint8_t* st = smem + s * kStageBytes;
          mbar_arrive_expect_tx(&sh->full[s], (pair ? 2 : 1) * kABytes + kBBytes);
          tma_load_2d(st, &tm_x, &sh->full[s], kb * BK, row0, pol);
          if (pair) tma_load_2d(st + kABytes, &tm_x, &sh->full[s], kb * BK, row0 + BM, pol);
          uint8_t* b = st + 2 * kABytes;
          tma_load_3d(b + 0 * kBChunk, &tm_w, &sh->full[s], n0, kb * BK, pg0, pol);
          tma_load_3d(b + 1 * kBChunk, &tm_w, &sh->full[s], n0 + 64, kb * BK, pg0, pol);
          tma_load_3d(b + 2 * kBChunk, &tm_w, &sh->full[s], n0, kb * BK, pg1, pol);
          tma_load_3d(b + 3 * kBChunk, &tm_w, &sh->full[s], n0 + 64, kb * BK, pg1, pol);
        }
      }
      if (!ok) {
        set_error(p.err, RIMURU_DEV_TIMEOUT);
        sh->abort = 1;
      }
      volatile int never = 0;  // every copy issued must land before the CTA exits
      const uint32_t first = it > static_cast<uint32_t>(kStages) ? it - kStages : 0u;
      for (uint32_t j = first; j < it; ++j)
        mbar_wait(&sh->full[j % kStages], (j / kStages) & 1u, &never);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------------ MMA issuer
      constexpr uint32_t idesc = idesc_bf16_f32(BM, BN, /*a_mn=*/false, /*b_mn=*/true);
      uint32_t it = 0, local = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < n_tiles; tile += gridDim.x, ++local) {
        const int pt = tile / p.n_blocks;
        const int e = p.tiles[2 * pt], row0 = p.tiles[2 * pt + 1];
        const bool pair = p.offsets[e + 1] - row0 > BM;
        if (!mbar_wait(&sh->tempty, (local & 1u) ^ 1u, abort)) {  // both accumulators free
          ok = false;
          break;
        }
        tc_fence_after();
        for (int kb = 0; kb < nkb; ++kb, ++it) {
          const uint32_t s = it % kStages, ph = (it / kStages) & 1u;
          if (!mbar_wait(&sh->full[s], ph, abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(smem + s * kStageBytes);
          const uint32_t b0 = a0 + 2 * kABytes;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint64_t bd = smem_desc_sw128(b0 + kk * 2048, kBChunk, 1024);
            const uint32_t accumulate = (kb | kk) != 0 ? 1u : 0u;
            umma_bf16(tmem_base, smem_desc_sw128(a0 + kk * 32, 16, 1024), bd, idesc, accumulate);
            if (pair)
              umma_bf16(tmem_base + BN, smem_desc_sw128(a0 + kABytes + kk * 32, 16, 1024), bd,
                        idesc, accumulate);
          }
          umma_commit(&sh->empty[s]);
        }
        if (!ok) break;
        umma_commit(&sh->tfull);
      }
      if (!ok) {
        set_error(p.err, RIMURU_DEV_TIMEOUT);
        sh->abort = 1;
      }
      umma_commit(&sh->drain);
      volatile int never = 0;
      mbar_wait(&sh->drain, 0, &never);
    }
  } else {
    // -------------------------------------------------------------- epilogue
    const int half = (warp - 2) >> 2;  // which row block / accumulator
    const int q = warp & 3;            // TMEM lane quadrant
    uint32_t local = 0;
    for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x, ++local) {
      const bool got = mbar_wait(&sh->tfull, local & 1u, abort);
      if (!__all_sync(0xffffffffu, got)) {
        if (lane == 0) {
          set_error(p.err, RIMURU_DEV_TIMEOUT);
          sh->abort = 1;
        }
        break;
      }
      tc_fence_after();
      const int pt = tile / p.n_blocks, nb = tile % p.n_blocks;
      const int e = p.tiles[2 * pt], row0 = p.tiles[2 * pt + 1];
      const int rows = min(2 * BM, p.offsets[e + 1] - row0);
      if (half * BM < rows) {  // the second accumulator holds nothing for a lone block
        const int r = half * BM + q * 32 + lane;
        const bool valid = r < rows;
        __nv_bfloat16* orow = p.out + static_cast<size_t>(row0 + r) * p.ldo;
        const uint32_t tb = tmem_base + half * BN + (static_cast<uint32_t>(q * 32) << 16);
        const int n0 = nb * (BN / 2);
#pragma unroll 1
        for (int c0 = 0; c0 < BN / 2; c0 += 32) {
          uint32_t g[32], u[32];
          tmem_ld32(tb + c0, g);
          tmem_ld32(tb + BN / 2 + c0, u);
          tmem_ld_wait();
          if (valid) {
            uint4* dst = reinterpret_cast<uint4*>(orow + n0 + c0);
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              uint32_t o[4];
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const int c = 8 * v + 2 * i;
                o[i] = pack_bf16x2(silu_mul(__uint_as_float(g[c]), __uint_as_float(u[c])),
                                   silu_mul(__uint_as_float(g[c + 1]), __uint_as_float(u[c + 1])));
              }
              dst[v] = make_uint4(o[0], o[1], o[2], o[3]);
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&sh->tempty);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

}  // namespace

cudaError_t launch_gemm1_swiglu_paired(const CUtensorMap& tm_x, const CUtensorMap& tm_w13,
                                       const GemmArgs& a, const LaunchOpts& o) {
  static bool configured = false;
  if (!configured) {
    cudaError_t st = cudaFuncSetAttribute(paired_gemm1_kernel,
                                          cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (st != cudaSuccess) return st;
    configured = true;
  }
  const long long tiles = static_cast<long long>(a.max_tiles) * a.n_blocks;
  const int grid = static_cast<int>(tiles < o.sm_count ? tiles : o.sm_count);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid > 0 ? grid : 1);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = o.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = o.pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, paired_gemm1_kernel, tm_x, tm_w13, a);
}

}  // namespace rimuru
