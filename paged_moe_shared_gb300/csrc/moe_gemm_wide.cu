// GEMM 1 + SwiGLU of the paged fused MoE layer for large batches, with
// 256-row tiles on one SM.
//
// The computation is that of paged_gemm_kernel<true, true> (moe_gemm.cu):
// h = silu(x_e w1_e) * (x_e w3_e), the A rows gathered from x with cp.async
// through `sorted`, w1 and w3 read in place from their pool pages through the
// 3-D tensor map over the pool (Rimuru, arXiv 2610.40305: abstract and the
// explainer page's paragraph on the fused MoE kernel).
//
// What changes is the tile: 256 rows x 256 MMA columns, computed as two
// M = 128 MMAs per 16-deep k step that read the same staged weight block.  A
// 64-deep k block then costs the SM 32 KiB of A and 32 KiB of weights for
// 2 x 128 x 256 x 64 multiply-adds, against 16 + 32 KiB for half of that work
// with 128-row tiles: a third fewer bytes into shared memory per MMA, and the
// bytes per SM are what bounds the 128-row kernel at large batches.  The two
// 128 x 256 fp32 accumulators fill all 512 TMEM columns, so there is no second
// accumulator for the epilogue of one tile to overlap the next tile's main
// loop; eight epilogue warps drain it, half 0 first, and the MMA issuer
// starts the next tile's half 0 as soon as that half is drained.
//
// A tile is one entry of the pair table written by moe_align (two 128-row
// blocks of one expert; an expert's odd last block alone, in which case the
// loads, MMAs and epilogue of half 1 are skipped) times one block of 128
// output columns (gate from the w1 page, up from the w3 page).
//
// Warps: 0 = weight TMA producer, 1 = TMEM owner + MMA issuer, 2-9 = epilogue
// (warp w reads TMEM lanes 32 (w % 4) .. 32 (w % 4) + 31 and output columns
// 64 ((w - 2) / 4) .. + 63 of the block), 10-13 = A loaders (warp 10 + i copies
// rows 64 i .. 64 i + 63 of each stage).
#include <atomic>

#include "device.cuh"
#include "kernels.h"

namespace rimuru {
namespace {

using namespace dev;

constexpr int BM = 128;                      // rows per accumulator half
constexpr int BK = 64;
constexpr int BN = 256;                      // MMA N: 128 gate + 128 up columns
constexpr int kStages = 3;
constexpr int kAHalfBytes = BM * BK * 2;     // 16 KiB
constexpr int kABytes = 2 * kAHalfBytes;     // 32 KiB: 256 rows
constexpr int kBChunk = BK * 64 * 2;         // 8 KiB: [64 k rows][64 cols] of one page
constexpr int kBBytes = 4 * kBChunk;         // 32 KiB
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kEpiWarps = 8;
constexpr int kLoaderWarps = 4;
constexpr int kFirstLoader = 2 + kEpiWarps;
constexpr int kThreads = 32 * (kFirstLoader + kLoaderWarps);  // 448
constexpr int kTmemCols = 2 * BN;            // the two halves' accumulators
// Epilogue staging: per epilogue warp one 32-row x 128-byte block of h, 16-byte
// chunks XOR-swizzled by row, so each store instruction writes four whole rows.
constexpr int kStageOutBytes = 32 * 128;
constexpr int kSmemBytes = kStages * kStageBytes + kEpiWarps * kStageOutBytes +
                           1024 /*align slack*/ + 256 /*barriers*/;
static_assert(kSmemBytes <= 232448, "shared memory per block");
static_assert(kThreads * 128 <= 65536, "registers: 128 per thread fit one SM");

// Dynamic unit scheduling: the producer takes each next unit from a global
// counter (units differ in cost: an expert's lone last block is half a tile)
// and publishes it in a small ring read by every other role in the same order.
constexpr int kSched = 4;
constexpr int kSchedReaders = 1 + kEpiWarps + kLoaderWarps;  // MMA thread + one per warp

struct Shared {
  uint64_t full[kStages];   // weight bytes + one arrival per loader thread
  uint64_t empty[kStages];  // the stage's MMAs are done
  uint64_t tfull;           // both accumulator halves hold the tile
  uint64_t tempty[2];       // half h drained by the eight epilogue warps
  uint64_t drain;
  uint64_t sfull[kSched];   // unit index published
  uint64_t sempty[kSched];  // every role has read it
  int sunit[kSched];
  uint32_t tmem_base;
  int abort;
};

__device__ __forceinline__ void fail(Shared* sh, int* err) {
  set_error(err, RIMURU_DEV_TIMEOUT);
  sh->abort = 1;
}

__global__ void __launch_bounds__(kThreads, 1)
    wide_gemm1_kernel(const __grid_constant__ CUtensorMap tm_w,
                      const __grid_constant__ CUtensorMap tm_out, const GemmArgs p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;                        // [stage][256 rows][128 B], 128-byte swizzle
  uint8_t* sB = smem + kStages * kABytes;    // [stage][4 chunks][64 k rows][128 B]
  uint8_t* sOut = smem + kStages * kStageBytes;  // [epilogue warp][32 rows][128 B]
  Shared* sh = reinterpret_cast<Shared*>(sOut + kEpiWarps * kStageOutBytes);
  volatile int* abort = &sh->abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sh->full[s], 1 + 32 * kLoaderWarps);
      mbar_init(&sh->empty[s], 1);
    }
    mbar_init(&sh->tfull, 1);
    mbar_init(&sh->tempty[0], kEpiWarps);
    mbar_init(&sh->tempty[1], kEpiWarps);
    mbar_init(&sh->drain, 1);
    for (int i = 0; i < kSched; ++i) {
      mbar_init(&sh->sfull[i], 1);
      mbar_init(&sh->sempty[i], kSchedReaders);
    }
    sh->abort = 0;
    fence_barrier_init();
    prefetch_tmap(&tm_w);
    prefetch_tmap(&tm_out);
  }
  if (warp == 1) {
    tmem_alloc(&sh->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = sh->tmem_base;

  grid_dep_wait();    // pair table, offsets and sorted come from earlier kernels
  grid_dep_launch();  // the next kernel may be scheduled now; it waits for our completion
  const int n_units = *p.num_tiles * p.n_blocks;  // (pair of row blocks, column block)
  const int nkb = p.num_k_blocks;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer
      const uint64_t pol_w = p.weights_evict_first ? policy_evict_first() : policy_evict_last();
      uint32_t it = 0;
      bool ok = true;
      int u = blockIdx.x;
      for (int i = 0; ok; ++i) {
        // publish unit u as this CTA's i-th (u >= n_units ends every role's loop)
        const uint32_t sl = i % kSched, sph = (i / kSched) & 1u;
        if (!mbar_wait(&sh->sempty[sl], sph ^ 1u, abort)) {
          ok = false;
          break;
        }
        sh->sunit[sl] = u;
        mbar_arrive(&sh->sfull[sl]);
        if (u >= n_units) break;
        // the next unit, fetched while this one's copies are issued
        const int next = static_cast<int>(gridDim.x) + atomicAdd(p.sched, 1);
        const int pt = u / p.n_blocks, nb = u % p.n_blocks;
        const int e = p.tiles[2 * pt];
        int pg0 = p.page_table[3 * e + RIMURU_PROJ_W1];
        int pg1 = p.page_table[3 * e + RIMURU_PROJ_W3];
        if (pg0 < 0 || pg0 >= p.num_pages || pg1 < 0 || pg1 >= p.num_pages) {
          set_error(p.err, RIMURU_DEV_BAD_PAGE);  // host checks make this unreachable
          pg0 = pg1 = 0;
        }
        const int n0 = nb * (BN / 2);
        for (int kb = 0; kb < nkb; ++kb, ++it) {
          const uint32_t s = it % kStages, ph = (it / kStages) & 1u;
          if (!mbar_wait(&sh->empty[s], ph ^ 1u, abort)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&sh->full[s], kBBytes);
          uint8_t* b = sB + s * kBBytes;
          tma_load_3d(b + 0 * kBChunk, &tm_w, &sh->full[s], n0, kb * BK, pg0, pol_w);
          tma_load_3d(b + 1 * kBChunk, &tm_w, &sh->full[s], n0 + 64, kb * BK, pg0, pol_w);
          tma_load_3d(b + 2 * kBChunk, &tm_w, &sh->full[s], n0, kb * BK, pg1, pol_w);
          tma_load_3d(b + 3 * kBChunk, &tm_w, &sh->full[s], n0 + 64, kb * BK, pg1, pol_w);
        }
        u = next;
      }
      if (!ok) fail(sh, p.err);
      // every copy this thread issued must have landed before the CTA exits
      volatile int never = 0;
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
      for (;; ++local) {
        const uint32_t sl = local % kSched, sph = (local / kSched) & 1u;
        if (!mbar_wait(&sh->sfull[sl], sph, abort)) {
          ok = false;
          break;
        }
        const int u = sh->sunit[sl];
        mbar_arrive(&sh->sempty[sl]);
        if (u >= n_units) break;
        const int pt = u / p.n_blocks;
        const int e = p.tiles[2 * pt], row0 = p.tiles[2 * pt + 1];
        const bool has1 = p.offsets[e + 1] - row0 > BM;
        // Accumulator half h is free once the epilogue drained it for the
        // previous tile (phase local - 1 of tempty[h]).  The epilogue drains
        // half 0 before half 1 and every warp arrives on tempty[1] of a tile
        // before tempty[0] of the next, so half 1's barrier is never more
        // than one phase behind the tile being issued.
        const uint32_t par = (local & 1u) ^ 1u;
        if (!mbar_wait(&sh->tempty[0], par, abort)) {
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
          // A arrived through cp.async (generic proxy); the MMA reads it
          // through the async proxy
          fence_proxy_async_smem();
          const uint32_t a0 = smem_u32(sA + s * kABytes);
          const uint32_t b0 = smem_u32(sB + s * kBBytes);
          // A: K-major, 128-byte rows, 8-row groups 1024 B apart; +32 B per 16 k.
          // B: MN-major, 64-column chunks kBChunk apart (LBO), 8-k-row groups
          // 1024 B apart (SBO); +16 rows * 128 B per 16 k.
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            umma_bf16(tmem_base, smem_desc_sw128(a0 + kk * 32, 16, 1024),
                      smem_desc_sw128(b0 + kk * 2048, kBChunk, 1024), idesc,
                      (kb != 0 || kk != 0) ? 1u : 0u);
          if (has1) {
            // half 1 of the previous tile may still be draining: half 0's
            // first MMAs are already queued while this thread waits for it
            if (kb == 0) {
              if (!mbar_wait(&sh->tempty[1], par, abort)) {
                ok = false;
                break;
              }
              tc_fence_after();
            }
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk)
              umma_bf16(tmem_base + BN, smem_desc_sw128(a0 + kAHalfBytes + kk * 32, 16, 1024),
                        smem_desc_sw128(b0 + kk * 2048, kBChunk, 1024), idesc,
                        (kb != 0 || kk != 0) ? 1u : 0u);
          }
          umma_commit(&sh->empty[s]);  // stage s is free once these MMAs are done
        }
        if (!ok) break;
        umma_commit(&sh->tfull);  // both halves ready for the epilogue
      }
      if (!ok) fail(sh, p.err);
      // all MMAs must be finished before TMEM is released
      umma_commit(&sh->drain);
      volatile int never = 0;
      mbar_wait(&sh->drain, 0, &never);
    }
  } else if (warp >= kFirstLoader) {
    // ----------------------------------------------------------- A loaders
    // Row r of a tile is token sorted[row0 + r] / top_k; eight lanes cover one
    // row's 128 bytes, each 16-byte chunk c of row r written at chunk
    // c ^ (r % 8) as the 128-byte swizzle of the MMA descriptor expects.  Rows
    // past the expert repeat its last row (never stored); the rows of an absent
    // half are not loaded.  Each thread's arrival on the stage's full barrier
    // fires when its copies have landed.
    const int lw = warp - kFirstLoader, half = lw >> 1;
    const int sub = lane >> 3, chunk = lane & 7;
    uint32_t it = 0;
    bool ok = true;
    for (uint32_t i = 0; ok; ++i) {
      const uint32_t sl = i % kSched, sph = (i / kSched) & 1u;
      if (!__all_sync(0xffffffffu, mbar_wait(&sh->sfull[sl], sph, abort))) {
        ok = false;
        break;
      }
      const int u = sh->sunit[sl];
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh->sempty[sl]);
      if (u >= n_units) break;
      const int pt = u / p.n_blocks;
      const int e = p.tiles[2 * pt];
      const int hrow0 = p.tiles[2 * pt + 1] + half * BM;  // first row of this warp's half
      const int rows = min(BM, p.offsets[e + 1] - hrow0);  // <= 0: half 1 absent
      const __nv_bfloat16* src[16];
      if (rows > 0) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int r = min(64 * (lw & 1) + 4 * i + sub, rows - 1);
          src[i] = p.x + static_cast<size_t>(p.sorted[hrow0 + r] / p.top_k) * p.ldx + chunk * 8;
        }
      }
      // x (T x H, a few tens of MB) is gathered k times per column block: the
      // row copies carry the same L2 evict-last priority as the weight boxes
      // (prefill GEMM 1 317 -> 311 us; its DRAM traffic did not change).
      const uint64_t pol_x = policy_evict_last();
      for (int kb = 0; kb < nkb; ++kb, ++it) {
        const uint32_t s = it % kStages, ph = (it / kStages) & 1u;
        bool got = true;
        if (lane == 0) got = mbar_wait(&sh->empty[s], ph ^ 1u, abort);
        if (!__shfl_sync(0xffffffffu, got, 0)) {
          ok = false;
          break;
        }
        if (rows > 0) {
          const uint32_t a_s = smem_u32(sA + s * kABytes);
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int r = 64 * lw + 4 * i + sub;  // 0..255
            cp_async16_hint(a_s + r * 128 + ((chunk ^ (r & 7)) << 4), src[i] + kb * BK, pol_x);
          }
        }
        cp_async_arrive_noinc(&sh->full[s]);
      }
    }
    if (!ok && lane == 0) fail(sh, p.err);
    cp_async_wait_all();  // no copy of this thread is in flight when the CTA exits
  } else {
    // -------------------------------------------------------------- epilogue
    // Each warp turns its 32 rows x 64 columns of h into bf16 in registers,
    // releases the accumulator half (the next tile's MMAs may start on it),
    // then writes the rows out through its staging block.
    const int q = warp & 3;                  // TMEM lane quadrant this warp may read
    const int cb = 64 * ((warp - 2) >> 2);   // this warp's first output column of the block
    const uint32_t blk_s = smem_u32(sOut + (warp - 2) * kStageOutBytes);
    for (uint32_t local = 0;; ++local) {
      const uint32_t sl = local % kSched, sph = (local / kSched) & 1u;
      if (!__all_sync(0xffffffffu, mbar_wait(&sh->sfull[sl], sph, abort))) {
        if (lane == 0) fail(sh, p.err);
        break;
      }
      const int u = sh->sunit[sl];
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh->sempty[sl]);
      if (u >= n_units) break;
      const bool got = mbar_wait(&sh->tfull, local & 1u, abort);
      if (!__all_sync(0xffffffffu, got)) {
        if (lane == 0) fail(sh, p.err);
        break;
      }
      tc_fence_after();
      const int pt = u / p.n_blocks, nb = u % p.n_blocks;
      const int e = p.tiles[2 * pt], row0 = p.tiles[2 * pt + 1];
      const int rem = p.offsets[e + 1] - row0;
      const int n0 = nb * (BN / 2) + cb;
#pragma unroll 1
      for (int h = 0; h < 2; ++h) {
        const int rows = min(BM, rem - h * BM);  // warp-uniform
        uint32_t packed[32];
        if (rows > 0) {
          const uint32_t tb = tmem_base + h * BN + (static_cast<uint32_t>(q * 32) << 16) + cb;
#pragma unroll
          for (int c0 = 0; c0 < 64; c0 += 32) {
            uint32_t g[32], v[32];
            tmem_ld32(tb + c0, g);
            tmem_ld32(tb + BN / 2 + c0, v);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; ++i)
              packed[c0 / 2 + i] =
                  pack_bf16x2(silu_mul(__uint_as_float(g[2 * i]), __uint_as_float(v[2 * i])),
                              silu_mul(__uint_as_float(g[2 * i + 1]), __uint_as_float(v[2 * i + 1])));
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh->tempty[h]);
        if (rows > 0) {
          // lane l holds row q*32 + l: stage it, then one TMA store of the block, or,
          // when it holds rows of the next expert, four whole rows per store instruction
          if (lane == 0) bulk_wait_read_all();  // an earlier block's TMA store has read it
          __syncwarp();
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const uint32_t at = blk_s + lane * 128 + ((c ^ (lane & 7)) << 4);
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(at), "r"(packed[4 * c]),
                         "r"(packed[4 * c + 1]), "r"(packed[4 * c + 2]), "r"(packed[4 * c + 3])
                         : "memory");
          }
          if (rows - q * 32 >= 32) {
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&tm_out, blk_s, n0, row0 + h * BM + q * 32);
              bulk_commit();
            }
            continue;
          }
          __syncwarp();
          const int chunk = lane & 7;
#pragma unroll 1  // blocks with rows of the next expert only; unrolled, the kernel spills
          for (int i = 0; i < 8; ++i) {
            const int rr = 4 * i + (lane >> 3);  // row within this warp's 32
            uint4 val;
            asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(val.x), "=r"(val.y), "=r"(val.z), "=r"(val.w)
                         : "r"(blk_s + rr * 128 + ((chunk ^ (rr & 7)) << 4))
                         : "memory");
            if (q * 32 + rr < rows)
              *reinterpret_cast<uint4*>(p.out + static_cast<size_t>(row0 + h * BM + q * 32 + rr) *
                                                    p.ldo +
                                        n0 + chunk * 8) = val;
          }
          __syncwarp();  // the staging block is read out before the next half reuses it
        }
      }
    }
  }

  if (warp >= 2 && warp < 2 + kEpiWarps && lane == 0) bulk_wait_all();  // h is complete
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

}  // namespace

cudaError_t launch_gemm1_wide(const CUtensorMap& tm_w13, const CUtensorMap& tm_h,
                              const GemmArgs& a, const LaunchOpts& o) {
  // the shared-memory opt-in is a per-device function attribute: set it once per device
  static std::atomic<bool> configured[64];
  int dev = 0;
  cudaError_t st = cudaGetDevice(&dev);
  if (st != cudaSuccess) return st;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!configured[dev].load(std::memory_order_acquire)) {
    st = cudaFuncSetAttribute(wide_gemm1_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              kSmemBytes);
    if (st != cudaSuccess) return st;
    configured[dev].store(true, std::memory_order_release);
  }
  const long long units = static_cast<long long>(a.max_tiles) * a.n_blocks;
  const int grid = static_cast<int>(units < o.sm_count ? units : o.sm_count);
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
  return cudaLaunchKernelEx(&cfg, wide_gemm1_kernel, tm_w13, tm_h, a);
}

}  // namespace rimuru
