// GEMM 2 of the paged fused MoE layer for large batches, on CTA pairs
// (tcgen05 cta_group::2).
//
// The computation is that of paged_gemm_kernel<false> (moe_gemm.cu): y = h w2_e
// with w2_e read in place from its pool page through the 3-D tensor map over
// the pool (page coordinate = page-table entry; Rimuru, abstract and the
// explainer page's paragraph on the fused MoE kernel).
//
// What changes is the operand traffic per SM.  A cluster of two CTAs on two
// SMs computes one 256-row x 256-column tile with M = 256 MMAs: each CTA
// stages its own 128 rows of h and only 128 of the tile's 256 weight columns,
// and the pair's MMAs read the other half from the peer.  A 64-deep k block
// costs each SM 32 KiB of loads instead of 48 KiB for the same MMA work, which
// matters because large batches are limited by shared-memory traffic, not by
// the tensor pipe; the smaller stages also let six of them be in flight.  Each
// CTA's TMEM holds the 128 x 256 fp32 accumulator of its own rows,
// double-buffered, so the epilogue still overlaps the next tile's main loop.
// The epilogue stages 32 rows x 64 columns of y at a time in the 128-byte
// swizzle pattern and writes them with one TMA store (prefill GEMM 2
// 167.6 -> 165.7 us against per-lane stores); a block that holds rows of the
// next expert goes out row by row from the same staging instead.
//
// A tile is one entry of the pair table written by moe_align (two 128-row
// blocks of the same expert; an expert's odd last block is paired with the
// rows that follow it, which are computed and not stored) times one column
// block.  Rank r stages columns 128 r .. 128 r + 127 of the 256-column block.
//
// Synchronisation: the full barrier of a stage lives in the rank-0 CTA and
// counts both CTAs' bytes (each producer arms it for its own loads); the MMA
// completion is multicast to the empty barrier of both CTAs and to both
// accumulator-full barriers; the accumulator-empty barrier lives in the rank-0
// CTA and counts one arrival per epilogue warp of either CTA.  Every wait is
// bounded; a timeout raises the abort flag of both CTAs.
//
// Warps: 0 = TMA producer, 1 = TMEM allocation (both CTAs) and MMA issue
// (rank 0), 2-5 = epilogue (warp w reads TMEM lanes 32 * (w % 4)).
#include <atomic>

#include "device.cuh"
#include "kernels.h"

namespace rimuru {
namespace {

using namespace dev;

constexpr int BM = 128;                      // rows per CTA, 256 per pair
constexpr int BK = 64;
constexpr int BN = 256;                      // MMA N
constexpr int kStages = 6;
constexpr int kABytes = BM * BK * 2;         // 16 KiB
constexpr int kBChunk = BK * 64 * 2;         // 8 KiB: [64 k rows][64 cols] of one page
constexpr int kBBytes = 2 * kBChunk;         // 16 KiB: this CTA's 128 columns
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kThreads = 192;
constexpr int kTmemCols = 2 * BN;            // two accumulators
constexpr int kEpiWarps = 4;
constexpr int kStageOutBytes = 32 * 128;     // GEMM 2 epilogue staging per warp
constexpr int kSmemBytes = kStages * kStageBytes + kEpiWarps * kStageOutBytes +
                           1024 /*align slack*/ + 256 /*barriers*/;
static_assert(kSmemBytes <= 232448, "shared memory per block");

struct Shared {
  uint64_t full[kStages];   // rank 0's are used: both CTAs' bytes of a stage
  uint64_t empty[kStages];  // each CTA's own: its stage may be refilled
  uint64_t tfull[2];        // each CTA's own: accumulator ready
  uint64_t tempty[2];       // rank 0's are used: accumulator drained by both CTAs
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

// Raise the abort flag of both CTAs of the pair.
__device__ __forceinline__ void abort_pair(Shared* sh, int* err) {
  set_error(err, RIMURU_DEV_TIMEOUT);
  sh->abort = 1;
  st_cluster_u32(cluster_addr(&sh->abort, cluster_rank() ^ 1u), 1u);
}

__global__ void __launch_bounds__(kThreads, 1)
    pair_gemm2_kernel(const __grid_constant__ CUtensorMap tm_act,
                     const __grid_constant__ CUtensorMap tm_w,
                     const __grid_constant__ CUtensorMap tm_out, const GemmArgs p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + kStages * kABytes;
  uint8_t* sOut = smem + kStages * kStageBytes;
  Shared* sh = reinterpret_cast<Shared*>(sOut + kEpiWarps * kStageOutBytes);
  volatile int* abort = &sh->abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sh->full[s], 2);  // one armed arrival per CTA
      mbar_init(&sh->empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&sh->tfull[a], 1);
      mbar_init(&sh->tempty[a], 2 * kEpiWarps);
    }
    mbar_init(&sh->drain, 1);
    sh->abort = 0;
    fence_barrier_init();
    prefetch_tmap(&tm_act);
    prefetch_tmap(&tm_w);
    prefetch_tmap(&tm_out);
  }
  if (warp == 1) {
    tmem_alloc_pair(&sh->tmem_base, kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync();  // both CTAs' barriers exist before any remote arrival
  tc_fence_after();
  const uint32_t tmem_base = sh->tmem_base;

  grid_dep_wait();    // pair table, offsets and activations come from earlier kernels
  grid_dep_launch();  // the next kernel may be scheduled now; it waits for our completion
  const int n_units = *p.num_tiles * p.n_blocks;  // (pair of row blocks, column block)
  const int nkb = p.num_k_blocks;
  const int cid = static_cast<int>(cluster_id_x()), ncl = static_cast<int>(num_clusters_x());

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer
      const uint64_t pol_w = p.weights_evict_first ? policy_evict_first() : policy_evict_last();
      const uint64_t pol_a = policy_evict_last();
      uint32_t it = 0;
      bool ok = true;
      for (int u = cid; ok && u < n_units; u += ncl) {
        const int pt = u / p.n_blocks, nb = u % p.n_blocks;
        const int e = p.tiles[2 * pt];
        const int row0 = p.tiles[2 * pt + 1] + static_cast<int>(rank) * BM;
        int pg = p.page_table[3 * e + RIMURU_PROJ_W2];
        const int n0 = nb * BN + static_cast<int>(rank) * (BN / 2);
        if (pg < 0 || pg >= p.num_pages) {
          set_error(p.err, RIMURU_DEV_BAD_PAGE);  // host checks make this unreachable
          pg = 0;
        }
        for (int kb = 0; kb < nkb; ++kb, ++it) {
          const uint32_t s = it % kStages, ph = (it / kStages) & 1u;
          if (!mbar_wait_cluster(&sh->empty[s], ph ^ 1u, abort)) {
            ok = false;
            break;
          }
          const uint32_t full0 = cluster_addr(&sh->full[s], 0);
          mbar_arrive_expect_tx_cluster(full0, kStageBytes);
          tma_load_2d_pair(sA + s * kABytes, &tm_act, full0, kb * BK, row0, pol_a);
          uint8_t* b = sB + s * kBBytes;
          tma_load_3d_pair(b, &tm_w, full0, n0, kb * BK, pg, pol_w);
          tma_load_3d_pair(b + kBChunk, &tm_w, full0, n0 + 64, kb * BK, pg, pol_w);
        }
      }
      if (!ok) {
        abort_pair(sh, p.err);
        // copies already issued land within microseconds: let them before the CTA can leave
        const uint64_t t0 = globaltimer();
        while (globaltimer() - t0 < 100000ull) {
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      // ------------------------------------------------------------ MMA issuer
      constexpr uint32_t idesc = idesc_bf16_f32(2 * BM, BN, /*a_mn=*/false, /*b_mn=*/true);
      uint32_t it = 0, local = 0;
      bool ok = true;
      for (int u = cid; ok && u < n_units; u += ncl, ++local) {
        const uint32_t acc = local & 1u, aph = (local >> 1) & 1u;
        if (!mbar_wait_cluster(&sh->tempty[acc], aph ^ 1u, abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem_base + acc * BN;
        for (int kb = 0; kb < nkb; ++kb, ++it) {
          const uint32_t s = it % kStages, ph = (it / kStages) & 1u;
          if (!mbar_wait_cluster(&sh->full[s], ph, abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(sA + s * kABytes);
          const uint32_t b0 = smem_u32(sB + s * kBBytes);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            // A: K-major, 128-byte rows, 8-row groups 1024 B apart; +32 B per 16 k.
            const uint64_t ad = smem_desc_sw128(a0 + kk * 32, 16, 1024);
            // B: MN-major, this CTA's two 64-column chunks kBChunk apart (LBO),
            // 8-k-row groups 1024 B apart (SBO); +16 rows * 128 B per 16 k.
            const uint64_t bd = smem_desc_sw128(b0 + kk * 2048, kBChunk, 1024);
            umma_bf16_pair(d, ad, bd, idesc, (kb != 0 || kk != 0) ? 1u : 0u);
          }
          umma_commit_pair(&sh->empty[s], 0x3);  // stage s is free in both CTAs
        }
        if (!ok) break;
        umma_commit_pair(&sh->tfull[acc], 0x3);  // accumulator ready in both CTAs
      }
      if (!ok) abort_pair(sh, p.err);
      // every MMA must be finished before either CTA releases TMEM or exits
      umma_commit_pair(&sh->drain, 0x1);
      volatile int never = 0;
      mbar_wait(&sh->drain, 0, &never);
    }
  } else {
    // -------------------------------------------------------------- epilogue
    const int q = warp & 3;  // TMEM lane quadrant this warp may read
    const uint32_t tempty0[2] = {cluster_addr(&sh->tempty[0], 0), cluster_addr(&sh->tempty[1], 0)};
    uint32_t local = 0;
    for (int u = cid; u < n_units; u += ncl, ++local) {
      const uint32_t acc = local & 1u, aph = (local >> 1) & 1u;
      const bool got = mbar_wait_cluster(&sh->tfull[acc], aph, abort);
      if (!__all_sync(0xffffffffu, got)) {
        if (lane == 0) abort_pair(sh, p.err);
        break;
      }
      tc_fence_after();
      const int pt = u / p.n_blocks, nb = u % p.n_blocks;
      const int e = p.tiles[2 * pt];
      const int row0 = p.tiles[2 * pt + 1] + static_cast<int>(rank) * BM;
      const int rows = min(BM, p.offsets[e + 1] - row0);  // <= 0: rows of the next expert
      const uint32_t tb = tmem_base + acc * BN + (static_cast<uint32_t>(q * 32) << 16);
      {
        // Rows q*32 .. q*32+31 go out in blocks of 64 columns through a
        // row-swizzled staging block: one TMA store when all 32 rows are the
        // expert's, else four full 128-byte row segments per store instruction.
        const uint32_t blk_s = smem_u32(sOut + (warp - 2) * kStageOutBytes);
        const int n0 = nb * BN;
#pragma unroll 1
        for (int c0 = 0; c0 < BN; c0 += 64) {
          uint32_t a0[32], a1[32];
          tmem_ld32(tb + c0, a0);
          tmem_ld32(tb + c0 + 32, a1);
          tmem_ld_wait();
          uint32_t packed[32];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            packed[i] = pack_bf16x2(__uint_as_float(a0[2 * i]), __uint_as_float(a0[2 * i + 1]));
            packed[16 + i] =
                pack_bf16x2(__uint_as_float(a1[2 * i]), __uint_as_float(a1[2 * i + 1]));
          }
          if (lane == 0) bulk_wait_read_all();  // an earlier block's TMA store has read it
          __syncwarp();                         // and so have the lanes' loads
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
              tma_store_2d(&tm_out, blk_s, n0 + c0, row0 + q * 32);
              bulk_commit();
            }
            continue;
          }
          __syncwarp();
          const int chunk = lane & 7;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int rr = 4 * i + (lane >> 3);  // row within this warp's 32
            uint4 val;
            asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(val.x), "=r"(val.y), "=r"(val.z), "=r"(val.w)
                         : "r"(blk_s + rr * 128 + ((chunk ^ (rr & 7)) << 4))
                         : "memory");
            if (q * 32 + rr < rows)
              *reinterpret_cast<uint4*>(p.out + static_cast<size_t>(row0 + q * 32 + rr) * p.ldo +
                                        n0 + c0 + chunk * 8) = val;
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(tempty0[acc]);
    }
  }

  if (warp >= 2 && lane == 0) bulk_wait_all();  // y is complete when the grid is
  // No CTA leaves, or gives back TMEM, while its peer may still use its
  // barriers, its shared memory or the pair's accumulators.
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, kTmemCols);
  }
}

int max_pair_clusters(const LaunchOpts& o) {
  // per device (the kernel's occupancy depends on the GPU), looked up once
  constexpr int kMaxDevices = 64;
  static std::atomic<int> cached[kMaxDevices];  // 0 = not looked up yet
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return o.sm_count / 2;
  int n = cached[dev].load(std::memory_order_relaxed);
  if (n == 0) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * (o.sm_count / 2));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, pair_gemm2_kernel, &cfg) != cudaSuccess || n < 1) {
      cudaGetLastError();
      n = o.sm_count / 2;
    }
    cached[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

cudaError_t launch_pair(const CUtensorMap& tm_act, const CUtensorMap& tm_w,
                        const CUtensorMap& tm_out, const GemmArgs& a, const LaunchOpts& o) {
  // the shared-memory opt-in is a per-device function attribute: set it once per device
  static std::atomic<bool> configured[64];
  int dev = 0;
  cudaError_t st = cudaGetDevice(&dev);
  if (st != cudaSuccess) return st;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!configured[dev].load(std::memory_order_acquire)) {
    st = cudaFuncSetAttribute(pair_gemm2_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              kSmemBytes);
    if (st != cudaSuccess) return st;
    configured[dev].store(true, std::memory_order_release);
  }
  const long long tiles = static_cast<long long>(a.max_tiles) * a.n_blocks;
  const int clusters_cap = max_pair_clusters(o);
  const int clusters = static_cast<int>(tiles < clusters_cap ? tiles : clusters_cap);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * (clusters > 0 ? clusters : 1));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = o.stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = o.pdl ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, pair_gemm2_kernel, tm_act, tm_w, tm_out, a);
}

}  // namespace

cudaError_t launch_gemm2_pair(const CUtensorMap& tm_h, const CUtensorMap& tm_w2,
                              const CUtensorMap& tm_y, const GemmArgs& a, const LaunchOpts& o) {
  return launch_pair(tm_h, tm_w2, tm_y, a, o);
}

}  // namespace rimuru
