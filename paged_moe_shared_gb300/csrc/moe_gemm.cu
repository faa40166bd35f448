// Paged grouped GEMMs of the fused MoE layer on sm_103a tensor cores.
//
// Rimuru (arXiv 2610.40305), abstract and the explainer page's paragraph on
// the fused MoE kernel: the MoE kernel reads each expert's weights from the
// scattered pages of the pool directly, instead of first copying them into a
// contiguous buffer as an ordinary fused MoE kernel would need.
//
// Here that becomes: the expert view is one 3-D TMA tensor map over the whole
// pool, [pages][rows][cols] with the page stride equal to the view's page
// size, so resolving the expert's page through the page table means setting
// the third TMA coordinate to page_table[expert][proj].  No descriptor is
// rewritten per expert and no weight byte is copied anywhere but into shared
// memory.
//
// Tile: 128 assignment rows x 256 MMA columns x 64-deep k blocks.
//   GEMM 1: columns 0..127 come from the w1 page, 128..255 from the w3 page
//           (same 128 output columns), so gate and up accumulate side by side
//           in TMEM and the epilogue writes h = silu(gate) * up in bf16.
//   GEMM 2: 256 consecutive columns of the w2 page; the epilogue writes y.
// A (activations, K-major) and B (weights, MN-major: rows of the page are k)
// are staged by TMA with 128-byte swizzle into a 4-deep ring; one thread
// issues tcgen05.mma into a double-buffered TMEM accumulator (2 x 256
// columns) so the epilogue of one tile overlaps the main loop of the next.
// Warp roles: warp 0 = TMA producer, warp 1 = TMEM owner + MMA issuer,
// warps 2-5 = epilogue (warp w reads TMEM lanes 32 * (w % 4) ..).
// GEMM 1 past the small-batch size (kGatherA) has no x_sorted to read: warps
// 6-9 copy each A stage's rows straight from x with cp.async, the producer
// loads only the weight boxes, and the stage's full barrier also counts the
// 128 loader threads.
#include <atomic>

#include "device.cuh"
#include "kernels.h"

namespace rimuru {
namespace {

using namespace dev;

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int BN = 256;                      // MMA N
constexpr int kStages = 4;
constexpr int kABytes = BM * BK * 2;         // 16 KiB
constexpr int kBChunk = BK * 64 * 2;         // 8 KiB: [64 k rows][64 cols] of one page
constexpr int kBBytes = 4 * kBChunk;         // 32 KiB
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kThreads = 192;
// GEMM 1 with its A rows gathered from x by four more warps (cp.async): 320.
constexpr int kLoaderWarps = 4;
constexpr int kThreadsGather = kThreads + 32 * kLoaderWarps;
constexpr int kTmemCols = 2 * BN;            // two accumulators
// Epilogue staging: per epilogue warp one 32-row x 64-column bf16 block (4 KiB),
// 128-byte rows with 16-byte chunks XOR-swizzled by row so that both the
// row-per-lane writes and the row-segment reads are free of bank conflicts.
constexpr int kStageOutBytes = 32 * 128;
constexpr int kSmemBytes = kStages * kStageBytes + 4 * kStageOutBytes + 1024 /*align slack*/ +
                           256 /*barriers*/;

struct Shared {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  int last;  // split-K: this CTA finished the last split of the current tile
};

template <bool kSwiGLU, bool kGatherA>
__global__ void __launch_bounds__(kGatherA ? kThreadsGather : kThreads, 1)
    paged_gemm_kernel(const __grid_constant__ CUtensorMap tm_act,
                      const __grid_constant__ CUtensorMap tm_w, const GemmArgs p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + kStages * kABytes;
  uint8_t* sOut = smem + kStages * kStageBytes;  // 4 epilogue blocks
  Shared* sh = reinterpret_cast<Shared*>(sOut + 4 * kStageOutBytes);
  volatile int* abort = &sh->abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      // the producer's armed arrival, plus one per loader thread when A is gathered
      mbar_init(&sh->full[s], kGatherA ? 1 + 32 * kLoaderWarps : 1);
      mbar_init(&sh->empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&sh->tfull[a], 1);
      mbar_init(&sh->tempty[a], 128);
    }
    mbar_init(&sh->drain, 1);
    sh->abort = 0;
    fence_barrier_init();
    if (!kGatherA) prefetch_tmap(&tm_act);
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

  if (threadIdx.x == 0 && p.prefetch_kb > 0) {
    // Weights do not depend on the kernel we follow (only which experts are
    // used does): start streaming the guessed first tile's weights into L2
    // while that kernel still runs.  A wrong guess costs bandwidth only.
    const int S = p.splits, nkb = p.num_k_blocks;
    const int tile = blockIdx.x / S, split = blockIdx.x - tile * S;
    const int mb = tile / p.n_blocks, nb = tile % p.n_blocks;
    // prefetch_bpe = 0: the tile table was written by a kernel that finished
    // before the one we follow started, so read it (at L2: no stale L1 line)
    const int e = p.prefetch_bpe > 0 ? mb / p.prefetch_bpe
                                     : (mb < __ldcg(p.num_tiles) ? __ldcg(p.tiles + 2 * mb)
                                                                : p.num_experts);
    const int kb0 = split * nkb / S;
    const int kb1 = min(kb0 + p.prefetch_kb, (split + 1) * nkb / S);
    if (e < p.num_experts) {
      const int pg0 = p.page_table[3 * e + (kSwiGLU ? RIMURU_PROJ_W1 : RIMURU_PROJ_W2)];
      const int pg1 = kSwiGLU ? p.page_table[3 * e + RIMURU_PROJ_W3] : pg0;
      if (pg0 >= 0 && pg0 < p.num_pages && pg1 >= 0 && pg1 < p.num_pages) {
        for (int kb = kb0; kb < kb1; ++kb) {
          if (kSwiGLU) {
            const int n0 = nb * (BN / 2);
            tma_prefetch_3d(&tm_w, n0, kb * BK, pg0);
            tma_prefetch_3d(&tm_w, n0 + 64, kb * BK, pg0);
            tma_prefetch_3d(&tm_w, n0, kb * BK, pg1);
            tma_prefetch_3d(&tm_w, n0 + 64, kb * BK, pg1);
          } else {
#pragma unroll
            for (int c = 0; c < 4; ++c) tma_prefetch_3d(&tm_w, nb * BN + 64 * c, kb * BK, pg0);
          }
        }
      }
    }
  }

  grid_dep_wait();  // tile table, offsets and activations come from earlier kernels
  grid_dep_launch();  // the next kernel may be scheduled now; it waits for our completion
  const int S = p.splits;
  const int n_units = *p.num_tiles * p.n_blocks * S;  // (tile, split) work units
  const int nkb = p.num_k_blocks;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer
      const uint64_t pol_w = p.weights_evict_first ? policy_evict_first() : policy_evict_last();
      const uint64_t pol_a = policy_evict_last();
      uint32_t it = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < n_units; u += gridDim.x) {
        const int tile = u / S, split = u - tile * S;
        const int kb0 = split * nkb / S, kb1 = (split + 1) * nkb / S;
        const int mb = tile / p.n_blocks, nb = tile % p.n_blocks;
        const int e = p.tiles[2 * mb], row0 = p.tiles[2 * mb + 1];
        int pg0, pg1, n0;
        if (kSwiGLU) {
          pg0 = p.page_table[3 * e + RIMURU_PROJ_W1];
          pg1 = p.page_table[3 * e + RIMURU_PROJ_W3];
          n0 = nb * (BN / 2);
        } else {
          pg0 = pg1 = p.page_table[3 * e + RIMURU_PROJ_W2];
          n0 = nb * BN;
        }
        if (pg0 < 0 || pg0 >= p.num_pages || pg1 < 0 || pg1 >= p.num_pages) {
          set_error(p.err, RIMURU_DEV_BAD_PAGE);  // host checks make this unreachable
          pg0 = pg1 = 0;
        }
        for (int kb = kb0; kb < kb1; ++kb, ++it) {
          const uint32_t s = it % kStages, ph = (it / kStages) & 1u;
          if (!mbar_wait(&sh->empty[s], ph ^ 1u, abort)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&sh->full[s], kGatherA ? kBBytes : kStageBytes);
          if (!kGatherA) tma_load_2d(sA + s * kABytes, &tm_act, &sh->full[s], kb * BK, row0, pol_a);
          uint8_t* b = sB + s * kBBytes;
          if (kSwiGLU) {
            tma_load_3d(b + 0 * kBChunk, &tm_w, &sh->full[s], n0, kb * BK, pg0, pol_w);
            tma_load_3d(b + 1 * kBChunk, &tm_w, &sh->full[s], n0 + 64, kb * BK, pg0, pol_w);
            tma_load_3d(b + 2 * kBChunk, &tm_w, &sh->full[s], n0, kb * BK, pg1, pol_w);
            tma_load_3d(b + 3 * kBChunk, &tm_w, &sh->full[s], n0 + 64, kb * BK, pg1, pol_w);
          } else {
#pragma unroll
            for (int c = 0; c < 4; ++c)
              tma_load_3d(b + c * kBChunk, &tm_w, &sh->full[s], n0 + 64 * c, kb * BK, pg0, pol_w);
          }
        }
      }
      if (!ok) {
        set_error(p.err, RIMURU_DEV_TIMEOUT);
        sh->abort = 1;
      }
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
      for (int u = blockIdx.x; ok && u < n_units; u += gridDim.x, ++local) {
        const int split = u % S;
        const int kb0 = split * nkb / S, kb1 = (split + 1) * nkb / S;
        const uint32_t acc = local & 1u, aph = (local >> 1) & 1u;
        if (!mbar_wait(&sh->tempty[acc], aph ^ 1u, abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem_base + acc * BN;
        for (int kb = kb0; kb < kb1; ++kb, ++it) {
          const uint32_t s = it % kStages, ph = (it / kStages) & 1u;
          if (!mbar_wait(&sh->full[s], ph, abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
          // A arrived through cp.async (generic proxy); the MMA reads it
          // through the async proxy
          if (kGatherA) fence_proxy_async_smem();
          const uint32_t a0 = smem_u32(sA + s * kABytes);
          const uint32_t b0 = smem_u32(sB + s * kBBytes);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            // A: K-major, 128-byte rows, 8-row groups 1024 B apart; +32 B per 16 k.
            const uint64_t ad = smem_desc_sw128(a0 + kk * 32, 16, 1024);
            // B: MN-major, 64-column chunks kBChunk apart (LBO), 8-k-row groups
            // 1024 B apart (SBO); +16 rows * 128 B per 16 k.
            const uint64_t bd = smem_desc_sw128(b0 + kk * 2048, kBChunk, 1024);
            umma_bf16(d, ad, bd, idesc, (kb != kb0 || kk != 0) ? 1u : 0u);
          }
          umma_commit(&sh->empty[s]);  // stage s is free once these MMAs are done
        }
        if (!ok) break;
        umma_commit(&sh->tfull[acc]);  // accumulator ready for the epilogue
      }
      if (!ok) {
        set_error(p.err, RIMURU_DEV_TIMEOUT);
        sh->abort = 1;
      }
      // all MMAs must be finished before TMEM is released
      umma_commit(&sh->drain);
      volatile int never = 0;
      mbar_wait(&sh->drain, 0, &never);
    }
  } else if (kGatherA && warp >= 6) {
    // ----------------------------------------------------------- A loaders
    // Warp 6 + w copies rows 32 w .. 32 w + 31 of each A stage straight from x:
    // row r of the tile is token sorted[row0 + r] / top_k.  Eight lanes cover
    // one row's 128 bytes, written at the 128-byte-swizzled position the MMA
    // descriptor expects (16-byte chunk c of row r at chunk c ^ (r % 8)).
    // Rows past the tile's expert repeat its last row (their results are not
    // stored).  Each thread's arrival on the stage's full barrier fires when
    // its copies have landed.
    const int lw = warp - 6, sub = lane >> 3, chunk = lane & 7;
    uint32_t it = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < n_units; u += gridDim.x) {
      const int tile = u / S, split = u - tile * S;
      const int kb0 = split * nkb / S, kb1 = (split + 1) * nkb / S;
      const int mb = tile / p.n_blocks;
      const int e = p.tiles[2 * mb], row0 = p.tiles[2 * mb + 1];
      const int rows = min(BM, p.offsets[e + 1] - row0);  // >= 1 for a listed tile
      const __nv_bfloat16* src[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int r = min(32 * lw + 4 * i + sub, rows - 1);
        src[i] = p.x + static_cast<size_t>(p.sorted[row0 + r] / p.top_k) * p.ldx + chunk * 8;
      }
      for (int kb = kb0; kb < kb1; ++kb, ++it) {
        const uint32_t s = it % kStages, ph = (it / kStages) & 1u;
        bool got = true;
        if (lane == 0) got = mbar_wait(&sh->empty[s], ph ^ 1u, abort);
        if (!__shfl_sync(0xffffffffu, got, 0)) {
          ok = false;
          break;
        }
        const uint32_t a_s = smem_u32(sA + s * kABytes);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int r = 32 * lw + 4 * i + sub;
          cp_async16(a_s + r * 128 + ((chunk ^ (r & 7)) << 4), src[i] + kb * BK);
        }
        cp_async_arrive_noinc(&sh->full[s]);
      }
    }
    if (!ok && lane == 0) {
      set_error(p.err, RIMURU_DEV_TIMEOUT);
      sh->abort = 1;
    }
    cp_async_wait_all();  // no copy of this thread is in flight when the CTA exits
  } else {
    // -------------------------------------------------------------- epilogue
    const int q = warp & 3;  // TMEM lane quadrant this warp may read
    uint32_t local = 0;
    const int et = (warp - 2) * 32 + lane;  // 0..127 across the epilogue warps
    for (int u = blockIdx.x; u < n_units; u += gridDim.x, ++local) {
      const int tile = u / S;
      const uint32_t acc = local & 1u, aph = (local >> 1) & 1u;
      bool got = mbar_wait(&sh->tfull[acc], aph, abort);
      if (S > 1) got = named_bar_and(got);  // the split path syncs the four warps: decide together
      if (!__all_sync(0xffffffffu, got)) {
        if (lane == 0) {
          set_error(p.err, RIMURU_DEV_TIMEOUT);
          sh->abort = 1;
        }
        break;
      }
      tc_fence_after();
      const int mb = tile / p.n_blocks, nb = tile % p.n_blocks;
      const int e = p.tiles[2 * mb], row0 = p.tiles[2 * mb + 1];
      const int rows = min(BM, p.offsets[e + 1] - row0);
      const uint32_t tb = tmem_base + acc * BN + (static_cast<uint32_t>(q * 32) << 16);
      if (S > 1) {
        // Split-K: write this split's fp32 accumulator rows to its slab, count
        // the tile's finished splits, and let the last CTA sum the slabs in
        // split order (deterministic) and apply the epilogue.
        const int r = q * 32 + lane;
        float* slab = p.part + static_cast<size_t>(u) * p.part_rows * BN;
#pragma unroll 1
        for (int c0 = 0; c0 < BN; c0 += 32) {
          uint32_t a[32];
          tmem_ld32(tb + c0, a);
          tmem_ld_wait();
          if (r < rows) {
            float4* dst = reinterpret_cast<float4*>(slab + static_cast<size_t>(r) * BN + c0);
#pragma unroll
            for (int v = 0; v < 8; ++v)
              dst[v] = make_float4(__uint_as_float(a[4 * v]), __uint_as_float(a[4 * v + 1]),
                                   __uint_as_float(a[4 * v + 2]), __uint_as_float(a[4 * v + 3]));
          }
        }
        __threadfence();
        named_bar_sync();
        if (et == 0) sh->last = (atomicAdd(&p.tile_cnt[tile], 1) == S - 1);
        named_bar_sync();
        if (sh->last) {
          __threadfence();
          const float* base = p.part + static_cast<size_t>(tile) * S * p.part_rows * BN;
          const size_t slab_elems = static_cast<size_t>(p.part_rows) * BN;
          if (kSwiGLU) {
            const int n0 = nb * (BN / 2);
            for (int idx = et; idx < rows * (BN / 2); idx += 128) {
              const int rr = idx / (BN / 2), c = idx % (BN / 2);
              float g = 0.f, v = 0.f;
              for (int sp = 0; sp < S; ++sp) {
                const float* row = base + sp * slab_elems + static_cast<size_t>(rr) * BN;
                g += __ldcg(row + c);
                v += __ldcg(row + BN / 2 + c);
              }
              p.out[static_cast<size_t>(row0 + rr) * p.ldo + n0 + c] =
                  __float2bfloat16_rn(silu_mul(g, v));
            }
          } else {
            const int n0 = nb * BN;
            for (int idx = et; idx < rows * BN; idx += 128) {
              const int rr = idx / BN, c = idx % BN;
              float y = 0.f;
              for (int sp = 0; sp < S; ++sp)
                y += __ldcg(base + sp * slab_elems + static_cast<size_t>(rr) * BN + c);
              p.out[static_cast<size_t>(row0 + rr) * p.ldo + n0 + c] = __float2bfloat16_rn(y);
            }
          }
        }
      } else if (kSwiGLU) {
        // GEMM 1: each lane writes its own row of h, 32 columns at a time.
        const int r = q * 32 + lane;
        const bool valid = r < rows;
        __nv_bfloat16* orow = p.out + static_cast<size_t>(row0 + r) * p.ldo;
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
      } else {
        // GEMM 2: rows q*32 .. q*32+31 go out in blocks of 64 columns; each
        // lane packs its own row into the staging block, then each store
        // instruction writes four complete 128-byte row segments.
        const uint32_t blk_s = smem_u32(sOut + q * kStageOutBytes);
        const int n0 = nb * BN;
#pragma unroll 1
        for (int c0 = 0; c0 < BN; c0 += 64) {
          uint32_t packed[32];
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            uint32_t a[32];
            tmem_ld32(tb + c0 + 32 * half, a);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; ++i)
              packed[16 * half + i] =
                  pack_bf16x2(__uint_as_float(a[2 * i]), __uint_as_float(a[2 * i + 1]));
          }
          __syncwarp();  // the previous block has been read out
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const uint32_t at = blk_s + lane * 128 + ((c ^ (lane & 7)) << 4);
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(at), "r"(packed[4 * c]),
                         "r"(packed[4 * c + 1]), "r"(packed[4 * c + 2]), "r"(packed[4 * c + 3])
                         : "memory");
          }
          __syncwarp();
          const int chunk = lane & 7;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int rr = 4 * i + (lane >> 3);  // row within this warp's 32
            uint4 v;
            asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                         : "r"(blk_s + rr * 128 + ((chunk ^ (rr & 7)) << 4))
                         : "memory");
            if (q * 32 + rr < rows)
              *reinterpret_cast<uint4*>(p.out + static_cast<size_t>(row0 + q * 32 + rr) * p.ldo +
                                        n0 + c0 + chunk * 8) = v;
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&sh->tempty[acc]);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

template <bool kSwiGLU, bool kGatherA>
cudaError_t launch_gemm(const CUtensorMap& tm_act, const CUtensorMap& tm_w, const GemmArgs& a,
                        const LaunchOpts& o) {
  // the shared-memory opt-in is a per-device function attribute: set it once per device
  static std::atomic<bool> configured[64];
  int dev = 0;
  cudaError_t st = cudaGetDevice(&dev);
  if (st != cudaSuccess) return st;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!configured[dev].load(std::memory_order_acquire)) {
    st = cudaFuncSetAttribute(paged_gemm_kernel<kSwiGLU, kGatherA>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              kSmemBytes);
    if (st != cudaSuccess) return st;
    configured[dev].store(true, std::memory_order_release);
  }
  const long long tiles = static_cast<long long>(a.max_tiles) * a.n_blocks * a.splits;
  const int grid = static_cast<int>(tiles < o.sm_count ? tiles : o.sm_count);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid > 0 ? grid : 1);
  cfg.blockDim = dim3(kGatherA ? kThreadsGather : kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = o.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = o.pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, paged_gemm_kernel<kSwiGLU, kGatherA>, tm_act, tm_w, a);
}

}  // namespace

cudaError_t launch_gemm1_swiglu(const CUtensorMap& tm_x, const CUtensorMap& tm_w13,
                                const GemmArgs& a, const LaunchOpts& o) {
  return launch_gemm<true, false>(tm_x, tm_w13, a, o);
}

cudaError_t launch_gemm1_swiglu_gather(const CUtensorMap& tm_w13, const GemmArgs& a,
                                       const LaunchOpts& o) {
  return launch_gemm<true, true>(tm_w13, tm_w13, a, o);  // the activation map is not used
}

cudaError_t launch_gemm2(const CUtensorMap& tm_h, const CUtensorMap& tm_w2, const GemmArgs& a,
                         const LaunchOpts& o) {
  return launch_gemm<false, false>(tm_h, tm_w2, a, o);
}

}  // namespace rimuru
