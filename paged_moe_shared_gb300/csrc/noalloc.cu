// rimuru_moe_forward_noalloc: the fused MoE forward for callers that cannot
// allocate device memory.  Its scratch (routing tables, the sorted activations,
// h and y, the layer's page table and an error word) lives in one file-scope
// __device__ array instead of a caller-provided workspace, and the call makes
// no cudaMalloc / cudaFree / cudaMallocHost / event creation of any kind.
//
// The array is a fixed kNoAllocScratchBytes on every GPU that loads the
// library and stays allocated until the process exits.  Every call shares it
// and it keeps the previous call's contents, so calls whose kernels overlap on
// the GPU (two streams, or two threads) race on it: serialise them.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstring>
#include <mutex>
#include <string>

#include "internal.h"
#include "kernels.h"

namespace rimuru {
namespace {

constexpr uint64_t kNoAllocScratchBytes = 16ull << 20;  // 16 MiB per device
constexpr uint64_t kErrBytes = 256;                     // device error word
constexpr uint64_t kTableBytes = 8192;                  // one layer: experts * 3 int32 (<= 512 experts)
constexpr int kMaxDevices = 64;

static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_setup_mu;
uint8_t* g_scratch_ptr[kMaxDevices] = {};

std::string msg_of(const char* what, cudaError_t e) {
  return std::string(what) + ": " + cudaGetErrorName(e) + " (" + cudaGetErrorString(e) + ")";
}

// Device address of the scratch array on the current device.  In host code the
// array's name is only a stand-in, so the real address is looked up once per
// device, with that device current, and cached.
int scratch_for_device(int device, uint8_t** out) {
  if (device < 0 || device >= kMaxDevices) return fail(RIMURU_ERR_CUDA, "device index out of range");
  std::lock_guard<std::mutex> g(g_setup_mu);
  if (!g_scratch_ptr[device]) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return fail(RIMURU_ERR_CUDA, msg_of("cudaGetSymbolAddress(scratch)", e));
    g_scratch_ptr[device] = static_cast<uint8_t*>(p);
  }
  *out = g_scratch_ptr[device];
  return RIMURU_OK;
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

int encode(CUtensorMap* m, void* base, int rank, const cuuint64_t* dims, const cuuint64_t* strides,
           const cuuint32_t* box) {
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
  if (!fn) return fail(RIMURU_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, static_cast<cuuint32_t>(rank), base, dims,
                  strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(RIMURU_ERR_CUDA, "cuTensorMapEncodeTiled failed with CUresult " + std::to_string(r));
  return RIMURU_OK;
}

}  // namespace
}  // namespace rimuru

using rimuru::fail;

extern "C" int rimuru_moe_forward_noalloc(const void* x_bf16, const float* logits, int num_tokens,
                                          rimuru_view_t view, int layer, void* out_bf16,
                                          int* dev_error, void* stream_ptr) {
  using namespace rimuru;
  clear_error();
  if (!view) return fail(RIMURU_ERR_ARG, "null view");
  View& v = view->v;
  if (!v.has_shape) return fail(RIMURU_ERR_STATE, "view has no MoE shape");
  if (layer < 0 || layer >= v.layers) return fail(RIMURU_ERR_RANGE, "layer out of range");
  if (num_tokens < 0) return fail(RIMURU_ERR_ARG, "negative token count");
  if (v.mapped_per_layer[layer] != v.experts * 3)
    return fail(RIMURU_ERR_UNMAPPED, "layer " + std::to_string(layer) + " has unmapped projections");
  if (num_tokens == 0) return RIMURU_OK;
  if (!x_bf16 || !logits || !out_bf16) return fail(RIMURU_ERR_ARG, "null device pointer");
  auto mis = [](const void* p, uintptr_t a) { return reinterpret_cast<uintptr_t>(p) % a != 0; };
  if (mis(x_bf16, 16) || mis(logits, 16) || mis(out_bf16, 16))
    return fail(RIMURU_ERR_ALIGN, "x, logits and out must be 16-byte aligned");
  if (dev_error && mis(dev_error, 4)) return fail(RIMURU_ERR_ALIGN, "dev_error must be 4-byte aligned");
  if (x_bf16 == out_bf16) return fail(RIMURU_ERR_ARG, "out may not alias x");

  rimuru_ws_layout L;
  int st = rimuru_moe_workspace_layout(view, num_tokens, &L);
  if (st != RIMURU_OK) return st;
  const uint64_t need = kErrBytes + kTableBytes + L.total;
  if (need > kNoAllocScratchBytes)
    return fail(RIMURU_ERR_WORKSPACE,
                std::to_string(num_tokens) + " tokens need " + std::to_string(need) +
                    " bytes of scratch; the built-in scratch holds " +
                    std::to_string(kNoAllocScratchBytes) +
                    " bytes (use rimuru_moe_forward with a caller-provided workspace for larger "
                    "batches)");

  int device = 0;
  cudaError_t e = cudaGetDevice(&device);
  if (e != cudaSuccess) return fail(RIMURU_ERR_CUDA, msg_of("cudaGetDevice", e));
  uint8_t* scratch = nullptr;
  st = scratch_for_device(device, &scratch);
  if (st != RIMURU_OK) return st;
  int sms = 0;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
  if (e != cudaSuccess || sms <= 0) return fail(RIMURU_ERR_CUDA, "could not query the SM count");

  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  int* err = dev_error ? dev_error : reinterpret_cast<int*>(scratch);
  int32_t* table = reinterpret_cast<int32_t*>(scratch + kErrBytes);
  uint8_t* ws = scratch + kErrBytes + kTableBytes;  // 256-byte aligned base

  const int T = num_tokens, E = v.experts, k = v.top_k, H = v.hidden, I = v.inter;
  const int A = T * k;
  // Left over from the previous call: the scratch error word (cleared here) and
  // the page table (this layer's entries are copied in on every call).  Every
  // other region is written by a kernel before it is read.
  if (!dev_error) e = cudaMemsetAsync(err, 0, sizeof(int), stream);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(table, v.page_table.data() + static_cast<size_t>(layer) * E * 3,
                        static_cast<size_t>(E) * 3 * sizeof(int32_t), cudaMemcpyHostToDevice, stream);
  if (e != cudaSuccess) return fail(RIMURU_ERR_CUDA, msg_of("scratch set-up", e));

  auto* ids = reinterpret_cast<int32_t*>(ws + L.ids);
  auto* w = reinterpret_cast<float*>(ws + L.weights);
  auto* chunk_hist = reinterpret_cast<int32_t*>(ws + L.chunk_hist);
  auto* offsets = reinterpret_cast<int32_t*>(ws + L.offsets);
  auto* sorted = reinterpret_cast<int32_t*>(ws + L.sorted);
  auto* inv = reinterpret_cast<int32_t*>(ws + L.inv);
  auto* tiles = reinterpret_cast<int32_t*>(ws + L.tiles);
  auto* num_tiles = reinterpret_cast<int32_t*>(ws + L.num_tiles);
  auto* xs = reinterpret_cast<__nv_bfloat16*>(ws + L.x_sorted);
  auto* h = reinterpret_cast<__nv_bfloat16*>(ws + L.h);
  auto* y = reinterpret_cast<__nv_bfloat16*>(ws + L.y);

  // TMA descriptors: activations in the scratch, expert view over the pool.
  CUtensorMap tm_x, tm_h, tm_w13, tm_w2;
  const uint64_t P = static_cast<uint64_t>(v.n_pages);
  {
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(A)};
    cuuint64_t str[1] = {static_cast<cuuint64_t>(H) * 2};
    cuuint32_t box[2] = {64, 128};
    if ((st = encode(&tm_x, xs, 2, dims, str, box)) != RIMURU_OK) return st;
  }
  {
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(I), static_cast<cuuint64_t>(A)};
    cuuint64_t str[1] = {static_cast<cuuint64_t>(I) * 2};
    cuuint32_t box[2] = {64, 128};
    if ((st = encode(&tm_h, h, 2, dims, str, box)) != RIMURU_OK) return st;
  }
  {
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(I), static_cast<cuuint64_t>(H), P};
    cuuint64_t str[2] = {static_cast<cuuint64_t>(I) * 2, v.page_bytes};
    cuuint32_t box[3] = {64, 64, 1};
    if ((st = encode(&tm_w13, v.pool->base, 3, dims, str, box)) != RIMURU_OK) return st;
  }
  {
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(I), P};
    cuuint64_t str[2] = {static_cast<cuuint64_t>(H) * 2, v.page_bytes};
    cuuint32_t box[3] = {64, 64, 1};
    if ((st = encode(&tm_w2, v.pool->base, 3, dims, str, box)) != RIMURU_OK) return st;
  }

  LaunchOpts o;
  o.stream = stream;
  o.sm_count = sms;
  const int tpc = kChunkAssign / k;
  GemmArgs g1{};
  g1.page_table = table;
  g1.tiles = tiles;
  g1.num_tiles = num_tiles;
  g1.offsets = offsets;
  g1.num_pages = static_cast<int>(v.n_pages);
  g1.max_tiles = L.max_tiles;
  g1.weights_evict_first = (A <= E * kTileM / 4) ? 1 : 0;
  g1.err = err;
  GemmArgs g2 = g1;
  g1.out = h;
  g1.ldo = I;
  g1.n_blocks = I / 128;
  g1.num_k_blocks = H / 64;
  g2.out = y;
  g2.ldo = H;
  g2.n_blocks = H / 256;
  g2.num_k_blocks = I / 64;

  e = launch_route(logits, T, E, k, v.renorm, tpc, ids, w, chunk_hist, err, o);
  if (e == cudaSuccess)
    e = launch_align(ids, chunk_hist, L.chunks, A, E, tpc * k, offsets, sorted, inv, tiles,
                     num_tiles, err, o);
  if (e == cudaSuccess)
    e = launch_gather(static_cast<const __nv_bfloat16*>(x_bf16), sorted, A, k, H, xs, o);
  if (e == cudaSuccess) e = launch_gemm1_swiglu(tm_x, tm_w13, g1, o);
  if (e == cudaSuccess) e = launch_gemm2(tm_h, tm_w2, g2, o);
  if (e == cudaSuccess)
    e = launch_combine(y, inv, w, T, k, H, static_cast<__nv_bfloat16*>(out_bf16), o);
  if (e != cudaSuccess) return fail(RIMURU_ERR_CUDA, msg_of("kernel launch", e));
  return RIMURU_OK;
}
