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
// Layout from the first 1 KiB boundary of the array (the array itself is only
// 256-byte aligned): the error word's 1 KiB, then 8 KiB for one layer's page
// table (experts * 3 int32, at most 512 experts), then the layer's workspace,
// whose regions are 1 KiB-aligned offsets from a 1 KiB-aligned base as in the
// ordinary forward.
constexpr uint64_t kAlignSlack = 1024;
constexpr uint64_t kErrBytes = 1024;
constexpr uint64_t kTableBytes = 8192;
constexpr uint64_t kHeaderBytes = kAlignSlack + kErrBytes + kTableBytes;
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
  if (num_tokens < 0 || num_tokens > (1 << 20))
    return fail(RIMURU_ERR_ARG, "num_tokens must be in [0, 2^20]");
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
  const uint64_t need = kHeaderBytes + L.total;
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
  st = check_device(&v, device);
  if (st != RIMURU_OK) return st;
  uint8_t* scratch = nullptr;
  st = scratch_for_device(device, &scratch);
  if (st != RIMURU_OK) return st;
  int sms = 0;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
  if (e != cudaSuccess || sms <= 0) return fail(RIMURU_ERR_CUDA, "could not query the SM count");

  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(scratch) + kAlignSlack - 1) & ~static_cast<uintptr_t>(kAlignSlack - 1));
  int* err = dev_error ? dev_error : reinterpret_cast<int*>(base);
  int32_t* table = reinterpret_cast<int32_t*>(base + kErrBytes);
  uint8_t* ws = base + kErrBytes + kTableBytes;  // 1 KiB-aligned, as the ordinary forward requires

  const int T = num_tokens, E = v.experts, k = v.top_k, H = v.hidden, I = v.inter;
  // Left over from the previous call: the scratch error word (cleared here) and
  // the page table (this layer's entries are copied in on every call).  Every
  // other region is written by a kernel before it is read.
  if (!dev_error) e = cudaMemsetAsync(err, 0, sizeof(int), stream);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(table, v.page_table.data() + static_cast<size_t>(layer) * E * 3,
                        static_cast<size_t>(E) * 3 * sizeof(int32_t), cudaMemcpyHostToDevice, stream);
  if (e != cudaSuccess) return fail(RIMURU_ERR_CUDA, msg_of("scratch set-up", e));

  CUtensorMap tm_w13, tm_w2;
  st = make_weight_maps(v.pool->base, v.page_bytes, v.n_pages, H, I, &tm_w13, &tm_w2);
  if (st != RIMURU_OK) return st;

  LayerLaunch a;
  a.x = x_bf16;
  a.logits = logits;
  a.out = out_bf16;
  a.T = T;
  a.E = E;
  a.k = k;
  a.H = H;
  a.I = I;
  a.renorm = v.renorm;
  a.num_pages = static_cast<int>(v.n_pages);
  a.ws = ws;
  a.layout = L;
  a.table = table;
  a.err = err;
  a.tm_w13 = &tm_w13;
  a.tm_w2 = &tm_w2;
  a.pool = static_cast<uint8_t*>(v.pool->base);
  a.page_bytes = v.page_bytes;
  a.decode_max_tokens = v.decode_max_tokens;
  a.stream = stream;
  a.sm_count = sms;
  return launch_layer(a);
}
