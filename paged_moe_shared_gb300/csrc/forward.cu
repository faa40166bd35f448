// C ABI of the forward path: workspace layout, per-view device state (page
// table + error word + TMA descriptors of the expert view), kernel launches
// and per-kernel event timing.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "internal.h"
#include "kernels.h"

namespace rimuru {

struct DeviceState {
  int device = -1;
  int32_t* d_table = nullptr;  // [layers][experts][3]
  int* d_err = nullptr;        // device error word
  int32_t* h_stage = nullptr;  // pinned staging copy of the table
  cudaEvent_t upload_done = nullptr;
  bool upload_pending = false;
  CUtensorMap tm_w13{};  // [pages][hidden][inter] over the pool
  CUtensorMap tm_w2{};   // [pages][inter][hidden] over the pool
  // profiling: per recorded forward, per kernel, a start/stop event pair
  bool prof_on = false;
  int prof_cap = 0;
  int prof_calls = 0;
  std::vector<cudaEvent_t> prof_ev;
};

namespace {

std::string cuda_msg(const char* what, cudaError_t e) {
  return std::string(what) + ": " + cudaGetErrorName(e) + " (" + cudaGetErrorString(e) + ")";
}

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

// bf16 tensor map with 128-byte swizzle; dims/strides innermost first,
// strides in bytes for dims 1.. (rank - 1).
int make_map(CUtensorMap* m, void* base, int rank, const cuuint64_t* dims,
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

int sm_count_of(int device) {
  static int cached_dev = -1, cached = 0;
  if (device != cached_dev) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) n = 0;
    cached = n;
    cached_dev = device;
  }
  return cached;
}

uint64_t align_up(uint64_t v, uint64_t a) { return (v + a - 1) / a * a; }

void layout_for(const View& v, int T, rimuru_ws_layout* L) {
  const uint64_t A = static_cast<uint64_t>(T) * v.top_k;
  const int tpc = kChunkAssign / v.top_k;
  const int chunks = T > 0 ? (T + tpc - 1) / tpc : 0;
  const uint64_t max_tiles = (A + kTileM - 1) / kTileM + (A < static_cast<uint64_t>(v.experts) ? A : v.experts);
  uint64_t at = 0;
  auto take = [&](uint64_t bytes) {
    uint64_t here = at;
    at = align_up(at + bytes, 1024);
    return here;
  };
  L->ids = take(A * 4);
  L->weights = take(A * 4);
  L->chunk_hist = take(static_cast<uint64_t>(chunks) * v.experts * 4);
  L->offsets = take(static_cast<uint64_t>(v.experts + 1) * 4);
  L->sorted = take(A * 4);
  L->inv = take(A * 4);
  L->tiles = take(max_tiles * 2 * 4);
  L->num_tiles = take(16);
  L->x_sorted = take(A * v.hidden * 2);
  L->h = take(A * v.inter * 2);
  L->y = take(A * v.hidden * 2);
  L->total = at;
  L->chunks = chunks;
  L->max_tiles = static_cast<int32_t>(max_tiles);
}

int ensure_device_state(View* v) {
  if (v->dev) return RIMURU_OK;
  auto* d = new (std::nothrow) DeviceState;
  if (!d) return fail(RIMURU_ERR_OOM, "host allocation failed");
  cudaError_t e = cudaGetDevice(&d->device);
  const size_t n = v->page_table.size();
  if (e == cudaSuccess) e = cudaMalloc(&d->d_table, n * sizeof(int32_t));
  if (e == cudaSuccess) e = cudaMalloc(&d->d_err, 4 * sizeof(int));
  if (e == cudaSuccess) e = cudaMemset(d->d_err, 0, 4 * sizeof(int));
  if (e == cudaSuccess) e = cudaMallocHost(&d->h_stage, n * sizeof(int32_t));
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&d->upload_done, cudaEventDisableTiming);
  if (e != cudaSuccess) {
    v->dev = d;
    destroy_device_state(v);
    return fail(RIMURU_ERR_CUDA, cuda_msg("device state of the view", e));
  }
  v->dev = d;
  // the expert view as two 3-D tensor maps over the whole pool
  const uint64_t H = v->hidden, I = v->inter, P = v->n_pages;
  cuuint64_t dims13[3] = {I, H, P};
  cuuint64_t str13[2] = {I * 2, v->page_bytes};
  cuuint64_t dims2[3] = {H, I, P};
  cuuint64_t str2[2] = {H * 2, v->page_bytes};
  cuuint32_t box[3] = {64, 64, 1};
  int st = make_map(&d->tm_w13, v->pool->base, 3, dims13, str13, box);
  if (st == RIMURU_OK) st = make_map(&d->tm_w2, v->pool->base, 3, dims2, str2, box);
  if (st != RIMURU_OK) {
    std::string msg = rimuru_last_error();
    destroy_device_state(v);
    return fail(st, msg);
  }
  v->table_dirty = true;
  return RIMURU_OK;
}

int upload_table(View* v, cudaStream_t stream) {
  DeviceState* d = v->dev;
  if (!v->table_dirty) return RIMURU_OK;
  int st = wait_table_upload(v);
  if (st != RIMURU_OK) return st;
  const size_t bytes = v->page_table.size() * sizeof(int32_t);
  std::memcpy(d->h_stage, v->page_table.data(), bytes);
  cudaError_t e = cudaMemcpyAsync(d->d_table, d->h_stage, bytes, cudaMemcpyHostToDevice, stream);
  if (e == cudaSuccess) e = cudaEventRecord(d->upload_done, stream);
  if (e != cudaSuccess) return fail(RIMURU_ERR_CUDA, cuda_msg("page table upload", e));
  d->upload_pending = true;
  v->table_dirty = false;
  return RIMURU_OK;
}

}  // namespace

// The host staging copy may only change once the previous upload has left it.
int wait_table_upload(View* v) {
  if (!v->dev || !v->dev->upload_pending) return RIMURU_OK;
  cudaError_t e = cudaEventSynchronize(v->dev->upload_done);
  if (e != cudaSuccess) return fail(RIMURU_ERR_CUDA, cuda_msg("waiting for the page table upload", e));
  v->dev->upload_pending = false;
  return RIMURU_OK;
}

void destroy_device_state(View* v) {
  DeviceState* d = v->dev;
  if (!d) return;
  if (d->upload_done) {
    if (d->upload_pending) cudaEventSynchronize(d->upload_done);
    cudaEventDestroy(d->upload_done);
  }
  for (cudaEvent_t ev : d->prof_ev) cudaEventDestroy(ev);
  if (d->d_table) cudaFree(d->d_table);
  if (d->d_err) cudaFree(d->d_err);
  if (d->h_stage) cudaFreeHost(d->h_stage);
  delete d;
  v->dev = nullptr;
}

}  // namespace rimuru

using rimuru::fail;

extern "C" {

uint64_t rimuru_moe_workspace_bytes(rimuru_view_t view, int num_tokens) {
  if (!view || !view->v.has_shape || num_tokens < 0) return 0;
  rimuru_ws_layout L;
  rimuru::layout_for(view->v, num_tokens, &L);
  return L.total;
}

int rimuru_moe_workspace_layout(rimuru_view_t view, int num_tokens, rimuru_ws_layout* out) {
  rimuru::clear_error();
  if (!view || !out) return fail(RIMURU_ERR_ARG, "null argument");
  if (!view->v.has_shape) return fail(RIMURU_ERR_STATE, "view has no MoE shape");
  if (num_tokens < 0) return fail(RIMURU_ERR_ARG, "negative token count");
  rimuru::layout_for(view->v, num_tokens, out);
  return RIMURU_OK;
}

int rimuru_device_sm_count(void) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return rimuru::sm_count_of(dev);
}

const char* rimuru_kernel_name(int k) {
  static const char* names[RIMURU_K_COUNT] = {"moe_route", "moe_align", "moe_gather",
                                              "moe_gemm1_swiglu", "moe_gemm2", "moe_combine"};
  return (k >= 0 && k < RIMURU_K_COUNT) ? names[k] : nullptr;
}

int rimuru_moe_forward(const void* x_bf16, const float* logits, int num_tokens, rimuru_view_t view,
                       int layer, void* out_bf16, void* workspace, uint64_t workspace_bytes,
                       void* stream_ptr) {
  rimuru::clear_error();
  if (!view) return fail(RIMURU_ERR_ARG, "null view");
  rimuru::View& v = view->v;
  if (!v.has_shape) return fail(RIMURU_ERR_STATE, "view has no MoE shape");
  if (layer < 0 || layer >= v.layers) return fail(RIMURU_ERR_RANGE, "layer out of range");
  if (num_tokens < 0 || num_tokens > (1 << 20))
    return fail(RIMURU_ERR_ARG, "num_tokens must be in [0, 2^20]");
  if (v.mapped_per_layer[layer] != v.experts * 3)
    return fail(RIMURU_ERR_UNMAPPED, "layer " + std::to_string(layer) + " has " +
                                         std::to_string(v.experts * 3 - v.mapped_per_layer[layer]) +
                                         " unmapped projections");
  if (num_tokens == 0) return RIMURU_OK;
  if (!x_bf16 || !logits || !out_bf16 || !workspace)
    return fail(RIMURU_ERR_ARG, "null device pointer");
  auto mis = [](const void* p, uintptr_t a) { return reinterpret_cast<uintptr_t>(p) % a != 0; };
  if (mis(x_bf16, 16) || mis(logits, 16) || mis(out_bf16, 16))
    return fail(RIMURU_ERR_ALIGN, "x, logits and out must be 16-byte aligned");
  if (mis(workspace, 1024)) return fail(RIMURU_ERR_ALIGN, "workspace must be 1024-byte aligned");
  if (x_bf16 == out_bf16) return fail(RIMURU_ERR_ARG, "out may not alias x");
  rimuru_ws_layout L;
  rimuru::layout_for(v, num_tokens, &L);
  if (workspace_bytes < L.total)
    return fail(RIMURU_ERR_WORKSPACE, "workspace needs " + std::to_string(L.total) + " bytes");

  int st = rimuru::ensure_device_state(&v);
  if (st != RIMURU_OK) return st;
  rimuru::DeviceState* d = v.dev;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  st = rimuru::upload_table(&v, stream);
  if (st != RIMURU_OK) return st;

  const int T = num_tokens, E = v.experts, k = v.top_k, H = v.hidden, I = v.inter;
  const int A = T * k;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
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

  // activation maps: x_sorted [A][H] and h [A][I], 64 x 128 boxes
  CUtensorMap tm_x, tm_h;
  {
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(A)};
    cuuint64_t str[1] = {static_cast<cuuint64_t>(H) * 2};
    cuuint32_t box[2] = {64, 128};
    st = rimuru::make_map(&tm_x, xs, 2, dims, str, box);
    if (st != RIMURU_OK) return st;
  }
  {
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(I), static_cast<cuuint64_t>(A)};
    cuuint64_t str[1] = {static_cast<cuuint64_t>(I) * 2};
    cuuint32_t box[2] = {64, 128};
    st = rimuru::make_map(&tm_h, h, 2, dims, str, box);
    if (st != RIMURU_OK) return st;
  }

  rimuru::LaunchOpts o;
  o.stream = stream;
  o.sm_count = rimuru::sm_count_of(d->device);
  if (o.sm_count <= 0) return fail(RIMURU_ERR_CUDA, "could not query the SM count");

  // per-kernel timing
  cudaEvent_t* ev = nullptr;
  if (d->prof_on && d->prof_calls < d->prof_cap) {
    ev = &d->prof_ev[static_cast<size_t>(d->prof_calls) * RIMURU_K_COUNT * 2];
    d->prof_calls += 1;
  }
  cudaError_t e = cudaSuccess;
  auto mark = [&](int kidx, int which) {
    if (ev && e == cudaSuccess) e = cudaEventRecord(ev[kidx * 2 + which], stream);
  };

  const int tpc = rimuru::kChunkAssign / k;
  rimuru::GemmArgs g1{};
  g1.page_table = d->d_table + static_cast<size_t>(layer) * E * 3;
  g1.tiles = tiles;
  g1.num_tiles = num_tiles;
  g1.offsets = offsets;
  g1.num_pages = static_cast<int>(v.n_pages);
  g1.max_tiles = L.max_tiles;
  g1.weights_evict_first = (A <= E * rimuru::kTileM / 4) ? 1 : 0;
  g1.err = d->d_err;
  rimuru::GemmArgs g2 = g1;
  g1.out = h;
  g1.ldo = I;
  g1.n_blocks = I / 128;
  g1.num_k_blocks = H / 64;
  g2.out = y;
  g2.ldo = H;
  g2.n_blocks = H / 256;
  g2.num_k_blocks = I / 64;

  mark(RIMURU_K_ROUTE, 0);
  if (e == cudaSuccess)
    e = rimuru::launch_route(logits, T, E, k, v.renorm, tpc, ids, w, chunk_hist, d->d_err, o);
  mark(RIMURU_K_ROUTE, 1);
  mark(RIMURU_K_ALIGN, 0);
  if (e == cudaSuccess)
    e = rimuru::launch_align(ids, chunk_hist, L.chunks, A, E, tpc * k, offsets, sorted, inv, tiles,
                             num_tiles, d->d_err, o);
  mark(RIMURU_K_ALIGN, 1);
  mark(RIMURU_K_GATHER, 0);
  if (e == cudaSuccess)
    e = rimuru::launch_gather(static_cast<const __nv_bfloat16*>(x_bf16), sorted, A, k, H, xs, o);
  mark(RIMURU_K_GATHER, 1);
  mark(RIMURU_K_GEMM1, 0);
  if (e == cudaSuccess) e = rimuru::launch_gemm1_swiglu(tm_x, d->tm_w13, g1, o);
  mark(RIMURU_K_GEMM1, 1);
  mark(RIMURU_K_GEMM2, 0);
  if (e == cudaSuccess) e = rimuru::launch_gemm2(tm_h, d->tm_w2, g2, o);
  mark(RIMURU_K_GEMM2, 1);
  mark(RIMURU_K_COMBINE, 0);
  if (e == cudaSuccess)
    e = rimuru::launch_combine(y, inv, w, T, k, H, static_cast<__nv_bfloat16*>(out_bf16), o);
  mark(RIMURU_K_COMBINE, 1);
  if (e != cudaSuccess) return fail(RIMURU_ERR_CUDA, rimuru::cuda_msg("kernel launch", e));
  return RIMURU_OK;
}

int rimuru_get_device_error(rimuru_view_t view, int* code, int clear) {
  rimuru::clear_error();
  if (!view || !code) return fail(RIMURU_ERR_ARG, "null argument");
  rimuru::View& v = view->v;
  if (!v.dev) {
    *code = RIMURU_DEV_OK;
    return RIMURU_OK;
  }
  int h = 0;
  cudaError_t e = cudaMemcpy(&h, v.dev->d_err, sizeof(int), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess && clear) e = cudaMemset(v.dev->d_err, 0, sizeof(int));
  if (e != cudaSuccess) return fail(RIMURU_ERR_CUDA, rimuru::cuda_msg("reading the device error", e));
  *code = h;
  return RIMURU_OK;
}

int rimuru_profile_enable(rimuru_view_t view, int enable, int capacity) {
  rimuru::clear_error();
  if (!view) return fail(RIMURU_ERR_ARG, "null view");
  rimuru::View& v = view->v;
  if (!v.has_shape) return fail(RIMURU_ERR_STATE, "view has no MoE shape");
  int st = rimuru::ensure_device_state(&v);
  if (st != RIMURU_OK) return st;
  rimuru::DeviceState* d = v.dev;
  if (!enable) {
    d->prof_on = false;
    return RIMURU_OK;
  }
  if (capacity <= 0 || capacity > (1 << 16)) return fail(RIMURU_ERR_ARG, "capacity out of range");
  const size_t need = static_cast<size_t>(capacity) * RIMURU_K_COUNT * 2;
  while (d->prof_ev.size() < need) {
    cudaEvent_t ev;
    cudaError_t e = cudaEventCreate(&ev);
    if (e != cudaSuccess) return fail(RIMURU_ERR_CUDA, rimuru::cuda_msg("cudaEventCreate", e));
    d->prof_ev.push_back(ev);
  }
  d->prof_cap = capacity;
  d->prof_calls = 0;
  d->prof_on = true;
  return RIMURU_OK;
}

int rimuru_profile_read(rimuru_view_t view, int k, int* launches, double* total_ms) {
  rimuru::clear_error();
  if (!view || !launches || !total_ms) return fail(RIMURU_ERR_ARG, "null argument");
  if (k < 0 || k >= RIMURU_K_COUNT) return fail(RIMURU_ERR_RANGE, "kernel index out of range");
  rimuru::View& v = view->v;
  *launches = 0;
  *total_ms = 0.0;
  if (!v.dev) return RIMURU_OK;
  rimuru::DeviceState* d = v.dev;
  for (int c = 0; c < d->prof_calls; ++c) {
    cudaEvent_t a = d->prof_ev[(static_cast<size_t>(c) * RIMURU_K_COUNT + k) * 2];
    cudaEvent_t b = d->prof_ev[(static_cast<size_t>(c) * RIMURU_K_COUNT + k) * 2 + 1];
    float ms = 0.f;
    cudaError_t e = cudaEventSynchronize(b);
    if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, a, b);
    if (e != cudaSuccess) return fail(RIMURU_ERR_CUDA, rimuru::cuda_msg("reading profile events", e));
    *launches += 1;
    *total_ms += ms;
  }
  return RIMURU_OK;
}

}  // extern "C"
