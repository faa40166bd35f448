// C ABI of the forward path: workspace layout, per-view device state (page
// table + error word + TMA descriptors of the expert view), kernel launches
// and per-kernel event timing.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
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
  unsigned prof_mask = 0;  // kernels bracketed by an event pair
  int prof_cap = 0;
  int prof_calls = 0;
  int prof_every = 1;   // record every prof_every-th forward
  long long prof_seen = 0;  // forwards since profiling was enabled
  std::vector<cudaEvent_t> prof_ev;
  std::vector<unsigned> prof_hits;  // per recorded forward: kernels that ran between their events
};

namespace {

std::string cuda_msg(const char* what, cudaError_t e) {
  return std::string(what) + ": " + cudaGetErrorName(e) + " (" + cudaGetErrorString(e) + ")";
}

// SM count per device, looked up once (callers may be on several threads).
int sm_count_of(int device) {
  constexpr int kMaxDevices = 64;
  static std::atomic<int> cached[kMaxDevices];  // 0 = not looked up yet
  if (device < 0 || device >= kMaxDevices) return 0;
  int n = cached[device].load(std::memory_order_relaxed);
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) n = 0;
    cached[device].store(n, std::memory_order_relaxed);
  }
  return n;
}

uint64_t align_up(uint64_t v, uint64_t a) { return (v + a - 1) / a * a; }

void layout_for(const View& v, int T, rimuru_ws_layout* L) {
  const uint64_t A = static_cast<uint64_t>(T) * v.top_k;
  const int tpc = tokens_per_chunk(v.top_k);
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
  // x rows in sorted order exist only for batches the small-batch kernel
  // handles; past that, GEMM 1 gathers its rows from x itself
  L->x_sorted = take(A <= static_cast<uint64_t>(kChunkAssign) ? A * v.hidden * 2 : 0);
  L->h = take(A * v.inter * 2);
  L->y = take(A * v.hidden * 2);
  // split-K bookkeeping (see split_count): counters for both GEMMs, one slab
  // of fp32 partials per work unit, sized for the larger of the two
  const long long t1 = static_cast<long long>(max_tiles) * (v.inter / 128);
  const long long t2 = static_cast<long long>(max_tiles) * (v.hidden / 256);
  const int s1 = split_count(t1, v.hidden / 64), s2 = split_count(t2, v.inter / 64);
  const uint64_t part_rows = A < static_cast<uint64_t>(kTileM) ? A : kTileM;
  const uint64_t units = std::max<uint64_t>(s1 > 1 ? t1 * s1 : 0, s2 > 1 ? t2 * s2 : 0);
  L->ptiles = take(max_tiles * 2 * 4);
  L->num_ptiles = take(16);
  L->tile_cnt = take((2 * std::max<uint64_t>(t1, t2) + kSchedCounters) * 4);
  // the decode path's fp32 partials share the region (only one path runs per forward)
  const uint64_t dec = decode_path_fits(T, v.top_k, v.hidden, v.inter)
                           ? decode_part_bytes(T, v.top_k, v.experts, v.inter)
                           : 0;
  L->part = take(std::max<uint64_t>(units * part_rows * 256 * 4, dec));
  L->plan = take(dec ? kDecodePlanInts * 4 : 0);
  L->total = at;
  L->chunks = chunks;
  L->max_tiles = static_cast<int32_t>(max_tiles);
}

// Device staging of the host-buffer forward, after the layer's own workspace.
struct HostStaging {
  uint64_t x, logits, out, total;
};

HostStaging host_staging(const View& v, int T) {
  rimuru_ws_layout L;
  layout_for(v, T, &L);
  HostStaging s;
  const uint64_t t = static_cast<uint64_t>(T);
  s.x = align_up(L.total, 1024);
  s.logits = align_up(s.x + t * v.hidden * 2, 1024);
  s.out = align_up(s.logits + t * v.experts * 4, 1024);
  s.total = align_up(s.out + t * v.hidden * 2, 1024);
  return s;
}

}  // namespace

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
  int st = make_weight_maps(v->pool->base, v->page_bytes, v->n_pages, v->hidden, v->inter,
                            &d->tm_w13, &d->tm_w2);
  if (st != RIMURU_OK) {
    std::string msg = rimuru_last_error();
    destroy_device_state(v);
    return fail(st, msg);
  }
  v->table_dirty = true;
  return RIMURU_OK;
}

int view_device_table(View* v, int32_t** table, int** err, const CUtensorMap** w13,
                      const CUtensorMap** w2, int* device) {
  int st = ensure_device_state(v);
  if (st != RIMURU_OK) return st;
  *table = v->dev->d_table;
  *err = v->dev->d_err;
  *w13 = &v->dev->tm_w13;
  *w2 = &v->dev->tm_w2;
  *device = v->dev->device;
  return RIMURU_OK;
}

namespace {

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

int check_device(View* v, int device) {
  Pool* pool = v->pool;
  int pd = pool->device.load(std::memory_order_acquire);
  if (pd == -2) {
    cudaPointerAttributes at{};
    pd = -1;
    if (cudaPointerGetAttributes(&at, pool->base) != cudaSuccess)
      cudaGetLastError();  // not a pointer CUDA knows of: clear the error this call left
    else if (at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged)
      pd = at.device;
    pool->device.store(pd, std::memory_order_release);
  }
  if (pd >= 0 && pd != device)
    return fail(RIMURU_ERR_ARG, "the pool lives on device " + std::to_string(pd) +
                                    " but device " + std::to_string(device) + " is current");
  if (v->dev && v->dev->device != device)
    return fail(RIMURU_ERR_ARG, "the view's device state lives on device " +
                                    std::to_string(v->dev->device) + " but device " +
                                    std::to_string(device) + " is current");
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
  static const char* names[RIMURU_K_COUNT] = {
      "moe_route",         "moe_align",         "moe_gather",       "moe_gemm1_swiglu",
      "moe_gemm2",         "moe_combine",       "moe_route_align_gather",
      "moe_decode_gemm1",  "moe_decode_reduce", "moe_decode_gemm2"};
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

  int cur = 0;
  cudaError_t ce = cudaGetDevice(&cur);
  if (ce != cudaSuccess) return fail(RIMURU_ERR_CUDA, rimuru::cuda_msg("cudaGetDevice", ce));
  int st = rimuru::check_device(&v, cur);
  if (st != RIMURU_OK) return st;
  st = rimuru::ensure_device_state(&v);
  if (st != RIMURU_OK) return st;
  rimuru::DeviceState* d = v.dev;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  st = rimuru::upload_table(&v, stream);
  if (st != RIMURU_OK) return st;

  rimuru::LayerLaunch a;
  a.x = x_bf16;
  a.logits = logits;
  a.out = out_bf16;
  a.T = num_tokens;
  a.E = v.experts;
  a.k = v.top_k;
  a.H = v.hidden;
  a.I = v.inter;
  a.renorm = v.renorm;
  a.num_pages = static_cast<int>(v.n_pages);
  a.ws = static_cast<uint8_t*>(workspace);
  a.layout = L;
  a.table = d->d_table + static_cast<size_t>(layer) * v.experts * 3;
  a.err = d->d_err;
  a.tm_w13 = &d->tm_w13;
  a.tm_w2 = &d->tm_w2;
  a.pool = static_cast<uint8_t*>(v.pool->base);
  a.page_bytes = v.page_bytes;
  a.decode_max_tokens = v.decode_max_tokens;
  a.stream = stream;
  a.sm_count = rimuru::sm_count_of(d->device);
  if (a.sm_count <= 0) return fail(RIMURU_ERR_CUDA, "could not query the SM count");
  if (d->prof_on && d->prof_calls < d->prof_cap && d->prof_seen++ % d->prof_every == 0) {
    a.ev = &d->prof_ev[static_cast<size_t>(d->prof_calls) * RIMURU_K_COUNT * 2];
    a.ev_mask = d->prof_mask;
    a.hits = &d->prof_hits[d->prof_calls];
    *a.hits = 0u;
    d->prof_calls += 1;
  }
  return rimuru::launch_layer(a);
}

uint64_t rimuru_moe_host_workspace_bytes(rimuru_view_t view, int num_tokens) {
  if (!view || !view->v.has_shape || num_tokens < 0) return 0;
  return rimuru::host_staging(view->v, num_tokens).total;
}

int rimuru_moe_forward_host(const void* x_host, const float* logits_host, int num_tokens,
                            rimuru_view_t view, int layer, void* out_host, void* workspace,
                            uint64_t workspace_bytes, void* stream_ptr) {
  rimuru::clear_error();
  if (!view) return fail(RIMURU_ERR_ARG, "null view");
  rimuru::View& v = view->v;
  if (!v.has_shape) return fail(RIMURU_ERR_STATE, "view has no MoE shape");
  if (num_tokens < 0 || num_tokens > (1 << 20))
    return fail(RIMURU_ERR_ARG, "num_tokens must be in [0, 2^20]");
  if (num_tokens > 0 && (!x_host || !logits_host || !out_host || !workspace))
    return fail(RIMURU_ERR_ARG, "null pointer");
  const rimuru::HostStaging s = rimuru::host_staging(v, num_tokens);
  if (num_tokens > 0 && workspace_bytes < s.total)
    return fail(RIMURU_ERR_WORKSPACE, "workspace needs " + std::to_string(s.total) + " bytes");
  if (num_tokens > 0 && reinterpret_cast<uintptr_t>(workspace) % 1024 != 0)
    return fail(RIMURU_ERR_ALIGN, "workspace must be 1024-byte aligned");
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const size_t xb = static_cast<size_t>(num_tokens) * v.hidden * 2;
  const size_t lb = static_cast<size_t>(num_tokens) * v.experts * 4;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  cudaError_t e = cudaSuccess;
  // Checks that need no copy come first: an unmapped layer or a bad layer index
  // is reported before anything is queued.
  if (layer < 0 || layer >= v.layers) return fail(RIMURU_ERR_RANGE, "layer out of range");
  if (v.mapped_per_layer[layer] != v.experts * 3)
    return fail(RIMURU_ERR_UNMAPPED, "layer " + std::to_string(layer) + " has unmapped projections");
  if (num_tokens == 0) return RIMURU_OK;
  e = cudaMemcpyAsync(ws + s.x, x_host, xb, cudaMemcpyHostToDevice, stream);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(ws + s.logits, logits_host, lb, cudaMemcpyHostToDevice, stream);
  if (e != cudaSuccess) return fail(RIMURU_ERR_CUDA, rimuru::cuda_msg("input copy", e));
  int st = rimuru_moe_forward(ws + s.x, reinterpret_cast<const float*>(ws + s.logits), num_tokens,
                              view, layer, ws + s.out, workspace, s.x, stream_ptr);
  if (st != RIMURU_OK) return st;
  e = cudaMemcpyAsync(out_host, ws + s.out, xb, cudaMemcpyDeviceToHost, stream);
  if (e != cudaSuccess) return fail(RIMURU_ERR_CUDA, rimuru::cuda_msg("output copy", e));
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

int rimuru_profile_enable(rimuru_view_t view, int kernel_mask, int capacity) {
  return rimuru_profile_enable_sampled(view, kernel_mask, capacity, 1);
}

int rimuru_profile_enable_sampled(rimuru_view_t view, int kernel_mask, int capacity, int every) {
  rimuru::clear_error();
  if (every < 1) return fail(RIMURU_ERR_ARG, "every must be >= 1");
  if (!view) return fail(RIMURU_ERR_ARG, "null view");
  rimuru::View& v = view->v;
  if (!v.has_shape) return fail(RIMURU_ERR_STATE, "view has no MoE shape");
  if (kernel_mask < 0 || kernel_mask >= (1 << RIMURU_K_COUNT))
    return fail(RIMURU_ERR_ARG, "kernel mask out of range");
  int st = rimuru::ensure_device_state(&v);
  if (st != RIMURU_OK) return st;
  rimuru::DeviceState* d = v.dev;
  if (kernel_mask == 0) {
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
  d->prof_hits.assign(static_cast<size_t>(capacity), 0u);
  d->prof_cap = capacity;
  d->prof_calls = 0;
  d->prof_every = every;
  d->prof_seen = 0;
  d->prof_mask = static_cast<unsigned>(kernel_mask);
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
  if (!(d->prof_mask >> k & 1u)) return RIMURU_OK;
  for (int c = 0; c < d->prof_calls; ++c) {
    if (!(d->prof_hits[c] >> k & 1u)) continue;  // kernel k is not part of this forward's path
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
