// Expert offloading for a stack of paged MoE layers: every expert lives in
// pinned host memory; a fixed number of them are resident in pages of the
// expert view at any time.  Routing decides which experts a layer needs;
// misses are copied host -> device on a side stream straight into pool pages
// (no staging buffer and no device-to-device copy), with least-recently-used
// eviction.  A prefetch for the next layer can be queued on the copy stream
// while the current layer computes (two sets of pages in flight: the ones
// being read and the ones being filled).
//
// Rimuru page (arXiv 2610.40305): expert offloading to CPU memory (Figure 1,
// panel b, and the explainer's motivation paragraph) and dual buffers that
// overlap expert prefetch with execution while avoiding a local
// device-to-device copy (Figure 8).  The pages name no eviction policy; LRU is
// this library's choice.
//
// Ordering rules (all on the GPU, the host never waits for a copy):
//  * a slot is overwritten only after the last forward that read it has
//    finished: the copy stream waits on that forward's completion event;
//  * a forward reads a layer's slots only after the copies into them have
//    landed: the compute stream waits on the layer's last copy event;
//  * the layer's page-table slice is uploaded on the compute stream just
//    before its expert kernels, from a pinned staging ring.
#include <cuda_runtime.h>

#include <algorithm>
#include <string>
#include <vector>

#include "internal.h"
#include "kernels.h"

namespace rimuru {

int ensure_device_state(View* v);  // forward.cu
int view_device_table(View* v, int32_t** table, int** err, const CUtensorMap** w13,
                      const CUtensorMap** w2, int* device);  // forward.cu

namespace {

constexpr int kDoneRing = 64;   // completion events of recent forwards
constexpr int kStageRing = 8;   // pinned staging slices for page-table uploads

std::string cuda_msg(const char* what, cudaError_t e) {
  return std::string(what) + ": " + cudaGetErrorName(e) + " (" + cudaGetErrorString(e) + ")";
}

}  // namespace

struct Offload {
  rimuru_view_t vh = nullptr;
  View* v = nullptr;
  int L = 0, E = 0, cap = 0;
  uint64_t matrix_bytes = 0;  // bytes of one projection (hidden * inter * 2)
  const uint8_t* host = nullptr;
  cudaStream_t copy = nullptr;
  bool own_copy = false;

  std::vector<int64_t> slot_page;  // [cap][3]
  std::vector<int> slot_key;       // l * E + e, or -1
  std::vector<int64_t> slot_seq;   // last forward that read the slot, or -1
  std::vector<int64_t> slot_op;    // operation that last claimed the slot
  std::vector<int> key_slot;       // [L * E]
  std::vector<int> prv, nxt;       // LRU list over slots; head = most recent
  int head = -1, tail = -1;
  int64_t op = 0, seq = 0;
  int policy = RIMURU_EVICT_LRU;
  int next_layer = 0;  // layer the next forward is expected to run (layer-cycle policy)

  std::vector<cudaEvent_t> done_ev;   // [kDoneRing]
  std::vector<cudaEvent_t> ready_ev;  // [L]
  std::vector<char> ready_pending;    // [L]
  int32_t* h_offsets = nullptr;       // pinned, E + 1
  cudaEvent_t offsets_ev = nullptr;
  std::vector<int32_t*> stage;        // pinned, [kStageRing][E * 3]
  std::vector<cudaEvent_t> stage_ev;
  int stage_next = 0;

  rimuru_offload_counters st{};
  rimuru_offload_counters& st_ = st;

  // Copies are merged while both ends continue the pending run.
  uint64_t pend_dst = 0, pend_src = 0, pend_len = 0;
  int64_t waited_seq = 0;  // the copy stream already waits for forwards up to this one

  cudaError_t flush() {
    if (pend_len == 0) return cudaSuccess;
    uint8_t* pool = static_cast<uint8_t*>(v->pool->base);
    cudaError_t e = cudaMemcpyAsync(pool + pend_dst, host + pend_src, pend_len,
                                    cudaMemcpyHostToDevice, copy);
    pend_len = 0;
    return e;
  }
  cudaError_t queue_copy(uint64_t dst, uint64_t src, uint64_t len) {
    if (pend_len && dst == pend_dst + pend_len && src == pend_src + pend_len &&
        len == v->page_bytes) {
      pend_len += len;
      return cudaSuccess;
    }
    cudaError_t e = flush();
    pend_dst = dst;
    pend_src = src;
    pend_len = len;
    return e;
  }

  void unlink(int s) {
    if (prv[s] >= 0) nxt[prv[s]] = nxt[s]; else head = nxt[s];
    if (nxt[s] >= 0) prv[nxt[s]] = prv[s]; else tail = prv[s];
    prv[s] = nxt[s] = -1;
  }
  void push_front(int s) {
    prv[s] = -1;
    nxt[s] = head;
    if (head >= 0) prv[head] = s; else tail = s;
    head = s;
  }
  void touch(int s) {
    if (head == s) return;
    unlink(s);
    push_front(s);
  }

  void set_entry(int layer, int expert, int proj, int32_t page) {
    const size_t at = (static_cast<size_t>(layer) * E + expert) * 3 + proj;
    const int32_t old = v->page_table[at];
    if (old >= 0) v->map_count[old] -= 1; else if (page >= 0) v->mapped_per_layer[layer] += 1;
    if (page >= 0) v->map_count[page] += 1; else if (old >= 0) v->mapped_per_layer[layer] -= 1;
    v->page_table[at] = page;
    v->table_dirty = true;
  }

  // The slot to refill, never one claimed by the current operation.
  //  LRU: the least recently used.
  //  Layer cycle (layers run 0, 1, ..., L-1, 0, ... as in every decode step of
  //  a model): the slot whose expert's layer comes last counting on from the
  //  next forward's layer, i.e. whose next use is furthest away (Belady's rule
  //  for a cyclic order); empty slots first, ties to the least recently used.
  //  Under LRU a cycle of L layers larger than the cache misses on every
  //  expert; this keeps a fixed part of the cycle resident.
  int victim() const {
    if (policy == RIMURU_EVICT_LRU) {
      int s = tail;
      while (s >= 0 && slot_op[s] == op) s = prv[s];
      return s;
    }
    int best = -1, best_d = -1;
    for (int s = tail; s >= 0; s = prv[s]) {
      if (slot_op[s] == op) continue;
      const int d = slot_key[s] < 0 ? L : ((slot_key[s] / E - next_layer) % L + L) % L;
      if (d > best_d) {
        best = s;
        best_d = d;
      }
    }
    return best;
  }

  // Make expert (layer, e) resident; `protect` slots claimed in this operation.
  int load(int layer, int e, bool demand, bool* was_hit) {
    const int key = layer * E + e;
    int s = key_slot[key];
    if (s >= 0) {
      touch(s);
      slot_op[s] = op;
      *was_hit = true;
      return RIMURU_OK;
    }
    *was_hit = false;
    s = victim();
    if (s < 0)
      return fail(RIMURU_ERR_OOM, "offload capacity is smaller than the experts one layer needs");
    const int old = slot_key[s];
    if (old >= 0) {
      for (int p = 0; p < 3; ++p) set_entry(old / E, old % E, p, -1);
      key_slot[old] = -1;
      st.evictions += 1;
    }
    cudaError_t err = cudaSuccess;
    if (slot_seq[s] > waited_seq) {  // a forward newer than any waited for read this slot
      err = flush();
      if (err == cudaSuccess)
        err = cudaStreamWaitEvent(copy, done_ev[static_cast<size_t>(slot_seq[s] % kDoneRing)], 0);
      waited_seq = slot_seq[s];
    }
    for (int p = 0; p < 3 && err == cudaSuccess; ++p) {
      const uint64_t dst = static_cast<uint64_t>(slot_page[static_cast<size_t>(s) * 3 + p]) * v->page_bytes;
      const uint64_t src = (static_cast<uint64_t>(key) * 3 + p) * v->page_bytes;
      err = queue_copy(dst, src, matrix_bytes);
    }
    if (err != cudaSuccess) return fail(RIMURU_ERR_CUDA, cuda_msg("expert copy", err));
    for (int p = 0; p < 3; ++p)
      set_entry(layer, e, p, static_cast<int32_t>(slot_page[static_cast<size_t>(s) * 3 + p]));
    slot_key[s] = key;
    key_slot[key] = s;
    slot_op[s] = op;
    touch(s);
    ready_pending[layer] = 1;
    st.bytes_h2d += static_cast<int64_t>(3 * matrix_bytes);
    if (!demand) st.prefetch_loads += 1;
    return RIMURU_OK;
  }

  // Wait (host) until no copy and no forward can still touch any slot.
  int quiesce() {
    cudaError_t e = flush();
    if (e == cudaSuccess) e = cudaStreamSynchronize(copy);
    if (e == cudaSuccess && seq > 0)
      e = cudaEventSynchronize(done_ev[static_cast<size_t>(seq % kDoneRing)]);
    return e == cudaSuccess ? RIMURU_OK : fail(RIMURU_ERR_CUDA, cuda_msg("waiting for the cache", e));
  }

  // Change the number of slots.  Shrinking drops the least recently used
  // slots (evicting their experts) and frees their pages, which the
  // allocator merges back into larger pages; growing takes new pages from the
  // view's level and adds empty slots as the next victims.
  int resize(int new_cap) {
    if (new_cap == cap) return RIMURU_OK;
    int st = quiesce();
    if (st != RIMURU_OK) return st;
    Pool& pool = *v->pool;
    std::lock_guard<std::mutex> g(pool.mu);
    const int lvl = pool.level_of(v->page_bytes);
    std::vector<int> keep;  // surviving slots, most recent first
    for (int s = head; s >= 0; s = nxt[s]) keep.push_back(s);
    std::vector<int64_t> fresh;
    if (new_cap < cap) {
      for (int i = new_cap; i < cap; ++i) {
        const int s = keep[i];
        if (slot_key[s] >= 0) {
          for (int p = 0; p < 3; ++p) set_entry(slot_key[s] / E, slot_key[s] % E, p, -1);
          key_slot[slot_key[s]] = -1;
          st_.evictions += 1;
        }
        for (int p = 0; p < 3; ++p) pool.release(lvl, v->id, slot_page[static_cast<size_t>(s) * 3 + p]);
      }
      keep.resize(new_cap);
    } else {
      for (int i = 0; i < 3 * (new_cap - cap); ++i) {
        int64_t pg = -1;
        if (pool.alloc(lvl, v->id, &pg) != RIMURU_OK) {
          for (int64_t f : fresh) pool.release(lvl, v->id, f);
          return fail(RIMURU_ERR_OOM, "the pool has no room for " + std::to_string(new_cap) +
                                          " resident experts");
        }
        fresh.push_back(pg);
      }
    }
    // rebuild the slot arrays in recency order; new empty slots go last
    std::vector<int64_t> page2, seq2, op2;
    std::vector<int> key2;
    for (int s : keep) {
      for (int p = 0; p < 3; ++p) page2.push_back(slot_page[static_cast<size_t>(s) * 3 + p]);
      key2.push_back(slot_key[s]);
      seq2.push_back(slot_seq[s]);
      op2.push_back(slot_op[s]);
    }
    for (size_t i = 0; i < fresh.size(); i += 3) {
      for (int p = 0; p < 3; ++p) page2.push_back(fresh[i + p]);
      key2.push_back(-1);
      seq2.push_back(-1);
      op2.push_back(-1);
    }
    cap = new_cap;
    slot_page.swap(page2);
    slot_key.swap(key2);
    slot_seq.swap(seq2);
    slot_op.swap(op2);
    prv.assign(cap, -1);
    nxt.assign(cap, -1);
    head = tail = -1;
    for (int s = cap - 1; s >= 0; --s) push_front(s);  // slot 0 most recent
    std::fill(key_slot.begin(), key_slot.end(), -1);
    for (int s = 0; s < cap; ++s)
      if (slot_key[s] >= 0) key_slot[slot_key[s]] = s;
    return RIMURU_OK;
  }

  int mark_ready(int layer) {
    cudaError_t e = flush();
    if (e == cudaSuccess) e = cudaEventRecord(ready_ev[layer], copy);
    return e == cudaSuccess ? RIMURU_OK : fail(RIMURU_ERR_CUDA, cuda_msg("copy event", e));
  }
};

// Releases everything the cache holds (the object itself is freed by the caller).
void release_offload(Offload* o) {
  if (o->copy) cudaStreamSynchronize(o->copy);
  for (cudaEvent_t e : o->done_ev) if (e) cudaEventSynchronize(e), cudaEventDestroy(e);
  for (cudaEvent_t e : o->ready_ev) if (e) cudaEventDestroy(e);
  for (cudaEvent_t e : o->stage_ev) if (e) cudaEventSynchronize(e), cudaEventDestroy(e);
  if (o->offsets_ev) cudaEventDestroy(o->offsets_ev);
  for (int32_t* p : o->stage) if (p) cudaFreeHost(p);
  if (o->h_offsets) cudaFreeHost(o->h_offsets);
  if (o->own_copy && o->copy) cudaStreamDestroy(o->copy);
  if (o->v) {
    for (int s = 0; s < static_cast<int>(o->slot_key.size()); ++s)
      if (o->slot_key[s] >= 0)
        for (int p = 0; p < 3; ++p) o->set_entry(o->slot_key[s] / o->E, o->slot_key[s] % o->E, p, -1);
    std::lock_guard<std::mutex> g(o->v->pool->mu);
    const int lvl = o->v->pool->level_of(o->v->page_bytes);
    for (int64_t pg : o->slot_page)
      if (pg >= 0) o->v->pool->release(lvl, o->v->id, pg);
  }
}

}  // namespace rimuru

struct rimuru_offload_s {
  rimuru::Offload o;
};

using rimuru::fail;

extern "C" {

int rimuru_offload_create(rimuru_view_t view, const void* host_pages, int capacity_experts,
                          void* copy_stream, rimuru_offload_t* out) {
  rimuru::clear_error();
  if (!view || !host_pages || !out) return fail(RIMURU_ERR_ARG, "null argument");
  rimuru::View& v = view->v;
  if (!v.has_shape) return fail(RIMURU_ERR_STATE, "view has no MoE shape");
  if (capacity_experts <= 0 || capacity_experts > v.layers * v.experts)
    return fail(RIMURU_ERR_ARG, "capacity must be in [1, layers * experts]");
  for (int l = 0; l < v.layers; ++l)
    if (v.mapped_per_layer[l] != 0)
      return fail(RIMURU_ERR_STATE, "the view's page table must be empty: the cache maps pages");
  cudaPointerAttributes pa{};
  if (cudaPointerGetAttributes(&pa, host_pages) != cudaSuccess || pa.type != cudaMemoryTypeHost) {
    cudaGetLastError();
    return fail(RIMURU_ERR_ARG, "host_pages must be pinned host memory (cudaHostAlloc / registered)");
  }
  auto* h = new (std::nothrow) rimuru_offload_s;
  if (!h) return fail(RIMURU_ERR_OOM, "host allocation failed");
  rimuru::Offload& o = h->o;
  o.L = v.layers;
  o.E = v.experts;
  o.cap = capacity_experts;
  o.matrix_bytes = static_cast<uint64_t>(v.hidden) * v.inter * 2;
  o.host = static_cast<const uint8_t*>(host_pages);
  o.slot_page.assign(static_cast<size_t>(o.cap) * 3, -1);
  // pages for every slot, from the view's allocator
  {
    std::lock_guard<std::mutex> g(v.pool->mu);
    const int lvl = v.pool->level_of(v.page_bytes);
    for (size_t i = 0; i < o.slot_page.size(); ++i) {
      int64_t pg = -1;
      if (v.pool->alloc(lvl, v.id, &pg) != RIMURU_OK) {
        std::string msg = "pool cannot hold " + std::to_string(o.cap) + " resident experts";
        for (size_t j = 0; j < i; ++j) v.pool->release(lvl, v.id, o.slot_page[j]);
        delete h;
        return fail(RIMURU_ERR_OOM, msg);
      }
      o.slot_page[i] = pg;
    }
  }
  o.v = &v;
  o.vh = view;
  o.slot_key.assign(o.cap, -1);
  o.slot_seq.assign(o.cap, -1);
  o.slot_op.assign(o.cap, -1);
  o.key_slot.assign(static_cast<size_t>(o.L) * o.E, -1);
  o.prv.assign(o.cap, -1);
  o.nxt.assign(o.cap, -1);
  for (int s = 0; s < o.cap; ++s) o.push_front(s);  // slot 0 ends at the tail: first victim
  cudaError_t e = cudaSuccess;
  if (copy_stream) {
    o.copy = static_cast<cudaStream_t>(copy_stream);
  } else {
    e = cudaStreamCreateWithFlags(&o.copy, cudaStreamNonBlocking);
    o.own_copy = (e == cudaSuccess);
  }
  o.done_ev.assign(rimuru::kDoneRing, nullptr);
  o.ready_ev.assign(o.L, nullptr);
  o.ready_pending.assign(o.L, 0);
  for (auto& ev : o.done_ev)
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
  for (auto& ev : o.ready_ev)
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&o.offsets_ev, cudaEventDisableTiming);
  if (e == cudaSuccess) e = cudaMallocHost(&o.h_offsets, sizeof(int32_t) * (o.E + 1));
  o.stage.assign(rimuru::kStageRing, nullptr);
  o.stage_ev.assign(rimuru::kStageRing, nullptr);
  for (int i = 0; i < rimuru::kStageRing && e == cudaSuccess; ++i) {
    e = cudaMallocHost(&o.stage[i], sizeof(int32_t) * o.E * 3);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&o.stage_ev[i], cudaEventDisableTiming);
  }
  if (e == cudaSuccess && rimuru::ensure_device_state(&v) != RIMURU_OK) {
    std::string msg = rimuru_last_error();
    rimuru::release_offload(&o);
    delete h;
    return fail(RIMURU_ERR_CUDA, msg);
  }
  if (e != cudaSuccess) {
    rimuru::release_offload(&o);
    delete h;
    return fail(RIMURU_ERR_CUDA, rimuru::cuda_msg("offload set-up", e));
  }
  *out = h;
  return RIMURU_OK;
}

int rimuru_offload_destroy(rimuru_offload_t off) {
  rimuru::clear_error();
  if (!off) return fail(RIMURU_ERR_ARG, "null handle");
  rimuru::release_offload(&off->o);
  delete off;
  return RIMURU_OK;
}

int rimuru_offload_prefetch(rimuru_offload_t off, int layer, const int32_t* experts, int n) {
  rimuru::clear_error();
  if (!off || (n > 0 && !experts)) return fail(RIMURU_ERR_ARG, "null argument");
  rimuru::Offload& o = off->o;
  if (layer < 0 || layer >= o.L) return fail(RIMURU_ERR_RANGE, "layer out of range");
  if (n < 0 || n > o.E) return fail(RIMURU_ERR_ARG, "expert count out of range");
  o.op += 1;
  bool loaded = false;
  for (int i = 0; i < n; ++i) {
    if (experts[i] < 0 || experts[i] >= o.E) return fail(RIMURU_ERR_RANGE, "expert out of range");
    bool hit = false;
    int st = o.load(layer, experts[i], /*demand=*/false, &hit);
    if (st != RIMURU_OK) return st;
    loaded |= !hit;
  }
  return loaded ? o.mark_ready(layer) : RIMURU_OK;
}

int rimuru_offload_forward(rimuru_offload_t off, const void* x_bf16, const float* logits,
                           int num_tokens, int layer, void* out_bf16, void* workspace,
                           uint64_t workspace_bytes, void* stream_ptr) {
  rimuru::clear_error();
  if (!off) return fail(RIMURU_ERR_ARG, "null handle");
  rimuru::Offload& o = off->o;
  rimuru::View& v = *o.v;
  if (layer < 0 || layer >= o.L) return fail(RIMURU_ERR_RANGE, "layer out of range");
  if (num_tokens < 0 || num_tokens > (1 << 20))
    return fail(RIMURU_ERR_ARG, "num_tokens must be in [0, 2^20]");
  if (num_tokens == 0) return RIMURU_OK;
  if (!x_bf16 || !logits || !out_bf16 || !workspace) return fail(RIMURU_ERR_ARG, "null device pointer");
  auto mis = [](const void* p, uintptr_t a) { return reinterpret_cast<uintptr_t>(p) % a != 0; };
  if (mis(x_bf16, 16) || mis(logits, 16) || mis(out_bf16, 16))
    return fail(RIMURU_ERR_ALIGN, "x, logits and out must be 16-byte aligned");
  if (mis(workspace, 1024)) return fail(RIMURU_ERR_ALIGN, "workspace must be 1024-byte aligned");
  if (x_bf16 == out_bf16) return fail(RIMURU_ERR_ARG, "out may not alias x");
  rimuru_ws_layout Lw;
  int st = rimuru_moe_workspace_layout(o.vh, num_tokens, &Lw);
  if (st != RIMURU_OK) return st;
  if (workspace_bytes < Lw.total)
    return fail(RIMURU_ERR_WORKSPACE, "workspace needs " + std::to_string(Lw.total) + " bytes");

  int32_t* table = nullptr;
  int* err = nullptr;
  const CUtensorMap *w13 = nullptr, *w2 = nullptr;
  int device = 0;
  st = rimuru::view_device_table(&v, &table, &err, &w13, &w2, &device);
  if (st != RIMURU_OK) return st;
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess || sms <= 0)
    return fail(RIMURU_ERR_CUDA, "could not query the SM count");
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);

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
  a.layout = Lw;
  a.table = table + static_cast<size_t>(layer) * v.experts * 3;
  a.err = err;
  a.tm_w13 = w13;
  a.tm_w2 = w2;
  a.stream = stream;
  a.sm_count = sms;

  // 1. routing on the device, then the per-expert counts back to the host
  st = rimuru::launch_layer_route(a);
  if (st != RIMURU_OK) return st;
  cudaError_t e = cudaMemcpyAsync(o.h_offsets, a.ws + Lw.offsets, sizeof(int32_t) * (o.E + 1),
                                  cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaEventRecord(o.offsets_ev, stream);
  if (e == cudaSuccess) e = cudaEventSynchronize(o.offsets_ev);
  if (e != cudaSuccess) return fail(RIMURU_ERR_CUDA, rimuru::cuda_msg("routing read-back", e));

  // 2. every routed expert resident (demand copies for the misses)
  o.op += 1;
  o.next_layer = layer;
  std::vector<int> routed;
  routed.reserve(o.E);
  for (int ex = 0; ex < o.E; ++ex)
    if (o.h_offsets[ex + 1] > o.h_offsets[ex]) routed.push_back(ex);
  bool loaded = false;
  for (int ex : routed) {
    bool hit = false;
    st = o.load(layer, ex, /*demand=*/true, &hit);
    if (st != RIMURU_OK) return st;
    if (hit) o.st.hits += 1; else o.st.misses += 1;
    loaded |= !hit;
  }
  if (loaded && (st = o.mark_ready(layer)) != RIMURU_OK) return st;
  if (o.ready_pending[layer]) {
    e = cudaStreamWaitEvent(stream, o.ready_ev[layer], 0);
    o.ready_pending[layer] = 0;
    if (e != cudaSuccess) return fail(RIMURU_ERR_CUDA, rimuru::cuda_msg("waiting for copies", e));
  }

  // 3. this layer's page-table slice, uploaded from the staging ring
  {
    const int i = o.stage_next;
    o.stage_next = (o.stage_next + 1) % rimuru::kStageRing;
    e = cudaEventSynchronize(o.stage_ev[i]);  // the slice used 8 uploads ago has left
    const size_t n = static_cast<size_t>(o.E) * 3;
    if (e == cudaSuccess) {
      std::copy(v.page_table.begin() + static_cast<size_t>(layer) * n,
                v.page_table.begin() + static_cast<size_t>(layer + 1) * n, o.stage[i]);
      e = cudaMemcpyAsync(const_cast<int32_t*>(a.table), o.stage[i], n * sizeof(int32_t),
                          cudaMemcpyHostToDevice, stream);
    }
    if (e == cudaSuccess) e = cudaEventRecord(o.stage_ev[i], stream);
    if (e != cudaSuccess) return fail(RIMURU_ERR_CUDA, rimuru::cuda_msg("page-table upload", e));
  }

  // 4. the expert kernels, then this forward's completion event
  st = rimuru::launch_layer_experts(a, /*after_route=*/false);
  if (st != RIMURU_OK) return st;
  o.seq += 1;
  e = cudaEventRecord(o.done_ev[static_cast<size_t>(o.seq % rimuru::kDoneRing)], stream);
  if (e != cudaSuccess) return fail(RIMURU_ERR_CUDA, rimuru::cuda_msg("completion event", e));
  for (int ex : routed) o.slot_seq[o.key_slot[layer * o.E + ex]] = o.seq;
  o.st.forwards += 1;
  o.next_layer = (layer + 1) % o.L;
  return RIMURU_OK;
}

int rimuru_offload_set_policy(rimuru_offload_t off, int policy) {
  rimuru::clear_error();
  if (!off) return fail(RIMURU_ERR_ARG, "null handle");
  if (policy != RIMURU_EVICT_LRU && policy != RIMURU_EVICT_LAYER_CYCLE)
    return fail(RIMURU_ERR_ARG, "unknown eviction policy");
  off->o.policy = policy;
  return RIMURU_OK;
}

int rimuru_offload_resize(rimuru_offload_t off, int capacity_experts) {
  rimuru::clear_error();
  if (!off) return fail(RIMURU_ERR_ARG, "null handle");
  rimuru::Offload& o = off->o;
  if (capacity_experts <= 0 || capacity_experts > o.L * o.E)
    return fail(RIMURU_ERR_ARG, "capacity must be in [1, layers * experts]");
  return o.resize(capacity_experts);
}

int rimuru_offload_capacity(rimuru_offload_t off, int* capacity_experts) {
  rimuru::clear_error();
  if (!off || !capacity_experts) return fail(RIMURU_ERR_ARG, "null argument");
  *capacity_experts = off->o.cap;
  return RIMURU_OK;
}

int rimuru_adjust(rimuru_offload_t off, rimuru_view_t kv_view, int64_t kv_blocks_wanted,
                  int min_capacity, int max_capacity, int* capacity_out) {
  rimuru::clear_error();
  if (!off || !kv_view || !capacity_out) return fail(RIMURU_ERR_ARG, "null argument");
  rimuru::Offload& o = off->o;
  rimuru::View& kv = kv_view->v;
  rimuru::Pool& pool = *o.v->pool;
  if (kv.pool != &pool) return fail(RIMURU_ERR_ARG, "the KV view belongs to another pool");
  if (o.v->page_bytes != pool.huge_page_bytes)
    return fail(RIMURU_ERR_UNSUPPORTED, "the adjuster needs expert pages equal to huge pages");
  if (kv_blocks_wanted < 0 || min_capacity < 1 || max_capacity < min_capacity ||
      max_capacity > o.L * o.E)
    return fail(RIMURU_ERR_ARG, "bad demand or capacity bounds");
  int64_t free_huge = 0, kv_free = 0;
  {
    std::lock_guard<std::mutex> g(pool.mu);
    free_huge = static_cast<int64_t>(pool.levels[0].free_list.size());
    const int lk = pool.level_of(kv.page_bytes);
    if (lk > 0) kv_free = static_cast<int64_t>(pool.levels[lk].free_list.size());
  }
  const int64_t per_huge = static_cast<int64_t>(pool.huge_page_bytes / kv.page_bytes);
  const int64_t need_blocks = std::max<int64_t>(0, kv_blocks_wanted - kv_free);
  const int64_t need_huge = (need_blocks + per_huge - 1) / per_huge;
  const int64_t spare = free_huge - need_huge;  // huge pages beyond what KV will take
  int64_t target = o.cap;
  if (spare < 0) target = o.cap - (-spare + 2) / 3;  // each slot frees three huge pages
  else target = o.cap + spare / 3;
  target = std::max<int64_t>(min_capacity, std::min<int64_t>(max_capacity, target));
  int st = o.resize(static_cast<int>(target));
  if (st != RIMURU_OK) return st;
  *capacity_out = o.cap;
  return RIMURU_OK;
}

int rimuru_offload_stats(rimuru_offload_t off, rimuru_offload_counters* out) {
  rimuru::clear_error();
  if (!off || !out) return fail(RIMURU_ERR_ARG, "null argument");
  *out = off->o.st;
  return RIMURU_OK;
}

int rimuru_offload_resident(rimuru_offload_t off, int layer, int expert, int* slot) {
  rimuru::clear_error();
  if (!off || !slot) return fail(RIMURU_ERR_ARG, "null argument");
  rimuru::Offload& o = off->o;
  if (layer < 0 || layer >= o.L || expert < 0 || expert >= o.E)
    return fail(RIMURU_ERR_RANGE, "layer or expert out of range");
  *slot = o.key_slot[layer * o.E + expert];
  return RIMURU_OK;
}

}  // extern "C"
