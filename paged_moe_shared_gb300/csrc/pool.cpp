// Shared page pool, memory views, the multi-level page allocator and the
// expert page table (host side only: nothing here touches device memory).
//
// Rimuru page (arXiv 2610.40305), abstract: a shared page pool, memory views
// with their own page size and page table, huge-page alignment and a
// multi-level page allocator that cuts pages and joins them back; Figure 7.
// Explainer page, memory-manager paragraph: huge pages are the LCM of the
// expert and SSM page sizes; a huge page is split into expert-sized pages and
// an expert-sized page into KV-sized pages, never a huge page directly into KV
// blocks; freeing walks the same chain back up.
#include <algorithm>
#include <cstring>
#include <limits>
#include <numeric>

#include "internal.h"

namespace rimuru {

namespace {
thread_local std::string g_last_error;
constexpr uint64_t kPoolAlign = 2ull << 20;  // pool base alignment
constexpr uint64_t kPageAlign = 256;         // every page size is a multiple of this
}  // namespace

int fail(int status, const std::string& msg) {
  g_last_error = msg;
  return status;
}
void clear_error() { g_last_error.clear(); }

// ------------------------------------------------------------------ levels

int Pool::level_of(uint64_t page_bytes) const {
  for (size_t i = 0; i < levels.size(); ++i)
    if (levels[i].page_bytes == page_bytes) return static_cast<int>(i);
  return -1;
}

int Pool::add_level(uint64_t page_bytes) {
  Level l;
  l.page_bytes = page_bytes;
  l.n_pages = static_cast<int64_t>(bytes / page_bytes);
  l.state.assign(static_cast<size_t>(l.n_pages), Level::ABSENT);
  l.owner.assign(static_cast<size_t>(l.n_pages), 0);
  auto pos = std::find_if(levels.begin(), levels.end(),
                          [&](const Level& o) { return o.page_bytes < page_bytes; });
  int idx = static_cast<int>(pos - levels.begin());
  levels.insert(pos, std::move(l));
  return idx;
}

// A FREE page of level lvl becomes SPLIT; its children at lvl + 1 become FREE.
int Pool::split_page(int lvl, int64_t id) {
  Level& L = levels[lvl];
  Level& C = levels[lvl + 1];
  L.state[id] = Level::SPLIT;
  L.free_list.erase(id);
  L.split += 1;
  int64_t per = static_cast<int64_t>(L.page_bytes / C.page_bytes);
  for (int64_t c = id * per; c < (id + 1) * per; ++c) {
    C.state[c] = Level::FREE;
    C.free_list.insert(c);
  }
  return RIMURU_OK;
}

// If every child of the parent of `id` (at level lvl) is FREE, the children
// vanish and the parent becomes FREE again; then the parent's own siblings
// are checked.  Level 0 pages have no parent.
void Pool::try_merge(int lvl, int64_t id) {
  while (lvl > 0) {
    Level& C = levels[lvl];
    Level& P = levels[lvl - 1];
    int64_t per = static_cast<int64_t>(P.page_bytes / C.page_bytes);
    int64_t parent = id / per;
    for (int64_t c = parent * per; c < (parent + 1) * per; ++c)
      if (C.state[c] != Level::FREE) return;
    for (int64_t c = parent * per; c < (parent + 1) * per; ++c) {
      C.state[c] = Level::ABSENT;
      C.free_list.erase(c);
    }
    P.state[parent] = Level::FREE;
    P.split -= 1;
    P.free_list.insert(parent);
    id = parent;
    lvl -= 1;
  }
}

int Pool::alloc(int lvl, int32_t owner_id, int64_t* id) {
  Level& L = levels[lvl];
  if (L.free_list.empty()) {
    if (lvl == 0) return fail(RIMURU_ERR_OOM, "pool has no free huge page");
    // take the lowest free page one level up (splitting further up if needed)
    Level& P = levels[lvl - 1];
    int64_t parent;
    if (!P.free_list.empty()) {
      parent = *P.free_list.begin();
    } else {
      int st = alloc(lvl - 1, 0, &parent);  // claim it, then turn it into a split page
      if (st != RIMURU_OK) return st;
      P.state[parent] = Level::FREE;
      P.owned -= 1;
    }
    split_page(lvl - 1, parent);
  }
  int64_t p = *L.free_list.begin();
  L.free_list.erase(L.free_list.begin());
  L.state[p] = Level::OWNED;
  L.owner[p] = owner_id;
  L.owned += 1;
  any_placed = true;
  *id = p;
  return RIMURU_OK;
}

int Pool::alloc_near(int lvl, int32_t owner_id, int64_t hint, int64_t* id) {
  Level& L = levels[lvl];
  if (lvl > 0 && hint == RIMURU_NEW_GROUP) {
    // first page of a group: cut a parent that nobody uses yet, if there is one
    Level& P = levels[lvl - 1];
    int64_t parent = -1;
    if (!P.free_list.empty()) {
      parent = *P.free_list.begin();
    } else if (lvl - 1 > 0) {  // cut a fresh parent out of the level above it
      int st = alloc(lvl - 1, 0, &parent);
      if (st != RIMURU_OK) parent = -1;
      else {
        P.state[parent] = Level::FREE;
        P.owned -= 1;
      }
    }
    if (parent >= 0) {
      split_page(lvl - 1, parent);
      const int64_t per = static_cast<int64_t>(P.page_bytes / L.page_bytes);
      const int64_t c = parent * per;
      L.free_list.erase(c);
      L.state[c] = Level::OWNED;
      L.owner[c] = owner_id;
      L.owned += 1;
      any_placed = true;
      *id = c;
      return RIMURU_OK;
    }
    clear_error();
    return alloc(lvl, owner_id, id);
  }
  if (lvl > 0 && hint >= 0 && hint < L.n_pages) {
    const int64_t per = static_cast<int64_t>(levels[lvl - 1].page_bytes / L.page_bytes);
    const int64_t parent = hint / per;
    for (int64_t c = parent * per; c < (parent + 1) * per; ++c) {
      if (L.state[c] == Level::FREE) {
        L.free_list.erase(c);
        L.state[c] = Level::OWNED;
        L.owner[c] = owner_id;
        L.owned += 1;
        any_placed = true;
        *id = c;
        return RIMURU_OK;
      }
    }
  }
  return alloc(lvl, owner_id, id);
}

int Pool::place(int lvl, int32_t owner_id, int64_t id) {
  Level& L = levels[lvl];
  if (id < 0 || id >= L.n_pages) return fail(RIMURU_ERR_RANGE, "page id out of range");
  if (L.state[id] == Level::ABSENT) {
    // the page above must be split first (and must itself be free or split)
    if (lvl == 0) return fail(RIMURU_ERR_STATE, "huge page state corrupt");
    int64_t per = static_cast<int64_t>(levels[lvl - 1].page_bytes / L.page_bytes);
    int64_t parent = id / per;
    Level& P = levels[lvl - 1];
    if (P.state[parent] == Level::ABSENT) {
      int st = place(lvl - 1, 0, parent);
      if (st != RIMURU_OK) return st;
      P.state[parent] = Level::FREE;
      P.owned -= 1;
      P.free_list.insert(parent);
    }
    if (P.state[parent] == Level::OWNED)
      return fail(RIMURU_ERR_STATE, "page lies inside a larger page that is owned");
    if (P.state[parent] == Level::FREE) split_page(lvl - 1, parent);
  }
  if (L.state[id] == Level::OWNED) return fail(RIMURU_ERR_STATE, "page already owned");
  if (L.state[id] == Level::SPLIT)
    return fail(RIMURU_ERR_STATE, "page is split into smaller pages in use");
  L.free_list.erase(id);
  L.state[id] = Level::OWNED;
  L.owner[id] = owner_id;
  L.owned += 1;
  any_placed = true;
  return RIMURU_OK;
}

int Pool::release(int lvl, int32_t owner_id, int64_t id) {
  Level& L = levels[lvl];
  if (id < 0 || id >= L.n_pages) return fail(RIMURU_ERR_RANGE, "page id out of range");
  if (L.state[id] != Level::OWNED || L.owner[id] != owner_id)
    return fail(RIMURU_ERR_STATE, "page is not owned by this view");
  L.state[id] = Level::FREE;
  L.owner[id] = 0;
  L.owned -= 1;
  L.free_list.insert(id);
  try_merge(lvl, id);
  return RIMURU_OK;
}

}  // namespace rimuru

using rimuru::fail;

// =================================================================== C ABI

extern "C" {

const char* rimuru_last_error(void) { return rimuru::g_last_error.c_str(); }

const char* rimuru_status_string(int s) {
  switch (s) {
    case RIMURU_OK: return "RIMURU_OK";
    case RIMURU_ERR_ARG: return "RIMURU_ERR_ARG";
    case RIMURU_ERR_ALIGN: return "RIMURU_ERR_ALIGN";
    case RIMURU_ERR_OOM: return "RIMURU_ERR_OOM";
    case RIMURU_ERR_UNMAPPED: return "RIMURU_ERR_UNMAPPED";
    case RIMURU_ERR_RANGE: return "RIMURU_ERR_RANGE";
    case RIMURU_ERR_WORKSPACE: return "RIMURU_ERR_WORKSPACE";
    case RIMURU_ERR_CUDA: return "RIMURU_ERR_CUDA";
    case RIMURU_ERR_DEVICE: return "RIMURU_ERR_DEVICE";
    case RIMURU_ERR_STATE: return "RIMURU_ERR_STATE";
    case RIMURU_ERR_UNSUPPORTED: return "RIMURU_ERR_UNSUPPORTED";
    default: return "RIMURU_UNKNOWN_STATUS";
  }
}

uint64_t rimuru_huge_page_bytes(uint64_t expert_page_bytes, uint64_t ssm_page_bytes) {
  if (expert_page_bytes == 0) return 0;
  if (ssm_page_bytes == 0) return expert_page_bytes;
  uint64_t g = std::gcd(expert_page_bytes, ssm_page_bytes);
  uint64_t a = expert_page_bytes / g;
  if (a > std::numeric_limits<uint64_t>::max() / ssm_page_bytes) return 0;
  return a * ssm_page_bytes;
}

int rimuru_pool_create(void* dev_base, uint64_t bytes, uint64_t huge_page_bytes,
                       rimuru_pool_t* out) {
  rimuru::clear_error();
  if (!out || !dev_base) return fail(RIMURU_ERR_ARG, "null pool base or output handle");
  if (bytes == 0 || huge_page_bytes == 0) return fail(RIMURU_ERR_ARG, "zero pool or page size");
  if (reinterpret_cast<uintptr_t>(dev_base) % rimuru::kPoolAlign != 0)
    return fail(RIMURU_ERR_ALIGN, "pool base must be 2 MiB aligned");
  if (huge_page_bytes % rimuru::kPageAlign != 0)
    return fail(RIMURU_ERR_ALIGN, "huge page size must be a multiple of 256 bytes");
  if (bytes % huge_page_bytes != 0)
    return fail(RIMURU_ERR_ALIGN, "pool size must be a multiple of the huge page size");
  auto* h = new (std::nothrow) rimuru_pool_s;
  if (!h) return fail(RIMURU_ERR_OOM, "host allocation failed");
  rimuru::Pool& p = h->p;
  p.base = dev_base;
  p.bytes = bytes;
  p.huge_page_bytes = huge_page_bytes;
  p.add_level(huge_page_bytes);
  rimuru::Level& top = p.levels[0];
  for (int64_t i = 0; i < top.n_pages; ++i) {
    top.state[i] = rimuru::Level::FREE;
    top.free_list.insert(i);
  }
  *out = h;
  return RIMURU_OK;
}

int rimuru_pool_destroy(rimuru_pool_t pool) {
  rimuru::clear_error();
  if (!pool) return fail(RIMURU_ERR_ARG, "null pool");
  {
    std::lock_guard<std::mutex> g(pool->p.mu);
    if (!pool->p.views.empty()) return fail(RIMURU_ERR_STATE, "pool still has views");
  }
  delete pool;
  return RIMURU_OK;
}

int rimuru_pool_num_levels(rimuru_pool_t pool, int* levels) {
  rimuru::clear_error();
  if (!pool || !levels) return fail(RIMURU_ERR_ARG, "null argument");
  std::lock_guard<std::mutex> g(pool->p.mu);
  *levels = static_cast<int>(pool->p.levels.size());
  return RIMURU_OK;
}

int rimuru_pool_level_stats(rimuru_pool_t pool, int level, rimuru_level_stats* out) {
  rimuru::clear_error();
  if (!pool || !out) return fail(RIMURU_ERR_ARG, "null argument");
  std::lock_guard<std::mutex> g(pool->p.mu);
  if (level < 0 || level >= static_cast<int>(pool->p.levels.size()))
    return fail(RIMURU_ERR_RANGE, "level out of range");
  const rimuru::Level& L = pool->p.levels[level];
  out->page_bytes = L.page_bytes;
  out->pages_total = L.n_pages;
  out->pages_free = static_cast<int64_t>(L.free_list.size());
  out->pages_owned = L.owned;
  out->pages_split = L.split;
  return RIMURU_OK;
}

int rimuru_view_create(rimuru_pool_t pool, uint64_t page_bytes, rimuru_view_t* out) {
  rimuru::clear_error();
  if (!pool || !out) return fail(RIMURU_ERR_ARG, "null argument");
  rimuru::Pool& p = pool->p;
  if (page_bytes == 0 || page_bytes % rimuru::kPageAlign != 0)
    return fail(RIMURU_ERR_ALIGN, "view page size must be a positive multiple of 256 bytes");
  if (p.huge_page_bytes % page_bytes != 0)
    return fail(RIMURU_ERR_ALIGN, "view page size must divide the huge page size");
  std::lock_guard<std::mutex> g(p.mu);
  int lvl = p.level_of(page_bytes);
  if (lvl < 0) {
    // the new size must sit in the divisibility chain of the existing levels
    for (const auto& L : p.levels) {
      bool ok = (L.page_bytes > page_bytes) ? (L.page_bytes % page_bytes == 0)
                                            : (page_bytes % L.page_bytes == 0);
      if (!ok)
        return fail(RIMURU_ERR_ALIGN, "view page size breaks the divisibility chain of the pool");
    }
    if (p.any_placed)
      return fail(RIMURU_ERR_STATE, "a view of a new page size must be created before pages are placed");
    p.add_level(page_bytes);
  }
  auto* h = new (std::nothrow) rimuru_view_s;
  if (!h) return fail(RIMURU_ERR_OOM, "host allocation failed");
  rimuru::View& v = h->v;
  v.pool = &p;
  v.id = p.next_view_id++;
  v.page_bytes = page_bytes;
  v.n_pages = static_cast<int64_t>(p.bytes / page_bytes);
  p.views.push_back(&v);
  *out = h;
  return RIMURU_OK;
}

int rimuru_view_destroy(rimuru_view_t view) {
  rimuru::clear_error();
  if (!view) return fail(RIMURU_ERR_ARG, "null view");
  rimuru::View& v = view->v;
  rimuru::Pool& p = *v.pool;
  rimuru::destroy_device_state(&v);
  {
    std::lock_guard<std::mutex> g(p.mu);
    int lvl = p.level_of(v.page_bytes);
    rimuru::Level& L = p.levels[lvl];
    for (int64_t i = 0; i < L.n_pages; ++i)
      if (L.state[i] == rimuru::Level::OWNED && L.owner[i] == v.id) p.release(lvl, v.id, i);
    p.views.erase(std::find(p.views.begin(), p.views.end(), &v));
  }
  delete view;
  return RIMURU_OK;
}

int rimuru_view_info(rimuru_view_t view, int64_t* num_pages, uint64_t* page_bytes) {
  rimuru::clear_error();
  if (!view) return fail(RIMURU_ERR_ARG, "null view");
  if (num_pages) *num_pages = view->v.n_pages;
  if (page_bytes) *page_bytes = view->v.page_bytes;
  return RIMURU_OK;
}

int rimuru_page_alloc(rimuru_view_t view, int64_t* page_id) {
  rimuru::clear_error();
  if (!view || !page_id) return fail(RIMURU_ERR_ARG, "null argument");
  rimuru::View& v = view->v;
  std::lock_guard<std::mutex> g(v.pool->mu);
  return v.pool->alloc(v.pool->level_of(v.page_bytes), v.id, page_id);
}

int rimuru_page_alloc_near(rimuru_view_t view, int64_t hint_page, int64_t* page_id) {
  rimuru::clear_error();
  if (!view || !page_id) return fail(RIMURU_ERR_ARG, "null argument");
  rimuru::View& v = view->v;
  std::lock_guard<std::mutex> g(v.pool->mu);
  return v.pool->alloc_near(v.pool->level_of(v.page_bytes), v.id, hint_page, page_id);
}

int rimuru_pool_fragmentation(rimuru_pool_t pool, int level, int64_t* partial_parents,
                              int64_t* stranded_free) {
  rimuru::clear_error();
  if (!pool || !partial_parents || !stranded_free) return fail(RIMURU_ERR_ARG, "null argument");
  rimuru::Pool& p = pool->p;
  std::lock_guard<std::mutex> g(p.mu);
  if (level < 1 || level >= static_cast<int>(p.levels.size()))
    return fail(RIMURU_ERR_RANGE, "level must name a level that is cut from a parent");
  const rimuru::Level& C = p.levels[level];
  const rimuru::Level& P = p.levels[level - 1];
  const int64_t per = static_cast<int64_t>(P.page_bytes / C.page_bytes);
  int64_t partial = 0, stranded = 0;
  for (int64_t q = 0; q < P.n_pages; ++q) {
    if (P.state[q] != rimuru::Level::SPLIT) continue;
    int64_t nfree = 0;
    for (int64_t c = q * per; c < (q + 1) * per; ++c) nfree += (C.state[c] == rimuru::Level::FREE);
    if (nfree > 0) {  // a split parent with free children cannot be merged back yet
      partial += 1;
      stranded += nfree;
    }
  }
  *partial_parents = partial;
  *stranded_free = stranded;
  return RIMURU_OK;
}

int rimuru_page_place(rimuru_view_t view, int64_t page_id) {
  rimuru::clear_error();
  if (!view) return fail(RIMURU_ERR_ARG, "null view");
  rimuru::View& v = view->v;
  std::lock_guard<std::mutex> g(v.pool->mu);
  return v.pool->place(v.pool->level_of(v.page_bytes), v.id, page_id);
}

int rimuru_page_free(rimuru_view_t view, int64_t page_id) {
  rimuru::clear_error();
  if (!view) return fail(RIMURU_ERR_ARG, "null view");
  rimuru::View& v = view->v;
  if (page_id >= 0 && page_id < static_cast<int64_t>(v.map_count.size()) && v.map_count[page_id] > 0)
    return fail(RIMURU_ERR_STATE, "page is still mapped as an expert projection");
  std::lock_guard<std::mutex> g(v.pool->mu);
  return v.pool->release(v.pool->level_of(v.page_bytes), v.id, page_id);
}

int rimuru_page_owned(rimuru_view_t view, int64_t page_id, int* owned) {
  rimuru::clear_error();
  if (!view || !owned) return fail(RIMURU_ERR_ARG, "null argument");
  rimuru::View& v = view->v;
  std::lock_guard<std::mutex> g(v.pool->mu);
  const rimuru::Level& L = v.pool->levels[v.pool->level_of(v.page_bytes)];
  if (page_id < 0 || page_id >= L.n_pages) return fail(RIMURU_ERR_RANGE, "page id out of range");
  *owned = (L.state[page_id] == rimuru::Level::OWNED && L.owner[page_id] == v.id) ? 1 : 0;
  return RIMURU_OK;
}

int rimuru_view_set_decode_tokens(rimuru_view_t view, int max_tokens) {
  rimuru::clear_error();
  if (!view) return fail(RIMURU_ERR_ARG, "null view");
  if (max_tokens < 0 || max_tokens > 4) return fail(RIMURU_ERR_ARG, "max_tokens must be in [0, 4]");
  view->v.decode_max_tokens = max_tokens;
  return RIMURU_OK;
}

int rimuru_view_set_moe_shape(rimuru_view_t view, int layers, int experts, int hidden, int inter,
                              int top_k, int renorm) {
  rimuru::clear_error();
  if (!view) return fail(RIMURU_ERR_ARG, "null view");
  rimuru::View& v = view->v;
  if (v.has_shape) return fail(RIMURU_ERR_STATE, "view already has an MoE shape");
  if (layers <= 0 || experts <= 0 || hidden <= 0 || inter <= 0 || top_k <= 0)
    return fail(RIMURU_ERR_ARG, "shape values must be positive");
  if (hidden % 128 != 0 || inter % 128 != 0)
    return fail(RIMURU_ERR_UNSUPPORTED, "hidden and inter must be multiples of 128");
  if (hidden % 256 != 0)
    return fail(RIMURU_ERR_UNSUPPORTED, "hidden must be a multiple of 256 (down-projection tile)");
  if (experts > 512) return fail(RIMURU_ERR_UNSUPPORTED, "at most 512 experts");
  if (top_k > experts || top_k > 32) return fail(RIMURU_ERR_UNSUPPORTED, "top_k must be <= min(experts, 32)");
  if (static_cast<uint64_t>(hidden) * static_cast<uint64_t>(inter) * 2u > v.page_bytes)
    return fail(RIMURU_ERR_UNSUPPORTED, "one projection must fit in one page of the view");
  if (v.n_pages > std::numeric_limits<int32_t>::max())
    return fail(RIMURU_ERR_UNSUPPORTED, "view has too many pages for an int32 page table");
  v.layers = layers;
  v.experts = experts;
  v.hidden = hidden;
  v.inter = inter;
  v.top_k = top_k;
  v.renorm = renorm ? 1 : 0;
  v.page_table.assign(static_cast<size_t>(layers) * experts * 3, -1);
  v.mapped_per_layer.assign(static_cast<size_t>(layers), 0);
  v.map_count.assign(static_cast<size_t>(v.n_pages), 0);
  v.table_dirty = true;
  v.has_shape = true;
  return RIMURU_OK;
}

static int check_entry(const rimuru::View& v, int layer, int expert, int proj) {
  if (!v.has_shape) return fail(RIMURU_ERR_STATE, "view has no MoE shape");
  if (layer < 0 || layer >= v.layers || expert < 0 || expert >= v.experts || proj < 0 || proj > 2)
    return fail(RIMURU_ERR_RANGE, "layer, expert or projection out of range");
  return RIMURU_OK;
}

int rimuru_expert_map(rimuru_view_t view, int layer, int expert, int proj, int64_t page_id) {
  rimuru::clear_error();
  if (!view) return fail(RIMURU_ERR_ARG, "null view");
  rimuru::View& v = view->v;
  int st = check_entry(v, layer, expert, proj);
  if (st != RIMURU_OK) return st;
  if (page_id < 0 || page_id >= v.n_pages) return fail(RIMURU_ERR_RANGE, "page id out of range");
  {
    std::lock_guard<std::mutex> g(v.pool->mu);
    const rimuru::Level& L = v.pool->levels[v.pool->level_of(v.page_bytes)];
    if (L.state[page_id] != rimuru::Level::OWNED || L.owner[page_id] != v.id)
      return fail(RIMURU_ERR_STATE, "page is not owned by this view");
  }
  st = rimuru::wait_table_upload(&v);
  if (st != RIMURU_OK) return st;
  size_t at = (static_cast<size_t>(layer) * v.experts + expert) * 3 + proj;
  int32_t old = v.page_table[at];
  if (old >= 0) v.map_count[old] -= 1;
  else v.mapped_per_layer[layer] += 1;
  v.page_table[at] = static_cast<int32_t>(page_id);
  v.map_count[page_id] += 1;
  v.table_dirty = true;
  return RIMURU_OK;
}

int rimuru_expert_unmap(rimuru_view_t view, int layer, int expert, int proj) {
  rimuru::clear_error();
  if (!view) return fail(RIMURU_ERR_ARG, "null view");
  rimuru::View& v = view->v;
  int st = check_entry(v, layer, expert, proj);
  if (st != RIMURU_OK) return st;
  st = rimuru::wait_table_upload(&v);
  if (st != RIMURU_OK) return st;
  size_t at = (static_cast<size_t>(layer) * v.experts + expert) * 3 + proj;
  int32_t old = v.page_table[at];
  if (old >= 0) {
    v.map_count[old] -= 1;
    v.mapped_per_layer[layer] -= 1;
    v.page_table[at] = -1;
    v.table_dirty = true;
  }
  return RIMURU_OK;
}

int rimuru_expert_lookup(rimuru_view_t view, int layer, int expert, int proj, int64_t* page_id) {
  rimuru::clear_error();
  if (!view || !page_id) return fail(RIMURU_ERR_ARG, "null argument");
  rimuru::View& v = view->v;
  int st = check_entry(v, layer, expert, proj);
  if (st != RIMURU_OK) return st;
  *page_id = v.page_table[(static_cast<size_t>(layer) * v.experts + expert) * 3 + proj];
  return RIMURU_OK;
}

}  // extern "C"
