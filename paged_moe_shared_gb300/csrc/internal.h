// Host-side state shared by the allocator (pool.cpp) and the forward path
// (forward.cu).  Not part of the public ABI.
#pragma once

#include <atomic>
#include <cstdint>
#include <memory>
#include <mutex>
#include <set>
#include <string>
#include <vector>

#include "../../include/rimuru.h"

namespace rimuru {

constexpr int kDefaultDecodeTokens = 0;

// Thread-local error message, returned by rimuru_last_error().
int fail(int status, const std::string& msg);
void clear_error();

// One level of the pool: every page of one size.  Page i covers bytes
// [i * page_bytes, (i + 1) * page_bytes) of the pool.
struct Level {
  enum State : uint8_t { ABSENT = 0, FREE = 1, OWNED = 2, SPLIT = 3 };
  uint64_t page_bytes = 0;
  int64_t n_pages = 0;
  std::vector<uint8_t> state;   // State per page
  std::vector<int32_t> owner;   // view id when OWNED
  std::set<int64_t> free_list;  // ascending: lowest free page first
  int64_t owned = 0, split = 0;
};

struct View;

struct Pool {
  void* base = nullptr;
  uint64_t bytes = 0;
  uint64_t huge_page_bytes = 0;
  std::vector<Level> levels;  // levels[0] = huge pages, page size strictly decreasing
  std::vector<View*> views;
  int next_view_id = 1;
  bool any_placed = false;
  std::mutex mu;
  // Device that holds the pool bytes: -2 = not looked up yet, -1 = unknown (the
  // pointer is not a device allocation CUDA knows of; no check is made).
  std::atomic<int> device{-2};

  int level_of(uint64_t page_bytes) const;  // -1 if none
  int add_level(uint64_t page_bytes);       // keeps the chain ordered; returns its index
  // allocator primitives (caller holds mu)
  int alloc(int lvl, int32_t owner, int64_t* id);
  // Prefer a free page cut from the same parent as `hint` (lowest id first).
  int alloc_near(int lvl, int32_t owner, int64_t hint, int64_t* id);
  int place(int lvl, int32_t owner, int64_t id);
  int release(int lvl, int32_t owner, int64_t id);
  int split_page(int lvl, int64_t id);  // FREE page at lvl -> children FREE at lvl + 1
  void try_merge(int lvl, int64_t id);  // merge id's siblings back into the parent
};

// Device-side resources of one expert view (created on first forward).
struct DeviceState;

struct View {
  Pool* pool = nullptr;
  int32_t id = 0;
  int level = 0;
  uint64_t page_bytes = 0;
  int64_t n_pages = 0;

  // MoE shape (set once)
  bool has_shape = false;
  int layers = 0, experts = 0, hidden = 0, inter = 0, top_k = 0, renorm = 1;
  // batches of at most this many tokens take the three-kernel decode path
  int decode_max_tokens = kDefaultDecodeTokens;
  std::vector<int32_t> page_table;       // [layers][experts][3], -1 = unmapped
  std::vector<int32_t> mapped_per_layer;  // number of mapped entries per layer
  std::vector<int32_t> map_count;        // per page: how many entries point at it
  bool table_dirty = true;

  DeviceState* dev = nullptr;  // owned; freed by destroy_device_state
};

void destroy_device_state(View* v);
// RIMURU_OK when `device` (the caller's current device) holds the view's pool
// and, once the view has device state, that state; RIMURU_ERR_ARG otherwise.
int check_device(View* v, int device);
// Block until the last page-table upload has left the host staging copy.
int wait_table_upload(View* v);

}  // namespace rimuru

struct rimuru_pool_s {
  rimuru::Pool p;
};
struct rimuru_view_s {
  rimuru::View v;
};
