/*
 * rimuru.h - C ABI of the GB300 paged fused-MoE library (librimuru.so).
 *
 * The library implements one hot path of Rimuru ("Rimuru: Unified Memory
 * Management for Modern LLM Serving via Elastic Expert Offloading", arXiv
 * 2610.40305): a fused MoE layer whose expert projection matrices are read in
 * place from non-contiguous pages of one shared device pool, through an expert
 * memory view (a page size plus a page table), with no gather into a
 * contiguous buffer.  Around it sits the host-side page allocator that places
 * pages of several views in that pool (huge pages split into expert-sized
 * pages, expert-sized pages split into KV-sized pages, and merged back).
 *
 * Conventions for every function below:
 *  - Return value: RIMURU_OK (0) or a negative rimuru_status.  No function
 *    aborts the process; on failure a message is available from
 *    rimuru_last_error() on the calling thread.
 *  - Ownership: the caller owns all device memory it passes in (the pool, x,
 *    logits, out, workspace).  The library owns its host metadata and, per
 *    expert view with an MoE shape, one small device buffer (page table plus a
 *    device error word) allocated on first use and freed by
 *    rimuru_view_destroy().
 *  - Pointers named dev_* or documented as device pointers must be device
 *    memory of the current CUDA device; host pointers are plain host memory.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  Forward calls are asynchronous on that stream.
 *  - Handles are not safe to use concurrently from several threads unless
 *    stated; the pool serialises its own allocator calls with a lock.
 */
#ifndef RIMURU_H_
#define RIMURU_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct rimuru_pool_s* rimuru_pool_t;
typedef struct rimuru_view_s* rimuru_view_t;

typedef enum rimuru_status {
  RIMURU_OK = 0,
  RIMURU_ERR_ARG = -1,         /* null handle/pointer, negative or zero size, bad index */
  RIMURU_ERR_ALIGN = -2,       /* pointer or size does not meet the stated alignment */
  RIMURU_ERR_OOM = -3,         /* no free page at any level that could be split */
  RIMURU_ERR_UNMAPPED = -4,    /* a projection of the requested layer has no page */
  RIMURU_ERR_RANGE = -5,       /* page id, layer, expert or projection out of range */
  RIMURU_ERR_WORKSPACE = -6,   /* workspace smaller than rimuru_moe_workspace_bytes() */
  RIMURU_ERR_CUDA = -7,        /* a CUDA runtime or driver call failed */
  RIMURU_ERR_DEVICE = -8,      /* a kernel reported an error through the device error word */
  RIMURU_ERR_STATE = -9,       /* call not valid in the current state (see each function) */
  RIMURU_ERR_UNSUPPORTED = -10 /* shape outside what the kernels handle */
} rimuru_status;

/* Projection index inside one expert (Table 1 of the Rimuru page lists the
 * three projection matrices of an expert: w1 and w3 [hidden, inter], w2
 * [inter, hidden]). */
enum { RIMURU_PROJ_W1 = 0, RIMURU_PROJ_W3 = 1, RIMURU_PROJ_W2 = 2 };

/* Device error codes written by kernels (read with rimuru_get_device_error). */
enum {
  RIMURU_DEV_OK = 0,
  RIMURU_DEV_BAD_PAGE = 1,      /* a page-table entry outside the view: tile skipped */
  RIMURU_DEV_NONFINITE = 2,     /* a router logit was NaN or infinite */
  RIMURU_DEV_TIMEOUT = 3,       /* a bounded wait inside a kernel gave up */
  RIMURU_DEV_BAD_SHAPE = 4      /* device-side tables disagree with the launch shape */
};

/* ------------------------------------------------------------------ errors */

/* Message for the last failing call on this thread ("" if none).  The
 * string stays valid until the next library call on the same thread. */
const char* rimuru_last_error(void);

/* Name of a rimuru_status value ("RIMURU_ERR_ARG", ...). */
const char* rimuru_status_string(int status);

/* ------------------------------------------------------------------- pool */

/*
 * Shared page pool (Rimuru page, abstract: one pool of device pages that
 * tensors of different types share; explainer page, memory-manager
 * paragraph: the pool is cut into huge pages).
 *
 * dev_base          device pointer to `bytes` bytes owned by the caller; must
 *                   be 2 MiB aligned (over-allocate and align up).
 * bytes             pool size; a positive multiple of huge_page_bytes.
 * huge_page_bytes   size of the top-level pages; a positive multiple of 256.
 *                   Use rimuru_huge_page_bytes() for the paper's rule.
 * out               receives the handle.
 * Errors: RIMURU_ERR_ARG (null, zero sizes), RIMURU_ERR_ALIGN (alignment or
 * bytes not a multiple of huge_page_bytes).
 * The pool never touches device memory: it only places pages.
 */
int rimuru_pool_create(void* dev_base, uint64_t bytes, uint64_t huge_page_bytes,
                       rimuru_pool_t* out);

/* Destroy a pool.  RIMURU_ERR_STATE while views of it still exist. */
int rimuru_pool_destroy(rimuru_pool_t pool);

/*
 * Huge-page size rule (explainer page, memory-manager paragraph: the pool is
 * cut into huge pages whose size is the least common multiple of the expert
 * page size and the state-space-model page size, so that no page of one type
 * straddles a huge-page boundary).  ssm_page_bytes == 0 means the model has
 * no SSM state and the result is expert_page_bytes.  Returns 0 on a zero
 * expert size or on overflow.
 */
uint64_t rimuru_huge_page_bytes(uint64_t expert_page_bytes, uint64_t ssm_page_bytes);

/* Allocator occupancy, for one level (page size) of the pool. */
typedef struct rimuru_level_stats {
  uint64_t page_bytes;   /* page size of this level */
  int64_t pages_total;   /* pool_bytes / page_bytes */
  int64_t pages_free;    /* pages of this level on its free list */
  int64_t pages_owned;   /* pages handed to views */
  int64_t pages_split;   /* pages cut into pages of the next level */
} rimuru_level_stats;

/* Number of levels (distinct page sizes: the huge page plus every view size). */
int rimuru_pool_num_levels(rimuru_pool_t pool, int* levels);
/* Stats of level `level` (0 = huge pages, larger = smaller pages). */
int rimuru_pool_level_stats(rimuru_pool_t pool, int level, rimuru_level_stats* out);

/* ------------------------------------------------------------------ views */

/*
 * Memory view (Rimuru page, abstract and Figure 6: every tensor type reads
 * the shared space with a page size and a page table of its own).  Page `i` of a view is the byte range
 * [i * page_bytes, (i + 1) * page_bytes) of the pool.
 *
 * page_bytes must divide huge_page_bytes, be a multiple of 256, and fit the
 * divisibility chain of the pool's other views (each level divides the one
 * above it).  A view whose size is new to the pool can only be created
 * before any page has been placed (RIMURU_ERR_STATE otherwise); views of an
 * existing size may be created at any time.
 */
int rimuru_view_create(rimuru_pool_t pool, uint64_t page_bytes, rimuru_view_t* out);

/* Destroy a view: frees its pages back to the allocator (merging them) and
 * its device page table.  The caller must make sure no forward using it is
 * still running on the GPU. */
int rimuru_view_destroy(rimuru_view_t view);

/* Pages in the view (pool_bytes / page_bytes) and its page size. */
int rimuru_view_info(rimuru_view_t view, int64_t* num_pages, uint64_t* page_bytes);

/*
 * Multi-level page allocator (Rimuru page, abstract, and Figure 7: pages
 * are cut into smaller pages and joined back; explainer page, memory-manager
 * paragraph: huge pages are cut into expert-sized pages, expert-sized pages
 * into KV-sized pages, huge pages never directly into KV blocks, and freeing
 * walks the same chain upwards).
 *
 * rimuru_page_alloc  hands out the lowest free page of the view's level,
 *                    splitting the lowest free page of the level above
 *                    (recursively) when the level has none.
 *                    RIMURU_ERR_OOM when nothing can be split.
 * rimuru_page_place  claims one given page id (splitting the pages above it
 *                    as needed).  RIMURU_ERR_STATE if any page containing it
 *                    or it itself is owned, or it is already split.
 * rimuru_page_free   returns a page the view owns; when every sibling cut
 *                    from the same parent is free they merge back into the
 *                    parent, recursively.  RIMURU_ERR_STATE if the view does
 *                    not own it or it is still mapped as an expert
 *                    projection.
 * The allocator only places pages: it never reads, writes or moves bytes.
 */
int rimuru_page_alloc(rimuru_view_t view, int64_t* page_id);
int rimuru_page_place(rimuru_view_t view, int64_t page_id);
int rimuru_page_free(rimuru_view_t view, int64_t page_id);

/*
 * Request-affine allocation (explainer page, memory-manager paragraph: the
 * allocator tries to cut one request's small pages from the same parent page
 * so that freeing them is simple).  Hands out the lowest free page cut from
 * the same parent page as `hint_page` (e.g. the request's previous KV
 * block).  hint_page == RIMURU_NEW_GROUP starts a group instead: the first
 * page of a parent that has not been cut yet (so the group can merge back
 * when it is freed).  When neither is possible, or hint_page == -1, it
 * behaves as rimuru_page_alloc.
 */
#define RIMURU_NEW_GROUP (-2)
int rimuru_page_alloc_near(rimuru_view_t view, int64_t hint_page, int64_t* page_id);

/* Fragmentation of level `level` (>= 1): parents (pages of level - 1) that
 * are split but still have free children, so cannot be merged back, and the
 * number of such free children. */
int rimuru_pool_fragmentation(rimuru_pool_t pool, int level, int64_t* partial_parents,
                              int64_t* stranded_free);

/* 1 if `page_id` of this view is currently owned by this view, else 0. */
int rimuru_page_owned(rimuru_view_t view, int64_t page_id, int* owned);

/* ------------------------------------------------------- expert page table */

/*
 * Declare that `view` holds the experts of an MoE model: `layers` layers of
 * `experts` experts, hidden size `hidden`, intermediate size `inter`, top
 * `top_k` routing with renormalised weights when `renorm` != 0.  Creates the
 * view's expert page table, int32 [layers][experts][3] (all unmapped).
 * Requirements: hidden and inter multiples of 128, hidden * inter * 2 <=
 * page_bytes (one projection per page), 1 <= top_k <= min(experts, 32),
 * experts <= 512.  RIMURU_ERR_UNSUPPORTED otherwise; RIMURU_ERR_STATE if the
 * view already has a shape.
 */
int rimuru_view_set_moe_shape(rimuru_view_t view, int layers, int experts, int hidden, int inter,
                              int top_k, int renorm);

/*
 * Batches of at most `max_tokens` tokens run the layer's decode path: three
 * kernels in place of five, for decode steps of one to a few tokens, where
 * each routed expert has a row or two and the layer is bound by its weight
 * bytes and by latency.  The path also needs T * top_k <= 64, the batch's x
 * rows within 32 KiB (T * hidden * 2) and its h within 96 KiB
 * (T * top_k * inter * 2); other batches take the general path whatever
 * `max_tokens` says.  0 turns the decode path off.  Default 0; at most 4.
 * RIMURU_ERR_ARG outside [0, 4].  The results of the two paths agree within
 * the layer's bf16 rounding, not bit for bit (their sums run in another
 * order).  Not thread-safe against a concurrent forward on the same view.
 */
int rimuru_view_set_decode_tokens(rimuru_view_t view, int max_tokens);

/*
 * Expert page table entry (explainer page, memory-manager paragraph: each
 * tensor type keeps a page table of its own; paragraph on the fused MoE
 * kernel: the kernel reads an expert's pages in place).  Maps projection `proj` (RIMURU_PROJ_W1/W3/W2) of `expert` in
 * `layer` to page `page_id` of this view, which must be owned by the view.
 * The projection is stored bf16 row-major starting at the page base: w1 and
 * w3 as [hidden][inter], w2 as [inter][hidden].
 * The device copy of the table is refreshed by the next forward call on its
 * stream; the caller must not call this while a forward that reads the old
 * entry may still be queued if it relies on the old mapping.
 */
int rimuru_expert_map(rimuru_view_t view, int layer, int expert, int proj, int64_t page_id);

/* Clear one entry (the page stays owned by the view). */
int rimuru_expert_unmap(rimuru_view_t view, int layer, int expert, int proj);

/* Read one entry (-1 if unmapped). */
int rimuru_expert_lookup(rimuru_view_t view, int layer, int expert, int proj, int64_t* page_id);

/* ---------------------------------------------------------------- forward */

/* Workspace (device bytes) a forward of `num_tokens` tokens needs; 0 on a
 * bad view.  The workspace holds routing ids/weights, the expert-sorted
 * permutation, the tile table and the bf16 intermediates. */
uint64_t rimuru_moe_workspace_bytes(rimuru_view_t view, int num_tokens);

/* Byte offsets of the named regions inside the workspace, for inspection
 * and tests (all relative to the workspace base).  A = num_tokens * top_k. */
typedef struct rimuru_ws_layout {
  uint64_t ids;        /* int32 [A]: expert of assignment f = t*k + j */
  uint64_t weights;    /* fp32 [A]: routing weight of assignment f */
  uint64_t chunk_hist; /* int32 [chunks][experts]: per-chunk expert counts */
  uint64_t offsets;    /* int32 [experts + 1]: expert e owns sorted rows offsets[e] .. offsets[e+1]-1 */
  uint64_t sorted;     /* int32 [A]: assignment f held by sorted row r (ascending f within an expert) */
  uint64_t inv;        /* int32 [A]: sorted row of assignment f */
  uint64_t tiles;      /* int32 [max_tiles][2]: (expert, first sorted row) of each 128-row block */
  uint64_t num_tiles;  /* int32: number of valid row blocks */
  uint64_t x_sorted;   /* bf16 [A][hidden]: x rows in sorted order, only when A <= 1024
                          (empty region otherwise: GEMM 1 then gathers rows from x) */
  uint64_t h;          /* bf16 [A][inter]: silu(x w1) * (x w3) in sorted order */
  uint64_t y;          /* bf16 [A][hidden]: h w2 in sorted order (unweighted) */
  uint64_t ptiles;     /* int32 [max_tiles][2]: (expert, first row) of each 256-row pair of blocks */
  uint64_t num_ptiles; /* int32: number of valid pair entries */
  uint64_t tile_cnt;   /* int32 [2][...]: split-K tile counters of the two GEMMs */
  uint64_t part;       /* fp32 partials: split-K tiles of the general path, or the
                          decode path's GEMM 1 partials (empty when neither runs) */
  uint64_t total;      /* bytes needed */
  int32_t chunks;      /* number of routing chunks */
  int32_t max_tiles;   /* capacity of the tile table */
  uint64_t plan;       /* int32 [1 + 3 * 64]: the decode path's routed experts (count,
                          then expert ids, first sorted rows, row counts); empty region
                          when the batch cannot take the decode path */
} rimuru_ws_layout;

int rimuru_moe_workspace_layout(rimuru_view_t view, int num_tokens, rimuru_ws_layout* out);

/*
 * The page-table-aware fused MoE layer (Rimuru page, abstract: the MoE
 * kernel reads expert weights from scattered pages directly, so nothing is
 * copied first; explainer page, paragraph on the fused MoE kernel).  For layer `layer` of `view`:
 *   routing  ids[t, 0..k-1]: the k largest logits of token t, larger first,
 *            lower expert index first on equal values; weights w[t, j] =
 *            softmax probabilities of the chosen experts, divided by their
 *            sum (renorm) or by the sum over all experts;
 *   grouping assignments f = t*k + j sorted by expert, ascending f within one
 *            expert;
 *   GEMM 1   h = silu(x w1_e) * (x w3_e), w1_e and w3_e read from their pages;
 *   GEMM 2   y = h w2_e, read from its page;
 *   combine  out[t] = sum_j w[t, j] * y[t*k + j], j ascending, in fp32.
 * Arguments:
 *   x_bf16      device, bf16 [num_tokens][hidden], 16-byte aligned
 *   logits      device, fp32 [num_tokens][experts], 16-byte aligned, finite
 *   num_tokens  >= 0 (0 returns at once), <= 1 << 20
 *   out_bf16    device, bf16 [num_tokens][hidden], 16-byte aligned; may not
 *               alias x
 *   workspace   device, >= rimuru_moe_workspace_bytes(view, num_tokens)
 *               bytes, 1024-byte aligned; contents on return are the
 *               intermediates described by rimuru_moe_workspace_layout()
 *   stream      cudaStream_t as void*
 * Every (layer, expert, projection) of `layer` must be mapped
 * (RIMURU_ERR_UNMAPPED otherwise).  The current device must be the one that
 * holds the pool (and the view's device state, once created): RIMURU_ERR_ARG
 * otherwise.  Host-side checks run before any launch; kernel-side problems set
 * the device error word and never trap.
 * CUDA graphs: the first forward after the view's mappings change copies the
 * page table to the device and may wait for an earlier copy; any other
 * forward only launches kernels on `stream` (with programmatic dependent
 * launch), so it can be recorded by stream capture and replayed.  Replays use
 * the pointers and the token count of the recorded call, and read the page
 * table as it is on the device when they run.
 */
int rimuru_moe_forward(const void* x_bf16, const float* logits, int num_tokens, rimuru_view_t view,
                       int layer, void* out_bf16, void* workspace, uint64_t workspace_bytes,
                       void* stream);

/*
 * rimuru_moe_forward for activations that live in host memory.  The pages
 * describe the layer on device-resident activations only; this entry point is
 * the same layer with the copies in and out made part of the call.
 * On `stream`, in order: x and logits are copied from the host buffers into
 * device staging regions at the end of the workspace, the layer runs exactly as
 * rimuru_moe_forward, and out is copied back to the host buffer.  The call
 * returns once everything is queued; out_host is valid after the stream has
 * been synchronised.
 * Arguments:
 *   x_host      host, bf16 [num_tokens][hidden]
 *   logits_host host, fp32 [num_tokens][experts], finite
 *   out_host    host, bf16 [num_tokens][hidden]
 *   workspace   device, >= rimuru_moe_host_workspace_bytes(view, num_tokens)
 *               bytes, 1024-byte aligned: the layer's workspace (same layout
 *               as rimuru_moe_workspace_layout) followed by the staging copies
 *               of x, logits and out
 *   others      as rimuru_moe_forward
 * Page-locked host buffers (cudaHostAlloc / cudaHostRegister) make the copies
 * asynchronous; with pageable buffers the copy calls may block the host until
 * they are done.  Host buffers must stay untouched until the stream is
 * synchronised.  Errors as rimuru_moe_forward; RIMURU_ERR_CUDA if a copy cannot
 * be queued.
 */
uint64_t rimuru_moe_host_workspace_bytes(rimuru_view_t view, int num_tokens);
int rimuru_moe_forward_host(const void* x_host, const float* logits_host, int num_tokens,
                            rimuru_view_t view, int layer, void* out_host, void* workspace,
                            uint64_t workspace_bytes, void* stream);

/*
 * The same layer as rimuru_moe_forward, for callers that cannot allocate
 * device memory.  The Rimuru pages have no counterpart of this entry point.
 *
 * Who needs it: a serving engine that hands nearly all device memory to its
 * own page pool at start-up (as a unified pool does) has nothing left for a
 * per-call cudaMalloc, and a host that accounts for every device byte itself
 * may not let a library allocate behind its back; cudaMalloc/cudaFree can
 * also synchronise the device, which a decode loop cannot afford.  Such a
 * caller passes only inputs and outputs here.
 *
 * Scratch: a fixed array of 16 MiB in the library's device memory (a
 * file-scope __device__ array), present on every GPU that loads the library
 * until the process exits.  It holds the routing tables, the sorted
 * activations, h, y, this layer's page table and an error word; the call
 * makes no cudaMalloc, cudaFree, cudaMallocHost or other allocating call.
 * A forward whose workspace (rimuru_moe_workspace_bytes) plus 10 KiB (1 KiB
 * of alignment slack, the error word's 1 KiB, 8 KiB of page table) does not
 * fit is rejected with RIMURU_ERR_WORKSPACE before anything is launched
 * (about 370 tokens at hidden 2048 / inter 768 / top-8).  The workspace part
 * starts on a 1 KiB boundary, as the ordinary forward requires.
 * First call on a device: it looks up the array's device address
 * (cudaGetSymbolAddress) with that device current and caches it; make that
 * first call before any stream capture.
 * Sharing: every call uses the same array and finds the previous call's
 * contents there (the kernels overwrite what they read; the error word is
 * cleared per call).  Calls whose kernels overlap on the GPU race on the
 * array: serialise them (one stream, or synchronise between streams).
 * Arguments are those of rimuru_moe_forward without the workspace, plus
 * dev_error: an optional device int that receives the first RIMURU_DEV_*
 * code a kernel reports (the caller zeroes it).  With dev_error NULL, error
 * reporting is off: the kernels record into a word of the scratch that no
 * call reads back, so a bad input (a non-finite logit) is not reported.
 * RIMURU_ERR_ARG when the current device is not the one that holds the pool;
 * num_tokens must be in [0, 2^20].
 */
int rimuru_moe_forward_noalloc(const void* x_bf16, const float* logits, int num_tokens,
                               rimuru_view_t view, int layer, void* out_bf16, int* dev_error,
                               void* stream);

/* ------------------------------------------------------ expert offloading */

/*
 * Expert offloading for a stack of layers (Rimuru page, Figure 1 panel b and
 * the explainer's motivation paragraph: experts kept in CPU memory with a
 * device cache of resident experts; Figure 8: two buffers so that expert
 * prefetch overlaps execution without a device-to-device copy).  Every
 * expert of every layer lives in pinned host memory; `capacity_experts` of
 * them are resident at a time, each in three pages of the expert view that
 * the cache allocates at creation.  A miss is copied host -> device on the
 * copy stream straight into the pages of the slot the eviction policy picks
 * (least recently used unless rimuru_offload_set_policy chooses otherwise;
 * the pages name no eviction policy).
 *
 * host_pages  pinned host memory (cudaHostAlloc or registered) holding
 *             layers * experts * 3 pages of the view's page size; projection
 *             p of expert e in layer l starts at page (l * experts + e) * 3 +
 *             p, bf16 row-major as for rimuru_expert_map.  Must outlive the
 *             cache and stay unchanged.
 * capacity_experts  resident experts (1 .. layers * experts); the pool must
 *             have 3 * capacity free pages of the view's size.
 * copy_stream stream for the host -> device copies (NULL: the cache creates
 *             one).
 * The view's page table must be empty: the cache maps and unmaps entries as
 * experts come and go.  Ordering is kept on the GPU: a slot is overwritten
 * only after the last forward that read it has finished, and a forward reads
 * a layer's slots only after their copies have landed.
 */
typedef struct rimuru_offload_s* rimuru_offload_t;

typedef struct rimuru_offload_counters {
  int64_t forwards;        /* rimuru_offload_forward calls */
  int64_t hits;            /* routed experts already resident when routing finished */
  int64_t misses;          /* routed experts copied in on demand */
  int64_t prefetch_loads;  /* experts copied in by rimuru_offload_prefetch */
  int64_t evictions;       /* resident experts replaced */
  int64_t bytes_h2d;       /* bytes copied host -> device */
} rimuru_offload_counters;

int rimuru_offload_create(rimuru_view_t view, const void* host_pages, int capacity_experts,
                          void* copy_stream, rimuru_offload_t* out);
/* Waits for the copy stream, unmaps and frees every slot page. */
int rimuru_offload_destroy(rimuru_offload_t off);

/* Queue copies on the copy stream that make the listed experts (host array
 * of n expert ids) of `layer` resident, evicting by the cache's policy.
 * Returns at once; call it for layer l + 1 before the forward of layer l so
 * the copies overlap that layer's kernels. */
int rimuru_offload_prefetch(rimuru_offload_t off, int layer, const int32_t* experts, int n);

/* The fused MoE layer of rimuru_moe_forward for `layer`, with experts brought
 * in as needed: routing runs first, the host reads the per-expert counts
 * back (this call waits for the routing kernels), every routed expert that
 * is not resident is copied in, the layer's page-table slice is uploaded,
 * and the expert kernels run once the copies they need have landed.
 * Arguments and errors as rimuru_moe_forward; RIMURU_ERR_OOM if one layer
 * routes to more experts than the capacity. */
int rimuru_offload_forward(rimuru_offload_t off, const void* x_bf16, const float* logits,
                           int num_tokens, int layer, void* out_bf16, void* workspace,
                           uint64_t workspace_bytes, void* stream);

int rimuru_offload_stats(rimuru_offload_t off, rimuru_offload_counters* out);

/* Eviction policy of the cache (the pages name none).
 *   RIMURU_EVICT_LRU          least recently used slot (the default).
 *   RIMURU_EVICT_LAYER_CYCLE  for stacks whose layers run in order 0, 1, ...,
 *                             L-1, 0, ... (every decode step of a model): the
 *                             slot whose expert's layer comes last counting on
 *                             from the next forward's layer (the layer after
 *                             the last forward, or that forward's own layer
 *                             while it loads), i.e. whose next use is furthest
 *                             away; empty slots first, ties to the least
 *                             recently used.  Where a cycle of layers does not
 *                             fit, LRU misses on every expert; this keeps a
 *                             fixed part of the cycle resident.
 * Slots claimed by the current prefetch or forward are never victims under
 * either policy.  Errors: RIMURU_ERR_ARG (null handle, unknown policy). */
enum { RIMURU_EVICT_LRU = 0, RIMURU_EVICT_LAYER_CYCLE = 1 };
int rimuru_offload_set_policy(rimuru_offload_t off, int policy);

/* Change the number of resident experts.  Shrinking waits (on the host) for
 * the cache's copies and for the last forward it recorded, evicts the least
 * recently used slots and frees their pages (the allocator merges them back
 * into huge pages); growing allocates pages of the view and adds empty
 * slots.  RIMURU_ERR_OOM (nothing changed) when the pool cannot grow the
 * cache.  Forwards must all run on one stream for the wait to cover them. */
int rimuru_offload_resize(rimuru_offload_t off, int capacity_experts);
int rimuru_offload_capacity(rimuru_offload_t off, int* capacity_experts);

/*
 * Workload-aware adjuster (Rimuru page, abstract and the explainer's
 * paragraph on the adjuster: pages move between tensor types with runtime
 * demand; the KV side grows when concurrency climbs and space returns to
 * the experts when requests finish, in step with the prefetching pipeline).
 * The pages give no policy; this one is: the KV view `kv_view` (same pool)
 * is about to need `kv_blocks_wanted` free blocks.  Free KV blocks count
 * first, then whole free huge pages; if they fall short the expert cache
 * shrinks by enough slots (three huge pages each), and whole free huge
 * pages beyond the KV need are given back to the cache, all within
 * [min_capacity, max_capacity].  Requires expert pages equal to the huge
 * page (the LCM rule gives that for both model shapes here).  Writes the
 * resulting capacity.
 */
int rimuru_adjust(rimuru_offload_t off, rimuru_view_t kv_view, int64_t kv_blocks_wanted,
                  int min_capacity, int max_capacity, int* capacity_out);
/* Slot holding (layer, expert), or -1 when it is not resident. */
int rimuru_offload_resident(rimuru_offload_t off, int layer, int expert, int* slot);

/* Device error word of the view (RIMURU_DEV_*).  Synchronises with the
 * device (cudaMemcpy) so call it after the forward's stream has been
 * synchronised; clear != 0 resets it to RIMURU_DEV_OK. */
int rimuru_get_device_error(rimuru_view_t view, int* code, int clear);

/* ------------------------------------------------------------- profiling */

/* Kernel slots of one forward.  A decode-sized batch (see
 * rimuru_view_set_decode_tokens) launches RIMURU_K_DECODE_GEMM1 (routing in
 * every CTA, GEMM 1 partials, W2 pages prefetched into L2),
 * RIMURU_K_DECODE_REDUCE (h) and RIMURU_K_DECODE_GEMM2 (GEMM 2 and the
 * combine).  Otherwise, when its T * top_k assignments fit one CTA (at most
 * 1024), a forward launches the kernel in slot RIMURU_K_ROUTE_ALIGN_GATHER
 * (routing, grouping and the gather of x rows), then GEMM 1, GEMM 2 and
 * combine; beyond that route, align, GEMM 1 (which gathers its rows from x
 * itself), GEMM 2 and combine.  No current launch sequence uses slot
 * RIMURU_K_GATHER (a separate gather kernel); the slot keeps the numbering
 * of the others and always reports 0 launches. */
enum {
  RIMURU_K_ROUTE = 0,
  RIMURU_K_ALIGN = 1,
  RIMURU_K_GATHER = 2,
  RIMURU_K_GEMM1 = 3,
  RIMURU_K_GEMM2 = 4,
  RIMURU_K_COMBINE = 5,
  RIMURU_K_ROUTE_ALIGN_GATHER = 6,
  RIMURU_K_DECODE_GEMM1 = 7,
  RIMURU_K_DECODE_REDUCE = 8,
  RIMURU_K_DECODE_GEMM2 = 9,
  RIMURU_K_COUNT = 10
};

/* Name of kernel slot `k` ("moe_route", ...), or NULL. */
const char* rimuru_kernel_name(int k);

/* Record a CUDA event pair around the launches of the kernels selected by
 * `kernel_mask` (bit RIMURU_K_* set) in the next `capacity` forwards of this
 * view; kernel_mask == 0 stops recording.  Enabling resets the records.  An
 * event pair between two kernels keeps the second from overlapping the
 * first, so bracket only the kernels being measured. */
int rimuru_profile_enable(rimuru_view_t view, int kernel_mask, int capacity);
/* The same, recording only every `every`-th forward (the first, then every
 * `every` forwards after it) until `capacity` forwards are recorded, so that a
 * long timed run is perturbed on a few of its forwards only.  every >= 1. */
int rimuru_profile_enable_sampled(rimuru_view_t view, int kernel_mask, int capacity, int every);

/* Launch count and summed device time (ms) of kernel slot `k` over the
 * recorded forwards (0 launches if `k` was not selected).  Synchronises on
 * the recorded events. */
int rimuru_profile_read(rimuru_view_t view, int k, int* launches, double* total_ms);

/* Number of SMs the kernels size their persistent grids for (0 if no
 * device is visible). */
int rimuru_device_sm_count(void);

/* Failure-path self-test (no counterpart in the pages; it checks this
 * library's own safety net).  Launches one kernel on the current device
 * whose threads wait on an mbarrier that nothing ever arrives on, using the
 * same bounded wait as every pipeline stage of the GEMM kernels, with a limit
 * of `timeout_us` microseconds (at most 2 s).  The kernel gives up, records
 * RIMURU_DEV_TIMEOUT in a device status word and returns; the call
 * synchronises the device and stores that word in *status_out (expected:
 * RIMURU_DEV_TIMEOUT).  Nothing traps and the context stays usable. */
int rimuru_selftest_bounded_wait(uint32_t timeout_us, int* status_out);

#ifdef __cplusplus
}
#endif

#endif /* RIMURU_H_ */
