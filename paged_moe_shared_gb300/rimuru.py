"""ctypes binding of librimuru.so: the same entry points as ``include/rimuru.h``.

Argument marshalling only.  Every step of the layer runs in the library's CUDA
kernels; nothing here computes.  A non-zero status raises ``RimuruError`` with the
library's own message.  If the shared library is missing the import fails: there is
no fallback.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.environ.get("RIMURU_LIB", os.path.join(_HERE, "lib", "librimuru.so"))

OK = 0
ERR_ARG = -1
ERR_ALIGN = -2
ERR_OOM = -3
ERR_UNMAPPED = -4
ERR_RANGE = -5
ERR_WORKSPACE = -6
ERR_CUDA = -7
ERR_DEVICE = -8
ERR_STATE = -9
ERR_UNSUPPORTED = -10

PROJ_W1, PROJ_W3, PROJ_W2 = 0, 1, 2
NEW_GROUP = -2
DEV_OK, DEV_BAD_PAGE, DEV_NONFINITE, DEV_TIMEOUT, DEV_BAD_SHAPE = 0, 1, 2, 3, 4
(K_ROUTE, K_ALIGN, K_GATHER, K_GEMM1, K_GEMM2, K_COMBINE, K_ROUTE_ALIGN_GATHER, K_DECODE_GEMM1,
 K_DECODE_REDUCE, K_DECODE_GEMM2, K_COUNT) = range(11)

# Every symbol include/rimuru.h declares.
EXPORTS = [
    "rimuru_last_error", "rimuru_status_string", "rimuru_pool_create", "rimuru_pool_destroy",
    "rimuru_huge_page_bytes", "rimuru_pool_num_levels", "rimuru_pool_level_stats",
    "rimuru_view_create", "rimuru_view_destroy", "rimuru_view_info", "rimuru_page_alloc",
    "rimuru_page_place", "rimuru_page_free", "rimuru_page_owned", "rimuru_view_set_moe_shape",
    "rimuru_view_set_decode_tokens",
    "rimuru_expert_map", "rimuru_expert_unmap", "rimuru_expert_lookup",
    "rimuru_moe_workspace_bytes", "rimuru_moe_workspace_layout", "rimuru_moe_forward",
    "rimuru_moe_forward_noalloc", "rimuru_moe_host_workspace_bytes", "rimuru_moe_forward_host",
    "rimuru_get_device_error", "rimuru_kernel_name", "rimuru_profile_enable",
    "rimuru_profile_enable_sampled",
    "rimuru_profile_read", "rimuru_device_sm_count", "rimuru_selftest_bounded_wait",
    "rimuru_offload_create", "rimuru_offload_destroy", "rimuru_offload_prefetch",
    "rimuru_offload_forward", "rimuru_offload_stats", "rimuru_offload_resident",
    "rimuru_offload_set_policy",
    "rimuru_page_alloc_near", "rimuru_pool_fragmentation", "rimuru_offload_resize",
    "rimuru_offload_capacity", "rimuru_adjust",
]


class RimuruError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{status_name(status)}: {msg}")
        self.status = status


class LevelStats(ctypes.Structure):
    _fields_ = [("page_bytes", ctypes.c_uint64), ("pages_total", ctypes.c_int64),
                ("pages_free", ctypes.c_int64), ("pages_owned", ctypes.c_int64),
                ("pages_split", ctypes.c_int64)]


class WsLayout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_uint64) for n in (
        "ids", "weights", "chunk_hist", "offsets", "sorted", "inv", "tiles", "num_tiles",
        "x_sorted", "h", "y", "ptiles", "num_ptiles", "tile_cnt", "part", "total")] + [
        ("chunks", ctypes.c_int32), ("max_tiles", ctypes.c_int32), ("plan", ctypes.c_uint64)]


class OffloadCounters(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in (
        "forwards", "hits", "misses", "prefetch_loads", "evictions", "bytes_h2d")]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"librimuru.so not built ({LIB_PATH}); run __graft_entry__.build()")
    lib = ctypes.CDLL(LIB_PATH)
    P, i32, i64, u64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_uint64
    sig = {
        "rimuru_last_error": ([], ctypes.c_char_p),
        "rimuru_status_string": ([i32], ctypes.c_char_p),
        "rimuru_pool_create": ([P, u64, u64, ctypes.POINTER(P)], i32),
        "rimuru_pool_destroy": ([P], i32),
        "rimuru_huge_page_bytes": ([u64, u64], u64),
        "rimuru_pool_num_levels": ([P, ctypes.POINTER(i32)], i32),
        "rimuru_pool_level_stats": ([P, i32, ctypes.POINTER(LevelStats)], i32),
        "rimuru_view_create": ([P, u64, ctypes.POINTER(P)], i32),
        "rimuru_view_destroy": ([P], i32),
        "rimuru_view_info": ([P, ctypes.POINTER(i64), ctypes.POINTER(u64)], i32),
        "rimuru_page_alloc": ([P, ctypes.POINTER(i64)], i32),
        "rimuru_page_place": ([P, i64], i32),
        "rimuru_page_alloc_near": ([P, i64, ctypes.POINTER(i64)], i32),
        "rimuru_pool_fragmentation": ([P, i32, ctypes.POINTER(i64), ctypes.POINTER(i64)], i32),
        "rimuru_page_free": ([P, i64], i32),
        "rimuru_page_owned": ([P, i64, ctypes.POINTER(i32)], i32),
        "rimuru_view_set_moe_shape": ([P, i32, i32, i32, i32, i32, i32], i32),
        "rimuru_view_set_decode_tokens": ([P, i32], i32),
        "rimuru_expert_map": ([P, i32, i32, i32, i64], i32),
        "rimuru_expert_unmap": ([P, i32, i32, i32], i32),
        "rimuru_expert_lookup": ([P, i32, i32, i32, ctypes.POINTER(i64)], i32),
        "rimuru_moe_workspace_bytes": ([P, i32], u64),
        "rimuru_moe_workspace_layout": ([P, i32, ctypes.POINTER(WsLayout)], i32),
        "rimuru_moe_forward": ([P, P, i32, P, i32, P, P, u64, P], i32),
        "rimuru_moe_forward_noalloc": ([P, P, i32, P, i32, P, P, P], i32),
        "rimuru_moe_host_workspace_bytes": ([P, i32], u64),
        "rimuru_moe_forward_host": ([P, P, i32, P, i32, P, P, u64, P], i32),
        "rimuru_get_device_error": ([P, ctypes.POINTER(i32), i32], i32),
        "rimuru_kernel_name": ([i32], ctypes.c_char_p),
        "rimuru_profile_enable": ([P, i32, i32], i32),
        "rimuru_profile_enable_sampled": ([P, i32, i32, i32], i32),
        "rimuru_profile_read": ([P, i32, ctypes.POINTER(i32), ctypes.POINTER(ctypes.c_double)], i32),
        "rimuru_device_sm_count": ([], i32),
        "rimuru_selftest_bounded_wait": ([ctypes.c_uint32, ctypes.POINTER(i32)], i32),
        "rimuru_offload_create": ([P, P, i32, P, ctypes.POINTER(P)], i32),
        "rimuru_offload_destroy": ([P], i32),
        "rimuru_offload_prefetch": ([P, i32, P, i32], i32),
        "rimuru_offload_forward": ([P, P, P, i32, i32, P, P, u64, P], i32),
        "rimuru_offload_stats": ([P, ctypes.POINTER(OffloadCounters)], i32),
        "rimuru_offload_set_policy": ([P, i32], i32),
        "rimuru_offload_resident": ([P, i32, i32, ctypes.POINTER(i32)], i32),
        "rimuru_offload_resize": ([P, i32], i32),
        "rimuru_offload_capacity": ([P, ctypes.POINTER(i32)], i32),
        "rimuru_adjust": ([P, P, i64, i32, i32, ctypes.POINTER(i32)], i32),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    return lib


lib = _load()


def status_name(status: int) -> str:
    return lib.rimuru_status_string(int(status)).decode()


def _check(status: int):
    if status != OK:
        raise RimuruError(status, lib.rimuru_last_error().decode())


def rimuru_last_error() -> str:
    return lib.rimuru_last_error().decode()


def rimuru_status_string(status: int) -> str:
    return status_name(status)


def rimuru_huge_page_bytes(expert_page_bytes: int, ssm_page_bytes: int = 0) -> int:
    return int(lib.rimuru_huge_page_bytes(expert_page_bytes, ssm_page_bytes))


def rimuru_pool_create(dev_base: int, nbytes: int, huge_page_bytes: int):
    h = ctypes.c_void_p()
    _check(lib.rimuru_pool_create(ctypes.c_void_p(dev_base), nbytes, huge_page_bytes, ctypes.byref(h)))
    return h


def rimuru_pool_destroy(pool) -> None:
    _check(lib.rimuru_pool_destroy(pool))


def rimuru_pool_num_levels(pool) -> int:
    n = ctypes.c_int()
    _check(lib.rimuru_pool_num_levels(pool, ctypes.byref(n)))
    return n.value


def rimuru_pool_level_stats(pool, level: int) -> dict:
    s = LevelStats()
    _check(lib.rimuru_pool_level_stats(pool, level, ctypes.byref(s)))
    return {f: getattr(s, f) for f, _ in LevelStats._fields_}


def rimuru_view_create(pool, page_bytes: int):
    h = ctypes.c_void_p()
    _check(lib.rimuru_view_create(pool, page_bytes, ctypes.byref(h)))
    return h


def rimuru_view_destroy(view) -> None:
    _check(lib.rimuru_view_destroy(view))


def rimuru_view_info(view):
    n, pb = ctypes.c_int64(), ctypes.c_uint64()
    _check(lib.rimuru_view_info(view, ctypes.byref(n), ctypes.byref(pb)))
    return n.value, pb.value


def rimuru_page_alloc(view) -> int:
    p = ctypes.c_int64()
    _check(lib.rimuru_page_alloc(view, ctypes.byref(p)))
    return p.value


def rimuru_page_alloc_near(view, hint_page: int) -> int:
    p = ctypes.c_int64()
    _check(lib.rimuru_page_alloc_near(view, hint_page, ctypes.byref(p)))
    return p.value


def rimuru_pool_fragmentation(pool, level: int):
    a, b = ctypes.c_int64(), ctypes.c_int64()
    _check(lib.rimuru_pool_fragmentation(pool, level, ctypes.byref(a), ctypes.byref(b)))
    return a.value, b.value


def rimuru_page_place(view, page_id: int) -> None:
    _check(lib.rimuru_page_place(view, page_id))


def rimuru_page_free(view, page_id: int) -> None:
    _check(lib.rimuru_page_free(view, page_id))


def rimuru_page_owned(view, page_id: int) -> bool:
    o = ctypes.c_int()
    _check(lib.rimuru_page_owned(view, page_id, ctypes.byref(o)))
    return bool(o.value)


def rimuru_view_set_moe_shape(view, layers: int, experts: int, hidden: int, inter: int,
                              top_k: int, renorm: bool = True) -> None:
    _check(lib.rimuru_view_set_moe_shape(view, layers, experts, hidden, inter, top_k, int(renorm)))


def rimuru_view_set_decode_tokens(view, max_tokens: int) -> None:
    _check(lib.rimuru_view_set_decode_tokens(view, max_tokens))


def rimuru_expert_map(view, layer: int, expert: int, proj: int, page_id: int) -> None:
    _check(lib.rimuru_expert_map(view, layer, expert, proj, page_id))


def rimuru_expert_unmap(view, layer: int, expert: int, proj: int) -> None:
    _check(lib.rimuru_expert_unmap(view, layer, expert, proj))


def rimuru_expert_lookup(view, layer: int, expert: int, proj: int) -> int:
    p = ctypes.c_int64()
    _check(lib.rimuru_expert_lookup(view, layer, expert, proj, ctypes.byref(p)))
    return p.value


def rimuru_moe_workspace_bytes(view, num_tokens: int) -> int:
    return int(lib.rimuru_moe_workspace_bytes(view, num_tokens))


def rimuru_moe_workspace_layout(view, num_tokens: int) -> dict:
    L = WsLayout()
    _check(lib.rimuru_moe_workspace_layout(view, num_tokens, ctypes.byref(L)))
    return {f: getattr(L, f) for f, _ in WsLayout._fields_}


def rimuru_moe_forward(x_ptr: int, logits_ptr: int, num_tokens: int, view, layer: int,
                       out_ptr: int, workspace_ptr: int, workspace_bytes: int,
                       stream: int = 0) -> None:
    """Pointers are raw device addresses (e.g. ``tensor.data_ptr()``); ``stream`` is a
    cudaStream_t as an integer (e.g. ``torch.cuda.current_stream().cuda_stream``)."""
    _check(lib.rimuru_moe_forward(ctypes.c_void_p(x_ptr), ctypes.c_void_p(logits_ptr), num_tokens,
                                  view, layer, ctypes.c_void_p(out_ptr),
                                  ctypes.c_void_p(workspace_ptr), workspace_bytes,
                                  ctypes.c_void_p(stream)))


def rimuru_moe_host_workspace_bytes(view, num_tokens: int) -> int:
    return int(lib.rimuru_moe_host_workspace_bytes(view, num_tokens))


def rimuru_moe_forward_host(x_host_ptr: int, logits_host_ptr: int, num_tokens: int, view,
                            layer: int, out_host_ptr: int, workspace_ptr: int,
                            workspace_bytes: int, stream: int = 0) -> None:
    """The forward on host buffers: x, logits and out are host addresses (page-locked for
    asynchronous copies); the copies in and out run on ``stream`` with the layer."""
    _check(lib.rimuru_moe_forward_host(ctypes.c_void_p(x_host_ptr),
                                       ctypes.c_void_p(logits_host_ptr), num_tokens, view, layer,
                                       ctypes.c_void_p(out_host_ptr),
                                       ctypes.c_void_p(workspace_ptr), workspace_bytes,
                                       ctypes.c_void_p(stream)))


def rimuru_moe_forward_noalloc(x_ptr: int, logits_ptr: int, num_tokens: int, view, layer: int,
                               out_ptr: int, dev_error_ptr: int = 0, stream: int = 0) -> None:
    """The forward without a workspace, for callers that cannot allocate device memory:
    scratch comes from the library's built-in 16 MiB device array.  ``dev_error_ptr`` is an
    optional device int32 address that receives the first kernel error code."""
    _check(lib.rimuru_moe_forward_noalloc(ctypes.c_void_p(x_ptr), ctypes.c_void_p(logits_ptr),
                                          num_tokens, view, layer, ctypes.c_void_p(out_ptr),
                                          ctypes.c_void_p(dev_error_ptr or None),
                                          ctypes.c_void_p(stream)))


def rimuru_get_device_error(view, clear: bool = False) -> int:
    c = ctypes.c_int()
    _check(lib.rimuru_get_device_error(view, ctypes.byref(c), int(clear)))
    return c.value


def rimuru_kernel_name(k: int):
    n = lib.rimuru_kernel_name(k)
    return n.decode() if n else None


PROFILE_ALL = (1 << K_COUNT) - 1


def rimuru_profile_enable(view, kernel_mask: int, capacity: int = 1024) -> None:
    """Bracket the kernels in ``kernel_mask`` (bit K_*) with CUDA events; 0 stops."""
    _check(lib.rimuru_profile_enable(view, int(kernel_mask), capacity))


def rimuru_profile_enable_sampled(view, kernel_mask: int, capacity: int, every: int) -> None:
    """Event pairs around the selected kernels of every ``every``-th forward only."""
    _check(lib.rimuru_profile_enable_sampled(view, int(kernel_mask), capacity, every))


def rimuru_profile_read(view, k: int):
    n, ms = ctypes.c_int(), ctypes.c_double()
    _check(lib.rimuru_profile_read(view, k, ctypes.byref(n), ctypes.byref(ms)))
    return n.value, ms.value


def rimuru_device_sm_count() -> int:
    return int(lib.rimuru_device_sm_count())


def rimuru_selftest_bounded_wait(timeout_us: int) -> int:
    """Run the bounded-wait self-test kernel; returns the device status it recorded."""
    st = ctypes.c_int()
    _check(lib.rimuru_selftest_bounded_wait(int(timeout_us), ctypes.byref(st)))
    return st.value


def rimuru_offload_create(view, host_pages_ptr: int, capacity_experts: int, copy_stream: int = 0):
    h = ctypes.c_void_p()
    _check(lib.rimuru_offload_create(view, ctypes.c_void_p(host_pages_ptr), capacity_experts,
                                     ctypes.c_void_p(copy_stream or None), ctypes.byref(h)))
    return h


def rimuru_offload_destroy(off) -> None:
    _check(lib.rimuru_offload_destroy(off))


def rimuru_offload_prefetch(off, layer: int, experts) -> None:
    arr = (ctypes.c_int32 * len(experts))(*[int(e) for e in experts])
    _check(lib.rimuru_offload_prefetch(off, layer, ctypes.cast(arr, ctypes.c_void_p), len(experts)))


def rimuru_offload_forward(off, x_ptr: int, logits_ptr: int, num_tokens: int, layer: int,
                           out_ptr: int, workspace_ptr: int, workspace_bytes: int,
                           stream: int = 0) -> None:
    _check(lib.rimuru_offload_forward(off, ctypes.c_void_p(x_ptr), ctypes.c_void_p(logits_ptr),
                                      num_tokens, layer, ctypes.c_void_p(out_ptr),
                                      ctypes.c_void_p(workspace_ptr), workspace_bytes,
                                      ctypes.c_void_p(stream)))


EVICT_LRU, EVICT_LAYER_CYCLE = 0, 1


def rimuru_offload_set_policy(off, policy: int) -> None:
    """Eviction policy of the offload cache: EVICT_LRU (default) or EVICT_LAYER_CYCLE."""
    _check(lib.rimuru_offload_set_policy(off, policy))


def rimuru_offload_stats(off) -> dict:
    c = OffloadCounters()
    _check(lib.rimuru_offload_stats(off, ctypes.byref(c)))
    return {f: getattr(c, f) for f, _ in OffloadCounters._fields_}


def rimuru_offload_resident(off, layer: int, expert: int) -> int:
    s = ctypes.c_int()
    _check(lib.rimuru_offload_resident(off, layer, expert, ctypes.byref(s)))
    return s.value


def rimuru_offload_resize(off, capacity_experts: int) -> None:
    _check(lib.rimuru_offload_resize(off, capacity_experts))


def rimuru_offload_capacity(off) -> int:
    c = ctypes.c_int()
    _check(lib.rimuru_offload_capacity(off, ctypes.byref(c)))
    return c.value


def rimuru_adjust(off, kv_view, kv_blocks_wanted: int, min_capacity: int, max_capacity: int) -> int:
    c = ctypes.c_int()
    _check(lib.rimuru_adjust(off, kv_view, kv_blocks_wanted, min_capacity, max_capacity,
                             ctypes.byref(c)))
    return c.value
