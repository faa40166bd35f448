"""A shared page pool in device memory, driven through the C ABI.

PyTorch only provides the device bytes (one allocation, aligned up to 2 MiB) and the
host-to-device copy; every page is placed by the library's allocator and every expert
projection is entered in the expert view's page table with ``rimuru_expert_map``.
"""
from __future__ import annotations

import numpy as np
import torch

from . import rimuru as R

POOL_ALIGN = 2 << 20
NAN_BITS = 0x7FC0  # bf16 quiet NaN: free pages read as NaN


class DevicePool:
    def __init__(self, pool_bytes: int, huge_page_bytes: int, device="cuda"):
        self.raw = torch.empty(pool_bytes + POOL_ALIGN, dtype=torch.uint8, device=device)
        start = self.raw.data_ptr()
        off = (-start) % POOL_ALIGN
        self.base = start + off
        self.mem = self.raw[off:off + pool_bytes]
        self.pool_bytes = pool_bytes
        self.handle = R.rimuru_pool_create(self.base, pool_bytes, huge_page_bytes)
        self.views = []

    def view(self, page_bytes: int):
        v = R.rimuru_view_create(self.handle, page_bytes)
        self.views.append(v)
        return v

    def upload(self, image: np.ndarray, stream=None) -> None:
        """Copy a host image of the whole pool (uint8, pool_bytes long) to the device."""
        assert image.dtype == np.uint8 and image.nbytes == self.pool_bytes
        src = torch.from_numpy(image)
        self.mem.copy_(src, non_blocking=False)

    def close(self) -> None:
        for v in reversed(self.views):
            R.rimuru_view_destroy(v)
        self.views = []
        if self.handle is not None:
            R.rimuru_pool_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:  # noqa: BLE001 - best effort at interpreter exit
            pass


def load_workload(w, device="cuda", layer: int = 0, layers: int = 1, extra_pages: int = 0):
    """Place a ``workloads.Workload`` in a new device pool: views first (expert view, then
    the KV view of a mixed pool), then every page through the allocator, then the bytes.
    ``extra_pages`` adds free expert-view pages (NaN-filled) after the workload's pool.
    Returns (pool, expert_view, kv_view or None)."""
    assert w.huge_page_bytes == w.page_bytes or extra_pages == 0
    pool = DevicePool(w.pool_bytes + extra_pages * w.page_bytes, w.huge_page_bytes, device)
    ev = pool.view(w.page_bytes)
    kv = pool.view(w.kv_page_bytes) if w.kv_page_bytes else None
    s = w.shape
    R.rimuru_view_set_moe_shape(ev, layers, s.E, s.H, s.I, s.k, s.renorm)
    for e in range(s.E):
        for p in range(3):
            pid = int(w.page_table[e, p])
            R.rimuru_page_place(ev, pid)
            R.rimuru_expert_map(ev, layer, e, p, pid)
    if kv is not None:
        for pid in w.kv_pages.tolist():
            R.rimuru_page_place(kv, int(pid))
    if extra_pages:
        pool.mem[:w.pool_bytes].copy_(torch.from_numpy(w.pool))
        pool.mem[w.pool_bytes:].view(torch.int16).fill_(NAN_BITS)
    else:
        pool.upload(w.pool)
    return pool, ev, kv


def replicate_layers(pool: DevicePool, ev, w, layers: int) -> None:
    """Give layers 1 .. layers-1 their own copy of layer 0's expert pages: each projection is
    copied on the device into a page taken from the allocator and mapped there, so every
    layer holds the same weights at different addresses."""
    pb = w.page_bytes
    for layer in range(1, layers):
        for e in range(w.shape.E):
            for p in range(3):
                src = int(w.page_table[e, p])
                dst = R.rimuru_page_alloc(ev)
                pool.mem[dst * pb:(dst + 1) * pb].copy_(pool.mem[src * pb:(src + 1) * pb])
                R.rimuru_expert_map(ev, layer, e, p, dst)
