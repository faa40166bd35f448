"""Workload-aware adjuster on a synthetic KV-demand trace.

Requests arrive and finish; each holds KV blocks of a KV view that shares the pool with the
expert cache.  Before the blocks of a step are allocated, rimuru_adjust shrinks the cache
(evicting least recently used experts and returning their pages, which merge back into
huge pages that the KV view then cuts into blocks) or grows it again when requests finish.
After every step the offloaded MoE layers still match the oracle, every page belongs to
exactly one owner, and the capacity follows the policy written out below.

Rimuru page: the adjuster moves pages between tensor types as demand changes (abstract;
explainer paragraph on the adjuster)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import workloads as wl
from gpu_harness import bf16_tensor, rel_err, to_f64
from oracle import Oracle
from paged_moe_shared_gb300 import rimuru as R
from paged_moe_shared_gb300.device_pool import DevicePool

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def expected_capacity(cap, free_huge, kv_free, wanted, per_huge, lo, hi):
    need_blocks = max(0, wanted - kv_free)
    need_huge = -(-need_blocks // per_huge)
    spare = free_huge - need_huge
    target = cap - (-spare + 2) // 3 if spare < 0 else cap + spare // 3
    return max(lo, min(hi, target))


def test_adjuster_follows_kv_demand_and_layers_stay_correct():
    shape = wl.MoEShape(H=256, I=128, E=8, k=2)
    L, T, huge_pages = 4, 16, 48
    pb = shape.H * shape.I * 2            # 64 KiB expert page = huge page
    kvb = 4096                            # 16 KV blocks per huge page
    per_huge = pb // kvb
    st = wl.offload_stack(shape, L, T, steps=7, seed=61)
    host = torch.from_numpy(st.host_pages).pin_memory()
    pool = DevicePool(huge_pages * pb, pb, DEV)
    ev = pool.view(pb)
    kv = pool.view(kvb)
    R.rimuru_view_set_moe_shape(ev, L, shape.E, shape.H, shape.I, shape.k, shape.renorm)
    pool.upload(wl.empty_pool(huge_pages * pb))
    lo, hi = 8, 12
    off = R.rimuru_offload_create(ev, host.data_ptr(), hi, 0)
    oracle = Oracle()
    ws_bytes = R.rimuru_moe_workspace_bytes(ev, T)
    ws_raw = torch.empty(ws_bytes + 1024, dtype=torch.uint8, device=DEV)
    ws_ptr = (ws_raw.data_ptr() + 1023) // 1024 * 1024
    stream = torch.cuda.current_stream().cuda_stream
    demand = [0, 96, 192, 336, 192, 48, 0]   # KV blocks held at each step
    per_request = 48
    requests = []                             # list of block lists
    caps = []
    try:
        for step, want in enumerate(demand):
            held = sum(len(r) for r in requests)
            # requests that finish leave first, newest last
            while held > want:
                for b in requests.pop(0):
                    R.rimuru_page_free(kv, b)
                held = sum(len(r) for r in requests)
            s0 = R.rimuru_pool_level_stats(pool.handle, 0)
            s1 = R.rimuru_pool_level_stats(pool.handle, 1)
            cap = R.rimuru_offload_capacity(off)
            exp = expected_capacity(cap, s0["pages_free"], s1["pages_free"], want - held,
                                    per_huge, lo, hi)
            got = R.rimuru_adjust(off, kv, want - held, lo, hi)
            assert got == exp == R.rimuru_offload_capacity(off), (step, got, exp)
            caps.append(got)
            while held < want:                 # new requests, one parent each where possible
                blocks = [R.rimuru_page_alloc_near(kv, R.NEW_GROUP)]
                while len(blocks) < per_request:
                    blocks.append(R.rimuru_page_alloc_near(kv, blocks[-1]))
                requests.append(blocks)
                held += per_request
            # ownership: expert view holds 3 pages per slot, KV view holds the blocks
            s0 = R.rimuru_pool_level_stats(pool.handle, 0)
            s1 = R.rimuru_pool_level_stats(pool.handle, 1)
            assert s0["pages_owned"] == 3 * got
            assert s1["pages_owned"] == held
            assert (s0["pages_free"] + s0["pages_owned"] + s0["pages_split"]) == huge_pages
            assert s0["pages_split"] * per_huge == s1["pages_free"] + s1["pages_owned"]
            # the layers still compute the right thing
            for l in range(L):
                x = bf16_tensor(st.x_bits[step][l])
                lg = torch.from_numpy(st.logits[step][l]).to(DEV)
                out = torch.empty_like(x)
                R.rimuru_offload_forward(off, x.data_ptr(), lg.data_ptr(), T, l, out.data_ptr(),
                                         ws_ptr, ws_bytes, stream)
                torch.cuda.synchronize()
                o = oracle.moe_forward(st.x_bits[step][l], st.logits[step][l], st.host_pages, pb,
                                       st.layer_table(l), shape.H, shape.I, shape.k, shape.renorm)
                assert rel_err(to_f64(out), o["out"]) <= 1e-2, (step, l)
            assert R.rimuru_get_device_error(ev, clear=True) == R.DEV_OK
    finally:
        R.rimuru_offload_destroy(off)
        pool.close()
    assert caps[0] == hi and min(caps) < hi and caps[-1] == hi, caps
