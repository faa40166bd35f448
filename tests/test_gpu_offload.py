"""Expert offloading: every layer's output against the oracle, and the cache's hit, miss,
prefetch and eviction counts against an independent model of the policy (least recently
used slot first; slots claimed by the same prefetch or forward are never evicted by it).

Rimuru page: experts kept in CPU memory with a device cache (Figure 1 panel b) and dual
buffers that overlap prefetch with execution (Figure 8).  The eviction policy is this
library's (the pages name none): least recently used, or the layer-cycle rule."""
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


class CacheModel:
    """Slots in recency order (index 0 = most recent); initially slot 0 is the oldest.
    Victims: the least recently used slot (LRU), or the slot whose layer comes last counting
    on from the next forward's layer (layer cycle), empty slots first, ties to the least
    recently used; never a slot claimed by the current operation."""

    def __init__(self, cap, policy=R.EVICT_LRU, L=1, E=1):
        self.order = list(range(cap - 1, -1, -1))
        self.slot_key = [None] * cap
        self.key_slot = {}
        self.claimed = {}
        self.op = 0
        self.policy, self.L, self.E = policy, L, E
        self.next_layer = 0
        self.c = dict(hits=0, misses=0, prefetch_loads=0, evictions=0, bytes_h2d=0, forwards=0)

    def _victim(self):
        free = [s for s in reversed(self.order) if self.claimed.get(s) != self.op]
        if not free:
            raise AssertionError("capacity too small")
        if self.policy == R.EVICT_LRU:
            return free[0]

        def dist(s):
            k = self.slot_key[s]
            return self.L if k is None else (k // self.E - self.next_layer) % self.L
        best = free[0]
        for s in free[1:]:
            if dist(s) > dist(best):
                best = s
        return best

    def _load(self, key, demand, nbytes):
        s = self.key_slot.get(key)
        if s is not None:
            self.order.remove(s)
            self.order.insert(0, s)
            self.claimed[s] = self.op
            return True
        s = self._victim()
        old = self.slot_key[s]
        if old is not None:
            del self.key_slot[old]
            self.c["evictions"] += 1
        self.slot_key[s] = key
        self.key_slot[key] = s
        self.claimed[s] = self.op
        self.order.remove(s)
        self.order.insert(0, s)
        self.c["bytes_h2d"] += nbytes
        if not demand:
            self.c["prefetch_loads"] += 1
        return False

    def prefetch(self, keys, nbytes):
        self.op += 1
        for k in keys:
            self._load(k, False, nbytes)

    def forward(self, layer, keys, nbytes):
        self.op += 1
        self.next_layer = layer
        for k in keys:
            hit = self._load(k, True, nbytes)
            self.c["hits" if hit else "misses"] += 1
        self.c["forwards"] += 1
        self.next_layer = (layer + 1) % self.L


def run_stack(st: wl.OffloadStack, cap: int, prefetch: bool, policy=R.EVICT_LRU):
    s = st.shape
    E = s.E
    pb = st.page_bytes
    oracle = Oracle()
    host = torch.from_numpy(st.host_pages).pin_memory()
    pool = DevicePool((3 * cap + 5) * pb, pb, DEV)
    ev = pool.view(pb)
    R.rimuru_view_set_moe_shape(ev, st.L, E, s.H, s.I, s.k, s.renorm)
    pool.upload(wl.empty_pool((3 * cap + 5) * pb))
    off = R.rimuru_offload_create(ev, host.data_ptr(), cap, 0)
    R.rimuru_offload_set_policy(off, policy)
    model = CacheModel(cap, policy, st.L, E)
    nbytes = 3 * s.H * s.I * 2
    ws_bytes = R.rimuru_moe_workspace_bytes(ev, st.T)
    ws_raw = torch.empty(ws_bytes + 1024, dtype=torch.uint8, device=DEV)
    ws_ptr = (ws_raw.data_ptr() + 1023) // 1024 * 1024
    stream = torch.cuda.current_stream().cuda_stream
    prev_routed = {}
    worst = 0.0
    try:
        for step in range(st.steps):
            for l in range(st.L):
                o = oracle.moe_forward(st.x_bits[step][l], st.logits[step][l], st.host_pages, pb,
                                       st.layer_table(l), s.H, s.I, s.k, s.renorm)
                routed = sorted(set(o["ids"].ravel().tolist()))
                if prefetch and l + 1 < st.L and (l + 1) in prev_routed:
                    guess = prev_routed[l + 1]
                    R.rimuru_offload_prefetch(off, l + 1, guess)
                    model.prefetch([(l + 1) * E + e for e in guess], nbytes)
                x = bf16_tensor(st.x_bits[step][l])
                lg = torch.from_numpy(st.logits[step][l]).to(DEV)
                out = torch.empty_like(x)
                R.rimuru_offload_forward(off, x.data_ptr(), lg.data_ptr(), st.T, l, out.data_ptr(),
                                         ws_ptr, ws_bytes, stream)
                model.forward(l, [l * E + e for e in routed], nbytes)
                torch.cuda.synchronize()
                assert R.rimuru_get_device_error(ev, clear=True) == R.DEV_OK
                err = rel_err(to_f64(out), o["out"])
                assert err <= 1e-2, (step, l, err)
                worst = max(worst, err)
                prev_routed[l] = routed
                for e in range(E):  # residency matches the model
                    assert (R.rimuru_offload_resident(off, l, e) >= 0) == ((l * E + e) in model.key_slot)
        counters = R.rimuru_offload_stats(off)
    finally:
        R.rimuru_offload_destroy(off)
        pool.close()
    return counters, model.c, worst


@pytest.mark.parametrize("prefetch,cap", [(False, 12), (True, 12), (True, 20)],
                         ids=["demand_only_12", "prefetch_12", "prefetch_20"])
def test_offloaded_stack_matches_oracle_and_lru_model(prefetch, cap):
    """6 tiny layers (8 experts, top-2), 16 tokens, 3 steps; 12 or 20 of 48 experts resident.
    With 12 slots (less than two layers' worth) prefetching layer l + 1 evicts what was
    prefetched for layer l, so only 20 slots let prefetched experts be hit."""
    shape = wl.MoEShape(H=256, I=128, E=8, k=2)
    st = wl.offload_stack(shape, L=6, T=16, steps=3, seed=51)
    counters, expected, worst = run_stack(st, cap=cap, prefetch=prefetch)
    assert counters == expected
    assert counters["misses"] + counters["prefetch_loads"] > 0 and counters["evictions"] > 0
    if prefetch:
        assert counters["prefetch_loads"] > 0
    if cap == 20:
        assert counters["hits"] > 0


@pytest.mark.parametrize("prefetch", [False, True], ids=["demand_only", "prefetch"])
def test_layer_cycle_policy_keeps_part_of_the_cycle_resident(prefetch):
    """The same stack over 4 steps with the layer-cycle policy: outputs against the oracle,
    counters against the model, and fewer host-to-device bytes than LRU, which misses on
    every expert of a cycle larger than the cache."""
    shape = wl.MoEShape(H=256, I=128, E=8, k=2)
    st = wl.offload_stack(shape, L=6, T=16, steps=4, seed=53)
    cyc, cyc_model, _ = run_stack(st, cap=24, prefetch=prefetch, policy=R.EVICT_LAYER_CYCLE)
    assert cyc == cyc_model
    lru, lru_model, _ = run_stack(st, cap=24, prefetch=prefetch, policy=R.EVICT_LRU)
    assert lru == lru_model
    assert cyc["bytes_h2d"] < lru["bytes_h2d"] and cyc["hits"] >= lru["hits"]


def test_capacity_below_one_layer_is_rejected():
    """Every token routes to 2 of 8 experts, so 16 tokens touch more than 3 experts."""
    shape = wl.MoEShape(H=256, I=128, E=8, k=2)
    st = wl.offload_stack(shape, L=2, T=16, steps=1, seed=52)
    with pytest.raises(R.RimuruError) as e:
        run_stack(st, cap=3, prefetch=False)
    assert e.value.status == R.ERR_OOM


def test_qwen3_shaped_stack_matches_oracle_and_lru_model():
    """Three layers of the Qwen3-30B-A3B shape at full size (3 MiB pages, so the merged
    adjacent host-to-pool copies and the per-layer page-table slice from the pinned ring run
    on real page sizes), 64 tokens, two steps, with 200 experts resident: one cycle of layers
    routes to about 378 experts, so experts are evicted and loaded again in every step, and
    a prefetch of layer l + 1 competes with layer l's own experts.  Every token of every
    layer against the oracle; the counters against the model of least-recently-used
    eviction (the stack configuration's policy)."""
    st = wl.offload_stack(wl.Q3, L=3, T=64, steps=2, seed=61, distinct_layers=1)
    counters, expected, worst = run_stack(st, cap=200, prefetch=True)
    assert counters == expected
    # least-recently-used eviction over a cycle larger than the cache evicts exactly what is
    # needed next, so the model (and the cache) report misses, prefetches and no hits
    assert counters["evictions"] > 0 and counters["misses"] > 0
    assert counters["prefetch_loads"] > 0
