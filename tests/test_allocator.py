"""Host-side pool, views, multi-level allocator and expert page table (CPU only).

The pool never touches device memory, so a fake 2 MiB-aligned address stands in for the
device base.  Rimuru page: shared pool, memory views with their own page size and page
table, huge pages = LCM(expert page, SSM page), a multi-level allocator that splits
huge -> expert -> KV pages and merges them back (abstract; Figure 7; explainer page,
memory-manager paragraph)."""
import numpy as np
import pytest

from paged_moe_shared_gb300 import rimuru as R

KiB, MiB = 1024, 1024 * 1024
FAKE_BASE = 64 * 2 * MiB


def stats(pool):
    return [R.rimuru_pool_level_stats(pool, l) for l in range(R.rimuru_pool_num_levels(pool))]


def check_conservation(pool, pool_bytes):
    st = stats(pool)
    covered = sum((s["pages_free"] + s["pages_owned"]) * s["page_bytes"] for s in st)
    assert covered == pool_bytes
    for up, lo in zip(st, st[1:]):
        per = up["page_bytes"] // lo["page_bytes"]
        assert up["pages_split"] * per == lo["pages_free"] + lo["pages_owned"] + lo["pages_split"]
    assert st[-1]["pages_split"] == 0


def test_huge_page_rule():
    assert R.rimuru_huge_page_bytes(3 * MiB, 0) == 3 * MiB            # no SSM state
    assert R.rimuru_huge_page_bytes(2 * MiB, 1 * MiB) == 2 * MiB      # Qwen3.5: SSM bf16
    assert R.rimuru_huge_page_bytes(2 * MiB, 2 * MiB) == 2 * MiB      # SSM fp32
    assert R.rimuru_huge_page_bytes(3 * MiB, 2 * MiB) == 6 * MiB
    assert R.rimuru_huge_page_bytes(0, 2 * MiB) == 0


def test_pool_argument_checks():
    with pytest.raises(R.RimuruError) as e:
        R.rimuru_pool_create(FAKE_BASE + 256, 8 * MiB, 2 * MiB)
    assert e.value.status == R.ERR_ALIGN
    with pytest.raises(R.RimuruError) as e:
        R.rimuru_pool_create(FAKE_BASE, 5 * MiB, 2 * MiB)
    assert e.value.status == R.ERR_ALIGN
    with pytest.raises(R.RimuruError) as e:
        R.rimuru_pool_create(0, 8 * MiB, 2 * MiB)
    assert e.value.status == R.ERR_ARG


def test_split_goes_through_every_level_and_merges_back():
    huge, exp, kvb = 6 * MiB, 3 * MiB, 32 * KiB
    pool = R.rimuru_pool_create(FAKE_BASE, 4 * huge, huge)
    ev = R.rimuru_view_create(pool, exp)
    kv = R.rimuru_view_create(pool, kvb)
    assert R.rimuru_pool_num_levels(pool) == 3
    p = R.rimuru_page_alloc(kv)
    s = stats(pool)
    # the KV page came from an expert-sized page, which came from a huge page
    assert s[0]["pages_split"] == 1 and s[1]["pages_split"] == 1
    assert s[1]["pages_free"] == 1 and s[2]["pages_owned"] == 1 and s[2]["pages_free"] == 95
    assert p == 0
    check_conservation(pool, 4 * huge)
    e0 = R.rimuru_page_alloc(ev)           # lowest free expert page: the other half
    assert e0 == 1
    R.rimuru_page_free(kv, p)              # 96 KV pages merge into expert page 0
    s = stats(pool)
    assert s[2]["pages_owned"] == 0 and s[2]["pages_free"] == 0 and s[1]["pages_split"] == 0
    R.rimuru_page_free(ev, e0)             # both halves free: the huge page is whole again
    s = stats(pool)
    assert s[0]["pages_free"] == 4 and s[0]["pages_split"] == 0 and s[1]["pages_free"] == 0
    check_conservation(pool, 4 * huge)
    R.rimuru_view_destroy(kv)
    R.rimuru_view_destroy(ev)
    R.rimuru_pool_destroy(pool)


def test_equal_huge_and_expert_size_is_one_level():
    pool = R.rimuru_pool_create(FAKE_BASE, 8 * 2 * MiB, 2 * MiB)
    ev = R.rimuru_view_create(pool, 2 * MiB)
    kv = R.rimuru_view_create(pool, 32 * KiB)
    assert R.rimuru_pool_num_levels(pool) == 2
    R.rimuru_page_place(kv, 64 * 5 + 3)    # inside huge page 5
    with pytest.raises(R.RimuruError) as e:
        R.rimuru_page_place(ev, 5)         # split into KV blocks: not available
    assert e.value.status == R.ERR_STATE
    R.rimuru_page_place(ev, 4)
    with pytest.raises(R.RimuruError) as e:
        R.rimuru_page_place(kv, 64 * 4)    # inside an owned expert page
    assert e.value.status == R.ERR_STATE
    with pytest.raises(R.RimuruError) as e:
        R.rimuru_page_place(ev, 4)         # already owned
    assert e.value.status == R.ERR_STATE
    with pytest.raises(R.RimuruError) as e:
        R.rimuru_page_place(ev, 8)         # out of range
    assert e.value.status == R.ERR_RANGE
    with pytest.raises(R.RimuruError) as e:
        R.rimuru_page_free(kv, 64 * 5 + 4) # free but not owned
    assert e.value.status == R.ERR_STATE
    check_conservation(pool, 16 * MiB)
    R.rimuru_view_destroy(kv)
    R.rimuru_view_destroy(ev)
    R.rimuru_pool_destroy(pool)


def test_view_sizes_must_chain_and_come_first():
    pool = R.rimuru_pool_create(FAKE_BASE, 4 * 6 * MiB, 6 * MiB)
    ev = R.rimuru_view_create(pool, 3 * MiB)
    with pytest.raises(R.RimuruError) as e:
        R.rimuru_view_create(pool, 2 * MiB)        # 3 MiB is not a multiple of 2 MiB
    assert e.value.status == R.ERR_ALIGN
    with pytest.raises(R.RimuruError) as e:
        R.rimuru_view_create(pool, 4 * MiB)        # does not divide the huge page
    assert e.value.status == R.ERR_ALIGN
    R.rimuru_page_alloc(ev)
    with pytest.raises(R.RimuruError) as e:
        R.rimuru_view_create(pool, 32 * KiB)       # new level after placement
    assert e.value.status == R.ERR_STATE
    ev2 = R.rimuru_view_create(pool, 3 * MiB)       # existing size: fine
    with pytest.raises(R.RimuruError) as e:
        R.rimuru_pool_destroy(pool)
    assert e.value.status == R.ERR_STATE
    R.rimuru_view_destroy(ev2)
    R.rimuru_view_destroy(ev)
    R.rimuru_pool_destroy(pool)


@pytest.mark.parametrize("seed", range(4))
def test_random_alloc_free_keeps_invariants(seed):
    rng = np.random.default_rng(seed)
    huge, exp, kvb = 6 * MiB, 3 * MiB, 256 * KiB
    n_huge = 6
    pool = R.rimuru_pool_create(FAKE_BASE, n_huge * huge, huge)
    views = {"huge": R.rimuru_view_create(pool, huge), "exp": R.rimuru_view_create(pool, exp),
             "kv": R.rimuru_view_create(pool, kvb)}
    size = {"huge": huge, "exp": exp, "kv": kvb}
    owned = {k: set() for k in views}
    for _ in range(600):
        kind = rng.choice(list(views))
        if owned[kind] and rng.random() < 0.45:
            p = int(rng.choice(sorted(owned[kind])))
            R.rimuru_page_free(views[kind], p)
            owned[kind].remove(p)
        else:
            try:
                p = R.rimuru_page_alloc(views[kind])
            except R.RimuruError as e:
                assert e.status == R.ERR_OOM
                continue
            assert p not in owned[kind]
            owned[kind].add(p)
        # owned byte ranges never overlap
        spans = sorted((p * size[k], (p + 1) * size[k]) for k in owned for p in owned[k])
        for (a0, a1), (b0, b1) in zip(spans, spans[1:]):
            assert a1 <= b0
        check_conservation(pool, n_huge * huge)
    for k in views:
        for p in sorted(owned[k]):
            R.rimuru_page_free(views[k], p)
    s = stats(pool)
    assert s[0]["pages_free"] == n_huge and all(x["pages_free"] == 0 for x in s[1:])
    for v in views.values():
        R.rimuru_view_destroy(v)
    R.rimuru_pool_destroy(pool)


def test_expert_page_table():
    pool = R.rimuru_pool_create(FAKE_BASE, 16 * 64 * KiB, 64 * KiB)
    ev = R.rimuru_view_create(pool, 64 * KiB)
    with pytest.raises(R.RimuruError) as e:
        R.rimuru_expert_map(ev, 0, 0, 0, 1)                 # no shape yet
    assert e.value.status == R.ERR_STATE
    with pytest.raises(R.RimuruError) as e:
        R.rimuru_view_set_moe_shape(ev, 1, 4, 256, 100, 2)  # inter not a multiple of 128
    assert e.value.status == R.ERR_UNSUPPORTED
    with pytest.raises(R.RimuruError) as e:
        R.rimuru_view_set_moe_shape(ev, 1, 4, 256, 256, 2)  # 128 KiB does not fit a 64 KiB page
    assert e.value.status == R.ERR_UNSUPPORTED
    with pytest.raises(R.RimuruError) as e:
        R.rimuru_view_set_moe_shape(ev, 1, 4, 256, 128, 5)  # top_k > experts
    assert e.value.status == R.ERR_UNSUPPORTED
    R.rimuru_view_set_moe_shape(ev, 2, 4, 256, 128, 2)
    with pytest.raises(R.RimuruError) as e:
        R.rimuru_expert_map(ev, 0, 0, 0, 3)                 # page not owned
    assert e.value.status == R.ERR_STATE
    R.rimuru_page_place(ev, 3)
    R.rimuru_expert_map(ev, 0, 0, R.PROJ_W1, 3)
    assert R.rimuru_expert_lookup(ev, 0, 0, R.PROJ_W1) == 3
    assert R.rimuru_expert_lookup(ev, 1, 0, R.PROJ_W1) == -1
    for bad in ((2, 0, 0), (0, 4, 0), (0, 0, 3), (-1, 0, 0)):
        with pytest.raises(R.RimuruError) as e:
            R.rimuru_expert_map(ev, *bad, 3)
        assert e.value.status == R.ERR_RANGE
    with pytest.raises(R.RimuruError) as e:
        R.rimuru_page_free(ev, 3)                           # still mapped
    assert e.value.status == R.ERR_STATE
    R.rimuru_expert_unmap(ev, 0, 0, R.PROJ_W1)
    R.rimuru_page_free(ev, 3)
    R.rimuru_view_destroy(ev)
    R.rimuru_pool_destroy(pool)


def test_forward_host_checks_run_before_any_device_work():
    pool = R.rimuru_pool_create(FAKE_BASE, 32 * 64 * KiB, 64 * KiB)
    ev = R.rimuru_view_create(pool, 64 * KiB)
    R.rimuru_view_set_moe_shape(ev, 1, 8, 256, 128, 2)
    fake = 1 << 30
    with pytest.raises(R.RimuruError) as e:
        R.rimuru_moe_forward(fake, fake, 16, ev, 0, fake + (1 << 20), fake, 1 << 30)
    assert e.value.status == R.ERR_UNMAPPED
    for ex in range(8):
        for p in range(3):
            pid = R.rimuru_page_alloc(ev)
            R.rimuru_expert_map(ev, 0, ex, p, pid)
    ws = R.rimuru_moe_workspace_bytes(ev, 16)
    lay = R.rimuru_moe_workspace_layout(ev, 16)
    assert lay["total"] == ws and lay["x_sorted"] % 1024 == 0 and lay["y"] + 32 * 256 * 2 <= ws
    with pytest.raises(R.RimuruError) as e:
        R.rimuru_moe_forward(fake, fake, 16, ev, 0, fake + (1 << 20), fake, ws - 1)
    assert e.value.status == R.ERR_WORKSPACE
    with pytest.raises(R.RimuruError) as e:
        R.rimuru_moe_forward(fake + 8, fake, 16, ev, 0, fake + (1 << 20), fake, ws)
    assert e.value.status == R.ERR_ALIGN
    with pytest.raises(R.RimuruError) as e:
        R.rimuru_moe_forward(fake, fake, 16, ev, 1, fake + (1 << 20), fake, ws)
    assert e.value.status == R.ERR_RANGE
    with pytest.raises(R.RimuruError) as e:
        R.rimuru_moe_forward(fake, fake, -1, ev, 0, fake + (1 << 20), fake, ws)
    assert e.value.status == R.ERR_ARG
    R.rimuru_moe_forward(fake, fake, 0, ev, 0, fake, fake, 0)   # zero tokens: nothing to do
    R.rimuru_view_destroy(ev)
    R.rimuru_pool_destroy(pool)


def test_host_buffer_forward_checks_and_staging_size():
    """rimuru_moe_forward_host: the staging regions follow the layer's workspace, and bad
    arguments are refused before any copy is queued."""
    pool = R.rimuru_pool_create(FAKE_BASE, 32 * 64 * KiB, 64 * KiB)
    ev = R.rimuru_view_create(pool, 64 * KiB)
    R.rimuru_view_set_moe_shape(ev, 1, 8, 256, 128, 2)
    fake = 1 << 30
    T = 16
    hws = R.rimuru_moe_host_workspace_bytes(ev, T)
    ws = R.rimuru_moe_workspace_bytes(ev, T)
    # x and out (T*H bf16) and logits (T*E fp32), each in its own 1 KiB-aligned region
    assert hws >= ws + 2 * T * 256 * 2 + T * 8 * 4 and hws % 1024 == 0
    assert R.rimuru_moe_host_workspace_bytes(ev, -1) == 0
    with pytest.raises(R.RimuruError) as e:
        R.rimuru_moe_forward_host(fake, fake, T, ev, 0, fake, fake, hws)
    assert e.value.status == R.ERR_UNMAPPED
    for ex in range(8):
        for p in range(3):
            R.rimuru_expert_map(ev, 0, ex, p, R.rimuru_page_alloc(ev))
    with pytest.raises(R.RimuruError) as e:
        R.rimuru_moe_forward_host(fake, fake, T, ev, 0, fake, fake, hws - 1)
    assert e.value.status == R.ERR_WORKSPACE
    with pytest.raises(R.RimuruError) as e:
        R.rimuru_moe_forward_host(fake, fake, T, ev, 0, fake, fake + 512, hws)
    assert e.value.status == R.ERR_ALIGN
    with pytest.raises(R.RimuruError) as e:
        R.rimuru_moe_forward_host(0, fake, T, ev, 0, fake, fake, hws)
    assert e.value.status == R.ERR_ARG
    with pytest.raises(R.RimuruError) as e:
        R.rimuru_moe_forward_host(fake, fake, T, ev, 3, fake, fake, hws)
    assert e.value.status == R.ERR_RANGE
    R.rimuru_moe_forward_host(0, 0, 0, ev, 0, 0, 0, 0)   # zero tokens: nothing to do
    with pytest.raises(R.RimuruError) as e:              # sampling stride must be >= 1
        R.rimuru_profile_enable_sampled(ev, 1, 10, 0)
    assert e.value.status == R.ERR_ARG
    R.rimuru_view_destroy(ev)
    R.rimuru_pool_destroy(pool)


def _kv_pool():
    pool = R.rimuru_pool_create(FAKE_BASE, 16 * 2 * MiB, 2 * MiB)
    ev = R.rimuru_view_create(pool, 2 * MiB)
    kv = R.rimuru_view_create(pool, 32 * KiB)   # 64 KV blocks per huge page
    return pool, ev, kv


@pytest.mark.parametrize("grouped", [False, True], ids=["plain", "grouped"])
def test_request_affinity_lets_finished_requests_merge_back(grouped):
    """Eight requests take 16 KV blocks each, interleaved one block at a time.  Grouped
    (first block: a fresh parent; next blocks: near the previous one) keeps each request in
    one parent, so freeing half of the requests returns whole huge pages; plain allocation
    interleaves the requests in two parents and frees none."""
    pool, ev, kv = _kv_pool()
    blocks = {r: [] for r in range(8)}
    for i in range(16):
        for r in range(8):
            if grouped:
                hint = blocks[r][-1] if blocks[r] else R.NEW_GROUP
                blocks[r].append(R.rimuru_page_alloc_near(kv, hint))
            else:
                blocks[r].append(R.rimuru_page_alloc(kv))
    parents = {r: {b // 64 for b in blocks[r]} for r in range(8)}
    if grouped:
        assert all(len(p) == 1 for p in parents.values())
        assert len(set().union(*parents.values())) == 8
    for r in (0, 2, 4, 6):
        for b in blocks[r]:
            R.rimuru_page_free(kv, b)
    s = stats(pool)
    partial, stranded = R.rimuru_pool_fragmentation(pool, 1)
    check_conservation(pool, 32 * MiB)
    if grouped:
        assert s[0]["pages_free"] == 16 - 4 and partial == 4 and stranded == 4 * 48
        # the freed huge pages are whole again and can hold experts
        for _ in range(12):
            R.rimuru_page_alloc(ev)
    else:
        assert s[0]["pages_free"] == 14 and partial == 2 and stranded == 64
    for r in (1, 3, 5, 7):
        for b in blocks[r]:
            R.rimuru_page_free(kv, b)
    assert R.rimuru_pool_fragmentation(pool, 1) == (0, 0)
    R.rimuru_view_destroy(kv)
    R.rimuru_view_destroy(ev)
    R.rimuru_pool_destroy(pool)


def test_alloc_near_prefers_the_hint_parent():
    pool, ev, kv = _kv_pool()
    a = R.rimuru_page_alloc_near(kv, R.NEW_GROUP)
    b = R.rimuru_page_alloc_near(kv, R.NEW_GROUP)
    assert a // 64 != b // 64
    c = R.rimuru_page_alloc_near(kv, a)
    assert c // 64 == a // 64 and c != a
    d = R.rimuru_page_alloc_near(kv, -1)   # plain: lowest free block
    assert d == min(set(range(128)) - {a, b, c})
    R.rimuru_view_destroy(kv)
    R.rimuru_view_destroy(ev)
    R.rimuru_pool_destroy(pool)
