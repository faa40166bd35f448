"""The seeded input generators: pool placement, free pages, KV blocks, the Zipf bias.

They hold none of the method's arithmetic; these checks pin the input recipe they implement
(pages of one projection each, NaN free pages, KV blocks cut from whole huge pages, a
popularity bias that is a power law in a seeded rank)."""
import numpy as np

import workloads as wl

SMALL = wl.MoEShape(H=256, I=128, E=8, k=2)


def pages(w):
    return w.pool.view(np.uint16).reshape(-1, w.page_bytes // 2)


def test_simple_pool_places_each_projection_on_its_own_page_and_fills_the_rest_with_nan():
    w = wl.tiny(3)
    p = pages(w)
    assert p.shape[0] == w.notes["pool_pages"] == 64
    used = w.page_table.ravel()
    assert sorted(used.tolist()) == sorted(set(used.tolist()))  # no page shared
    w1, w3, w2 = wl.make_expert_weights(3, w.shape)
    for e in range(w.shape.E):
        for proj, mat in enumerate((w1[e], w3[e], w2[e])):
            np.testing.assert_array_equal(p[w.page_table[e, proj]], mat.ravel())
    free = np.setdiff1d(np.arange(p.shape[0]), used)
    assert len(free) == 64 - 3 * w.shape.E
    assert (p[free] == wl.BF16_NAN).all()


def test_placement_is_seeded():
    a, b, c = wl.tiny(5), wl.tiny(5), wl.tiny(6)
    np.testing.assert_array_equal(a.page_table, b.page_table)
    assert not np.array_equal(a.page_table, c.page_table)
    np.testing.assert_array_equal(a.x_bits, b.x_bits)
    np.testing.assert_array_equal(a.logits, b.logits)


def test_mixed_pool_cuts_kv_blocks_from_whole_huge_pages():
    w = wl.build_mixed(SMALL, 4, seed=2, kv_huge_pages=10, free_huge_pages=3,
                       kv_page_bytes=16 * wl.KiB)
    p = pages(w)
    per = w.page_bytes // w.kv_page_bytes
    assert p.shape[0] == 3 * SMALL.E + 10 + 3 == w.notes["huge_pages"]
    kv_huge = np.unique(w.kv_pages // per)
    assert len(kv_huge) == 10 and len(w.kv_pages) == 10 * per
    for hp in kv_huge:  # every block of a KV huge page is listed, in order
        np.testing.assert_array_equal(w.kv_pages[w.kv_pages // per == hp],
                                      np.arange(hp * per, hp * per + per))
    experts = w.page_table.ravel()
    assert not np.intersect1d(experts, kv_huge).size
    kv_vals = wl.bf16_bits_to_f32(p[kv_huge])
    assert np.isfinite(kv_vals).all() and 0.8 < kv_vals.std() < 1.2  # N(0, 1) noise
    free = np.setdiff1d(np.arange(p.shape[0]), np.concatenate([experts, kv_huge]))
    assert len(free) == 3 and (p[free] == wl.BF16_NAN).all()


def test_zipf_bias_is_a_power_law_in_a_seeded_rank():
    E = 128
    r = wl.zipf_ranks(4, E)
    assert sorted(r.tolist()) == list(range(1, E + 1))
    b = wl.zipf_bias(4, E, s=1.1, gamma=2.0)
    assert b[r == 1][0] == 0.0
    # exp(b) = r^(-gamma * s): the ratio of two experts' factors depends only on their ranks
    np.testing.assert_allclose(np.exp(b), r.astype(np.float64) ** (-2.0 * 1.1), rtol=1e-12)
    order = np.argsort(r)
    assert (np.diff(b[order]) < 0).all()


def test_bf16_bits_round_to_nearest_even():
    vals = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 65504.0], np.float32)
    bits = wl.to_bf16_bits(vals)
    # 1 + 2^-8 is halfway between 1 and 1 + 2^-7: ties go to the even mantissa (1.0);
    # 1 + 3 * 2^-8 is halfway between 1 + 2^-7 and 1 + 2^-6: the even one is 1 + 2^-6
    np.testing.assert_array_equal(wl.bf16_bits_to_f32(bits),
                                  np.array([1.0, 1.0, 1.0 + 2 ** -6, -2.5, 65536.0], np.float32))


def test_prefill_inputs_reuse_the_decode_pool():
    """The bench measures prefill on the decode layer's pool: at the same seed and pool size
    the prefill workload has the same pool bytes and page table, and q3_prefill_inputs gives
    its x and logits."""
    a = wl.q3_prefill_zipf(3, T=96, pool_pages=400)
    b = wl.q3_decode(3, T=8, pool_pages=400)
    x, lg = wl.q3_prefill_inputs(3, T=96)
    assert np.array_equal(a.pool, b.pool) and np.array_equal(a.page_table, b.page_table)
    assert np.array_equal(a.x_bits, x) and np.array_equal(a.logits, lg)
    c = wl.with_inputs(b, "q3_prefill_zipf", 96, x, lg)
    assert c.pool is b.pool and c.T == 96 and c.A == 96 * 8


def test_covering_sample_reaches_every_block():
    """covering_tokens picks tokens whose assignment rows include each expert's first and
    last row and one row of each of its 128-row blocks (random skewed routing, stable
    grouping by numpy)."""
    from gpu_harness import covering_tokens
    rng = np.random.default_rng(5)
    T, k, E = 3000, 4, 16
    p = 1.0 / np.arange(1, E + 1) ** 1.5
    ids = np.stack([rng.choice(E, k, replace=False, p=p / p.sum()) for _ in range(T)])
    srt = np.argsort(ids.ravel(), kind="stable").astype(np.int32)
    offs = np.concatenate([[0], np.cumsum(np.bincount(ids.ravel(), minlength=E))])
    toks = covering_tokens(offs, srt, k, seed=1)
    hit = np.isin(srt // k, toks)
    for e in range(E):
        a, b = offs[e], offs[e + 1]
        if b > a:
            assert hit[a] and hit[b - 1]
            for r0 in range(a, b, 128):
                assert hit[r0:min(b, r0 + 128)].any()
    assert len(toks) < T // 4
