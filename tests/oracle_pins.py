"""Pins that tie the CPU oracle to something other than itself.

Each ``pin_*`` function takes an ``oracle.Oracle`` and raises ``AssertionError`` when the
oracle disagrees with a value or property fixed by the pages or by mathematics:
hand-derived golden cases (``tests/golden``), closed forms (k = E is the dense softmax
mixture; k = 1 is the argmax expert's FFN), library routines (numpy's stable argsort and
lexsort, scipy's softmax and expit), brute force on tiny inputs, and invariants of the
paging scheme (placement shuffles, NaN in unused pages).

The same functions are run against deliberately broken builds of the oracle in
``test_oracle_mutants.py`` to show that each plausible mistake fails at least one pin.
"""
from __future__ import annotations

import json
import os

import numpy as np
from scipy.special import expit, softmax

import workloads as wl

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _dense_ffn(x, w1, w3, w2):
    """(silu(x w1) * (x w3)) w2 in float64 with silu = g * expit(g) (scipy)."""
    g = x @ w1
    u = x @ w3
    return (g * expit(g) * u) @ w2


def _weights_f64(weights):
    w1, w3, w2 = weights
    f = lambda a: wl.bf16_bits_to_f32(a).astype(np.float64)
    return f(w1), f(w3), f(w2)


# ---------------------------------------------------------------- routing
def pin_route_golden(o):
    g = _golden("route_cases.json")
    for c in g["cases"]:
        logits = np.array([c["logits"]], np.float32)
        ids, w = o.route(logits, c["k"], bool(c["renorm"]))
        assert ids[0].tolist() == c["ids"], (c["name"], ids[0].tolist(), c["ids"])
        np.testing.assert_allclose(w[0], np.array(c["w"]), rtol=0, atol=1e-7, err_msg=c["name"])


def _rank_topk(row, k):
    """Brute force: rank of i = number of j that come before i (larger value, or equal
    value and lower index).  Slot r holds the expert of rank r."""
    E = len(row)
    rank = [sum(1 for j in range(E) if row[j] > row[i] or (row[j] == row[i] and j < i))
            for i in range(E)]
    by_rank = {r: i for i, r in enumerate(rank)}
    return [by_rank[r] for r in range(k)]


def pin_route_bruteforce(o):
    rng = np.random.default_rng(11)
    for E in (3, 5, 8):
        for k in range(1, E + 1):
            logits = rng.integers(-2, 3, size=(20, E)).astype(np.float32)  # many ties
            ids, _ = o.route(logits, k, True)
            for t in range(logits.shape[0]):
                assert ids[t].tolist() == _rank_topk(logits[t].tolist(), k), (E, k, t)


def pin_route_lexsort(o):
    rng = np.random.default_rng(12)
    logits = (rng.standard_normal((64, 128)) * 0.5).astype(np.float32)
    logits[:, 5] = logits[:, 9]  # exact ties
    ids, _ = o.route(logits, 8, True)
    for t in range(64):
        order = np.lexsort((np.arange(128), -logits[t].astype(np.float64)))
        assert ids[t].tolist() == order[:8].tolist(), t


def pin_route_weights(o):
    rng = np.random.default_rng(13)
    logits = (rng.standard_normal((32, 8)) * 3).astype(np.float32)
    # k = E: the weights are the full softmax (scipy), in expert order
    ids, w = o.route(logits, 8, True)
    p = softmax(logits.astype(np.float64), axis=1)
    for t in range(32):
        np.testing.assert_allclose(w[t], p[t, ids[t]], rtol=0, atol=1e-7)
    # renormalised top-k weights sum to one and follow the softmax ratios
    ids, w = o.route(logits, 3, True)
    np.testing.assert_allclose(w.astype(np.float64).sum(1), 1.0, rtol=0, atol=3e-7)
    for t in range(32):
        q = p[t, ids[t]] / p[t, ids[t]].sum()
        np.testing.assert_allclose(w[t], q, rtol=0, atol=1e-7)
    # without renormalisation the weights are the plain softmax entries
    ids, w = o.route(logits, 3, False)
    for t in range(32):
        np.testing.assert_allclose(w[t], p[t, ids[t]], rtol=0, atol=1e-7)


# ---------------------------------------------------------------- grouping
def pin_align_library(o):
    rng = np.random.default_rng(14)
    for E, A in ((8, 32), (128, 512), (16, 1000), (4, 0)):
        ids = rng.integers(0, E, size=A).astype(np.int32)
        if A:
            ids[: A // 3] = E // 2  # one heavy expert
        s, off = o.align(ids, E)
        assert s.tolist() == np.argsort(ids, kind="stable").tolist()
        assert off.tolist() == [0] + np.cumsum(np.bincount(ids, minlength=E)).tolist()


# ---------------------------------------------------------------- bf16 and pages
def pin_bf16_decode(o):
    known = {0x3F80: 1.0, 0xC000: -2.0, 0x4049: 3.140625, 0x3F81: 1.0 + 2.0 ** -7,
             0x0001: 2.0 ** -133, 0x8000: -0.0, 0x0080: 2.0 ** -126, 0x7F7F: 3.3895313892515355e38}
    for bits, val in known.items():
        assert o.bf16_to_f64(bits) == val, hex(bits)
    assert o.bf16_to_f64(0x7F80) == float("inf")
    assert np.isnan(o.bf16_to_f64(0x7FC0))
    rng = np.random.default_rng(15)
    bits = rng.integers(0, 2 ** 16, size=4096, dtype=np.uint32).astype(np.uint16)
    with np.errstate(invalid="ignore"):
        ref = wl.bf16_bits_to_f32(bits).astype(np.float64)  # numpy reinterpretation
    got = np.array([o.bf16_to_f64(int(b)) for b in bits])
    fin = np.isfinite(ref)
    assert np.array_equal(got[fin], ref[fin])
    assert np.array_equal(np.isnan(got), np.isnan(ref))


def pin_page_to_matrix(o):
    rng = np.random.default_rng(16)
    page_bytes, rows, cols = 4096, 24, 40
    pool = wl.empty_pool(8 * page_bytes)
    bits = wl.to_bf16_bits(rng.standard_normal((rows, cols)))
    wl.write_page(pool, page_bytes, 5, bits)
    m = o.page_to_matrix(pool, page_bytes, 5, rows, cols)
    assert np.array_equal(m, wl.bf16_bits_to_f32(bits).astype(np.float64))
    # a page that is only NaN decodes to NaN
    assert np.isnan(o.page_to_matrix(pool, page_bytes, 6, rows, cols)).all()


# ---------------------------------------------------------------- the layer
def _golden_pair_workload(g, case):
    H, I, E = g["H"], g["I"], g["E"]
    a, b, c = (np.array(g[n], np.float64) for n in ("a", "b", "c"))
    s1, s2 = case["expert1"]["w1_sign"], case["expert1"]["w2_sign"]
    w1 = wl.to_bf16_bits(np.stack([a, s1 * a]))
    w3 = wl.to_bf16_bits(np.stack([b, b]))
    w2 = wl.to_bf16_bits(np.stack([c, s2 * c]))
    pool = wl.empty_pool(g["pool_pages"] * g["page_bytes"])
    pt = np.array(g["page_table"], np.int32)
    for e in range(E):
        wl.write_page(pool, g["page_bytes"], int(pt[e, 0]), w1[e])
        wl.write_page(pool, g["page_bytes"], int(pt[e, 1]), w3[e])
        wl.write_page(pool, g["page_bytes"], int(pt[e, 2]), w2[e])
    x = wl.to_bf16_bits(np.array(g["x"]))
    logits = np.array(case.get("logits", g["logits"]), np.float32)
    return x, logits, pool, pt


def pin_ffn_golden_pairs(o):
    g = _golden("ffn_pairs.json")
    for case in g["cases"]:
        x, logits, pool, pt = _golden_pair_workload(g, case)
        k = case.get("k", g["k"])
        r = o.moe_forward(x, logits, pool, g["page_bytes"], pt, g["H"], g["I"], k, True)
        np.testing.assert_allclose(r["out"], np.array(case["out"]), rtol=1e-12, atol=1e-12,
                                   err_msg=case["name"])


def _small(seed, T, H, I, E, k, pool_pages=None, slots_seed=None):
    shape = wl.MoEShape(H=H, I=I, E=E, k=k)
    weights = wl.make_expert_weights(seed, shape, std=0.3)
    x = wl.make_x(seed, T, H)
    logits = wl.make_logits(seed, x, E, gate_std=0.5)
    pool_pages = pool_pages or 3 * E + 5
    return shape, weights, x, logits, pool_pages


def pin_dense_mixture(o):
    """k = E: the layer is sum_e softmax(l)_e FFN_e(x) (closed form, no routing, no paging)."""
    for seed, (T, H, I, E) in enumerate([(5, 16, 8, 4), (3, 24, 16, 6)]):
        shape, weights, x, logits, pages = _small(seed, T, H, I, E, E)
        w = wl.build_simple("pin", shape, T, pages, seed, weights=weights, x_bits=x, logits=logits,
                            page_bytes=H * I * 2 + 64)
        r = o.moe_forward(x, logits, w.pool, w.page_bytes, w.page_table, H, I, E, True)
        W1, W3, W2 = _weights_f64(weights)
        xf = wl.bf16_bits_to_f32(x).astype(np.float64)
        p = softmax(logits.astype(np.float64), axis=1)
        ref = sum(p[:, e:e + 1] * _dense_ffn(xf, W1[e], W3[e], W2[e]) for e in range(E))
        np.testing.assert_allclose(r["out"], ref, rtol=1e-10, atol=1e-12)


def pin_k1_argmax(o):
    """k = 1 with renormalisation: the output is the FFN of the argmax expert."""
    T, H, I, E = 9, 16, 8, 5
    shape, weights, x, logits, pages = _small(3, T, H, I, E, 1)
    w = wl.build_simple("pin", shape, T, pages, 3, weights=weights, x_bits=x, logits=logits)
    r = o.moe_forward(x, logits, w.pool, w.page_bytes, w.page_table, H, I, 1, True)
    W1, W3, W2 = _weights_f64(weights)
    xf = wl.bf16_bits_to_f32(x).astype(np.float64)
    for t in range(T):
        e = int(np.argmax(logits[t]))  # numpy picks the first maximum
        ref = _dense_ffn(xf[t:t + 1], W1[e], W3[e], W2[e])
        np.testing.assert_allclose(r["out"][t:t + 1], ref, rtol=1e-10, atol=1e-12)


def pin_bruteforce_tiny(o):
    """T <= 4, E <= 4, H = I = 16, every k: per-token loop over brute-force top-k."""
    H = I = 16
    for seed in range(4):
        for E in (2, 3, 4):
            for k in range(1, E + 1):
                T = 1 + (seed + E + k) % 4
                shape, weights, x, logits, pages = _small(100 + seed, T, H, I, E, k)
                w = wl.build_simple("pin", shape, T, pages, seed, weights=weights, x_bits=x,
                                    logits=logits)
                r = o.moe_forward(x, logits, w.pool, w.page_bytes, w.page_table, H, I, k, True)
                W1, W3, W2 = _weights_f64(weights)
                xf = wl.bf16_bits_to_f32(x).astype(np.float64)
                for t in range(T):
                    sel = _rank_topk(logits[t].tolist(), k)
                    p = softmax(logits[t].astype(np.float64))[sel]
                    p = p / p.sum()
                    ref = sum(p[j] * _dense_ffn(xf[t:t + 1], W1[e], W3[e], W2[e])
                              for j, e in enumerate(sel))
                    np.testing.assert_allclose(r["out"][t:t + 1], ref, rtol=1e-10, atol=1e-12)


def pin_shuffle_invariance(o):
    """Where the pages sit does not change the result (bit for bit), and unused NaN pages are
    never read; pointing one entry of the page table at a NaN page poisons the output."""
    T, H, I, E, k = 6, 32, 16, 6, 2
    shape, weights, x, logits, _ = _small(5, T, H, I, E, k)
    outs = []
    for seed, pages in ((1, 3 * E), (2, 3 * E + 7), (3, 4 * E + 1)):
        w = wl.build_simple("pin", shape, T, pages, seed, weights=weights, x_bits=x, logits=logits)
        r = o.moe_forward(x, logits, w.pool, w.page_bytes, w.page_table, H, I, k, True)
        assert np.isfinite(r["out"]).all()
        outs.append(r["out"])
    for other in outs[1:]:
        assert np.array_equal(outs[0], other)
    # redirect the w2 page of an expert that token 0 uses to a NaN page
    w = wl.build_simple("pin", shape, T, 3 * E + 1, 4, weights=weights, x_bits=x, logits=logits)
    used = set(w.page_table.ravel().tolist())
    nan_page = next(p for p in range(3 * E + 1) if p not in used)
    e0 = o.route(logits, k, True)[0][0, 0]
    pt = w.page_table.copy()
    pt[e0, 2] = nan_page
    r = o.moe_forward(x, logits, w.pool, w.page_bytes, pt, H, I, k, True)
    assert np.isnan(r["out"][0]).all()


def pin_token_subset(o):
    """Computing a subset of tokens gives the same rows as computing them all."""
    T, H, I, E, k = 10, 16, 8, 4, 2
    shape, weights, x, logits, pages = _small(7, T, H, I, E, k)
    w = wl.build_simple("pin", shape, T, pages, 7, weights=weights, x_bits=x, logits=logits)
    full = o.moe_forward(x, logits, w.pool, w.page_bytes, w.page_table, H, I, k, True)
    sub = o.moe_forward(x, logits, w.pool, w.page_bytes, w.page_table, H, I, k, True,
                        tokens=[7, 2])
    assert np.array_equal(sub["out"][[2, 7]], full["out"][[2, 7]])
    assert np.isnan(sub["out"][[0, 1, 3]]).all()


ALL_PINS = [
    pin_route_golden, pin_route_bruteforce, pin_route_lexsort, pin_route_weights,
    pin_align_library, pin_bf16_decode, pin_page_to_matrix, pin_ffn_golden_pairs,
    pin_dense_mixture, pin_k1_argmax, pin_bruteforce_tiny, pin_shuffle_invariance,
    pin_token_subset,
]


def failing_pins(o):
    """Names of the pins that this oracle build fails (an exception counts as a failure)."""
    bad = []
    for pin in ALL_PINS:
        try:
            pin(o)
        except Exception as exc:  # noqa: BLE001 - any failure counts
            bad.append((pin.__name__, type(exc).__name__))
    return bad
