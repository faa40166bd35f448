"""CUDA path against the CPU oracle, element by element, through the C ABI.

Bar (from the layer's definition): routing ids, offsets and the expert-sorted permutation
bit-exact; routing weights within 1e-6; h, y and out within
max|gpu - oracle| / max|oracle| <= 1e-2 (bf16 inputs and intermediates, fp32 accumulation);
NaN anywhere counts as a failure.  Every unused pool page holds NaN, so a read outside an
expert's own pages shows up in the output.
"""
from __future__ import annotations

import numpy as np
import pytest

import workloads as wl
from gpu_harness import Runner, covering_tokens, rel_err
from oracle import Oracle

pytestmark = pytest.mark.gpu

TOL = 1e-2
W_TOL = 1e-6


@pytest.fixture(scope="module")
def oracle():
    return Oracle()


def check(res, w, o_res, tokens=None, hidden=True):
    s = w.shape
    assert res["dev_err"] == 0, f"device error {res['dev_err']}"
    np.testing.assert_array_equal(res["ids"], o_res["ids"])
    assert np.max(np.abs(res["w"] - o_res["w"])) <= W_TOL
    np.testing.assert_array_equal(res["offsets"], o_res["offsets"])
    np.testing.assert_array_equal(res["sorted"], o_res["sorted"])
    A = w.T * s.k
    assert np.array_equal(res["inv"][res["sorted"]], np.arange(A))
    counts = np.diff(o_res["offsets"])
    blocks = (counts + 127) // 128
    assert res["num_tiles"] == blocks.sum()
    exp_tiles = [(e, o_res["offsets"][e] + 128 * b) for e in range(s.E) for b in range(blocks[e])]
    assert [tuple(t) for t in res["tiles"].tolist()] == exp_tiles
    # pair table: each expert's blocks two by two (an odd last block alone), expert order
    exp_pairs = [(e, o_res["offsets"][e] + 256 * b) for e in range(s.E)
                 for b in range((blocks[e] + 1) // 2)]
    assert res["num_ptiles"] == len(exp_pairs)
    assert [tuple(t) for t in res["ptiles"].tolist()] == exp_pairs
    toks = np.arange(w.T) if tokens is None else np.asarray(tokens)
    err = rel_err(res["out"][toks], o_res["out"][toks])
    assert err <= TOL, f"out rel err {err:.3e}"
    if hidden:
        rows = np.nonzero(np.isin(res["sorted"] // s.k, toks))[0]
        f = res["sorted"][rows]
        eh = rel_err(res["h"][rows], o_res["h"][f])
        ey = rel_err(res["y"][rows], o_res["y"][f])
        assert eh <= TOL, f"h rel err {eh:.3e}"
        assert ey <= TOL, f"y rel err {ey:.3e}"
    return err


def run_oracle(oracle, w, tokens=None, hidden=True):
    s = w.shape
    return oracle.moe_forward(w.x_bits, w.logits, w.pool, w.page_bytes, w.page_table, s.H, s.I, s.k,
                              s.renorm, tokens=tokens, want_hidden=hidden)


def run_gpu(w, decode_tokens=None):
    r = Runner(w, decode_tokens=decode_tokens)
    try:
        r.forward()
        return r.results()
    finally:
        r.close()


# ------------------------------------------------------------------ tiny layer
@pytest.mark.parametrize("seed", range(5))
def test_tiny(oracle, seed):
    w = wl.tiny(seed)
    check(run_gpu(w), w, run_oracle(oracle, w))


@pytest.mark.parametrize("T", [1, 2, 13, 300, 1000])
def test_tiny_ragged_token_counts(oracle, T):
    """Several 128-row tiles per expert with ragged tails, and single tokens."""
    w = wl.tiny(7, T=T)
    check(run_gpu(w), w, run_oracle(oracle, w))


@pytest.mark.parametrize("T,fused", [(512, True), (513, False)])
def test_small_batch_kernel_boundary(oracle, T, fused):
    """Up to 1024 assignments (T * k) route, align and gather in one kernel; past that,
    route and align are kernels of their own and GEMM 1 gathers its rows from x.  Both sides of the boundary against the oracle, and the kernels
    each side launched, read from the library's per-kernel profile."""
    from paged_moe_shared_gb300 import rimuru as R

    w = wl.tiny(8, T=T)
    r = Runner(w)
    try:
        R.rimuru_profile_enable(r.ev, R.PROFILE_ALL, 1)
        r.forward()
        res = r.results()
        launched = {R.rimuru_kernel_name(i): R.rimuru_profile_read(r.ev, i)[0]
                    for i in range(R.K_COUNT)}
        R.rimuru_profile_enable(r.ev, 0, 1)
    finally:
        r.close()
    small = {"moe_route_align_gather": 1, "moe_route": 0, "moe_align": 0, "moe_gather": 0}
    large = {"moe_route_align_gather": 0, "moe_route": 1, "moe_align": 1, "moe_gather": 0}
    for name, n in (small if fused else large).items():
        assert launched[name] == n, (name, launched)
    for name in ("moe_gemm1_swiglu", "moe_gemm2", "moe_combine"):
        assert launched[name] == 1
    check(res, w, run_oracle(oracle, w))


@pytest.mark.parametrize("k", [1, 3, 8])
def test_tiny_top_k(oracle, k):
    """k = 1 (argmax expert), k = 3, and k = E = 8 (every expert, dense mixture)."""
    shape = wl.MoEShape(H=256, I=128, E=8, k=k)
    w = wl.build_simple("tiny_k", shape, 40, pool_pages=64, seed=11)
    check(run_gpu(w), w, run_oracle(oracle, w))


def test_tiny_without_renormalisation(oracle):
    shape = wl.MoEShape(H=256, I=128, E=8, k=2, renorm=False)
    w = wl.build_simple("tiny_norenorm", shape, 33, pool_pages=64, seed=12)
    check(run_gpu(w), w, run_oracle(oracle, w))


def test_one_hot_expert_and_empty_experts(oracle):
    """Every token's first choice is expert 5 (bias), so one expert holds three tiles and
    several experts get nothing."""
    shape = wl.TINY
    x = wl.make_x(13, 300, shape.H)
    bias = np.zeros(shape.E)
    bias[5] = 50.0
    bias[[0, 1, 2]] = -50.0
    w = wl.build_simple("tiny_hot", shape, 300, pool_pages=64, seed=13, x_bits=x,
                        logits=wl.make_logits(13, x, shape.E, bias=bias))
    o = run_oracle(oracle, w)
    assert np.diff(o["offsets"])[5] == 300 and (np.diff(o["offsets"]) == 0).sum() >= 3
    check(run_gpu(w), w, o)


def test_tied_logits_take_the_lower_index(oracle):
    """Integer-valued logits with many exact ties."""
    shape = wl.TINY
    x = wl.make_x(14, 64, shape.H)
    logits = np.random.default_rng(14).integers(-1, 2, size=(64, shape.E)).astype(np.float32)
    w = wl.build_simple("tiny_ties", shape, 64, pool_pages=64, seed=14, x_bits=x, logits=logits)
    check(run_gpu(w), w, run_oracle(oracle, w))


def test_page_placement_does_not_change_the_output():
    """Same layer, three page placements (and pool sizes): bit-identical GPU output."""
    shape = wl.TINY
    weights = wl.make_expert_weights(21, shape)
    x = wl.make_x(21, 64, shape.H)
    logits = wl.make_logits(21, x, shape.E)
    outs = []
    for seed, pages in ((1, 24), (2, 64), (3, 100)):
        w = wl.build_simple("tiny_shuffle", shape, 64, pool_pages=pages, seed=seed, weights=weights,
                            x_bits=x, logits=logits)
        outs.append(run_gpu(w)["out"])
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])


def test_repeated_forwards_are_bitwise_identical():
    w = wl.tiny(22, T=300)
    r = Runner(w)
    try:
        r.forward()
        a = r.results()
        r.forward()
        r.forward()
        b = r.results()
    finally:
        r.close()
    for key in ("out", "h", "y", "ids", "w", "sorted", "inv"):
        assert np.array_equal(a[key], b[key]), key


def test_nonfinite_logits_raise_the_device_error():
    from paged_moe_shared_gb300 import rimuru as R
    w = wl.tiny(23)
    w.logits[3, 2] = np.nan
    res = run_gpu(w)
    assert res["dev_err"] == R.DEV_NONFINITE
    assert ((res["ids"] >= 0) & (res["ids"] < w.shape.E)).all()


# ------------------------------------------------------------ full-size layers
@pytest.fixture(scope="module")
def q3_decode():
    return wl.q3_decode(0)


def test_q3_decode_full(oracle, q3_decode):
    """Qwen3-30B-A3B-shaped layer, 64 decode tokens, every output element."""
    w = q3_decode
    check(run_gpu(w), w, run_oracle(oracle, w))


def zipf_exponent(counts, ranks):
    """Slope of log(count) against log(rank) over the experts that received tokens."""
    nz = counts > 0
    return -np.polyfit(np.log(ranks[nz]), np.log(counts[nz]), 1)[0]


def sample_covering(oracle, w, seed):
    """Routing and grouping of the whole batch from the oracle, then a token sample whose
    assignment rows reach every 128-row block of every expert and each expert's first and
    last row (so every GEMM tile is compared, not a random subset of them)."""
    s = w.shape
    ids, _ = oracle.route(w.logits, s.k, s.renorm)
    srt, offs = oracle.align(ids, s.E)
    return covering_tokens(offs, srt, s.k, seed)


def assert_rows_cover_every_block(res, tokens, k):
    """Every 128-row block of every expert holds a checked row, and so do the first and
    last rows of every expert (read back from the GPU's own grouping)."""
    rows = np.nonzero(np.isin(res["sorted"] // k, tokens))[0]
    hit = np.zeros(res["sorted"].size, bool)
    hit[rows] = True
    offs = res["offsets"]
    for e in range(offs.size - 1):
        a, b = int(offs[e]), int(offs[e + 1])
        if b > a:
            assert hit[a] and hit[b - 1], e
            for r0 in range(a, b, 128):
                assert hit[r0:min(b, r0 + 128)].any(), (e, r0)


def test_q3_prefill_zipf_sampled(oracle):
    """8192 prefill tokens with Zipf(1.1)-skewed routing: routing, permutation and tiles for
    all tokens; h, y and out for a token sample that reaches every row block of every
    expert (the oracle computes those tokens one by one)."""
    w = wl.q3_prefill_zipf(0)
    tokens = sample_covering(oracle, w, 0)
    o = run_oracle(oracle, w, tokens=tokens)
    counts = np.diff(o["offsets"])
    s = zipf_exponent(counts, wl.zipf_ranks(0, w.shape.E))
    assert 0.9 <= s <= 1.3, f"realised popularity exponent {s:.2f}"
    res = run_gpu(w)
    assert_rows_cover_every_block(res, tokens, w.shape.k)
    check(res, w, o, tokens=tokens)


def test_q3_prefill_heavy_skew_sampled(oracle):
    """A steeper bias (gamma 2): 38 of 128 experts get every assignment, the rest are empty,
    and the hottest expert holds all 8192 tokens (64 row blocks)."""
    w = wl.q3_prefill_zipf(0, gamma=2.0)
    tokens = sample_covering(oracle, w, 2)
    o = run_oracle(oracle, w, tokens=tokens)
    counts = np.diff(o["offsets"])
    assert (counts == 0).sum() >= 1 and counts.max() == w.T
    res = run_gpu(w)
    assert_rows_cover_every_block(res, tokens, w.shape.k)
    check(res, w, o, tokens=tokens)


@pytest.mark.parametrize("T", [1, 16, 256])
def test_q35_mixed_pool(oracle, T):
    """Qwen3.5-35B-A3B-shaped layer (256 experts, I = 512) in a pool whose huge pages are
    partly split into 32 KiB KV blocks full of random data."""
    w = wl.q35_mixed_pool(0, T=T)
    check(run_gpu(w), w, run_oracle(oracle, w))


def test_q35_mixed_pool_4096_sampled(oracle):
    w = wl.q35_mixed_pool(0, T=4096)
    tokens = sample_covering(oracle, w, 1)
    res = run_gpu(w)
    assert_rows_cover_every_block(res, tokens, w.shape.k)
    check(res, w, run_oracle(oracle, w, tokens=tokens), tokens=tokens)


def _wide_inter_t1():
    # I = 1024 gives GEMM 2 sixteen k blocks, enough for it to split too
    shape = wl.MoEShape(H=256, I=1024, E=4, k=1)
    return wl.build_simple("wide_inter", shape, 1, pool_pages=16, seed=9)


def _gathered_split():
    # 1200 assignments (past the small-batch kernel, so GEMM 1 gathers its rows) over 8
    # experts with H = 1024: few enough tiles for GEMM 1 to split its 16 k blocks in two
    shape = wl.MoEShape(H=1024, I=128, E=8, k=2)
    return wl.build_simple("gathered_split", shape, 600, pool_pages=32, seed=10)


@pytest.mark.parametrize("make", [lambda: wl.q35_mixed_pool(0, T=1), lambda: wl.q3_decode(0, T=1),
                                  _wide_inter_t1, _gathered_split],
                         ids=["q35_T1_gemm1_split", "q3_T1_gemm1_split", "wide_inter_gemm2_split",
                              "gathered_gemm1_split"])
def test_split_k_is_used_for_few_tiles_and_is_deterministic(oracle, make):
    """With few tiles the GEMMs split K over several CTAs and sum the fp32 partials in split
    order, so repeated forwards agree bit for bit."""
    w = make()
    r = Runner(w, decode_tokens=0)  # the general path (one token would take the decode path)
    try:
        assert r.layout["total"] > r.layout["part"]  # a partial-sum region exists
        r.forward()
        a = r.results()
        r.forward()
        b = r.results()
    finally:
        r.close()
    check(a, w, run_oracle(oracle, w))
    for key in ("out", "h", "y"):
        assert np.array_equal(a[key], b[key]), key
    from paged_moe_shared_gb300 import rimuru as R
    r = Runner(w, decode_tokens=0)
    try:
        R.rimuru_profile_enable(r.ev, R.PROFILE_ALL, 1)
        r.forward()
        r.results()
        assert R.rimuru_profile_read(r.ev, R.K_DECODE_GEMM1)[0] == 0
        assert R.rimuru_profile_read(r.ev, R.K_GEMM1)[0] == 1
    finally:
        r.close()


def test_cta_pair_gemm2_with_odd_and_even_block_counts(oracle):
    """1500 tokens of the tiny layer (3000 assignments, at least two 128-row blocks per
    expert on average) run both GEMMs over the table of pairs of row blocks of one expert:
    GEMM 1 as 256-row tiles on one SM, GEMM 2 on CTA pairs. A bias makes one expert hot
    (many blocks) and others small, so some pairs hold a lone last block (GEMM 1 skips the
    empty half; GEMM 2 computes rows that are not stored)."""
    shape = wl.TINY
    x = wl.make_x(17, 1500, shape.H)
    bias = np.array([3.0, 0.0, -1.0, 0.5, -2.0, 1.0, 0.0, -0.5])
    w = wl.build_simple("tiny_paired", shape, 1500, pool_pages=64, seed=17, x_bits=x,
                        logits=wl.make_logits(17, x, shape.E, bias=bias))
    o = run_oracle(oracle, w)
    blocks = (np.diff(o["offsets"]) + 127) // 128
    assert (blocks % 2 == 1).any() and (blocks % 2 == 0).any() and blocks.max() >= 4
    check(run_gpu(w), w, o)


def test_cta_pair_gemm2_partial_last_pairs_of_every_kind(oracle):
    """An expert's last pair of row blocks on the CTA-pair GEMM 2 (and the 256-row GEMM 1)
    holds 1 to 256 of its rows; the rows after them belong to the next expert and must not
    be overwritten.  Router logits fix each expert's row count so that the last pairs hold
    1, 16, 17, 255, 256 (a full pair), 129, 128 and 150 rows: a lone block of one row, lone
    blocks ending on and just past a 16-row boundary, full and ragged second blocks."""
    shape = wl.TINY
    T = 1500
    counts = [257, 16, 529, 511, 256, 385, 128, 918]
    assert sum(counts) == T * shape.k and max(counts) <= T
    slots = np.repeat(np.arange(shape.E), counts)
    x = wl.make_x(23, T, shape.H)
    logits = (-2.0 + 0.1 * np.random.default_rng(23).standard_normal((T, shape.E))).astype(np.float32)
    logits[np.arange(T), slots[:T]] = 4.0
    logits[np.arange(T), slots[T:]] = 3.0
    w = wl.build_simple("tiny_partial_pairs", shape, T, pool_pages=64, seed=23, x_bits=x,
                        logits=logits)
    o = run_oracle(oracle, w)
    assert np.diff(o["offsets"]).tolist() == counts
    last = [c - 256 * ((c - 1) // 256) for c in counts]
    assert last == [1, 16, 17, 255, 256, 129, 128, 150]
    check(run_gpu(w), w, o)


# ------------------------------------------------------------ decode-sized batches
# Batches of up to the view's decode-token limit take three kernels: GEMM 1 partials over
# balanced k-block units with routing in every CTA, the reduction to h, and GEMM 2 with the
# combine.  Each case runs against the oracle, and against the general path on the same
# inputs (within the bf16 rounding both paths share, not bit for bit).
def decode_launches(r):
    from paged_moe_shared_gb300 import rimuru as R
    R.rimuru_profile_enable(r.ev, R.PROFILE_ALL, 1)
    r.forward()
    res = r.results()
    launched = {R.rimuru_kernel_name(i): R.rimuru_profile_read(r.ev, i)[0] for i in range(R.K_COUNT)}
    R.rimuru_profile_enable(r.ev, 0, 1)
    return res, launched


DECODE = {
    "q3_t1": lambda: wl.q3_decode(0, T=1),
    "q3_t2": lambda: wl.q3_decode(1, T=2),
    "q3_t4": lambda: wl.q3_decode(2, T=4),
    "q35_t1": lambda: wl.q35_mixed_pool(1, T=1),
    "q35_t2": lambda: wl.q35_mixed_pool(2, T=2),
    "q35_t4": lambda: wl.q35_mixed_pool(3, T=4),
    "tiny_t1": lambda: wl.tiny(4, T=1),
    "tiny_t3": lambda: wl.tiny(5, T=3),
    # 64 assignments (the most the path takes) over 64 experts, E past one warp's lanes
    "k32_t2": lambda: wl.build_simple("k32_t2", wl.MoEShape(H=256, I=128, E=64, k=32), 2,
                                      pool_pages=200, seed=6),
    # 512 experts (16 logits per lane in the routing warp), k = 10
    "e512_k10_t4": lambda: wl.build_simple("e512", wl.MoEShape(H=1024, I=256, E=512, k=10), 4,
                                           pool_pages=1540, seed=7),
    # 32 KiB of x rows (the most the path stages) and 24 column blocks of h
    "h4096_i1536_t4": lambda: wl.build_simple("h4096", wl.MoEShape(H=4096, I=1536, E=32, k=4), 4,
                                              pool_pages=100, seed=8),
    # every token routed to the same expert (4 rows in one unit)
    "one_expert_t4": lambda: wl.build_simple(
        "hot", wl.TINY, 4, pool_pages=64, seed=9,
        logits=np.tile(np.array([[0, 0, 9, 0, 0, 0, 8, 0]], np.float32), (4, 1))),
}


@pytest.mark.parametrize("name", sorted(DECODE))
def test_decode_path_against_oracle_and_general_path(oracle, name):
    w = DECODE[name]()
    r = Runner(w, decode_tokens=4)
    try:
        res, launched = decode_launches(r)
        r.forward()
        again = r.results()
    finally:
        r.close()
    assert launched["moe_decode_gemm1"] == 1 and launched["moe_decode_reduce"] == 1
    assert launched["moe_decode_gemm2"] == 1
    assert sum(launched.values()) == 3
    o = run_oracle(oracle, w, hidden=True)
    check(res, w, o)
    for key in ("out", "h", "y", "ids", "w", "sorted", "inv"):  # deterministic
        assert np.array_equal(res[key], again[key]), key
    res2 = run_gpu(w, decode_tokens=0)
    check(res2, w, o)
    assert rel_err(res["out"], res2["out"]) <= TOL


def test_decode_path_nonfinite_logits_raise_the_device_error():
    from paged_moe_shared_gb300 import rimuru as R
    w = wl.tiny(24, T=2)
    w.logits[1, 4] = np.inf
    res = run_gpu(w, decode_tokens=4)
    assert res["dev_err"] == R.DEV_NONFINITE
    assert ((res["ids"] >= 0) & (res["ids"] < w.shape.E)).all()


def test_decode_path_token_limit_setting(oracle):
    """rimuru_view_set_decode_tokens moves the boundary between the two paths (up to 4
    tokens), 0 turns the decode path off, and values outside [0, 4] are rejected."""
    from paged_moe_shared_gb300 import rimuru as R
    w = wl.q35_mixed_pool(6, T=3)
    o = run_oracle(oracle, w)
    for limit, expect in ((4, True), (3, True), (2, False), (0, False)):
        r = Runner(w, decode_tokens=limit)
        try:
            res, launched = decode_launches(r)
        finally:
            r.close()
        assert (launched["moe_decode_gemm1"] == 1) == expect, limit
        check(res, w, o)
    r = Runner(wl.tiny(1, T=1))
    try:
        for bad in (-1, 5):
            with pytest.raises(R.RimuruError) as e:
                R.rimuru_view_set_decode_tokens(r.ev, bad)
            assert e.value.status == R.ERR_ARG
    finally:
        r.close()


def test_decode_path_replays_from_a_cuda_graph():
    """One-token forwards recorded by stream capture replay to the bits of plain forwards,
    on the recorded inputs and on new ones written into the same buffers."""
    import torch

    from paged_moe_shared_gb300 import rimuru as R
    w = wl.q35_mixed_pool(7, T=1)
    r = Runner(w, decode_tokens=4)
    try:
        s = torch.cuda.Stream()
        r.forward(s)
        s.synchronize()
        plain = r.out.clone()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            r.forward(s)
        r.out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(r.out, plain)
        w2 = wl.q35_mixed_pool(8, T=1)
        r.x.copy_(torch.from_numpy(w2.x_bits.view(np.int16)).view(torch.bfloat16))
        r.logits.copy_(torch.from_numpy(w2.logits))
        g.replay()
        torch.cuda.synchronize()
        replayed = r.out.clone()
        r.forward(s)
        s.synchronize()
        assert torch.equal(replayed, r.out)
        assert R.rimuru_get_device_error(r.ev) == R.DEV_OK
    finally:
        r.close()


# ------------------------------------------------------ activation and routing extremes
# Weights scaled so that the gate pre-activation g spans about +-100: silu(g) saturates to g
# on the positive side, and below g = -87 the exponential in 1 + e^-g overflows fp32, where
# silu must give 0 (times the up value), not NaN.  Router logits of magnitude ~1e3 make the
# top-k softmax weights one-hot to within fp32 (the lower slots underflow to 0 or to
# subnormals).  Each case takes another GEMM path: the small-batch kernel with TMA rows,
# split-K, the gathered 128-row GEMM 1, and the 256-row / CTA-pair GEMMs.
EXTREME = {
    "decode_t4": (wl.TINY, 4, 2.5),
    "small_batch_t64": (wl.TINY, 64, 2.5),
    "split_k_h1024_t16": (wl.MoEShape(H=1024, I=128, E=8, k=2), 16, 1.25),
    "gathered_t600": (wl.TINY, 600, 2.5),
    "wide_pair_t1500": (wl.TINY, 1500, 2.5),
}


@pytest.mark.parametrize("name", sorted(EXTREME))
def test_silu_saturation_and_large_logits(oracle, name):
    shape, T, std = EXTREME[name]
    seed = 31
    x = wl.make_x(seed, T, shape.H)
    logits = wl.make_logits(seed, x, shape.E, gate_std=60.0)
    assert np.abs(logits).max() > 1e3
    weights = wl.make_expert_weights(seed, shape, std=std)
    w = wl.build_simple("extreme_" + name, shape, T, pool_pages=3 * shape.E + 8, seed=seed,
                        weights=weights, x_bits=x, logits=logits)
    o = run_oracle(oracle, w, hidden=True)
    # the gate pre-activations of the routed pairs reach both tails
    xf = wl.bf16_bits_to_f32(x).astype(np.float64)
    g = np.stack([xf[t] @ wl.bf16_bits_to_f32(weights[0][e]).astype(np.float64)
                  for t, e in zip(np.repeat(np.arange(T), shape.k), o["ids"].ravel())])
    assert g.min() < -87.5 and g.max() > 87.5, (g.min(), g.max())
    assert (o["w"].max(axis=1) > 0.999).mean() > 0.5  # mostly one-hot routing weights
    check(run_gpu(w), w, o)


# ------------------------------------------------- other sizes of the same layer family
# Each case changes what the kernels tile over: a wider H and I (more k blocks and column
# blocks), an I of 11 column blocks (an odd count), H = 14 down-projection
# tiles, 512 experts (the largest E the view accepts) with k = 10 (two combine groups), and
# non-renormalised weights at the Qwen3.5-35B shape.
SWEEP = {
    "h4096_i1536_e32_k4_t64": (wl.MoEShape(H=4096, I=1536, E=32, k=4), 64, 16),
    "h2048_i1408_e60_k4_t300": (wl.MoEShape(H=2048, I=1408, E=60, k=4), 300, 24),
    "h3584_i2560_e16_k4_t40": (wl.MoEShape(H=3584, I=2560, E=16, k=4), 40, 12),
    "h1024_i256_e512_k10_t64": (wl.MoEShape(H=1024, I=256, E=512, k=10), 64, None),
    # the largest top-k the kernels take (32 slots: one per lane) on both launch sequences
    "h256_i128_e64_k32_t32": (wl.MoEShape(H=256, I=128, E=64, k=32), 32, None),
    "h256_i128_e64_k32_t40": (wl.MoEShape(H=256, I=128, E=64, k=32), 40, None),
}


@pytest.mark.parametrize("name", sorted(SWEEP))
def test_layer_shape_sweep(oracle, name):
    shape, T, n_sample = SWEEP[name]
    w = wl.build_simple(name, shape, T, pool_pages=3 * shape.E + 16, seed=23)
    tokens = None
    if n_sample is not None:
        tokens = np.sort(np.random.default_rng(23).choice(T, n_sample, replace=False))
    check(run_gpu(w), w, run_oracle(oracle, w, tokens=tokens), tokens=tokens)


def test_q35_mixed_pool_without_renormalisation(oracle):
    """Top-8 of 256 experts with weights left as full-softmax probabilities."""
    shape = wl.MoEShape(H=2048, I=512, E=256, k=8, renorm=False)
    w = wl.build_mixed(shape, 256, seed=3)
    o = run_oracle(oracle, w)
    assert np.all(o["w"].sum(axis=1) < 1.0)
    check(run_gpu(w), w, o)


# ------------------------------------------------------------- host-buffer entry point
@pytest.mark.parametrize("pinned", [True, False], ids=["pinned", "pageable"])
def test_host_buffer_forward_equals_device_forward(oracle, pinned):
    """rimuru_moe_forward_host copies x and logits in, runs the same launches and copies out
    back: its output is bitwise the device-buffer forward's, and within the bar of the oracle."""
    import torch

    from paged_moe_shared_gb300 import rimuru as R

    w = wl.tiny(5, T=300)
    r = Runner(w)
    try:
        r.forward()
        ref = r.results()
        hws = R.rimuru_moe_host_workspace_bytes(r.ev, w.T)
        raw = torch.empty(hws + 1024, dtype=torch.uint8, device="cuda:0")
        ws = (raw.data_ptr() + 1023) // 1024 * 1024
        hx = torch.from_numpy(w.x_bits.view(np.int16).copy())
        hl = torch.from_numpy(np.ascontiguousarray(w.logits))
        ho = torch.zeros(w.T, w.shape.H, dtype=torch.int16)
        if pinned:
            hx, hl, ho = hx.pin_memory(), hl.pin_memory(), ho.pin_memory()
        s = torch.cuda.Stream()
        for _ in range(2):  # the second call finds the first call's staging contents
            R.rimuru_moe_forward_host(hx.data_ptr(), hl.data_ptr(), w.T, r.ev, 0, ho.data_ptr(),
                                      ws, hws, s.cuda_stream)
            s.synchronize()
            assert R.rimuru_get_device_error(r.ev) == R.DEV_OK
            assert torch.equal(ho, r.out.cpu().view(torch.int16))
        # rows of the layer's own workspace hold the same intermediates as the device call
        ids = raw[ws - raw.data_ptr():][r.layout["ids"]:r.layout["ids"] + w.T * w.shape.k * 4]
        assert np.array_equal(ids.view(torch.int32).cpu().numpy().reshape(w.T, w.shape.k),
                              ref["ids"])
    finally:
        r.close()
    check(ref, w, run_oracle(oracle, w))


def test_forward_replays_from_a_cuda_graph(oracle):
    """A forward recorded by stream capture (after one plain forward has uploaded the page
    table) replays to the same bits as plain forwards, including after the inputs change."""
    import torch

    from paged_moe_shared_gb300 import rimuru as R

    w = wl.q35_mixed_pool(4, T=16)
    r = Runner(w)
    try:
        s = torch.cuda.Stream()
        r.forward(s)
        s.synchronize()
        plain = r.out.clone()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            r.forward(s)
        r.out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(r.out, plain)
        # new inputs in the same buffers: the replay computes on them
        w2 = wl.q35_mixed_pool(5, T=16)
        r.x.copy_(torch.from_numpy(w2.x_bits.view(np.int16)).view(torch.bfloat16))
        r.logits.copy_(torch.from_numpy(w2.logits))
        g.replay()
        torch.cuda.synchronize()
        replayed = r.out.clone()
        r.forward(s)
        s.synchronize()
        assert torch.equal(replayed, r.out)
        assert R.rimuru_get_device_error(r.ev) == R.DEV_OK
    finally:
        r.close()
    check(run_gpu(w), w, run_oracle(oracle, w))



def test_sampled_profiling_records_every_nth_forward():
    """rimuru_profile_enable_sampled(every = 3, capacity = 4) over ten forwards brackets the
    selected kernel in forwards 0, 3, 6 and 9 only; kernels not selected report nothing."""
    from paged_moe_shared_gb300 import rimuru as R

    w = wl.tiny(3, T=16)
    r = Runner(w)
    try:
        R.rimuru_profile_enable_sampled(r.ev, 1 << R.K_GEMM1, 4, 3)
        for _ in range(10):
            r.forward()
        n, ms = R.rimuru_profile_read(r.ev, R.K_GEMM1)
        assert n == 4 and ms > 0
        assert R.rimuru_profile_read(r.ev, R.K_GEMM2) == (0, 0.0)
        R.rimuru_profile_enable(r.ev, 0, 1)
        assert R.rimuru_get_device_error(r.ev) == R.DEV_OK
    finally:
        r.close()
