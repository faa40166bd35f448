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
from gpu_harness import Runner, rel_err
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


def run_gpu(w):
    r = Runner(w)
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


def test_q3_prefill_zipf_sampled(oracle):
    """8192 prefill tokens with Zipf(1.1)-skewed routing: routing, permutation and tiles for
    all tokens; h, y and out for 48 sampled tokens (the oracle computes them one by one)."""
    w = wl.q3_prefill_zipf(0)
    tokens = np.sort(np.random.default_rng(0).choice(w.T, 48, replace=False))
    o = run_oracle(oracle, w, tokens=tokens)
    counts = np.diff(o["offsets"])
    s = zipf_exponent(counts, wl.zipf_ranks(0, w.shape.E))
    assert 0.9 <= s <= 1.3, f"realised popularity exponent {s:.2f}"
    check(run_gpu(w), w, o, tokens=tokens)


def test_q3_prefill_heavy_skew_sampled(oracle):
    """A steeper bias (gamma 2): 38 of 128 experts get every assignment, the rest are empty,
    and the hottest expert holds all 8192 tokens (64 row blocks)."""
    w = wl.q3_prefill_zipf(0, gamma=2.0)
    tokens = np.sort(np.random.default_rng(2).choice(w.T, 32, replace=False))
    o = run_oracle(oracle, w, tokens=tokens)
    counts = np.diff(o["offsets"])
    assert (counts == 0).sum() >= 1 and counts.max() == w.T
    check(run_gpu(w), w, o, tokens=tokens)


@pytest.mark.parametrize("T", [1, 16, 256])
def test_q35_mixed_pool(oracle, T):
    """Qwen3.5-35B-A3B-shaped layer (256 experts, I = 512) in a pool whose huge pages are
    partly split into 32 KiB KV blocks full of random data."""
    w = wl.q35_mixed_pool(0, T=T)
    check(run_gpu(w), w, run_oracle(oracle, w))


def test_q35_mixed_pool_4096_sampled(oracle):
    w = wl.q35_mixed_pool(0, T=4096)
    tokens = np.sort(np.random.default_rng(1).choice(w.T, 32, replace=False))
    check(run_gpu(w), w, run_oracle(oracle, w, tokens=tokens), tokens=tokens)


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
    r = Runner(w)
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
