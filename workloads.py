"""Seeded synthetic inputs for the paged fused-MoE layer.

This module only draws random numbers and lays bytes out in a host copy of the
shared pool.  It holds none of the layer's arithmetic (no routing, no GEMM, no
activation, no combine), so both the CPU oracle and the CUDA path can take their
inputs from it without sharing any of the method.

Shapes follow Table 1 of the Rimuru page (per-expert projection, KV and state shapes of
two models): Qwen3-30B-A3B experts w1, w3 [2048, 768] and w2 [768, 2048];
Qwen3.5-35B-A3B experts w1, w3 [2048, 512], w2 [512, 2048]; KV [2, 4, 128] per
token.  Pages of the pool follow the explainer's description of memory views
(one page size and one page table per tensor type over one shared pool) and of
huge pages split into expert-sized and KV-sized pages.

Recipes (all seeded, all bf16 bit patterns stored as uint16):
  * x ~ N(0, 1); router gate Wg [E, H] ~ N(0, 0.02); logits = x @ Wg.T computed
    in float64 from the bf16 x and rounded to fp32 (optionally plus a per-expert
    bias that makes expert popularity Zipf-like);
  * expert weights ~ N(0, 0.02), one projection per expert-view page, row-major;
  * every pool byte that holds no expert or KV data is the bf16 NaN 0x7FC0, so an
    out-of-page read shows up as NaN in the output;
  * KV blocks (mixed pool) hold N(0, 1) bf16 noise.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace

import numpy as np
import torch

KiB = 1024
MiB = 1024 * 1024
BF16_NAN = 0x7FC0


def to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """fp32/fp64 array -> bf16 bit patterns (round to nearest even), via torch."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> fp32 (exact widening)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


@dataclass
class MoEShape:
    H: int
    I: int
    E: int
    k: int
    renorm: bool = True


@dataclass
class Workload:
    """One synthetic layer: inputs, the host copy of the pool and its page table."""
    name: str
    shape: MoEShape
    T: int
    x_bits: np.ndarray            # uint16 [T, H]
    logits: np.ndarray            # float32 [T, E]
    pool: np.ndarray              # uint8 [pool_bytes]
    page_bytes: int               # expert-view page size
    huge_page_bytes: int
    page_table: np.ndarray        # int32 [E, 3] expert-view page ids (w1, w3, w2)
    kv_page_bytes: int = 0
    kv_pages: np.ndarray = field(default_factory=lambda: np.zeros(0, np.int64))
    free_value: int = BF16_NAN
    notes: dict = field(default_factory=dict)

    @property
    def pool_bytes(self) -> int:
        return int(self.pool.nbytes)

    @property
    def A(self) -> int:
        return self.T * self.shape.k


def _rng(seed: int, stream: str) -> np.random.Generator:
    # independent, reproducible stream per component
    tag = int.from_bytes(stream.encode(), "little") % (2**63)
    return np.random.default_rng(np.random.SeedSequence([seed, tag]))


def make_x(seed: int, T: int, H: int) -> np.ndarray:
    return to_bf16_bits(_rng(seed, "x").standard_normal((T, H), dtype=np.float32))


def make_logits(seed: int, x_bits: np.ndarray, E: int, gate_std: float = 0.02,
                bias: np.ndarray | None = None) -> np.ndarray:
    H = x_bits.shape[1]
    wg = _rng(seed, "gate").standard_normal((E, H)) * gate_std
    x = bf16_bits_to_f32(x_bits).astype(np.float64)
    logits = x @ wg.T
    if bias is not None:
        logits = logits + bias[None, :]
    return logits.astype(np.float32)


def zipf_ranks(seed: int, E: int) -> np.ndarray:
    """Popularity rank (1 = most popular) of each expert: a seeded permutation of 1..E."""
    return _rng(seed, "zipf").permutation(E) + 1


def zipf_bias(seed: int, E: int, s: float = 1.1, gamma: float = 0.5) -> np.ndarray:
    """Per-expert logit bias b_e = gamma * ln(r_e^-s).  With x Wg noise of std ~0.9 and
    top-8 of 128 experts, gamma = 0.5 makes the realised per-expert assignment counts fall
    off as rank^-1.1 (fitted exponent ~1.11 at 8192 tokens)."""
    r = zipf_ranks(seed, E)
    return gamma * (-s) * np.log(r.astype(np.float64))


def make_expert_weights(seed: int, shape: MoEShape, std: float = 0.02):
    """Contiguous bf16 weights: w1, w3 [E, H, I] and w2 [E, I, H] (uint16 bits)."""
    g = _rng(seed, "experts")
    E, H, I = shape.E, shape.H, shape.I
    w1 = np.empty((E, H, I), np.uint16)
    w3 = np.empty((E, H, I), np.uint16)
    w2 = np.empty((E, I, H), np.uint16)
    for e in range(E):
        w1[e] = to_bf16_bits(g.standard_normal((H, I), dtype=np.float32) * std)
        w3[e] = to_bf16_bits(g.standard_normal((H, I), dtype=np.float32) * std)
        w2[e] = to_bf16_bits(g.standard_normal((I, H), dtype=np.float32) * std)
    return w1, w3, w2


def empty_pool(pool_bytes: int, fill_bits: int = BF16_NAN) -> np.ndarray:
    pool = np.empty(pool_bytes // 2, np.uint16)
    pool.fill(fill_bits)
    return pool.view(np.uint8)


def write_page(pool: np.ndarray, page_bytes: int, page_id: int, bits: np.ndarray) -> None:
    raw = np.ascontiguousarray(bits, dtype=np.uint16).view(np.uint8).ravel()
    assert raw.nbytes <= page_bytes
    start = page_id * page_bytes
    pool[start:start + raw.nbytes] = raw


def place_experts(pool: np.ndarray, page_bytes: int, slots: np.ndarray, w1, w3, w2) -> np.ndarray:
    """Write expert e's (w1, w3, w2) to pages slots[3e], slots[3e+1], slots[3e+2]."""
    E = w1.shape[0]
    pt = np.asarray(slots[:3 * E], np.int32).reshape(E, 3)
    for e in range(E):
        write_page(pool, page_bytes, int(pt[e, 0]), w1[e])
        write_page(pool, page_bytes, int(pt[e, 1]), w3[e])
        write_page(pool, page_bytes, int(pt[e, 2]), w2[e])
    return pt


def build_simple(name: str, shape: MoEShape, T: int, pool_pages: int, seed: int,
                 bias: np.ndarray | None = None, weights=None, page_bytes: int | None = None,
                 x_bits: np.ndarray | None = None, logits: np.ndarray | None = None) -> Workload:
    """A pool whose huge page is the expert page; the 3E projections sit at seeded random
    slots of a ``pool_pages``-page pool and every other page is NaN."""
    H, I, E = shape.H, shape.I, shape.E
    if page_bytes is None:
        page_bytes = H * I * 2
    assert 3 * E <= pool_pages
    if x_bits is None:
        x_bits = make_x(seed, T, H)
    if logits is None:
        logits = make_logits(seed, x_bits, E, bias=bias)
    if weights is None:
        weights = make_expert_weights(seed, shape)
    pool = empty_pool(pool_pages * page_bytes)
    slots = _rng(seed, "placement").permutation(pool_pages)
    pt = place_experts(pool, page_bytes, slots, *weights)
    return Workload(name, shape, T, x_bits, logits, pool, page_bytes, page_bytes, pt,
                    notes={"pool_pages": pool_pages, "seed": seed})


def build_mixed(shape: MoEShape, T: int, seed: int, kv_huge_pages: int | None = None,
                free_huge_pages: int = 64, kv_page_bytes: int = 32 * KiB,
                weights=None) -> Workload:
    """Mixed pool: huge page = expert page; a seeded-random subset of huge pages is split
    into KV blocks of ``kv_page_bytes`` holding N(0,1) bf16 noise, the expert pages sit in
    the other huge pages in seeded order, and ``free_huge_pages`` stay NaN."""
    H, I, E = shape.H, shape.I, shape.E
    page_bytes = H * I * 2
    n_exp = 3 * E
    if kv_huge_pages is None:
        kv_huge_pages = n_exp
    n_huge = n_exp + kv_huge_pages + free_huge_pages
    pool = empty_pool(n_huge * page_bytes)
    order = _rng(seed, "placement").permutation(n_huge)
    kv_huge = np.sort(order[:kv_huge_pages])
    exp_slots = order[kv_huge_pages:kv_huge_pages + n_exp]
    g = _rng(seed, "kv")
    per = page_bytes // kv_page_bytes
    kv_pages = []
    for hp in kv_huge:
        noise = to_bf16_bits(g.standard_normal(page_bytes // 2, dtype=np.float32))
        write_page(pool, page_bytes, int(hp), noise)
        kv_pages.extend(range(int(hp) * per, int(hp) * per + per))
    if weights is None:
        weights = make_expert_weights(seed, shape)
    pt = place_experts(pool, page_bytes, exp_slots, *weights)
    x_bits = make_x(seed, T, H)
    logits = make_logits(seed, x_bits, E)
    return Workload("q35_mixed_pool", shape, T, x_bits, logits, pool, page_bytes, page_bytes, pt,
                    kv_page_bytes=kv_page_bytes, kv_pages=np.asarray(kv_pages, np.int64),
                    notes={"huge_pages": n_huge, "kv_huge_pages": kv_huge_pages,
                           "free_huge_pages": free_huge_pages, "seed": seed})


@dataclass
class OffloadStack:
    """Host image of every expert page of an L-layer stack plus per-(step, layer) inputs.
    Projection p of expert e in layer l is host page (l * E + e) * 3 + p."""
    shape: MoEShape
    L: int
    T: int
    steps: int
    page_bytes: int
    host_pages: np.ndarray        # uint8 [L * E * 3 * page_bytes]
    x_bits: list                  # [steps][L] uint16 [T, H]
    logits: list                  # [steps][L] float32 [T, E]

    def layer_table(self, layer: int) -> np.ndarray:
        E = self.shape.E
        return (np.arange(E * 3, dtype=np.int32) + layer * E * 3).reshape(E, 3)


def offload_stack(shape: MoEShape, L: int, T: int, steps: int, seed: int,
                  distinct_layers: int | None = None, host: np.ndarray | None = None,
                  distinct_inputs: int | None = None) -> OffloadStack:
    """Seeded stack.  With ``distinct_layers = d``, layer l copies the values of layer l % d
    with the lowest mantissa bit flipped when (l // d) is odd (cheap to make for 48 layers of
    Qwen3 size); None gives every layer its own draws.  ``host`` may be a caller buffer
    (e.g. pinned) of the right size.  With ``distinct_inputs = n`` only n (x, logits) pairs
    are drawn and (step, layer) uses pair (step * L + layer) % n."""
    H, I, E = shape.H, shape.I, shape.E
    pb = H * I * 2
    if host is None:
        host = np.empty(L * E * 3 * pb, np.uint8)
    assert host.dtype == np.uint8 and host.size == L * E * 3 * pb
    words = host.view(np.uint16).reshape(L, E, 3, H * I)
    d = L if distinct_layers is None else distinct_layers
    for l in range(L):
        if l < d:
            w1, w3, w2 = make_expert_weights(seed * 1000 + l, shape)
            words[l, :, 0] = w1.reshape(E, -1)
            words[l, :, 1] = w3.reshape(E, -1)
            words[l, :, 2] = w2.reshape(E, -1)
        else:
            np.bitwise_xor(words[l % d], np.uint16(l // d & 1), out=words[l])
    n = steps * L if distinct_inputs is None else distinct_inputs
    px = [make_x(seed * 7919 + i, T, H) for i in range(n)]
    pl = [make_logits(seed * 7919 + i, px[i], E) for i in range(n)]
    xs = [[px[(s * L + l) % n] for l in range(L)] for s in range(steps)]
    lg = [[pl[(s * L + l) % n] for l in range(L)] for s in range(steps)]
    return OffloadStack(shape, L, T, steps, pb, host, xs, lg)


def with_inputs(w: Workload, name: str, T: int, x_bits: np.ndarray, logits: np.ndarray,
                notes: dict | None = None) -> Workload:
    """The same pool and page table with another batch of inputs (no copy of the pool)."""
    return replace(w, name=name, T=T, x_bits=x_bits, logits=logits,
                   notes={**w.notes, **(notes or {})})


def q3_prefill_inputs(seed: int = 0, T: int = 8192, gamma: float = 0.5):
    """x and logits of q3_prefill_zipf without building its pool (which equals
    q3_decode's pool at the same seed and pool size)."""
    x = make_x(seed, T, Q3.H)
    return x, make_logits(seed, x, Q3.E, bias=zipf_bias(seed, Q3.E, 1.1, gamma))


# Named configurations -------------------------------------------------------------

TINY = MoEShape(H=256, I=128, E=8, k=2)
Q3 = MoEShape(H=2048, I=768, E=128, k=8)
Q35 = MoEShape(H=2048, I=512, E=256, k=8)


def tiny(seed: int = 0, T: int = 16) -> Workload:
    """hidden 256, intermediate 128, 8 experts, top-2, 16 tokens; 64 KiB pages in a 64-page pool."""
    return build_simple("tiny", TINY, T, pool_pages=64, seed=seed)


def q3_decode(seed: int = 0, T: int = 64, pool_pages: int = 1024) -> Workload:
    """Qwen3-30B-A3B-shaped layer, 64 decode tokens; 384 pages of 3 MiB in a 1024-page pool."""
    return build_simple("q3_decode", Q3, T, pool_pages=pool_pages, seed=seed)


def q3_prefill_zipf(seed: int = 0, T: int = 8192, gamma: float = 0.5,
                    pool_pages: int = 1024) -> Workload:
    """Same layer, 8192 prefill tokens, expert popularity skewed by a Zipf(1.1) logit bias."""
    w = build_simple("q3_prefill_zipf", Q3, T, pool_pages=pool_pages, seed=seed,
                     bias=zipf_bias(seed, Q3.E, 1.1, gamma))
    w.notes["zipf_gamma"] = gamma
    return w


def q35_mixed_pool(seed: int = 0, T: int = 16) -> Workload:
    """Qwen3.5-35B-A3B-shaped layer (E 256, I 512) whose 2 MiB expert pages interleave with
    huge pages split into 32 KiB KV blocks (16 tokens x [2, 4, 128] bf16)."""
    return build_mixed(Q35, T, seed)


CONFIGS = {
    "tiny": tiny,
    "q3_decode": q3_decode,
    "q3_prefill_zipf": q3_prefill_zipf,
    "q35_mixed_pool": q35_mixed_pool,
}
