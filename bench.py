"""Benchmark of the paged fused-MoE layer (one GB300, or N independent replicas).

python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

A step is one pass of the whole layer (route, align, GEMM 1 + SwiGLU with the gather of its
rows, GEMM 2, combine) over one batch of synthetic tokens, through the C ABI on device-resident
inputs.
The default workload is the Qwen3-30B-A3B-shaped layer with 64 decode tokens; its expert
pages (about 1.2 GB touched per step) exceed the 129 MB L2, so no flush is needed between
steps.  On one GPU the default line also carries the 8192-token prefill of the same layer, the
Qwen3.5-shaped layer at 1 / 16 / 256 / 4096 tokens and the 48-layer offloaded stack.  Rank 0 prints one JSON line.  ``--impl reference`` times the CPU oracle on the
host cores instead (a deliberately slow baseline, not a target).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged fused-MoE tokens/s; % of HBM / bf16 tensor roofline (Qwen3-30B-A3B)"
DEFAULT_STEPS = {"q3_decode": 2000, "q3_prefill_zipf": 100, "q35_mixed_pool": 500, "tiny": 2000,
                 "q3_stack_offload": 32}
# kernels one layer launches, in order
LAYER_KERNELS = ("moe_route", "moe_align", "moe_gemm1_swiglu", "moe_gemm2", "moe_combine")
PROFILE_EVERY = 10      # timed forwards per forward whose dominant kernel is bracketed
REF_DEFAULT_STEPS = 20  # oracle steps when --impl reference is given no --steps
REF_SECONDS = 120.0     # host time the oracle arm aims for, warm-up included
WORKLOAD_TEXT = {
    "q3_decode": "Qwen3-30B-A3B-shaped MoE layer, decode: hidden 2048, moe intermediate 768, "
                 "128 experts, top-8 renormalised, 64 tokens; each w1/w3/w2 one 3 MiB page "
                 "shuffled across a 1024-page pool, unused pages NaN",
    "q3_prefill_zipf": "same Qwen3-30B-A3B-shaped layer, prefill: 8192 tokens, router logits "
                       "= x.Wg + per-expert Zipf(s=1.1) bias",
    "q35_mixed_pool": "Qwen3.5-35B-A3B-shaped MoE layer: hidden 2048, intermediate 512, 256 "
                      "experts, top-8; 2 MiB expert pages interleaved with huge pages split "
                      "into 32 KiB KV blocks",
    "tiny": "tiny paged MoE layer: hidden 256, intermediate 128, 8 experts, top-2, 16 tokens",
    "q3_stack_offload": "48-layer stack of Qwen3-30B-A3B-shaped MoE layers (MoE only), 256 "
                        "decode tokens per step, expert view capped at 25% of all expert pages; "
                        "misses copied from pinned host memory on a side stream, next layer "
                        "prefetched during the current one, LRU eviction",
}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained", p["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


class ClockSampler:
    """nvidia-smi sampling of SM clocks, throttle reasons and utilisation while the GPU legs
    run.  A sample is under load when nvidia-smi saw a kernel executing in its period
    (utilization.gpu > 0); the median SM clock is taken over those samples."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,"
              "utilization.gpu")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"rimuru_clocks_{os.getpid()}_{id(self)}.csv")

    def start(self):
        try:
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.close()
        mhz, loaded, maxmhz, reasons = [], [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 10:
                    continue
                try:
                    clk = float(parts[1])
                    maxmhz = max(maxmhz, float(parts[2]))
                    util = float(parts[9])
                except ValueError:
                    continue
                mhz.append(clk)
                if util > 0:
                    loaded.append(clk)
                for n, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        os.remove(self.path)
        if not mhz:
            return None
        return {"sm_mhz": statistics.median(loaded or mhz), "sm_max_mhz": maxmhz,
                "reasons": sorted(reasons), "samples": len(mhz),
                "samples_under_load": len(loaded),
                "window": "every GPU leg of this run (timed region, bracketed pass, e2e, "
                          "graph replays, and the prefill and sweep blocks of a default "
                          "one-GPU run; its offload block runs before the window)"}


def source_digest(*rel_paths):
    h = hashlib.sha256()
    for p in rel_paths:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


GEMM_SOURCES = ("paged_moe_shared_gb300/csrc/moe_gemm.cu",
                "paged_moe_shared_gb300/csrc/moe_gemm_2sm.cu",
                "paged_moe_shared_gb300/csrc/moe_gemm_wide.cu",
                "paged_moe_shared_gb300/csrc/device.cuh")


def ncu_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on the current
    kernel source; otherwise None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        t = json.load(f)
    rec = t.get(workload, {}).get(kernel)
    if not rec or rec.get("source_digest") != source_digest(*GEMM_SOURCES):
        return None
    return rec.get("dram_bytes_per_launch")


def make_workload(args):
    import workloads as wl
    kw = {"seed": args.seed}
    if args.tokens is not None:
        kw["T"] = args.tokens
    if args.pool_pages is not None:
        kw["pool_pages"] = args.pool_pages
    if args.zipf_gamma is not None:
        kw["gamma"] = args.zipf_gamma
    return wl.CONFIGS[args.workload](**kw)


def kernel_work(w, counts):
    """Algorithmic bytes and flops per launch of each kernel (no padding, no re-reads)."""
    s = w.shape
    T, H, I, E, k = w.T, s.H, s.I, s.E, s.k
    A = T * k
    U = int((counts > 0).sum())
    return {
        "moe_route": {"bytes": T * E * 4 + A * 8, "flops": 0},
        "moe_align": {"bytes": A * 4 * 3, "flops": 0},
        "moe_route_align_gather": {"bytes": T * E * 4 + A * 8 + A * 4 * 3 + 2 * A * H * 2,
                                   "flops": 0},
        "moe_gemm1_swiglu": {"bytes": U * 2 * H * I * 2 + A * H * 2 + A * I * 2,
                             "flops": 2 * A * H * 2 * I},
        "moe_gemm2": {"bytes": U * I * H * 2 + A * I * 2 + A * H * 2, "flops": 2 * A * I * H},
        "moe_combine": {"bytes": A * H * 2 + T * H * 2 + A * 8, "flops": 2 * A * H},
        # decode path: decode_gemm1 streams W1/W3 into shared memory and prefetches the W2
        # pages into L2 (it moves every weight byte of the layer from HBM), decode_gemm2
        # reads W2 back from L2
        "moe_decode_gemm1": {"bytes": U * 3 * H * I * 2 + T * E * 4 + T * H * 2,
                             "flops": 2 * A * H * 2 * I},
        "moe_decode_reduce": {"bytes": A * I * 2, "flops": 0},
        "moe_decode_gemm2": {"bytes": U * I * H * 2 + A * I * 2 + T * H * 2,
                             "flops": 2 * A * I * H + 2 * A * H},
        "layer": {"bytes": U * 3 * H * I * 2 + T * H * 2 + T * E * 4 + T * H * 2,
                  "flops": 6 * A * H * I},
        "U": U,
    }


def run_offload(args, rank, world, local_rank):
    """48-layer offloaded stack: a step runs all layers once over T tokens; before layer l's
    forward every expert of layer l + 1 is prefetched (routing at 256 tokens touches nearly
    all of them).  Bound by the host-to-device link, measured in the same run.  The line's
    value uses least-recently-used eviction (the configuration's policy); the layer-cycle
    policy is measured on the same stack and reported beside it."""
    import torch

    import workloads as wl
    from paged_moe_shared_gb300 import rimuru as R
    from paged_moe_shared_gb300.device_pool import DevicePool

    torch.cuda.set_device(local_rank)
    dev = f"cuda:{local_rank}"
    shape = wl.Q3
    L, T = 48, (args.tokens or 256)
    E, H, I = shape.E, shape.H, shape.I
    cap = L * E // 4
    pb = H * I * 2
    host = torch.empty(L * E * 3 * pb, dtype=torch.uint8, pin_memory=True)
    st = wl.offload_stack(shape, L, T, 1, args.seed, distinct_layers=1, host=host.numpy(),
                          distinct_inputs=8)
    pool = DevicePool((3 * cap + 16) * pb, pb, dev)
    pool.mem.view(torch.int16).fill_(wl.BF16_NAN)
    ev = pool.view(pb)
    R.rimuru_view_set_moe_shape(ev, L, E, H, I, shape.k, shape.renorm)
    xs = [torch.from_numpy(st.x_bits[0][i].view(np.int16)).view(torch.bfloat16).to(dev)
          for i in range(8)]
    lgs = [torch.from_numpy(st.logits[0][i]).to(dev) for i in range(8)]
    out = torch.empty_like(xs[0])
    ws_bytes = R.rimuru_moe_workspace_bytes(ev, T)
    ws_raw = torch.empty(ws_bytes + 1024, dtype=torch.uint8, device=dev)
    ws_ptr = (ws_raw.data_ptr() + 1023) // 1024 * 1024
    stream = torch.cuda.current_stream()
    all_experts = list(range(E))
    K = args.steps
    clocks = ClockSampler(local_rank)
    clocks.start()

    def run_policy(policy):
        off = R.rimuru_offload_create(ev, host.data_ptr(), cap, 0)
        R.rimuru_offload_set_policy(off, policy)

        def one_step(step):
            for l in range(L):
                R.rimuru_offload_prefetch(off, (l + 1) % L, all_experts)
                i = (step * L + l) % 8
                R.rimuru_offload_forward(off, xs[i].data_ptr(), lgs[i].data_ptr(), T, l,
                                         out.data_ptr(), ws_ptr, ws_bytes, stream.cuda_stream)

        try:
            for w in range(args.warmup):
                one_step(w)
            torch.cuda.synchronize()
            c0 = R.rimuru_offload_stats(off)
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for k_ in range(K):
                one_step(args.warmup + k_)
            e1.record(stream)
            torch.cuda.synchronize()
            wall = time.perf_counter() - t0
            ms = e0.elapsed_time(e1)
            c1 = R.rimuru_offload_stats(off)
            if R.rimuru_get_device_error(ev) != R.DEV_OK:
                raise RuntimeError("device error in the timed region")
        finally:
            R.rimuru_offload_destroy(off)
        return ms, {k: c1[k] - c0[k] for k in c1}, wall

    ms_lru, d_lru, wall_lru = run_policy(R.EVICT_LRU)
    ms_cyc, d_cyc, wall_cyc = run_policy(R.EVICT_LAYER_CYCLE)
    clk = clocks.stop()
    # the link, measured the way the cache uses it: pinned host -> device, large copies
    src = host[: 1 << 30]
    dst = torch.empty(1 << 30, dtype=torch.uint8, device=dev)
    for _ in range(2):
        dst.copy_(src, non_blocking=True)
    b0, b1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    b0.record(stream)
    for _ in range(5):
        dst.copy_(src, non_blocking=True)
    b1.record(stream)
    torch.cuda.synchronize()
    link_gbs = 5 * (1 << 30) / (b0.elapsed_time(b1) / 1e3) / 1e9
    pool.close()

    def roof(d, ms):
        a = d["bytes_h2d"] / (ms / 1e3) / 1e9
        return {"bound": "h2d", "achieved": round(a, 1), "peak": round(link_gbs, 1),
                "unit": "GB/s", "frac": round(a / link_gbs, 4), "traffic": None,
                "peak_source": "pinned host->device copy measured in this run"}

    return {
        "metric": "offloaded 48-layer paged MoE stack tokens/s (Qwen3-30B-A3B layers)",
        "value": round(T * K / (ms_lru / 1e3), 1), "unit": "tokens/s", "n_gpus": 1, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(ms_lru / K, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"q3_stack_offload: {WORKLOAD_TEXT['q3_stack_offload']}",
                   "layers": L, "tokens": T, "resident_experts": cap, "eviction": "lru",
                   "host_pages_gib": round(host.numel() / 2**30, 1),
                   "l2": "inputs larger than L2 (the stack reads 54 GiB of expert pages)"},
        "roofline": roof(d_lru, ms_lru),
        "cache": {k: int(v) for k, v in d_lru.items()},
        "wall_s": round(wall_lru, 3),
        "layer_cycle": {"value": round(T * K / (ms_cyc / 1e3), 1), "unit": "tokens/s",
                        "ms_per_step": round(ms_cyc / K, 3), "eviction": "layer_cycle",
                        "roofline": roof(d_cyc, ms_cyc),
                        "cache": {k: int(v) for k, v in d_cyc.items()},
                        "wall_s": round(wall_cyc, 3)},
        "clocks": clk,
        "gpu_launches": len(LAYER_KERNELS) * L * K,
    }


def max_over_ranks(ms, dist, device):
    """The slowest rank's time: the job has finished only when every replica has."""
    if dist is None:
        return ms
    import torch
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


L2_BYTES = 129e6


def layers_to_cycle(w) -> int:
    """Copies of the layer to cycle over so that one cycle reads at least 3x the L2 size:
    1 when even the fewest experts a step can touch, min(E, T*k), already read that much."""
    s = w.shape
    step_bytes = min(s.E, w.T * s.k) * 3 * s.H * s.I * 2
    if step_bytes >= 2 * L2_BYTES:
        return 1
    return int(min(256, -(-3 * L2_BYTES // step_bytes)))


def workload_config(w, args_workload, seed, U, n_layers, layer_bytes, world):
    """The `config` object of a line: the same dict from both arms for the same workload."""
    return {"workload": f"{args_workload}: {WORKLOAD_TEXT[args_workload]}", "tokens": w.T,
            "experts_touched": int(U), "seed": seed,
            "l2": "inputs larger than L2: the expert pages read per step exceed 129 MB"
            if n_layers == 1 else
            f"a layer's pages fit in L2, so steps cycle over {n_layers} copies of the "
            f"layer (same weights, distinct pool pages): "
            f"{n_layers * layer_bytes / 1e6:.0f} MB per cycle",
            "parallelism": "replicas" if world > 1 else "single GPU"}


def roofline_of(work, kernel, ms, peaks, bound):
    """Algorithmic work of one launch over its mean CUDA-event duration, against the
    measured peak: HBM copy GB/s, or bf16 TFLOP/s both as a burst (a kernel timed on its
    own, short loop: this one governs here) and sustained (a seconds-long loop)."""
    t = ms / 1e3
    if bound == "hbm":
        a = work[kernel]["bytes"] / t / 1e9
        return {"bound": "hbm", "achieved": round(a, 1), "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": round(a / peaks["hbm_gbs"], 4),
                "peak_source": peaks["source"] + " (HBM copy)"}
    a = work[kernel]["flops"] / t / 1e12
    return {"bound": "tensor", "achieved": round(a, 1), "peak": peaks["bf16_tflops"],
            "unit": "TFLOP/s", "frac": round(a / peaks["bf16_tflops"], 4),
            "peak_sustained": peaks["bf16_tflops_sustained"],
            "frac_of_sustained": round(a / peaks["bf16_tflops_sustained"], 4),
            "peak_source": peaks["source"] + " (bf16 burst; the loop timed here is short)"}


class Layer:
    """A workload placed in a device pool, with its inputs, output and workspace."""

    def __init__(self, w, dev, n_layers=1, pool=None, ev=None, decode_tokens=None):
        import torch

        from paged_moe_shared_gb300 import rimuru as R
        from paged_moe_shared_gb300.device_pool import load_workload, replicate_layers
        self.R = R
        self.w = w
        self.dev = dev
        self.n_layers = n_layers
        self.own_pool = pool is None
        if pool is None:
            extra = (n_layers - 1) * 3 * w.shape.E
            pool, ev, _ = load_workload(w, dev, layers=n_layers, extra_pages=extra)
            replicate_layers(pool, ev, w, n_layers)
        self.pool, self.ev = pool, ev
        if decode_tokens is not None:
            R.rimuru_view_set_decode_tokens(ev, decode_tokens)
        self.counter = 0
        self.x = torch.from_numpy(w.x_bits.view(np.int16)).view(torch.bfloat16).to(dev)
        self.logits = torch.from_numpy(w.logits).to(dev)
        self.out = torch.empty_like(self.x)
        self.ws_bytes = R.rimuru_moe_workspace_bytes(ev, w.T)
        self.ws_raw = torch.empty(self.ws_bytes + 1024, dtype=torch.uint8, device=dev)
        self.ws_ptr = (self.ws_raw.data_ptr() + 1023) // 1024 * 1024
        self.stream = torch.cuda.current_stream()

    def step(self, on=None):
        layer = self.counter % self.n_layers
        self.counter += 1
        self.R.rimuru_moe_forward(self.x.data_ptr(), self.logits.data_ptr(), self.w.T, self.ev,
                                  layer, self.out.data_ptr(), self.ws_ptr, self.ws_bytes,
                                  (on or self.stream).cuda_stream)

    def counts(self):
        import torch
        lay = self.R.rimuru_moe_workspace_layout(self.ev, self.w.T)
        at = self.ws_ptr - self.ws_raw.data_ptr() + lay["offsets"]
        offs = self.ws_raw[at:at + (self.w.shape.E + 1) * 4].view(torch.int32).cpu().numpy()
        return np.diff(offs)

    def close(self):
        if self.own_pool:
            self.pool.close()


def measure(L, args, K, world, dist, dev, full=True):
    """Time K forwards of one layer (after args.warmup untimed ones): `value`, the per-kernel
    table, the dominant kernel in a bracketed pass, and (full) e2e and CUDA-graph legs."""
    import torch
    R = L.R
    w = L.w

    def barrier():
        if dist is not None:
            dist.barrier()

    for _ in range(args.warmup):
        L.step()
    torch.cuda.synchronize()
    if R.rimuru_get_device_error(L.ev) != R.DEV_OK:
        raise RuntimeError("device error during warm-up")
    work = kernel_work(w, L.counts())

    # -------------------------------------------- per-kernel table (untimed, all kernels)
    # Event pairs between kernels stop each kernel from overlapping its predecessor, so this
    # pass is separate from the timed region; it gives every kernel's share.
    Kp = min(K, 200)
    R.rimuru_profile_enable(L.ev, R.PROFILE_ALL, Kp)
    for _ in range(Kp):
        L.step()
    torch.cuda.synchronize()
    R.rimuru_profile_enable(L.ev, 0, 1)
    per_kernel = {}
    for kidx in range(R.K_COUNT):
        n, ms = R.rimuru_profile_read(L.ev, kidx)
        if n:  # kernels the layer's path does not launch report no launches
            per_kernel[R.rimuru_kernel_name(kidx)] = {"launches": n, "ms_per_launch": ms / n}
    launches_per_step = sum(v["launches"] for v in per_kernel.values()) // Kp
    gemms = [n for n in ("moe_gemm1_swiglu", "moe_gemm2", "moe_decode_gemm1", "moe_decode_gemm2")
             if n in per_kernel]
    dom = max(gemms, key=lambda n: per_kernel[n]["ms_per_launch"])
    names = [R.rimuru_kernel_name(i) for i in range(R.K_COUNT)]
    dom_idx = names.index(dom)

    # ---------------------------------------------------------------- timed region
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    t0.record(L.stream)
    for _ in range(K):
        L.step()
    t1.record(L.stream)
    torch.cuda.synchronize()
    barrier()
    ms_total = max_over_ranks(t0.elapsed_time(t1), dist, dev)
    if R.rimuru_get_device_error(L.ev) != R.DEV_OK:
        raise RuntimeError("device error in the timed region")
    ms_step = ms_total / K

    # ------------------------------------------- dominant kernel, bracketed pass
    # Right after the timed region, the same forwards with the dominant kernel bracketed by
    # an event pair on the launching stream in every one of them (a pair keeps that kernel
    # from overlapping its neighbours, so the timed region above is left unbracketed).
    Kb = max(K, 10)
    R.rimuru_profile_enable(L.ev, 1 << dom_idx, Kb)
    for _ in range(Kb):
        L.step()
    torch.cuda.synchronize()
    n_dom, ms_dom = R.rimuru_profile_read(L.ev, dom_idx)
    R.rimuru_profile_enable(L.ev, 0, 1)
    dom_ms = ms_dom / max(n_dom, 1)

    res = {"value": world * w.T * K / (ms_total / 1e3), "ms_per_step": ms_step, "work": work,
           "per_kernel": per_kernel, "dom": dom, "dom_ms": dom_ms, "n_dom": n_dom,
           "launches_per_step": launches_per_step, "Kp": Kp}
    if not full:
        return res

    # ---------------------------------------------------------------- end to end
    # Through rimuru_moe_forward_host: each step copies its x and logits in from pinned host
    # memory, runs the layer and copies out back to the host, all inside the timed region.
    # Steps alternate between two streams with their own workspace and host buffers (double
    # buffering, as a serving loop would), so one step's copies overlap the other's kernels;
    # the single-stream figure is reported beside it.
    Ke = min(K, args.e2e_steps)
    hws = R.rimuru_moe_host_workspace_bytes(L.ev, w.T)
    lanes = []
    for _ in range(2):
        raw = torch.empty(hws + 1024, dtype=torch.uint8, device=dev)
        lanes.append({
            "stream": torch.cuda.Stream(dev), "raw": raw,
            "ws": (raw.data_ptr() + 1023) // 1024 * 1024,
            "x": torch.from_numpy(w.x_bits.view(np.int16)).view(torch.bfloat16).pin_memory(),
            "logits": torch.from_numpy(w.logits).pin_memory(),
            "out": torch.empty(tuple(L.x.shape), dtype=torch.bfloat16).pin_memory()})

    def host_step(lane):
        layer = L.counter % L.n_layers
        L.counter += 1
        R.rimuru_moe_forward_host(lane["x"].data_ptr(), lane["logits"].data_ptr(), w.T, L.ev,
                                  layer, lane["out"].data_ptr(), lane["ws"], hws,
                                  lane["stream"].cuda_stream)

    def timed_host_steps(n_lanes):
        for i in range(3):
            host_step(lanes[i % n_lanes])
        torch.cuda.synchronize()
        barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(L.stream)
        for ln in lanes[:n_lanes]:
            ln["stream"].wait_event(e0)
        for i in range(Ke):
            host_step(lanes[i % n_lanes])
        for ln in lanes[:n_lanes]:
            L.stream.wait_stream(ln["stream"])
        e1.record(L.stream)
        torch.cuda.synchronize()
        barrier()
        return max_over_ranks(e0.elapsed_time(e1), dist, dev)

    ms_e2e_serial = timed_host_steps(1)
    ms_e2e = timed_host_steps(2)
    if R.rimuru_get_device_error(L.ev) != R.DEV_OK:
        raise RuntimeError("device error in the end-to-end steps")
    ref_out = L.out.cpu()
    for ln in lanes:  # same inputs, deterministic layer: the host results equal the device's
        if not torch.equal(ln["out"].view(torch.int16), ref_out.view(torch.int16)):
            raise RuntimeError("host-buffer forward disagrees with the device-buffer forward")
    res["e2e"] = {"value": round(world * w.T * Ke / (ms_e2e / 1e3), 1), "unit": "tokens/s",
                  "h2d_bytes_per_step": int(L.x.numel() * 2 + L.logits.numel() * 4),
                  "d2h_bytes_per_step": int(L.out.numel() * 2), "steps": Ke,
                  "ms_per_step": round(ms_e2e / Ke, 5),
                  "api": "rimuru_moe_forward_host (pinned host buffers)", "streams": 2,
                  "single_stream_value": round(world * w.T * Ke / (ms_e2e_serial / 1e3), 1)}
    del lanes

    # ------------------------------------------------------------ CUDA-graph replay
    # The same device-resident forwards recorded once by stream capture and replayed, as a
    # decode loop with fixed buffers would run them (reported beside `value`, which
    # launches every forward from the host).
    G = max(L.n_layers, 10)
    gs = torch.cuda.Stream(dev)
    gs.wait_stream(L.stream)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=gs):
        for _ in range(G):
            L.step(gs)
    reps = max(1, K // G)
    g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(gs):  # replay() launches on the current stream
        for _ in range(3):
            graph.replay()
        torch.cuda.synchronize()
        barrier()
        g0.record(gs)
        for _ in range(reps):
            graph.replay()
        g1.record(gs)
    torch.cuda.synchronize()
    barrier()
    ms_graph = max_over_ranks(g0.elapsed_time(g1), dist, dev)
    if R.rimuru_get_device_error(L.ev) != R.DEV_OK:
        raise RuntimeError("device error in the graph replays")
    res["cuda_graph"] = {"value": round(world * w.T * reps * G / (ms_graph / 1e3), 1),
                         "unit": "tokens/s", "ms_per_step": round(ms_graph / (reps * G), 5),
                         "forwards_per_graph": G, "replays": reps}
    del graph
    return res


def summarise(m, peaks, bound=None):
    """roofline (dominant kernel), layer_roofline and the per-kernel table of a measurement."""
    work, dom = m["work"], m["dom"]
    if bound is None:  # whichever of the kernel's byte time and flop time is longer
        bound = ("hbm" if work[dom]["bytes"] / (peaks["hbm_gbs"] * 1e9)
                 >= work[dom]["flops"] / (peaks["bf16_tflops"] * 1e12) else "tensor")
    roof = roofline_of(work, dom, m["dom_ms"], peaks, bound)
    roof.update({"kernel": dom, "ms_per_launch": round(m["dom_ms"], 5),
                 "launches_timed": m["n_dom"],
                 "timing": "CUDA events on the launching stream around every launch of this "
                           "kernel in a pass of forwards right after the timed region"})
    per_kernel = m["per_kernel"]
    total_k = sum(v["ms_per_launch"] for v in per_kernel.values())
    table = {}
    for name, v in per_kernel.items():
        tk = v["ms_per_launch"] / 1e3
        row = {"launches": v["launches"], "ms_per_launch": round(v["ms_per_launch"], 5),
               "share": round(v["ms_per_launch"] / total_k, 4) if total_k else None}
        if tk > 0:
            row["GB/s"] = round(work[name]["bytes"] / tk / 1e9, 1)
            if work[name]["flops"]:
                row["TFLOP/s"] = round(work[name]["flops"] / tk / 1e12, 1)
        table[name] = row
    lt = m["ms_per_step"] / 1e3
    layer = {"hbm_frac": round(work["layer"]["bytes"] / lt / 1e9 / peaks["hbm_gbs"], 4),
             "tensor_frac": round(work["layer"]["flops"] / lt / 1e12 / peaks["bf16_tflops"], 4),
             "tensor_frac_of_sustained": round(work["layer"]["flops"] / lt / 1e12
                                               / peaks["bf16_tflops_sustained"], 4)}
    return roof, layer, table


def run_ours(args, rank, world, local_rank):
    import torch

    import workloads as wl

    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    torch.cuda.set_device(local_rank)
    dev = f"cuda:{local_rank}"
    extra_blocks = (args.workload == "q3_decode" and not args.no_prefill and args.tokens is None
                    and args.pool_pages is None and world == 1)
    offload_block = None
    if extra_blocks:
        # the offloaded stack first, before this process holds anything else: its 54 GiB of
        # pinned host memory copied to the device ran slower when allocated after the other legs
        try:
            oargs = argparse.Namespace(**{**vars(args), "steps": 8, "warmup": 3,
                                          "tokens": None})
            off = run_offload(oargs, rank, world, local_rank)
            offload_block = {k: off[k] for k in ("metric", "value", "unit", "ms_per_step",
                                                 "steps", "warmup", "config", "roofline",
                                                 "cache", "layer_cycle", "gpu_launches")}
        except Exception as exc:  # host memory for the pinned stack, or the link
            offload_block = {"unavailable": f"{type(exc).__name__}: {exc}"[:300]}
    peaks = load_peaks()
    w = make_workload(args)
    # A layer whose expert pages fit in L2 would be re-read from L2 on every step; such
    # workloads cycle over identical copies of the layer at different pool addresses.
    n_layers = layers_to_cycle(w)
    L = Layer(w, dev, n_layers, decode_tokens=args.decode_tokens)
    clocks = ClockSampler(local_rank)  # from here on the run is GPU work (and host launches)
    clocks.start()
    K = args.steps
    m = measure(L, args, K, world, dist, dev)
    roof, layer_roof, table = summarise(m, peaks)
    roof["traffic"] = ncu_traffic(m["dom"], args.workload)
    work = m["work"]
    result = {
        "metric": METRIC, "value": round(m["value"], 1), "unit": "tokens/s", "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": round(m["ms_per_step"], 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": workload_config(w, args.workload, args.seed, work["U"], n_layers,
                                  work["layer"]["bytes"], world),
        "roofline": roof,
        "layer_roofline": layer_roof,
        "kernels": table,
        "kernels_note": f"per-kernel event pairs around every launch, {m['Kp']} untimed steps",
        "gpu_launches": m["launches_per_step"] * K,
        "e2e": m["e2e"],
        "cuda_graph": m["cuda_graph"],
    }

    # ------------------------------------------------------------ prefill block
    # The Qwen3-30B-A3B-shaped decode layer's pool is also the prefill layer's (same seed and
    # pool size give the same weights and placement), so the default run measures the
    # 8192-token Zipf prefill on the same pool, against the bf16 tensor peak.
    if args.workload == "q3_decode" and not args.no_prefill and args.tokens is None \
            and args.pool_pages is None:
        pre = {}
        for gamma in (0.5, 2.0):
            x, lg = wl.q3_prefill_inputs(args.seed, 8192, gamma)
            wp = wl.with_inputs(w, "q3_prefill_zipf", 8192, x, lg, {"zipf_gamma": gamma})
            Lp = Layer(wp, dev, 1, pool=L.pool, ev=L.ev)
            mp = measure(Lp, args, K, world, dist, dev, full=(gamma == 0.5))
            proof, player, ptable = summarise(mp, peaks, bound="tensor")
            c = Lp.counts()
            entry = {"value": round(mp["value"], 1), "unit": "tokens/s",
                     "ms_per_step": round(mp["ms_per_step"], 5), "steps": K,
                     "config": {**workload_config(wp, "q3_prefill_zipf", args.seed,
                                                  mp["work"]["U"], 1,
                                                  mp["work"]["layer"]["bytes"], world),
                                "zipf_gamma": gamma, "experts_empty": int((c == 0).sum()),
                                "assignments_per_expert": [int(c.min()), int(c.max())]},
                     "layer_roofline": player, "gpu_launches": mp["launches_per_step"] * K}
            if gamma == 0.5:
                proof["traffic"] = ncu_traffic(mp["dom"], "q3_prefill_zipf")
                entry.update({"roofline": proof, "kernels": ptable, "e2e": mp["e2e"],
                              "cuda_graph": mp["cuda_graph"]})
                if rank == 0 and not args.no_cpu_baseline:
                    entry["cpu_baseline"] = cpu_baseline(wp, args.cpu_seconds / 2)
                pre["gamma_0.5"] = entry
            else:
                entry["roofline"] = {k: proof[k] for k in ("kernel", "achieved", "frac",
                                                           "frac_of_sustained", "unit")}
                pre["gamma_2"] = entry
            Lp.close()
        result["prefill"] = {**pre["gamma_0.5"], "heavy_skew": pre["gamma_2"]}

    # --------------------------------------------- Qwen3.5 sweep and offload blocks
    # One GPU only (a replica run would multiply the offload stack's 54 GiB of pinned host
    # memory): the Qwen3.5-shaped layer in a pool shared with KV blocks at 1 / 16 / 256 /
    # 4096 tokens, and the 48-layer offloaded stack on its configured LRU policy, so that the
    # default line records them too.
    if extra_blocks:
        sweep = {}
        Ks = min(K, 500)
        for T in (1, 16, 256, 4096):
            ws = wl.q35_mixed_pool(args.seed, T=T)
            nl = layers_to_cycle(ws)
            Ls = Layer(ws, dev, nl)
            ms_ = measure(Ls, args, Ks, world, dist, dev, full=False)
            sroof, slayer, _ = summarise(ms_, peaks)
            sweep[f"T{T}"] = {"value": round(ms_["value"], 1), "unit": "tokens/s",
                              "ms_per_step": round(ms_["ms_per_step"], 5), "steps": Ks,
                              "layers_cycled": nl, "layer_roofline": slayer,
                              "roofline": {k: sroof[k] for k in ("kernel", "achieved", "frac",
                                                                 "unit", "bound")},
                              "gpu_launches": ms_["launches_per_step"] * Ks}
            Ls.close()
        result["q35_sweep"] = {"workload": f"q35_mixed_pool: {WORKLOAD_TEXT['q35_mixed_pool']}",
                               **sweep}
        result["offload"] = offload_block

    result["clocks"] = clocks.stop()
    if rank == 0 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(w, args.cpu_seconds)
    L.close()
    if dist is not None:
        dist.destroy_process_group()
    return result


def oracle_sample(w, tokens):
    import oracle
    o = oracle.Oracle()
    s = w.shape
    t0 = time.perf_counter()
    o.moe_forward(w.x_bits, w.logits, w.pool, w.page_bytes, w.page_table, s.H, s.I, s.k,
                  s.renorm, tokens=tokens)
    return time.perf_counter() - t0, o.max_threads()


def sample_tokens(w, budget_s):
    """Tokens per oracle step: enough to take roughly budget_s on the host cores, at most T."""
    n = min(w.T, 8)
    dt, cores = oracle_sample(w, np.arange(n))
    while n < w.T and dt < budget_s / 4:
        n = min(w.T, n * 4)
        dt, cores = oracle_sample(w, np.arange(n))
    return n, dt, cores


def cpu_baseline(w, budget_s):
    n, dt, cores = sample_tokens(w, budget_s)
    reps, total = 1, dt
    while total < budget_s * 0.5 and reps < 10000:
        d, _ = oracle_sample(w, np.arange(n))
        total += d
        reps += 1
    return {"value": round(n * reps / total, 3), "unit": "tokens/s", "cores": cores,
            "kind": "oracle",
            "sample": f"{n} of {w.T} tokens (all routing for {w.T}), {reps} pass(es), "
                      f"{total:.1f} s of CPU time"}


def run_reference(args):
    import oracle
    w = make_workload(args)
    # the same config object as the GPU arm: routing (for the experts touched) and the L2 rule
    o = oracle.Oracle()
    ids, _ = o.route(w.logits, w.shape.k, w.shape.renorm)
    counts = np.bincount(ids.ravel(), minlength=w.shape.E)
    U = int((counts > 0).sum())
    n_layers = layers_to_cycle(w)
    # every step is a sample of the workload's tokens, sized so that warm-up plus timed
    # steps take about REF_SECONDS on the host cores (one token per step at the least)
    per_step = REF_SECONDS / max(args.steps + args.warmup, 1)
    n, dt, cores = sample_tokens(w, budget_s=4 * per_step)
    while n > 1 and dt > per_step:
        n = max(1, n // 2)
        dt, cores = oracle_sample(w, np.arange(n))
    toks = np.arange(n)
    for _ in range(args.warmup):
        oracle_sample(w, toks)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_sample(w, toks)
    total = time.perf_counter() - t0
    value = n * args.steps / total
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "tokens/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(total / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(w, args.workload, args.seed, U, n_layers,
                                  kernel_work(w, counts)["layer"]["bytes"], 1),
        "where": "host cores",
        "cpu_baseline": {"value": round(value, 3), "unit": "tokens/s", "cores": cores,
                         "kind": "oracle",
                         "sample": f"{n} of {w.T} tokens per step (routing for all {w.T})"},
        "e2e": {"value": round(value, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="q3_decode", choices=sorted(WORKLOAD_TEXT))
    ap.add_argument("--tokens", type=int, default=None)
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--pool-pages", type=int, default=None,
                    help="pool size in expert pages (q3 workloads; default 1024)")
    ap.add_argument("--zipf-gamma", type=float, default=None,
                    help="scale of the Zipf logit bias (q3_prefill_zipf; default 0.5)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=500)
    ap.add_argument("--cpu-seconds", type=float, default=16.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--decode-tokens", type=int, default=None,
                    help="largest batch that takes the decode path (library default 4; 0: off)")
    ap.add_argument("--no-prefill", action="store_true",
                    help="q3_decode: skip the 8192-token prefill block of the default line")
    args = ap.parse_args()
    if args.steps is None:
        args.steps = REF_DEFAULT_STEPS if args.impl == "reference" else DEFAULT_STEPS[args.workload]
    args.warmup = max(args.warmup, 3)
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    local_rank = int(os.environ.get("LOCAL_RANK", 0))
    if world != args.gpus:
        world = max(world, 1)
    if args.impl == "reference":
        if rank != 0:
            return
        print(json.dumps(run_reference(args)), flush=True)
        return
    if args.workload == "q3_stack_offload":
        res = run_offload(args, rank, world, local_rank)
    else:
        res = run_ours(args, rank, world, local_rank)
    if rank == 0:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
