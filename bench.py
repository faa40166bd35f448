"""Benchmark of the paged fused-MoE layer (one GB300, or N independent replicas).

python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

A step is one pass of the whole layer (route, align, GEMM 1 + SwiGLU with the gather of its
rows, GEMM 2, combine) over one batch of synthetic tokens, through the C ABI on device-resident
inputs.
The default workload is the Qwen3-30B-A3B-shaped layer with 64 decode tokens; its expert
pages (about 1.2 GB touched per step) exceed the 129 MB L2, so no flush is needed between
steps.  Rank 0 prints one JSON line.  ``--impl reference`` times the CPU oracle on the
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
    """nvidia-smi sampling of SM clocks and throttle reasons while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"rimuru_clocks_{os.getpid()}.csv")

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
        mhz, maxmhz, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    mhz.append(float(parts[1]))
                    maxmhz = max(maxmhz, float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        os.remove(self.path)
        if not mhz:
            return None
        return {"sm_mhz": statistics.median(mhz), "sm_max_mhz": maxmhz,
                "reasons": sorted(reasons), "samples": len(mhz)}


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
        "layer": {"bytes": U * 3 * H * I * 2 + T * H * 2 + T * E * 4 + T * H * 2,
                  "flops": 6 * A * H * I},
        "U": U,
    }


def run_offload(args, rank, world, local_rank):
    """48-layer offloaded stack: a step runs all layers once over T tokens; before layer l's
    forward every expert of layer l + 1 is prefetched (routing at 256 tokens touches nearly
    all of them).  Bound by the host-to-device link, measured in the same run."""
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
    off = R.rimuru_offload_create(ev, host.data_ptr(), cap, 0)
    policy = R.EVICT_LAYER_CYCLE if args.evict == "layer_cycle" else R.EVICT_LRU
    R.rimuru_offload_set_policy(off, policy)
    xs = [torch.from_numpy(st.x_bits[0][i].view(np.int16)).view(torch.bfloat16).to(dev)
          for i in range(8)]
    lgs = [torch.from_numpy(st.logits[0][i]).to(dev) for i in range(8)]
    out = torch.empty_like(xs[0])
    ws_bytes = R.rimuru_moe_workspace_bytes(ev, T)
    ws_raw = torch.empty(ws_bytes + 1024, dtype=torch.uint8, device=dev)
    ws_ptr = (ws_raw.data_ptr() + 1023) // 1024 * 1024
    stream = torch.cuda.current_stream()
    all_experts = list(range(E))

    def one_step(step):
        for l in range(L):
            R.rimuru_offload_prefetch(off, (l + 1) % L, all_experts)
            i = (step * L + l) % 8
            R.rimuru_offload_forward(off, xs[i].data_ptr(), lgs[i].data_ptr(), T, l, out.data_ptr(),
                                     ws_ptr, ws_bytes, stream.cuda_stream)

    for w in range(args.warmup):
        one_step(w)
    torch.cuda.synchronize()
    c0 = R.rimuru_offload_stats(off)
    K = args.steps
    clocks = ClockSampler(local_rank)
    clocks.start()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for k_ in range(K):
        one_step(args.warmup + k_)
    e1.record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    clk = clocks.stop()
    ms = e0.elapsed_time(e1)
    c1 = R.rimuru_offload_stats(off)
    if R.rimuru_get_device_error(ev) != R.DEV_OK:
        raise RuntimeError("device error in the timed region")
    d = {k: c1[k] - c0[k] for k in c1}
    # the link, measured the same way the cache uses it: pinned host -> device, large copies
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
    achieved = d["bytes_h2d"] / (ms / 1e3) / 1e9
    R.rimuru_offload_destroy(off)
    pool.close()
    return {
        "metric": "offloaded 48-layer paged MoE stack tokens/s (Qwen3-30B-A3B layers)",
        "value": round(T * K / (ms / 1e3), 1), "unit": "tokens/s", "n_gpus": 1, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(ms / K, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"q3_stack_offload: {WORKLOAD_TEXT['q3_stack_offload']}",
                   "layers": L, "tokens": T, "resident_experts": cap, "eviction": args.evict,
                   "host_pages_gib": round(host.numel() / 2**30, 1),
                   "l2": "inputs larger than L2 (the stack reads 54 GiB of expert pages)"},
        "roofline": {"bound": "h2d", "achieved": round(achieved, 1), "peak": round(link_gbs, 1),
                     "unit": "GB/s", "frac": round(achieved / link_gbs, 4), "traffic": None,
                     "peak_source": "pinned host->device copy measured in this run"},
        "cache": {k: int(v) for k, v in d.items()},
        "wall_s": round(wall, 3), "clocks": clk,
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


def run_ours(args, rank, world, local_rank):
    import torch

    import workloads as wl
    from paged_moe_shared_gb300 import rimuru as R
    from paged_moe_shared_gb300.device_pool import load_workload, replicate_layers

    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    torch.cuda.set_device(local_rank)
    dev = f"cuda:{local_rank}"
    w = make_workload(args)
    # A layer whose expert pages fit in L2 would be re-read from L2 on every step; such
    # workloads cycle over identical copies of the layer at different pool addresses.
    n_layers = layers_to_cycle(w)
    extra = (n_layers - 1) * 3 * w.shape.E
    pool, ev, _ = load_workload(w, dev, layers=n_layers, extra_pages=extra)
    replicate_layers(pool, ev, w, n_layers)
    counter = [0]
    x = torch.from_numpy(w.x_bits.view(np.int16)).view(torch.bfloat16).to(dev)
    logits = torch.from_numpy(w.logits).to(dev)
    out = torch.empty_like(x)
    ws_bytes = R.rimuru_moe_workspace_bytes(ev, w.T)
    ws_raw = torch.empty(ws_bytes + 1024, dtype=torch.uint8, device=dev)
    ws_ptr = (ws_raw.data_ptr() + 1023) // 1024 * 1024
    stream = torch.cuda.current_stream()

    def step(on=None):
        layer = counter[0] % n_layers
        counter[0] += 1
        R.rimuru_moe_forward(x.data_ptr(), logits.data_ptr(), w.T, ev, layer, out.data_ptr(),
                             ws_ptr, ws_bytes, (on or stream).cuda_stream)

    def barrier():
        if dist is not None:
            dist.barrier()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if R.rimuru_get_device_error(ev) != R.DEV_OK:
        raise RuntimeError("device error during warm-up")
    lay = R.rimuru_moe_workspace_layout(ev, w.T)
    at = ws_ptr - ws_raw.data_ptr() + lay["offsets"]
    offs = ws_raw[at:at + (w.shape.E + 1) * 4].view(torch.int32).cpu().numpy()
    counts = np.diff(offs)
    work = kernel_work(w, counts)

    # -------------------------------------------- per-kernel table (untimed, all kernels)
    # Event pairs between kernels stop each kernel from overlapping its predecessor, so this
    # pass is separate from the timed region and only picks the dominant kernel.
    Kp = min(args.steps, 200)
    R.rimuru_profile_enable(ev, R.PROFILE_ALL, Kp)
    for _ in range(Kp):
        step()
    torch.cuda.synchronize()
    R.rimuru_profile_enable(ev, 0, 1)
    per_kernel = {}
    for kidx in range(R.K_COUNT):
        n, ms = R.rimuru_profile_read(ev, kidx)
        if n:  # kernels the layer's path does not launch report no launches
            per_kernel[R.rimuru_kernel_name(kidx)] = {"launches": n, "ms_per_launch": ms / n}
    launches_per_step = sum(v["launches"] for v in per_kernel.values()) // Kp
    dom = max(("moe_gemm1_swiglu", "moe_gemm2"), key=lambda n: per_kernel[n]["ms_per_launch"])
    dom_idx = [R.rimuru_kernel_name(i) for i in range(R.K_COUNT)].index(dom)

    # ---------------------------------------------------------------- timed region
    # The dominant kernel is bracketed by events (for the roofline) in one forward out of
    # PROFILE_EVERY: an event pair keeps the kernel from overlapping its neighbours, so
    # bracketing every forward would slow the measured step.
    K = args.steps
    R.rimuru_profile_enable_sampled(ev, 1 << dom_idx, -(-K // PROFILE_EVERY), PROFILE_EVERY)
    clocks = ClockSampler(local_rank)
    clocks.start()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    t0.record(stream)
    for _ in range(K):
        step()
    t1.record(stream)
    torch.cuda.synchronize()
    barrier()
    clk = clocks.stop()
    ms_total = t0.elapsed_time(t1)
    R.rimuru_profile_enable(ev, 0, 1)
    n_dom, ms_dom = R.rimuru_profile_read(ev, dom_idx)
    dom_ms_live = ms_dom / max(n_dom, 1)
    if R.rimuru_get_device_error(ev) != R.DEV_OK:
        raise RuntimeError("device error in the timed region")
    ms_total = max_over_ranks(ms_total, dist, dev)
    ms_step = ms_total / K
    value = world * w.T * K / (ms_total / 1e3)

    # ---------------------------------------------------------------- end to end
    # Through rimuru_moe_forward_host: each step copies its x and logits in from pinned host
    # memory, runs the layer and copies out back to the host, all inside the timed region.
    # Steps alternate between two streams with their own workspace and host buffers (double
    # buffering, as a serving loop would), so one step's copies overlap the other's kernels;
    # the single-stream figure is reported beside it.
    Ke = min(K, args.e2e_steps)
    hws = R.rimuru_moe_host_workspace_bytes(ev, w.T)
    lanes = []
    for _ in range(2):
        raw = torch.empty(hws + 1024, dtype=torch.uint8, device=dev)
        lanes.append({
            "stream": torch.cuda.Stream(dev), "raw": raw,
            "ws": (raw.data_ptr() + 1023) // 1024 * 1024,
            "x": torch.from_numpy(w.x_bits.view(np.int16)).view(torch.bfloat16).pin_memory(),
            "logits": torch.from_numpy(w.logits).pin_memory(),
            "out": torch.empty(tuple(x.shape), dtype=torch.bfloat16).pin_memory()})

    def host_step(lane):
        layer = counter[0] % n_layers
        counter[0] += 1
        R.rimuru_moe_forward_host(lane["x"].data_ptr(), lane["logits"].data_ptr(), w.T, ev,
                                  layer, lane["out"].data_ptr(), lane["ws"], hws,
                                  lane["stream"].cuda_stream)

    def timed_host_steps(n_lanes):
        for i in range(3):
            host_step(lanes[i % n_lanes])
        torch.cuda.synchronize()
        barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for ln in lanes[:n_lanes]:
            ln["stream"].wait_event(e0)
        for i in range(Ke):
            host_step(lanes[i % n_lanes])
        for ln in lanes[:n_lanes]:
            stream.wait_stream(ln["stream"])
        e1.record(stream)
        torch.cuda.synchronize()
        barrier()
        return max_over_ranks(e0.elapsed_time(e1), dist, dev)

    ms_e2e_serial = timed_host_steps(1)
    ms_e2e = timed_host_steps(2)
    if R.rimuru_get_device_error(ev) != R.DEV_OK:
        raise RuntimeError("device error in the end-to-end steps")
    ref_out = out.cpu()
    for ln in lanes:  # same inputs, deterministic layer: the host results equal the device's
        if not torch.equal(ln["out"].view(torch.int16), ref_out.view(torch.int16)):
            raise RuntimeError("host-buffer forward disagrees with the device-buffer forward")
    e2e_value = world * w.T * Ke / (ms_e2e / 1e3)

    # ------------------------------------------------------------ CUDA-graph replay
    # The same device-resident forwards recorded once by stream capture and replayed, as a
    # decode loop with fixed buffers would run them (reported beside `value`, which
    # launches every forward from the host).
    G = max(n_layers, 10)
    gs = torch.cuda.Stream(dev)
    gs.wait_stream(stream)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=gs):
        for _ in range(G):
            step(gs)
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
    if R.rimuru_get_device_error(ev) != R.DEV_OK:
        raise RuntimeError("device error in the graph replays")
    graph_value = world * w.T * reps * G / (ms_graph / 1e3)
    del graph

    # ---------------------------------------------------------------- roofline
    peaks = load_peaks()
    # the binding roofline of the dominant kernel: whichever of its byte time and its
    # flop time at the measured peaks is longer
    decode_like = (work[dom]["bytes"] / (peaks["hbm_gbs"] * 1e9)
                   >= work[dom]["flops"] / (peaks["bf16_tflops_sustained"] * 1e12))
    t_dom = dom_ms_live / 1e3
    if decode_like:
        achieved = work[dom]["bytes"] / t_dom / 1e9
        roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4)}
    else:
        achieved = work[dom]["flops"] / t_dom / 1e12
        roof = {"bound": "tensor", "achieved": round(achieved, 1),
                "peak": peaks["bf16_tflops_sustained"], "unit": "TFLOP/s",
                "frac": round(achieved / peaks["bf16_tflops_sustained"], 4)}
    roof["kernel"] = dom
    roof["ms_per_launch"] = round(dom_ms_live, 5)
    roof["launches_timed"] = n_dom
    roof["timed_one_launch_in"] = PROFILE_EVERY
    roof["traffic"] = ncu_traffic(dom, args.workload)
    roof["peak_source"] = peaks["source"] + (" (sustained bf16)" if not decode_like else " (HBM copy)")
    total_k = sum(v["ms_per_launch"] for v in per_kernel.values())
    for name, v in per_kernel.items():
        v["share"] = round(v["ms_per_launch"] / total_k, 4) if total_k else None
        tk = v["ms_per_launch"] / 1e3
        if tk > 0:
            v["GB/s"] = round(work[name]["bytes"] / tk / 1e9, 1)
            if work[name]["flops"]:
                v["TFLOP/s"] = round(work[name]["flops"] / tk / 1e12, 1)
        v["ms_per_launch"] = round(v["ms_per_launch"], 5)
    layer_t = ms_step / 1e3
    layer_roof = {"hbm_frac": round(work["layer"]["bytes"] / layer_t / 1e9 / peaks["hbm_gbs"], 4),
                  "tensor_frac": round(work["layer"]["flops"] / layer_t / 1e12
                                       / peaks["bf16_tflops_sustained"], 4)}

    result = {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": round(ms_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": f"{args.workload}: {WORKLOAD_TEXT[args.workload]}", "tokens": w.T,
                   "experts_touched": work["U"], "seed": args.seed,
                   "l2": "inputs larger than L2: the expert pages read per step exceed 129 MB"
                   if n_layers == 1 else
                   f"a layer's pages fit in L2, so steps cycle over {n_layers} copies of the "
                   f"layer (same weights, distinct pool pages): "
                   f"{n_layers * work['layer']['bytes'] / 1e6:.0f} MB per cycle",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "roofline": roof,
        "layer_roofline": layer_roof,
        "kernels": per_kernel,
        "kernels_note": f"per-kernel event pairs around every launch, {Kp} untimed steps",
        "gpu_launches": launches_per_step * K,
        "e2e": {"value": round(e2e_value, 1), "unit": "tokens/s",
                "h2d_bytes_per_step": int(x.numel() * 2 + logits.numel() * 4),
                "d2h_bytes_per_step": int(out.numel() * 2), "steps": Ke,
                "ms_per_step": round(ms_e2e / Ke, 5),
                "api": "rimuru_moe_forward_host (pinned host buffers)", "streams": 2,
                "single_stream_value": round(world * w.T * Ke / (ms_e2e_serial / 1e3), 1)},
        "cuda_graph": {"value": round(graph_value, 1), "unit": "tokens/s",
                       "ms_per_step": round(ms_graph / (reps * G), 5),
                       "forwards_per_graph": G, "replays": reps},
        "clocks": clk,
    }
    if rank == 0 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(w, args.cpu_seconds)
    pool.close()
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
    import workloads as wl
    w = make_workload(args)
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
        "config": {"workload": f"{args.workload}: {WORKLOAD_TEXT[args.workload]}", "tokens": w.T,
                   "parallelism": "host cores"},
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
    ap.add_argument("--cpu-seconds", type=float, default=20.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--evict", default="layer_cycle", choices=["layer_cycle", "lru"],
                    help="eviction policy of the offload cache (q3_stack_offload)")
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
