"""Runs one forward of the paged fused-MoE layer through the C ABI and returns every
intermediate the workspace holds (routing ids and weights, offsets, the permutation and
its inverse, the tile table, h, y; x_sorted for batches of at most 1024 assignments) plus the
output, all as numpy arrays."""
from __future__ import annotations

import numpy as np
import torch

from paged_moe_shared_gb300 import rimuru as R
from paged_moe_shared_gb300.device_pool import load_workload

DEV = "cuda:0"


def bf16_tensor(bits: np.ndarray, device=DEV) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


class Runner:
    """A workload placed on the device once; ``forward`` can be called repeatedly."""

    def __init__(self, w, device=DEV, decode_tokens=None):
        self.w = w
        self.pool, self.ev, self.kv = load_workload(w, device)
        if decode_tokens is not None:  # batches up to this size take the decode path (0: never)
            R.rimuru_view_set_decode_tokens(self.ev, decode_tokens)
        self.x = bf16_tensor(w.x_bits, device)
        self.logits = torch.from_numpy(np.ascontiguousarray(w.logits)).to(device)
        self.out = torch.empty_like(self.x)
        self.ws_bytes = R.rimuru_moe_workspace_bytes(self.ev, w.T)
        self.ws_raw = torch.empty(self.ws_bytes + 1024, dtype=torch.uint8, device=device)
        off = (-self.ws_raw.data_ptr()) % 1024
        self.ws = self.ws_raw[off:off + self.ws_bytes]
        self.layout = R.rimuru_moe_workspace_layout(self.ev, w.T)

    def forward(self, stream=None):
        s = stream if stream is not None else torch.cuda.current_stream()
        R.rimuru_moe_forward(self.x.data_ptr(), self.logits.data_ptr(), self.w.T, self.ev, 0,
                             self.out.data_ptr(), self.ws.data_ptr(), self.ws_bytes, s.cuda_stream)

    def region(self, name, dtype, count):
        off = self.layout[name]
        nbytes = count * torch.tensor([], dtype=dtype).element_size()
        return self.ws[off:off + nbytes].view(dtype)

    def results(self):
        torch.cuda.synchronize()
        w = self.w
        s = w.shape
        A = w.T * s.k
        r = {
            "out": to_f64(self.out),
            "ids": self.region("ids", torch.int32, A).cpu().numpy().reshape(w.T, s.k),
            "w": self.region("weights", torch.float32, A).cpu().numpy().reshape(w.T, s.k),
            "offsets": self.region("offsets", torch.int32, s.E + 1).cpu().numpy(),
            "sorted": self.region("sorted", torch.int32, A).cpu().numpy(),
            "inv": self.region("inv", torch.int32, A).cpu().numpy(),
            "num_tiles": int(self.region("num_tiles", torch.int32, 1).cpu().item()),
            "h": to_f64(self.region("h", torch.bfloat16, A * s.I).view(A, s.I)),
            "y": to_f64(self.region("y", torch.bfloat16, A * s.H).view(A, s.H)),
            "x_sorted": (self.region("x_sorted", torch.bfloat16, A * s.H).view(A, s.H)
                         if A <= 1024 else None),
            "dev_err": R.rimuru_get_device_error(self.ev, clear=True),
        }
        r["tiles"] = self.region("tiles", torch.int32, 2 * r["num_tiles"]).cpu().numpy().reshape(-1, 2)
        r["num_ptiles"] = int(self.region("num_ptiles", torch.int32, 1).cpu().item())
        r["ptiles"] = (self.region("ptiles", torch.int32, 2 * r["num_ptiles"]).cpu().numpy()
                       .reshape(-1, 2))
        return r

    def close(self):
        self.pool.close()


def rel_err(got: np.ndarray, ref: np.ndarray) -> float:
    """max |got - ref| / max |ref|; NaN anywhere in got makes it infinite."""
    if not np.isfinite(got).all():
        return float("inf")
    return float(np.max(np.abs(got - ref)) / max(np.max(np.abs(ref)), 1e-30))


def covering_tokens(offsets: np.ndarray, sorted_: np.ndarray, k: int, seed: int,
                    block: int = 128) -> np.ndarray:
    """Tokens to check when a layer is too large for the oracle to compute in full.

    The sample is chosen so that the checked assignment rows (every row of every chosen
    token) include, for each expert that received tokens, its first and last row in the
    expert-sorted order and at least one row of each of its ``block``-row blocks: every
    GEMM tile (both halves of a 256-row pair, an expert's lone last block, every column
    block and every k block, since a checked row spans them all) is then compared.
    ``offsets`` / ``sorted_`` are the oracle's grouping of the full batch."""
    rng = np.random.default_rng(seed)
    A = sorted_.size
    covered = np.zeros(A, bool)
    tok_of_row = sorted_ // k
    # rows of every token: row_of[f] = position of assignment f in the sorted order
    row_of = np.empty(A, np.int64)
    row_of[sorted_] = np.arange(A)
    chosen = set()

    def take(row):
        t = int(tok_of_row[row])
        if t not in chosen:
            chosen.add(t)
            covered[row_of[t * k:(t + 1) * k]] = True

    E = offsets.size - 1
    for e in range(E):
        a, b = int(offsets[e]), int(offsets[e + 1])
        if b > a:
            take(a)
            take(b - 1)
    for e in range(E):
        a, b = int(offsets[e]), int(offsets[e + 1])
        for r0 in range(a, b, block):
            r1 = min(b, r0 + block)
            if not covered[r0:r1].any():
                take(int(rng.integers(r0, r1)))
    return np.array(sorted(chosen), dtype=np.int64)
