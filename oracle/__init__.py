"""CPU oracle for the page-table-aware fused MoE layer (Rimuru, arXiv 2610.40305).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  The product path (``paged_moe_shared_gb300``) never imports it and
shares no code with it.

The arithmetic lives in ``rimuru_oracle.c`` (plain C, double precision, naive
loops); this module only compiles it with gcc and marshals numpy arrays.
Which passage of the pages each step follows is stated in the C file's header:
memory views and page tables (abstract; Figure 6), the page-table-aware kernel
reading experts in place (explainer page, paragraph on the fused MoE kernel),
expert projection shapes (Table 1).  Routing, grouping, SwiGLU and combine are
the standard top-k MoE FFN that the pages name but do not spell out.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "rimuru_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

OK = 0
ERR_ARG = -1
ERR_PAGE = -2
ERR_NONFINITE = -3
ERR_NOMEM = -4


def compile_oracle(src: str = _SRC, out: str = _LIB_PATH, extra_flags=()) -> str:
    """Compile the oracle C source into a shared library with gcc (OpenMP if available)."""
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-Wall", *extra_flags]
    tmp = out + ".tmp%d" % os.getpid()
    try:
        subprocess.run(base + ["-fopenmp", "-o", tmp, src, "-lm"], check=True,
                       capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base + ["-o", tmp, src, "-lm"], check=True, capture_output=True)
    os.replace(tmp, out)
    return out


def build() -> str:
    """Build liboracle.so next to the source if it is missing or stale."""
    if (not os.path.exists(_LIB_PATH)
            or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)):
        compile_oracle()
    return _LIB_PATH


def _bind(lib):
    P = ctypes.c_void_p
    i32, u64, i64 = ctypes.c_int, ctypes.c_uint64, ctypes.c_int64
    lib.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
    lib.oracle_bf16_to_f64.restype = ctypes.c_double
    lib.oracle_page_to_matrix.argtypes = [P, u64, u64, i64, i32, i32, P]
    lib.oracle_page_to_matrix.restype = i32
    lib.oracle_route.argtypes = [P, i32, i32, i32, i32, P, P]
    lib.oracle_route.restype = i32
    lib.oracle_align.argtypes = [P, i32, i32, P, P]
    lib.oracle_align.restype = i32
    lib.oracle_moe_forward.argtypes = [P, P, i32, i32, i32, i32, i32, i32, P, u64, u64, P, P,
                                       i32, i32, P, P, P, P, P, P, P]
    lib.oracle_moe_forward.restype = i32
    lib.oracle_max_threads.argtypes = []
    lib.oracle_max_threads.restype = i32
    return lib


def load(path: str | None = None):
    """Load the oracle library (building it first when ``path`` is None)."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
    return _lib


class OracleError(RuntimeError):
    pass


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data) if a is not None else None


def _check(st: int, what: str):
    if st != OK:
        raise OracleError(f"{what} failed with status {st}")


class Oracle:
    """numpy front end of one oracle library (the default build, or a variant)."""

    def __init__(self, lib=None):
        self.lib = lib if lib is not None else load()

    def bf16_to_f64(self, bits: int) -> float:
        return self.lib.oracle_bf16_to_f64(int(bits))

    def max_threads(self) -> int:
        return self.lib.oracle_max_threads()

    def page_to_matrix(self, pool: np.ndarray, page_bytes: int, page_id: int, rows: int,
                       cols: int) -> np.ndarray:
        pool = np.ascontiguousarray(pool, dtype=np.uint8)
        out = np.empty((rows, cols), np.float64)
        _check(self.lib.oracle_page_to_matrix(_ptr(pool), pool.nbytes, page_bytes, page_id,
                                              rows, cols, _ptr(out)), "page_to_matrix")
        return out

    def route(self, logits: np.ndarray, k: int, renorm: bool = True):
        logits = np.ascontiguousarray(logits, dtype=np.float32)
        T, E = logits.shape
        ids = np.empty((T, k), np.int32)
        w = np.empty((T, k), np.float32)
        _check(self.lib.oracle_route(_ptr(logits), T, E, k, int(renorm), _ptr(ids), _ptr(w)),
               "route")
        return ids, w

    def align(self, ids: np.ndarray, E: int):
        ids = np.ascontiguousarray(ids, dtype=np.int32).ravel()
        A = ids.size
        sorted_ = np.empty(A, np.int32)
        offsets = np.empty(E + 1, np.int32)
        _check(self.lib.oracle_align(_ptr(ids), A, E, _ptr(sorted_), _ptr(offsets)), "align")
        return sorted_, offsets

    def moe_forward(self, x_bits: np.ndarray, logits: np.ndarray, pool: np.ndarray,
                    page_bytes: int, page_table: np.ndarray, H: int, I: int, k: int,
                    renorm: bool = True, tokens=None, want_hidden: bool = False,
                    nthreads: int = 0):
        """Run the layer.  ``x_bits`` is uint16 [T, H] (bf16 bit patterns), ``logits`` fp32
        [T, E], ``pool`` the host bytes of the pool, ``page_table`` int32 [E, 3].

        Returns a dict with ids, w, sorted, offsets, out (float64 [T, H]; rows of tokens
        not in ``tokens`` are NaN) and, if ``want_hidden``, h [T*k, I] and y [T*k, H]."""
        x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
        logits = np.ascontiguousarray(logits, dtype=np.float32)
        pool = np.ascontiguousarray(pool, dtype=np.uint8).ravel()
        pt = np.ascontiguousarray(page_table, dtype=np.int32)
        T, E = logits.shape
        assert x_bits.shape == (T, H) and pt.shape == (E, 3)
        A = T * k
        ids = np.empty((T, k), np.int32)
        w = np.empty((T, k), np.float32)
        sorted_ = np.empty(A, np.int32)
        offsets = np.empty(E + 1, np.int32)
        out = np.full((T, H), np.nan, np.float64)
        h = np.full((A, I), np.nan, np.float64) if want_hidden else None
        y = np.full((A, H), np.nan, np.float64) if want_hidden else None
        if tokens is None:
            tok, ntok = None, -1
        else:
            tok = np.ascontiguousarray(tokens, dtype=np.int32)
            ntok = tok.size
        st = self.lib.oracle_moe_forward(
            _ptr(x_bits), _ptr(logits), T, H, I, E, k, int(renorm), _ptr(pool), pool.nbytes,
            page_bytes, _ptr(pt), _ptr(tok) if tok is not None else None, ntok, int(nthreads),
            _ptr(ids), _ptr(w), _ptr(sorted_), _ptr(offsets), _ptr(h) if h is not None else None,
            _ptr(y) if y is not None else None, _ptr(out))
        _check(st, "moe_forward")
        res = dict(ids=ids, w=w, sorted=sorted_, offsets=offsets, out=out)
        if want_hidden:
            res["h"] = h
            res["y"] = y
        return res
