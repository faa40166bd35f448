"""The allocation-free forward (rimuru_moe_forward_noalloc) against the ordinary one.

Some callers cannot allocate device memory at all: a serving engine that gives nearly all
device memory to its own page pool up front, or a host that accounts for every device byte
itself.  For them the library keeps a fixed 16 MiB scratch array in its own device memory.
The allocation-free call runs the same kernels on the same inputs as the workspace forward,
so its output must be bitwise the same, also when the scratch still holds a previous call's
contents of another size.  This file is collected last so that, if it fails, a run that
stops at the first failure has already run every other test; it must also pass on its own
in a fresh process."""
import numpy as np
import pytest
import torch

import workloads as wl
from gpu_harness import Runner
from paged_moe_shared_gb300 import rimuru as R

pytestmark = pytest.mark.gpu


def noalloc(r, out, err=None):
    """One allocation-free forward of the Runner's layer into `out`; returns the device
    error word the caller passed (or None)."""
    stream = torch.cuda.current_stream().cuda_stream
    R.rimuru_moe_forward_noalloc(r.x.data_ptr(), r.logits.data_ptr(), r.w.T, r.ev, 0,
                                 out.data_ptr(), err.data_ptr() if err is not None else 0, stream)
    torch.cuda.synchronize()
    return None if err is None else int(err.item())


def bits(t):
    return t.view(torch.int16).cpu()


@pytest.mark.parametrize("make", [lambda: wl.tiny(31, T=300), lambda: wl.q3_decode(0)],
                         ids=["tiny_300_tokens", "q3_decode_64_tokens"])
def test_noalloc_equals_the_workspace_forward_twice_in_a_row(make):
    w = make()
    r = Runner(w)
    try:
        r.forward()
        assert r.results()["dev_err"] == R.DEV_OK
        ref = bits(r.out)
        err = torch.zeros(1, dtype=torch.int32, device="cuda:0")
        for _ in range(2):
            out = torch.full_like(r.out, float("nan"))
            assert noalloc(r, out, err) == R.DEV_OK
            assert torch.equal(bits(out), ref)
    finally:
        r.close()


def test_noalloc_sizes_in_sequence_through_the_shared_scratch():
    """Batches of several sizes one after another, each finding the previous call's scratch
    contents: 16 and 300 tokens take the small-batch routing kernel, 600 tokens (1200
    assignments) separate route and align launches with GEMM 1 gathering rows from x, and
    1100 tokens (2200 assignments) the 256-row GEMM 1 and the CTA-pair GEMM 2.  Each output
    equals the workspace forward's bit for bit."""
    runners = {T: Runner(wl.tiny(40 + T, T=T)) for T in (300, 16, 600, 1100)}
    try:
        ref = {}
        for T, r in runners.items():
            r.forward()
            assert r.results()["dev_err"] == R.DEV_OK
            ref[T] = bits(r.out)
        err = torch.zeros(1, dtype=torch.int32, device="cuda:0")
        for T in (300, 16, 600, 1100, 300, 600):
            r = runners[T]
            out = torch.full_like(r.out, float("nan"))
            assert noalloc(r, out, err) == R.DEV_OK
            assert torch.equal(bits(out), ref[T]), T
    finally:
        for r in runners.values():
            r.close()


def test_noalloc_reports_kernel_errors_into_the_callers_word():
    """A NaN logit is a bad input the host does not check; the routing kernel records
    RIMURU_DEV_NONFINITE in the error word the caller passed."""
    w = wl.tiny(34, T=16)
    w.logits[5, 3] = np.nan
    r = Runner(w)
    try:
        err = torch.zeros(1, dtype=torch.int32, device="cuda:0")
        out = torch.empty_like(r.out)
        assert noalloc(r, out, err) == R.DEV_NONFINITE
    finally:
        r.close()


def test_noalloc_rejects_batches_beyond_the_scratch():
    w = wl.tiny(32, T=16)
    r = Runner(w)
    try:
        too_many = 1 << 16  # 65536 tokens of the tiny layer need far more than 16 MiB
        assert R.rimuru_moe_workspace_bytes(r.ev, too_many) > 16 << 20
        with pytest.raises(R.RimuruError) as e:
            R.rimuru_moe_forward_noalloc(r.x.data_ptr(), r.logits.data_ptr(), too_many, r.ev, 0,
                                         r.out.data_ptr(), 0, 0)
        assert e.value.status == R.ERR_WORKSPACE
        assert "16777216" in str(e.value)
        with pytest.raises(R.RimuruError) as e:
            R.rimuru_moe_forward_noalloc(r.x.data_ptr(), r.logits.data_ptr(), (1 << 20) + 1,
                                         r.ev, 0, r.out.data_ptr(), 0, 0)
        assert e.value.status == R.ERR_ARG
    finally:
        r.close()


def test_noalloc_leaves_free_device_memory_unchanged():
    w = wl.tiny(33, T=64)
    r = Runner(w)
    try:
        out = torch.empty_like(r.out)
        noalloc(r, out)
        free0, _ = torch.cuda.mem_get_info()
        for _ in range(3):
            noalloc(r, out)
        free1, _ = torch.cuda.mem_get_info()
        assert free1 == free0
    finally:
        r.close()
