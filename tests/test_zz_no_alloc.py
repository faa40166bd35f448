"""The allocation-free forward (rimuru_moe_forward_noalloc) against the ordinary one.

Some callers cannot allocate device memory at all: a serving engine that gives nearly all
device memory to its own page pool up front, or a host that accounts for every device byte
itself.  For them the library keeps a fixed 16 MiB scratch array in its own device memory.
This file is collected last so that, if it fails, a run that stops at the first failure has
already run every other test; it must also pass on its own in a fresh process."""
import numpy as np
import pytest
import torch

import workloads as wl
from gpu_harness import Runner, rel_err
from paged_moe_shared_gb300 import rimuru as R

pytestmark = pytest.mark.gpu

TOL = 1e-2


@pytest.mark.parametrize("make", [lambda: wl.tiny(31, T=300), lambda: wl.q3_decode(0)],
                         ids=["tiny_300_tokens", "q3_decode_64_tokens"])
def test_noalloc_matches_the_workspace_forward_twice_in_a_row(make):
    w = make()
    r = Runner(w)
    try:
        r.forward()
        ref = r.results()
        assert ref["dev_err"] == R.DEV_OK
        stream = torch.cuda.current_stream().cuda_stream
        err = torch.zeros(1, dtype=torch.int32, device="cuda:0")
        outs = []
        for _ in range(2):
            out = torch.full_like(r.out, float("nan"))
            R.rimuru_moe_forward_noalloc(r.x.data_ptr(), r.logits.data_ptr(), w.T, r.ev, 0,
                                         out.data_ptr(), err.data_ptr(), stream)
            torch.cuda.synchronize()
            assert int(err.item()) == R.DEV_OK
            got = out.float().cpu().numpy().astype(np.float64)
            assert rel_err(got, ref["out"]) <= TOL
            outs.append(got)
        # same kernels on the same inputs: the two calls agree exactly
        assert np.array_equal(outs[0], outs[1])
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
    finally:
        r.close()


def test_noalloc_leaves_free_device_memory_unchanged():
    w = wl.tiny(33, T=64)
    r = Runner(w)
    try:
        stream = torch.cuda.current_stream().cuda_stream
        out = torch.empty_like(r.out)
        R.rimuru_moe_forward_noalloc(r.x.data_ptr(), r.logits.data_ptr(), w.T, r.ev, 0,
                                     out.data_ptr(), 0, stream)
        torch.cuda.synchronize()
        free0, _ = torch.cuda.mem_get_info()
        for _ in range(3):
            R.rimuru_moe_forward_noalloc(r.x.data_ptr(), r.logits.data_ptr(), w.T, r.ev, 0,
                                         out.data_ptr(), 0, stream)
        torch.cuda.synchronize()
        free1, _ = torch.cuda.mem_get_info()
        assert free1 == free0
    finally:
        r.close()
