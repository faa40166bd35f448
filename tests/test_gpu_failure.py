"""Failure detection on the GPU without faulting it: a wait that nothing satisfies must run
out after its short limit, report RIMURU_DEV_TIMEOUT through the device status word, and
leave the context usable for the next forward."""
import numpy as np
import pytest

import workloads as wl
from gpu_harness import Runner, rel_err
from oracle import Oracle
from paged_moe_shared_gb300 import rimuru as R

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_reports():
    assert R.rimuru_selftest_bounded_wait(20_000) == R.DEV_TIMEOUT   # 20 ms limit


def test_forward_still_correct_after_a_timeout():
    assert R.rimuru_selftest_bounded_wait(5_000) == R.DEV_TIMEOUT
    w = wl.tiny(41)
    r = Runner(w)
    try:
        r.forward()
        res = r.results()
    finally:
        r.close()
    s = w.shape
    o = Oracle().moe_forward(w.x_bits, w.logits, w.pool, w.page_bytes, w.page_table, s.H, s.I,
                             s.k, s.renorm)
    assert res["dev_err"] == R.DEV_OK
    assert rel_err(res["out"], o["out"]) <= 1e-2
