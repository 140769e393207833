"""Failure detection without a GPU fault: a barrier wait that nothing
completes runs out after a short limit, the kernel reports it in the device
error word and returns, and the context keeps working afterwards."""
import time

import pytest
import torch

import paged_kv_cache_220_gb300 as pkv
from paged_kv_cache_220_gb300 import build as pkv_build
from paged_kv_cache_220_gb300 import synth, workload
from _oracle_side import assert_close, expected

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives():
    pkv_build.build()
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    t0 = time.perf_counter()
    pkv.selftest_wait_timeout(flag, limit_us=50000)
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    assert int(flag.item()) == pkv.DEVERR_WAIT_TIMEOUT
    assert 0.04 < dt < 5.0
    # the same context still runs the decode correctly
    w = synth.tiny()
    pw = workload.build(w)
    out = [torch.empty_like(pw.layers[0].q)]
    workload.step(pw, out, None, 0)
    torch.cuda.synchronize()
    assert_close(out[0].cpu(), expected(w, 0, range(w.num_seqs)), "after timeout")


def test_selftest_rejects_bad_limits():
    pkv_build.build()
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(pkv.PagedKVError):
        pkv.selftest_wait_timeout(flag, limit_us=0)
