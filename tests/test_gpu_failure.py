"""The failure path the pipeline kernels share, on the GPU without a fault:
a bounded wait on a barrier that nothing completes gives up after its limit,
sets the device error bit, and leaves the context usable (a decode step
afterwards still matches the oracle within the stated bar)."""
import time

import numpy as np
import pytest
import torch

from paged_kv_cache_309_gb300 import pa
from paged_kv_cache_309_gb300 import workloads as wl
from tests.gpu_util import need_gpu
from tests.test_gpu_decode import ATOL, RTOL, gpu_decode_step, oracle_rows, oracle_write

pytestmark = pytest.mark.gpu

PA_DEVERR_WAIT_TIMEOUT = 0x1


def test_bounded_wait_times_out_and_context_stays_usable():
    need_gpu()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    t0 = time.monotonic()
    pa.pa_selftest_bounded_wait(err)
    torch.cuda.synchronize()
    elapsed = time.monotonic() - t0
    assert int(err.item()) == PA_DEVERR_WAIT_TIMEOUT
    assert 1.5 < elapsed < 60.0, elapsed  # the 2 s wait limit ran out, then the kernel returned
    # the context still works: a decode step on the tiny workload matches the oracle
    w = wl.tiny_decode()
    got, dev_err, _ = gpu_decode_step(w)
    assert dev_err == 0
    oracle_write(w)
    rows = [(b, h) for b in range(w.num_seqs) for h in range(w.num_q_heads)]
    ref = oracle_rows(w, rows)
    for (b, h), r in ref.items():
        assert np.all(np.abs(got[b, h] - r) <= ATOL + RTOL * np.abs(r)), (b, h)
