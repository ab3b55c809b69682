"""Failure path on the GPU without a fault: a kernel whose bounded wait runs
out (an mbarrier that nothing completes) gives up after the wait limit,
records the timeout, releases its tensor memory and returns; the host reads
the status through dsa_last_device_error and the context keeps working."""
import time

import pytest

from gpu_util import bf, i32, need_gpu, torch
from synth import WORKLOADS, make_sparse_inputs, scaled_down

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


def test_wait_runs_out_and_context_survives():
    import dsa_sparse_mla_prefill_gb300 as dsa
    w = scaled_down(WORKLOADS["tiny_uniform_512"], (300,), (300,), k=64, seed=21)
    x = make_sparse_inputs(w)
    q, kv, idx = bf(x.q), bf(x.kv), i32(x.idx)
    before = dsa.dsa_sparse_prefill(q, kv, idx, w.k, w.scale)
    st, counts = dsa.dsa_last_device_error()
    assert st == dsa.DSA_OK, counts
    t0 = time.time()
    dsa.dsa_debug_wait_timeout()
    st, counts = dsa.dsa_last_device_error()
    elapsed = time.time() - t0
    assert st == dsa.DSA_ERR_DEVICE and counts[1] >= 1, (st, counts)
    assert 1.5 < elapsed < 60, elapsed      # the 2 s wait limit, then the kernel returned
    # the counters were cleared by the read, and the context still computes
    after = dsa.dsa_sparse_prefill(q, kv, idx, w.k, w.scale)
    torch.cuda.synchronize()
    st, counts = dsa.dsa_last_device_error()
    assert st == dsa.DSA_OK and counts == [0, 0, 0, 0], counts
    assert torch.equal(before[0], after[0]) and torch.equal(before[1], after[1])
