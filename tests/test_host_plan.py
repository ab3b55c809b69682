"""The chunk plan of the host-buffer call (dsa_sparse_prefill_host_plan, host
only): the chunks cover the tokens exactly, none is larger than the buffer
sets hold, the middle ones are a multiple of the SM count, and the first and
last ramp one, two, four ... tokens per SM."""
import pytest

import dsa_sparse_mla_prefill_gb300 as dsa


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from dsa_sparse_mla_prefill_gb300 import build as b
    b.build()


@pytest.mark.parametrize("T,cap,sms", [(16384, 1216, 152), (16384, 1024, 152), (3000, 1216, 152), (1000, 300, 152),
                                       (1000, 97, 152), (1000, 5000, 152), (1, 1, 152), (152, 152, 152),
                                       (100_000, 4096, 148), (777, 64, 16)])
def test_plan_properties(T, cap, sms):
    plan = dsa.dsa_sparse_prefill_host_plan(T, cap, sms)
    assert sum(plan) == T and all(n >= 1 for n in plan)
    c = min(cap, T)
    assert max(plan) <= c
    full = c // sms * sms if c >= sms else c
    # the ramp: sms, 2 sms, 4 sms, ... up front, mirrored at the end
    r = 0
    while r < len(plan) and plan[r] == sms << r and (sms << r) < full:
        r += 1
    assert plan[len(plan) - r:] == plan[:r][::-1]
    middle = plan[r:len(plan) - r]
    assert all(n == full for n in middle[:-1])           # full chunks, then the rest
    if c >= sms:
        assert full % sms == 0


def test_plan_edges_and_errors():
    assert dsa.dsa_sparse_prefill_host_plan(0, 100, 152) == []
    with pytest.raises(dsa.DSAError):
        dsa.dsa_sparse_prefill_host_plan(100, 0, 152)
    with pytest.raises(dsa.DSAError):
        dsa.dsa_sparse_prefill_host_plan(100, 10, 0)
    # the plan the benchmark's end-to-end step runs (16384 tokens, 1216-token buffers, 152 SMs)
    assert dsa.dsa_sparse_prefill_host_plan(16384, 1216, 152) == [152, 304, 608] + [1216] * 11 + [880, 608, 304, 152]
