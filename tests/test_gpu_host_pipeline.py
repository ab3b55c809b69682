"""dsa_sparse_prefill_host (host buffers, copies overlapped with the kernel in
chunks) against the device call on the same inputs: the same kernel runs on
every token, so out and lse must be bit for bit equal, for ragged chunks, more
chunks than buffer sets, kv on the host or on the device, and two calls in a
row through one workspace.  The device call itself is checked against the
oracle in test_gpu_sparse.py."""
import numpy as np
import pytest

from gpu_util import bf, i32, need_gpu, torch
from synth import WORKLOADS, make_sparse_inputs, scaled_down

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


def pinned(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.view(dtype)
    return t.pin_memory()


@pytest.mark.parametrize("T,chunk,kv_on_host", [
    (1000, 300, True), (1000, 300, False), (1000, 97, True), (1000, 5000, True),
    (3000, 1216, True),     # ramped first and last chunks (one and two tokens per SM), then full ones
])
def test_host_call_equals_device_call(T, chunk, kv_on_host):
    import dsa_sparse_mla_prefill_gb300 as dsa
    w = scaled_down(WORKLOADS["v32_h32_16k"], (T,), (T + 200,), k=256, ld=264, seed=17)
    x = make_sparse_inputs(w)
    q, kv, idx = bf(x.q), bf(x.kv), i32(x.idx)
    ref_o, ref_l = dsa.dsa_sparse_prefill(q, kv, idx, w.k, w.scale)
    hq = pinned(x.q.view(np.int16), torch.bfloat16)
    hkv = pinned(x.kv.view(np.int16), torch.bfloat16) if kv_on_host else kv
    hidx = pinned(x.idx)
    ws = torch.empty(dsa.dsa_sparse_prefill_host_workspace(w.T, w.N, w.d_qk, w.H, w.d_qk, w.ld, chunk, kv_on_host),
                     dtype=torch.uint8, device="cuda")
    for rep in range(2):   # the second call reuses the workspace and the library's streams
        ho = torch.full((w.T, w.H, 512), float("nan"), dtype=torch.bfloat16).pin_memory()
        hl = torch.full((w.T, w.H), float("nan"), dtype=torch.float32).pin_memory()
        dsa.dsa_sparse_prefill_host(hq, hkv, hidx, w.k, w.scale, ho, hl, ws, chunk_tokens=chunk)
        torch.cuda.current_stream().synchronize()
        st, counts = dsa.dsa_last_device_error()
        assert st == 0, counts
        assert torch.equal(ho, ref_o.cpu()), rep
        assert torch.equal(hl, ref_l.cpu()), rep


@pytest.mark.parametrize("T,chunk,kv_on_host,empty_rows", [
    (1000, 97, True, False), (3000, 1216, True, False), (3000, 1216, False, False),
    (3000, 300, True, True),    # tokens without a valid index (zero output, lse = -inf) mid-stream
    (100, 16, True, False),     # fewer tokens than SMs: one block of counters
    (1, 1, True, False),
])
def test_streamed_call_equals_device_call(T, chunk, kv_on_host, empty_rows):
    """A workspace that holds every token (sized with chunk_tokens >= T) selects the
    streamed form: one kernel launch over all tokens, chunk_tokens then sets only the
    upload granularity.  Same bits as the device call."""
    import dsa_sparse_mla_prefill_gb300 as dsa
    w = scaled_down(WORKLOADS["v32_h32_16k"], (T,), (T + 200,), k=256, ld=264, seed=19)
    x = make_sparse_inputs(w)
    idx_np = x.idx.copy()
    if empty_rows:
        idx_np[T // 3: T // 3 + 40] = -1
        idx_np[-7:] = -1
    q, kv, idx = bf(x.q), bf(x.kv), i32(idx_np)
    ref_o, ref_l = dsa.dsa_sparse_prefill(q, kv, idx, w.k, w.scale)
    hq = pinned(x.q.view(np.int16), torch.bfloat16)
    hkv = pinned(x.kv.view(np.int16), torch.bfloat16) if kv_on_host else kv
    hidx = pinned(idx_np)
    nbytes = dsa.dsa_sparse_prefill_host_workspace(w.T, w.N, w.d_qk, w.H, w.d_qk, w.ld, w.T, kv_on_host)
    ring = dsa.dsa_sparse_prefill_host_workspace(w.T, w.N, w.d_qk, w.H, w.d_qk, w.ld, chunk, kv_on_host)
    assert chunk >= T or nbytes != ring
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    for rep in range(2):   # the counters are cleared by the call itself
        ho = torch.full((w.T, w.H, 512), float("nan"), dtype=torch.bfloat16).pin_memory()
        hl = torch.full((w.T, w.H), float("nan"), dtype=torch.float32).pin_memory()
        dsa.dsa_sparse_prefill_host(hq, hkv, hidx, w.k, w.scale, ho, hl, ws, chunk_tokens=chunk)
        torch.cuda.current_stream().synchronize()
        st, counts = dsa.dsa_last_device_error()
        assert st == 0, counts
        assert torch.equal(ho, ref_o.cpu()), rep
        assert torch.equal(hl, ref_l.cpu()), rep


@pytest.mark.parametrize("base,H", [("v32_h32_16k", 16), ("nope_2x8192", 16), ("nope_2x8192", 32)])
def test_streamed_call_other_instances(base, H):
    """The streamed kernel instances of the other shapes (H = 16; D_QK = 512 without RoPE
    columns, two requests), against the device call, bit for bit."""
    import dsa_sparse_mla_prefill_gb300 as dsa
    w0 = WORKLOADS[base]
    qs = (700,) if len(w0.q_lens) == 1 else (400, 500)
    w = scaled_down(w0, qs, tuple(q + 150 for q in qs), k=256, ld=272, H=H, seed=21)
    x = make_sparse_inputs(w)
    q, kv, idx = bf(x.q), bf(x.kv), i32(x.idx)
    ref_o, ref_l = dsa.dsa_sparse_prefill(q, kv, idx, w.k, w.scale)
    hq = pinned(x.q.view(np.int16), torch.bfloat16)
    hkv = pinned(x.kv.view(np.int16), torch.bfloat16)
    hidx = pinned(x.idx)
    ws = torch.empty(dsa.dsa_sparse_prefill_host_workspace(w.T, w.N, w.d_qk, w.H, w.d_qk, w.ld, w.T, True),
                     dtype=torch.uint8, device="cuda")
    ho = torch.full((w.T, w.H, 512), float("nan"), dtype=torch.bfloat16).pin_memory()
    hl = torch.full((w.T, w.H), float("nan"), dtype=torch.float32).pin_memory()
    dsa.dsa_sparse_prefill_host(hq, hkv, hidx, w.k, w.scale, ho, hl, ws, chunk_tokens=200)
    torch.cuda.current_stream().synchronize()
    st, counts = dsa.dsa_last_device_error()
    assert st == 0, counts
    assert torch.equal(ho, ref_o.cpu()) and torch.equal(hl, ref_l.cpu())


def test_streamed_call_orders_with_the_callers_stream():
    """As below, for the streamed form: the kernel starts only after the caller's
    earlier work, and the caller's later work sees the outputs."""
    import dsa_sparse_mla_prefill_gb300 as dsa
    w = scaled_down(WORKLOADS["v32_h32_16k"], (600,), (700,), k=128, ld=128, seed=20)
    x = make_sparse_inputs(w)
    s = torch.cuda.Stream()
    kv_src = bf(x.kv)
    kv = torch.zeros_like(kv_src)
    hq = pinned(x.q.view(np.int16), torch.bfloat16)
    hidx = pinned(x.idx)
    ho = torch.empty((w.T, w.H, 512), dtype=torch.bfloat16).pin_memory()
    hl = torch.empty((w.T, w.H), dtype=torch.float32).pin_memory()
    ws = torch.empty(dsa.dsa_sparse_prefill_host_workspace(w.T, w.N, w.d_qk, w.H, w.d_qk, w.ld, w.T, False),
                     dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        torch.cuda._sleep(20_000_000)
        kv.copy_(kv_src)
        dsa.dsa_sparse_prefill_host(hq, kv, hidx, w.k, w.scale, ho, hl, ws, chunk_tokens=128, stream=s)
        done = torch.cuda.Event()
        done.record(s)
    done.synchronize()
    ref_o, ref_l = dsa.dsa_sparse_prefill(bf(x.q), kv_src, i32(x.idx), w.k, w.scale)
    assert torch.equal(ho, ref_o.cpu()) and torch.equal(hl, ref_l.cpu())


def test_host_call_orders_with_the_callers_stream():
    """Work queued on the caller's stream before the call (here: writing the kv the call
    reads, on the device) is seen by it, and work queued after it sees its outputs."""
    import dsa_sparse_mla_prefill_gb300 as dsa
    w = scaled_down(WORKLOADS["v32_h32_16k"], (600,), (700,), k=128, ld=128, seed=18)
    x = make_sparse_inputs(w)
    s = torch.cuda.Stream()
    kv_src = bf(x.kv)
    kv = torch.zeros_like(kv_src)
    hq = pinned(x.q.view(np.int16), torch.bfloat16)
    hidx = pinned(x.idx)
    ho = torch.empty((w.T, w.H, 512), dtype=torch.bfloat16).pin_memory()
    hl = torch.empty((w.T, w.H), dtype=torch.float32).pin_memory()
    ws = torch.empty(dsa.dsa_sparse_prefill_host_workspace(w.T, w.N, w.d_qk, w.H, w.d_qk, w.ld, 128, False),
                     dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        torch.cuda._sleep(20_000_000)   # keep the stream busy so the copy below lands late
        kv.copy_(kv_src)
        dsa.dsa_sparse_prefill_host(hq, kv, hidx, w.k, w.scale, ho, hl, ws, chunk_tokens=128, stream=s)
        done = torch.cuda.Event()
        done.record(s)
    done.synchronize()
    ref_o, ref_l = dsa.dsa_sparse_prefill(bf(x.q), kv_src, i32(x.idx), w.k, w.scale)
    assert torch.equal(ho, ref_o.cpu()) and torch.equal(hl, ref_l.cpu())
