"""dsa_sparse_prefill_host_noalloc: the host-buffer call for programs that
cannot allocate device memory (their allocator has reserved the GPU, or their
runtime forbids allocation while serving), with its chunk buffers in the
library's fixed device scratch array instead of a caller workspace.

It is called through the C ABI (ctypes on the raw symbol) and must agree with
dsa_sparse_prefill_host, which takes a workspace, within the parity tolerance,
on two calls in a row (the second call finds the first call's data in the
shared scratch).  This file is collected last on purpose."""
import ctypes

import numpy as np
import pytest

import dsa_sparse_mla_prefill_gb300 as dsa
import oracle.dsa_oracle as O
from synth import WORKLOADS, make_sparse_inputs, scaled_down


def _call_noalloc(torch, hq, hkv, hidx, k, scale, ho, hl, chunk, stream):
    T, H, d_qk = hq.shape
    N, ld_kv = hkv.shape
    return dsa.lib().dsa_sparse_prefill_host_noalloc(
        ctypes.c_void_p(hq.data_ptr()), ctypes.c_void_p(hkv.data_ptr()), 0 if hkv.is_cuda else 1, N, ld_kv,
        ctypes.c_void_p(hidx.data_ptr()), T, H, d_qk, 512, k, hidx.shape[1], ctypes.c_float(scale),
        ctypes.c_void_p(ho.data_ptr()), ctypes.c_void_p(hl.data_ptr()), chunk, ctypes.c_void_p(stream.cuda_stream))


def test_noalloc_rejects_shapes_beyond_the_scratch():
    """No GPU needed: the size check comes before any CUDA call."""
    from dsa_sparse_mla_prefill_gb300 import build as b
    b.build()
    lib = dsa.lib()
    # 16384 tokens of H = 32, top-2048, in one chunk: far more than 64 MiB of buffers
    need = lib.dsa_sparse_prefill_host_workspace(16384, 16384, 576, 32, 576, 512, 2048, 16384, 1)
    assert need > dsa.HOST_NOALLOC_SCRATCH_BYTES
    st = lib.dsa_sparse_prefill_host_noalloc(ctypes.c_void_p(16), ctypes.c_void_p(16), 1, 16384, 576,
                                             ctypes.c_void_p(16), 16384, 32, 576, 512, 2048, 2048,
                                             ctypes.c_float(0.07), ctypes.c_void_p(16), ctypes.c_void_p(16), 16384,
                                             ctypes.c_void_p(0))
    assert st == dsa.DSA_ERR_UNSUPPORTED
    # and the headline chunk shape the header names fits
    assert lib.dsa_sparse_prefill_host_workspace(16384, 16384, 576, 32, 576, 512, 2048, 152, 1) <= \
        dsa.HOST_NOALLOC_SCRATCH_BYTES


@pytest.mark.gpu
@pytest.mark.parametrize("kv_on_host", [True, False])
def test_noalloc_equals_workspace_call_twice(kv_on_host):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dsa_sparse_mla_prefill_gb300 import build as b
    b.build()
    w = scaled_down(WORKLOADS["v32_h32_16k"], (1000,), (1200,), k=256, ld=264, seed=23)
    x = make_sparse_inputs(w)

    def pinned(a, dtype=None):
        t = torch.from_numpy(np.ascontiguousarray(a))
        return (t.view(dtype) if dtype is not None else t).pin_memory()

    hq = pinned(x.q.view(np.int16), torch.bfloat16)
    hidx = pinned(x.idx)
    hkv = pinned(x.kv.view(np.int16), torch.bfloat16)
    if not kv_on_host:
        hkv = hkv.cuda()
    chunk = 300
    # the existing entry point, with a caller workspace
    ws = torch.empty(dsa.dsa_sparse_prefill_host_workspace(w.T, w.N, w.d_qk, w.H, w.d_qk, w.ld, chunk, kv_on_host),
                     dtype=torch.uint8, device="cuda")
    ref_o = torch.full((w.T, w.H, 512), float("nan"), dtype=torch.bfloat16).pin_memory()
    ref_l = torch.full((w.T, w.H), float("nan"), dtype=torch.float32).pin_memory()
    dsa.dsa_sparse_prefill_host(hq, hkv, hidx, w.k, w.scale, ref_o, ref_l, ws, chunk_tokens=chunk)
    torch.cuda.synchronize()
    ro = ref_o.float().numpy().astype(np.float64)
    rl = ref_l.numpy().astype(np.float64)
    stream = torch.cuda.current_stream()
    for rep in range(2):
        ho = torch.full((w.T, w.H, 512), float("nan"), dtype=torch.bfloat16).pin_memory()
        hl = torch.full((w.T, w.H), float("nan"), dtype=torch.float32).pin_memory()
        st = _call_noalloc(torch, hq, hkv, hidx, w.k, w.scale, ho, hl, chunk, stream)
        assert st == dsa.DSA_OK, dsa.status_string(st)
        stream.synchronize()
        st, counts = dsa.dsa_last_device_error()
        assert st == 0, counts
        res = O.compare(ho.float().numpy().astype(np.float64), hl.numpy().astype(np.float64), ro, rl)
        assert res["ok"], (rep, res)
