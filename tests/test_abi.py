"""The C-ABI library without a GPU: it loads, exports every function that
include/dsa.h declares, and its host-side helpers and argument checks work
(none of these calls reaches the GPU)."""
import ctypes
import os
import re

import numpy as np
import pytest

import dsa_sparse_mla_prefill_gb300 as dsa
import oracle.dsa_oracle as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from dsa_sparse_mla_prefill_gb300 import build as b
    b.build()
    return dsa.lib()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "dsa.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*(dsa_[a-z0-9_]+)\s*\(",
                                 src, flags=re.M)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(dsa.EXPORTED)


def test_status_strings(lib):
    assert dsa.status_string(0) == "DSA_OK"
    assert dsa.status_string(2) == "DSA_ERR_UNSUPPORTED"
    assert dsa.status_string(99) == "DSA_ERR_UNKNOWN"
    assert lib.dsa_version() >= 100


@pytest.mark.parametrize("G,k,ub", [(8, 2048, 128), (4, 2048, 128), (2, 4, 4), (3, 100, 16), (1, 1, 128)])
def test_union_pad_matches_oracle(lib, G, k, ub):
    assert dsa.dsa_union_pad(G, k, ub) == O.union_pad(G, k, ub)


@pytest.mark.parametrize("lens,G", [([16384], 8), ([8192, 8192], 8), ([5, 3, 17], 4), ([1, 1, 1], 8), ([0, 9], 2)])
def test_num_groups_matches_oracle(lib, lens, G):
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    assert dsa.dsa_num_groups(cu, int(cu[-1]), G) == len(O.groups(cu, G))


def _vp(x=0):
    return ctypes.c_void_p(x)


def test_argument_validation_without_gpu(lib):
    # unsupported head count / dims are rejected before any CUDA call
    assert lib.dsa_sparse_prefill(_vp(16), _vp(16), 10, 576, _vp(16), 4, 24, 576, 512, 8, 8, 1.0, _vp(16),
                                  _vp(16), None) == dsa.DSA_ERR_UNSUPPORTED
    assert lib.dsa_sparse_prefill(_vp(16), _vp(16), 10, 576, _vp(16), 4, 16, 448, 512, 8, 8, 1.0, _vp(16),
                                  _vp(16), None) == dsa.DSA_ERR_UNSUPPORTED
    # k beyond the supported top-k, ld < k, misaligned kv stride
    assert lib.dsa_sparse_prefill(_vp(16), _vp(16), 10, 576, _vp(16), 4, 16, 576, 512, 4096, 4096, 1.0, _vp(16),
                                  _vp(16), None) == dsa.DSA_ERR_UNSUPPORTED
    assert lib.dsa_sparse_prefill(_vp(16), _vp(16), 10, 576, _vp(16), 4, 16, 576, 512, 8, 4, 1.0, _vp(16),
                                  _vp(16), None) == dsa.DSA_ERR_INVALID_ARG
    assert lib.dsa_sparse_prefill(_vp(16), _vp(16), 10, 580, _vp(16), 4, 16, 576, 512, 8, 8, 1.0, _vp(16),
                                  _vp(16), None) == dsa.DSA_ERR_INVALID_ARG
    # null pointers and misalignment
    assert lib.dsa_sparse_prefill(None, _vp(16), 10, 576, _vp(16), 4, 16, 576, 512, 8, 8, 1.0, _vp(16),
                                  _vp(16), None) == dsa.DSA_ERR_INVALID_ARG
    assert lib.dsa_sparse_prefill(_vp(18), _vp(16), 10, 576, _vp(16), 4, 16, 576, 512, 8, 8, 1.0, _vp(16),
                                  _vp(16), None) == dsa.DSA_ERR_INVALID_ARG
    # empty problem is a no-op
    assert lib.dsa_sparse_prefill(None, None, 0, 576, None, 0, 16, 576, 512, 8, 8, 1.0, None, None,
                                  None) == dsa.DSA_OK
    # grouped: G*H must be 128 and G <= 8
    assert lib.dsa_grouped_prefill(_vp(16), _vp(16), 10, 576, _vp(16), _vp(16), _vp(16), 16, 4, None, 0, 8, 16,
                                   576, 512, 1.0, _vp(16), _vp(16), None) == dsa.DSA_ERR_UNSUPPORTED
    assert lib.dsa_grouped_prefill(_vp(16), _vp(16), 10, 576, _vp(16), _vp(16), _vp(16), 16, 16, None, 0, 8, 8,
                                   576, 512, 1.0, _vp(16), _vp(16), None) == dsa.DSA_ERR_UNSUPPORTED
    # grouped: the softmax scale must be positive and finite
    for bad in (0.0, -0.5, float("inf"), float("nan")):
        assert lib.dsa_grouped_prefill(_vp(16), _vp(16), 10, 576, _vp(16), _vp(16), _vp(16), 16, 8, None, 0, 8,
                                       16, 576, 512, bad, _vp(16), _vp(16), None) == dsa.DSA_ERR_INVALID_ARG
    # union build: G > 8 unsupported, union_pad must be a multiple of 16 and >= min(G*k, N)
    assert lib.dsa_union_build(_vp(16), 8, 4, 4, 9, None, 0, 100, _vp(16), _vp(16), _vp(16), 48,
                               None) == dsa.DSA_ERR_UNSUPPORTED
    assert lib.dsa_union_build(_vp(16), 8, 4, 4, 2, None, 0, 100, _vp(16), _vp(16), _vp(16), 8,
                               None) == dsa.DSA_ERR_INVALID_ARG
    assert lib.dsa_union_build(_vp(16), 8, 4, 4, 2, None, 0, 100, _vp(16), _vp(16), _vp(16), 20,
                               None) == dsa.DSA_ERR_INVALID_ARG
    # a bitmap that does not fit in shared memory
    assert lib.dsa_union_build(_vp(16), 8, 4, 4, 2, None, 0, 1 << 20, _vp(16), _vp(16), _vp(16), 16,
                               None) == dsa.DSA_ERR_UNSUPPORTED
    # request offsets that do not add up to T
    cu = (ctypes.c_int32 * 3)(0, 3, 7)
    assert lib.dsa_union_build(_vp(16), 8, 4, 4, 2, cu, 2, 100, _vp(16), _vp(16), _vp(16), 16,
                               None) == dsa.DSA_ERR_INVALID_ARG
    # masked MHA geometry allow-list
    assert lib.dsa_masked_mha_prefill(_vp(16), _vp(16), _vp(16), _vp(16), 4, None, None, 0, 8, 4, 576, 512, 1.0,
                                      _vp(16), _vp(16), None) == dsa.DSA_ERR_UNSUPPORTED
    # masked MHA: the softmax scale must be positive and finite
    for bad in (0.0, -1.0, float("inf"), float("nan")):
        assert lib.dsa_masked_mha_prefill(_vp(16), _vp(16), _vp(16), _vp(16), 4, None, None, 0, 8, 4, 192, 128,
                                          bad, _vp(16), _vp(16), None) == dsa.DSA_ERR_INVALID_ARG
    # strided masked MHA: geometry, RoPE width, the shared RoPE buffer, strides
    H = 4
    sok = dict(q=_vp(16), qt=H * 256, qh=256, k=_vp(16), kt=H * 512, kh=512, pe=None, pet=0, v=_vp(16),
               vt=H * 512, vh=512, T=8, dqk=256, dr=0, dv=256)

    def mstr(**kw):
        a = dict(sok, **kw)
        return lib.dsa_masked_mha_prefill_strided(a["q"], a["qt"], a["qh"], a["k"], a["kt"], a["kh"], a["pe"],
                                                  a["pet"], a["v"], a["vt"], a["vh"], _vp(16), 4, None, None, 0,
                                                  a["T"], H, a["dqk"], a["dr"], a["dv"], 0.0625, _vp(16), _vp(16),
                                                  None)
    assert mstr(dqk=576, dv=512) == dsa.DSA_ERR_UNSUPPORTED
    assert mstr(dqk=256, dv=128) == dsa.DSA_ERR_UNSUPPORTED
    assert mstr(dr=32) == dsa.DSA_ERR_UNSUPPORTED
    assert mstr(dr=64) == dsa.DSA_ERR_INVALID_ARG                      # RoPE columns without their buffer
    assert mstr(dr=64, pe=_vp(16), pet=32) == dsa.DSA_ERR_INVALID_ARG   # RoPE row stride below 64
    assert mstr(dr=64, pe=ctypes.c_void_p(24), pet=64) == dsa.DSA_ERR_INVALID_ARG  # misaligned RoPE buffer
    assert mstr(kh=516, kt=H * 516) == dsa.DSA_ERR_INVALID_ARG          # head stride not a multiple of 8
    assert mstr(kh=128, kt=H * 128) == dsa.DSA_ERR_INVALID_ARG          # heads overlap (256 columns read)
    assert mstr(vt=H * 512 - 8) == dsa.DSA_ERR_INVALID_ARG              # rows overlap
    assert mstr(qh=248, qt=H * 248) == dsa.DSA_ERR_INVALID_ARG          # q heads overlap
    assert mstr(q=ctypes.c_void_p(40)) == dsa.DSA_ERR_INVALID_ARG       # misaligned q
    assert mstr(T=0) == dsa.DSA_OK
    # host-memory per-token call: workspace size, chunking, alignment, shapes
    ws = lib.dsa_sparse_prefill_host_workspace(1000, 1200, 576, 16, 576, 512, 64, 300, 1)
    assert ws >= 1200 * 576 * 2 + 3 * 300 * (16 * 576 * 2 + 64 * 4 + 16 * 512 * 2 + 16 * 4)
    assert lib.dsa_sparse_prefill_host_workspace(1000, 1200, 576, 16, 576, 512, 64, 0, 1) == -1
    # chunk_tokens >= T sizes the streamed form: the table, one buffer set for all T tokens and the
    # counter words (one per token at most, plus `ready`), each part rounded up to 256 bytes
    up = lambda x: (x + 255) // 256 * 256
    per_tok = [16 * 576 * 2, 64 * 4, 16 * 512 * 2, 16 * 4]
    streamed = up(1200 * 576 * 2) + sum(up(1000 * b) for b in per_tok) + up(4 * 1001)
    assert lib.dsa_sparse_prefill_host_workspace(1000, 1200, 576, 16, 576, 512, 64, 1000, 1) == streamed
    assert lib.dsa_sparse_prefill_host_workspace(1000, 1200, 576, 16, 576, 512, 64, 5000, 1) == streamed
    assert lib.dsa_sparse_prefill_host_workspace(1000, 1200, 576, 16, 576, 512, 64, 1000, 0) == streamed - up(1200 * 576 * 2)
    # the ring form: the table and three chunk buffer sets
    assert ws == up(1200 * 576 * 2) + 3 * sum(up(300 * b) for b in per_tok)

    def hostcall(T=1000, H=16, ws_ptr=256, ws_bytes=ws, chunk=300, kv=_vp(16)):
        return lib.dsa_sparse_prefill_host(_vp(16), kv, 1, 1200, 576, _vp(16), T, H, 576, 512, 64, 64, 0.1,
                                           _vp(16), _vp(16), ctypes.c_void_p(ws_ptr), ws_bytes, chunk, None)
    assert hostcall(ws_bytes=ws - 1) == dsa.DSA_ERR_INVALID_ARG
    assert hostcall(chunk=0) == dsa.DSA_ERR_INVALID_ARG
    assert hostcall(ws_ptr=128) == dsa.DSA_ERR_INVALID_ARG
    assert hostcall(ws_ptr=0) == dsa.DSA_ERR_INVALID_ARG
    assert hostcall(kv=None) == dsa.DSA_ERR_INVALID_ARG
    assert hostcall(H=24) == dsa.DSA_ERR_UNSUPPORTED
    assert hostcall(T=0) == dsa.DSA_OK
    # FP8 rows: row width, RoPE width, row stride, alignment
    assert lib.dsa_kv_fp8_row_bytes(64) == 656 and lib.dsa_kv_fp8_row_bytes(0) == 528
    assert lib.dsa_kv_fp8_row_bytes(32) == -1
    assert lib.dsa_kv_fp8_quantize(_vp(16), 10, 576, 32, _vp(16), None) == dsa.DSA_ERR_UNSUPPORTED
    assert lib.dsa_kv_fp8_quantize(_vp(16), 10, 570, 64, _vp(16), None) == dsa.DSA_ERR_INVALID_ARG   # ld < 576
    assert lib.dsa_kv_fp8_quantize(_vp(16), 10, 580, 64, _vp(16), None) == dsa.DSA_ERR_INVALID_ARG   # ld % 8
    assert lib.dsa_kv_fp8_quantize(ctypes.c_void_p(8), 10, 576, 64, _vp(16), None) == dsa.DSA_ERR_INVALID_ARG
    assert lib.dsa_kv_fp8_dequantize(None, 10, 64, _vp(16), 576, None) == dsa.DSA_ERR_INVALID_ARG
    assert lib.dsa_kv_fp8_dequantize(_vp(16), 0, 64, _vp(16), 576, None) == dsa.DSA_OK
    # key mask: one-sided offsets are rejected
    assert lib.dsa_topk_to_key_mask(_vp(16), 8, 4, 4, cu, None, 2, _vp(16), 4, None) == dsa.DSA_ERR_INVALID_ARG
    # local -> physical rows: block size, table width, KV lengths, request offsets
    kl = (ctypes.c_int32 * 2)(40, 8)
    cu2 = (ctypes.c_int32 * 3)(0, 3, 8)
    ok_args = dict(idx=_vp(16), T=8, k=4, ld=4, cq=cu2, kl=kl, nreq=2, bt=_vp(16), mb=3, B=16, N=100, out=_vp(16))

    def l2g(**kw):
        a = dict(ok_args, **kw)
        return lib.dsa_local_to_global(a["idx"], a["T"], a["k"], a["ld"], a["cq"], a["kl"], a["nreq"], a["bt"],
                                       a["mb"], a["B"], a["N"], a["out"], None)
    assert l2g(B=0) == dsa.DSA_ERR_INVALID_ARG
    assert l2g(mb=0) == dsa.DSA_ERR_INVALID_ARG
    assert l2g(k=5) == dsa.DSA_ERR_INVALID_ARG                       # k > ld
    assert l2g(kl=None) == dsa.DSA_ERR_INVALID_ARG
    assert l2g(kl=(ctypes.c_int32 * 2)(49, 8)) == dsa.DSA_ERR_INVALID_ARG   # more positions than 3 blocks of 16
    assert l2g(kl=(ctypes.c_int32 * 2)(-1, 8)) == dsa.DSA_ERR_INVALID_ARG
    assert l2g(cq=(ctypes.c_int32 * 3)(0, 3, 7)) == dsa.DSA_ERR_INVALID_ARG  # offsets do not add up to T
    assert l2g(bt=None) == dsa.DSA_ERR_INVALID_ARG
    assert l2g(out=ctypes.c_void_p(18)) == dsa.DSA_ERR_INVALID_ARG           # misaligned output
    assert l2g(T=0, cq=None, nreq=0) == dsa.DSA_OK


def test_python_binding_refuses_cpu_tensors(lib):
    import torch
    with pytest.raises(ValueError):
        dsa.dsa_sparse_prefill(torch.zeros(2, 16, 576, dtype=torch.bfloat16), torch.zeros(4, 576, dtype=torch.bfloat16),
                               torch.zeros(2, 8, dtype=torch.int32), 8, 1.0)
