"""GB300 (sm_103a) DeepSeek-Sparse-Attention prefill over an MLA latent KV cache.

A thin ctypes binding over ``libdsa.so`` (C ABI in ``include/dsa.h``).  The
functions carry the C names and only marshal arguments: they check tensor
dtypes/devices, allocate outputs with torch when none are given, pass raw
device pointers and the current CUDA stream, and raise ``DSAError`` on a
non-zero status.  All arithmetic happens in the library's CUDA kernels;
there is no CPU fallback: without the built library every call raises.

Forms (see the header for the exact contracts):
  dsa_sparse_prefill      per-token sparse attention over each token's top-k rows
  dsa_sparse_prefill_host the same from and to host memory, copies overlapped with the kernel
  dsa_sparse_prefill_host_noalloc  the same without a workspace (fixed library scratch)
  dsa_union_build         sorted union per group + head-group membership mask
  dsa_grouped_prefill     G = 128/H tokens as 128 pseudo-heads over the union
  dsa_topk_to_key_mask    packed per-token key mask from the top-k rows
  dsa_masked_mha_prefill  masked dense MHA with per-head q/k/v
  dsa_masked_mha_prefill_strided  the same on strided views, RoPE key columns shared
  dsa_choose_form         predicted time of each form and the fastest (host only)
  dsa_kv_fp8_quantize / dsa_kv_fp8_dequantize  FP8 latent rows of the KV cache
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdsa.so")
MAX_REQUESTS = 512

DSA_OK, DSA_ERR_INVALID_ARG, DSA_ERR_UNSUPPORTED, DSA_ERR_CUDA, DSA_ERR_DEVICE = range(5)


class DSAError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} ({status})")


_lib_handle = None

_VP = ctypes.c_void_p
_I = ctypes.c_int
_F = ctypes.c_float
_I32P = ctypes.POINTER(ctypes.c_int32)
_L = ctypes.c_int64

FORMS = ("per_token", "grouped", "masked")


class FormCalibration(ctypes.Structure):
    _fields_ = [(n, ctypes.c_double) for n in (
        "hbm_gbs", "bf16_tflops", "per_token_frac", "per_token_ms0", "union_frac", "union_ms0",
        "grouped_frac_576", "grouped_frac_512", "grouped_ms0", "masked_frac_192", "masked_frac_256", "masked_ms0",
        "key_mask_frac", "key_mask_ms0", "union_growth")]


class FormQuery(ctypes.Structure):
    _fields_ = [("num_req", ctypes.c_int), ("q_lens", ctypes.POINTER(ctypes.c_int32)),
                ("kv_lens", ctypes.POINTER(ctypes.c_int32)), ("H", ctypes.c_int), ("k", ctypes.c_int),
                ("d_qk", ctypes.c_int), ("masked_d_qk", ctypes.c_int), ("masked_d_v", ctypes.c_int),
                ("union_rows", ctypes.c_double)]


class FormEstimate(ctypes.Structure):
    _fields_ = [("ms", ctypes.c_double * 3), ("form", ctypes.c_int), ("union_rows", ctypes.c_double)]


_SIGNATURES = {
    "dsa_status_string": (ctypes.c_char_p, [_I]),
    "dsa_version": (_I, []),
    "dsa_union_pad": (ctypes.c_int64, [_I, _I, _I]),
    "dsa_num_groups": (_I, [_I32P, _I, _I, _I, ctypes.POINTER(ctypes.c_int)]),
    "dsa_union_build": (_I, [_VP, _I, _I, _I, _I, _I32P, _I, _I, _VP, _VP, _VP, _I, _VP]),
    "dsa_sparse_prefill": (_I, [_VP, _VP, _I, _I, _VP, _I, _I, _I, _I, _I, _I, _F, _VP, _VP, _VP]),
    "dsa_grouped_prefill": (_I, [_VP, _VP, _I, _I, _VP, _VP, _VP, _I, _I, _I32P, _I, _I, _I, _I, _I, _F, _VP,
                                 _VP, _VP]),
    "dsa_topk_to_key_mask": (_I, [_VP, _I, _I, _I, _I32P, _I32P, _I, _VP, _I, _VP]),
    "dsa_local_to_global": (_I, [_VP, _I, _I, _I, _I32P, _I32P, _I, _VP, _I, _I, _I, _VP, _VP]),
    "dsa_masked_mha_prefill": (_I, [_VP, _VP, _VP, _VP, _I, _I32P, _I32P, _I, _I, _I, _I, _I, _F, _VP, _VP,
                                    _VP]),
    "dsa_masked_mha_prefill_strided": (_I, [_VP, _L, _L, _VP, _L, _L, _VP, _L, _VP, _L, _L, _VP, _I, _I32P, _I32P,
                                            _I, _I, _I, _I, _I, _I, _F, _VP, _VP, _VP]),
    "dsa_sparse_prefill_host_workspace": (_L, [_I, _I, _I, _I, _I, _I, _I, _I, _I]),
    "dsa_sparse_prefill_host_plan": (_I, [_I, _I, _I, _I32P, _I, ctypes.POINTER(ctypes.c_int)]),
    "dsa_sparse_prefill_host": (_I, [_VP, _VP, _I, _I, _I, _VP, _I, _I, _I, _I, _I, _I, _F, _VP, _VP, _VP, _L, _I,
                                     _VP]),
    "dsa_sparse_prefill_host_noalloc": (_I, [_VP, _VP, _I, _I, _I, _VP, _I, _I, _I, _I, _I, _I, _F, _VP, _VP, _I,
                                             _VP]),
    "dsa_kv_fp8_row_bytes": (_L, [_I]),
    "dsa_kv_fp8_quantize": (_I, [_VP, _I, _I, _I, _VP, _VP]),
    "dsa_kv_fp8_dequantize": (_I, [_VP, _I, _I, _VP, _I, _VP]),
    "dsa_sparse_prefill_fp8": (_I, [_VP, _VP, _I, _I, _VP, _I, _I, _I, _I, _I, _I, _F, _VP, _VP, _VP]),
    "dsa_form_calibration_default": (_I, [ctypes.POINTER(FormCalibration)]),
    "dsa_choose_form": (_I, [ctypes.POINTER(FormQuery), ctypes.POINTER(FormCalibration),
                             ctypes.POINTER(FormEstimate)]),
    "dsa_last_device_error": (_I, [_VP, ctypes.POINTER(ctypes.c_uint32)]),
    "dsa_debug_trace": (_I, [_VP, _I]),
    "dsa_debug_wait_timeout": (_I, [_VP]),
}

EXPORTED = tuple(_SIGNATURES)


def lib() -> ctypes.CDLL:
    """The loaded ``libdsa.so`` (raises if it has not been built)."""
    global _lib_handle
    if _lib_handle is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with `python -m dsa_sparse_mla_prefill_gb300.build` "
                               "(the library has no CPU fallback)")
        h = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(h, name)
            fn.restype = res
            fn.argtypes = args
        _lib_handle = h
    return _lib_handle


def status_string(status: int) -> str:
    return lib().dsa_status_string(int(status)).decode()


def _check(status: int, where: str):
    if status != DSA_OK:
        raise DSAError(status, where)


def _host_i32(arr):
    """Host int32 array for a cu_seqlens argument (None stays None)."""
    if arr is None:
        return None, None
    try:
        import torch
        if isinstance(arr, torch.Tensor):
            arr = arr.detach().cpu().numpy()
    except ImportError:  # pragma: no cover
        pass
    a = np.ascontiguousarray(np.asarray(arr, dtype=np.int32))
    return a, a.ctypes.data_as(_I32P)


def _stream(stream, device):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _need(t, dtype, name, ndim=None):
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {t.dim()}")
    return t


def dsa_union_pad(G: int, k: int, union_block: int = 128) -> int:
    return int(lib().dsa_union_pad(G, k, union_block))


def dsa_num_groups(cu_seqlens_q, T: int, G: int) -> int:
    arr, ptr = _host_i32(cu_seqlens_q)
    n = ctypes.c_int(0)
    nreq = 0 if arr is None else len(arr) - 1
    _check(lib().dsa_num_groups(ptr, nreq, T, G, ctypes.byref(n)), "dsa_num_groups")
    return n.value


def dsa_union_build(idx, k: int, G: int, N: int, cu_seqlens_q=None, union_pad: int | None = None,
                    union_block: int = 128, out=None, stream=None):
    """Returns (union_idx [groups, union_pad] int32, union_len [groups] int32,
    mask [groups, union_pad] uint8)."""
    import torch
    _need(idx, torch.int32, "idx", 2)
    T, ld = idx.shape
    if union_pad is None:
        union_pad = dsa_union_pad(G, k, union_block)
    ng = dsa_num_groups(cu_seqlens_q, T, G)
    if out is None:
        u = torch.empty((ng, union_pad), dtype=torch.int32, device=idx.device)
        ul = torch.empty((ng,), dtype=torch.int32, device=idx.device)
        m = torch.empty((ng, union_pad), dtype=torch.uint8, device=idx.device)
    else:
        u, ul, m = out
    arr, ptr = _host_i32(cu_seqlens_q)
    nreq = 0 if arr is None else len(arr) - 1
    _check(lib().dsa_union_build(idx.data_ptr(), T, k, ld, G, ptr, nreq, N, u.data_ptr(), ul.data_ptr(),
                                 m.data_ptr(), union_pad, _stream(stream, idx.device)), "dsa_union_build")
    return u, ul, m


def dsa_sparse_prefill(q, kv, idx, k: int, scale: float, d_v: int = 512, out=None, lse=None, stream=None):
    """Per-token sparse prefill.  q [T, H, d_qk] bf16, kv [N, ld_kv] bf16 (the
    first d_qk columns are the latent key, the first d_v the value), idx
    [T, ld] int32 global rows.  Returns (out [T, H, d_v] bf16, lse [T, H] fp32)."""
    import torch
    _need(q, torch.bfloat16, "q", 3)
    _need(kv, torch.bfloat16, "kv", 2)
    _need(idx, torch.int32, "idx", 2)
    T, H, d_qk = q.shape
    N, ld_kv = kv.shape
    if idx.shape[0] != T:
        raise ValueError("idx rows must match q tokens")
    if out is None:
        out = torch.empty((T, H, d_v), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((T, H), dtype=torch.float32, device=q.device)
    _check(lib().dsa_sparse_prefill(q.data_ptr(), kv.data_ptr(), N, ld_kv, idx.data_ptr(), T, H, d_qk, d_v, k,
                                    idx.shape[1], float(scale), out.data_ptr(), lse.data_ptr(),
                                    _stream(stream, q.device)), "dsa_sparse_prefill")
    return out, lse


def _host_tensor(t, dtype, name, ndim):
    import torch
    if not isinstance(t, torch.Tensor) or t.dtype != dtype or t.dim() != ndim:
        raise TypeError(f"{name} must be a {ndim}-D {dtype} tensor")
    if t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous host tensor (pinned for overlapped copies)")
    return t


def dsa_sparse_prefill_host_workspace(T: int, N: int, ld_kv: int, H: int, d_qk: int, ld: int, chunk_tokens: int,
                                      kv_on_host: bool = True, d_v: int = 512) -> int:
    """Device workspace bytes dsa_sparse_prefill_host needs for these shapes."""
    n = lib().dsa_sparse_prefill_host_workspace(T, N, ld_kv, H, d_qk, d_v, ld, chunk_tokens, int(bool(kv_on_host)))
    if n < 0:
        raise DSAError(DSA_ERR_INVALID_ARG, "dsa_sparse_prefill_host_workspace")
    return int(n)


def dsa_sparse_prefill_host_plan(T: int, chunk_tokens: int, num_sms: int) -> list:
    """Chunk sizes the host-buffer call uses for T tokens on num_sms SMs (host only)."""
    n = ctypes.c_int(0)
    st = lib().dsa_sparse_prefill_host_plan(T, chunk_tokens, num_sms, None, 0, ctypes.byref(n))
    if st != DSA_OK and n.value == 0:
        _check(st, "dsa_sparse_prefill_host_plan")   # bad sizes
    buf = (ctypes.c_int32 * max(1, n.value))()
    _check(lib().dsa_sparse_prefill_host_plan(T, chunk_tokens, num_sms, buf, n.value, ctypes.byref(n)),
           "dsa_sparse_prefill_host_plan")
    return [int(buf[i]) for i in range(n.value)]


def dsa_sparse_prefill_host(q, kv, idx, k: int, scale: float, out, lse, workspace, chunk_tokens: int = 2048,
                            stream=None):
    """Per-token sparse prefill from and to host memory: q [T, H, d_qk] bf16, idx [T, ld] int32,
    out [T, H, 512] bf16 and lse [T, H] fp32 are host tensors (pinned, for the copies to overlap
    the kernel), kv [N, ld_kv] bf16 a host or CUDA tensor, workspace a CUDA uint8 tensor of
    dsa_sparse_prefill_host_workspace bytes.  A workspace sized with chunk_tokens >= T selects
    the streamed form (one kernel launch, copies in chunks of at most chunk_tokens); a smaller
    one the ring of chunk launches.  Asynchronous on `stream` (synchronize before reading out
    and lse)."""
    import torch
    _host_tensor(q, torch.bfloat16, "q", 3)
    _host_tensor(idx, torch.int32, "idx", 2)
    _host_tensor(out, torch.bfloat16, "out", 3)
    _host_tensor(lse, torch.float32, "lse", 2)
    if kv.dtype != torch.bfloat16 or kv.dim() != 2 or not kv.is_contiguous():
        raise TypeError("kv must be a contiguous 2-D bf16 tensor")
    _need(workspace, torch.uint8, "workspace", 1)
    T, H, d_qk = q.shape
    N, ld_kv = kv.shape
    if idx.shape[0] != T or out.shape[0] != T or lse.shape != (T, H):
        raise ValueError("q, idx, out and lse must cover the same tokens")
    _check(lib().dsa_sparse_prefill_host(q.data_ptr(), kv.data_ptr(), 0 if kv.is_cuda else 1, N, ld_kv,
                                         idx.data_ptr(), T, H, d_qk, out.shape[2], k, idx.shape[1], float(scale),
                                         out.data_ptr(), lse.data_ptr(), workspace.data_ptr(), workspace.numel(),
                                         int(chunk_tokens), _stream(stream, workspace.device)),
           "dsa_sparse_prefill_host")
    return out, lse


HOST_NOALLOC_SCRATCH_BYTES = 64 << 20


def dsa_sparse_prefill_host_noalloc(q, kv, idx, k: int, scale: float, out, lse, chunk_tokens: int = 152,
                                    stream=None):
    """dsa_sparse_prefill_host for callers that cannot allocate device memory: the same
    arguments without a workspace; the library's fixed 64 MiB device scratch holds the
    chunks in flight.  Shapes whose buffers need more (dsa_sparse_prefill_host_workspace)
    raise DSAError(DSA_ERR_UNSUPPORTED); lower chunk_tokens then.  Calls that overlap on
    the GPU share the scratch and race: keep them on one stream."""
    import torch
    _host_tensor(q, torch.bfloat16, "q", 3)
    _host_tensor(idx, torch.int32, "idx", 2)
    _host_tensor(out, torch.bfloat16, "out", 3)
    _host_tensor(lse, torch.float32, "lse", 2)
    if kv.dtype != torch.bfloat16 or kv.dim() != 2 or not kv.is_contiguous():
        raise TypeError("kv must be a contiguous 2-D bf16 tensor")
    T, H, d_qk = q.shape
    N, ld_kv = kv.shape
    if idx.shape[0] != T or out.shape[0] != T or lse.shape != (T, H):
        raise ValueError("q, idx, out and lse must cover the same tokens")
    dev = kv.device if kv.is_cuda else torch.device("cuda", torch.cuda.current_device())
    _check(lib().dsa_sparse_prefill_host_noalloc(q.data_ptr(), kv.data_ptr(), 0 if kv.is_cuda else 1, N, ld_kv,
                                                 idx.data_ptr(), T, H, d_qk, out.shape[2], k, idx.shape[1],
                                                 float(scale), out.data_ptr(), lse.data_ptr(), int(chunk_tokens),
                                                 _stream(stream, dev)),
           "dsa_sparse_prefill_host_noalloc")
    return out, lse


def dsa_grouped_prefill(q, kv, union_idx, union_len, mask, G: int, scale: float, cu_seqlens_q=None,
                        d_v: int = 512, out=None, lse=None, stream=None):
    """Grouped sparse prefill over (union_idx, union_len, mask) from dsa_union_build."""
    import torch
    _need(q, torch.bfloat16, "q", 3)
    _need(kv, torch.bfloat16, "kv", 2)
    _need(union_idx, torch.int32, "union_idx", 2)
    _need(union_len, torch.int32, "union_len", 1)
    _need(mask, torch.uint8, "mask", 2)
    T, H, d_qk = q.shape
    N, ld_kv = kv.shape
    if out is None:
        out = torch.empty((T, H, d_v), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((T, H), dtype=torch.float32, device=q.device)
    arr, ptr = _host_i32(cu_seqlens_q)
    nreq = 0 if arr is None else len(arr) - 1
    _check(lib().dsa_grouped_prefill(q.data_ptr(), kv.data_ptr(), N, ld_kv, union_idx.data_ptr(),
                                     union_len.data_ptr(), mask.data_ptr(), union_idx.shape[1], G, ptr, nreq, T,
                                     H, d_qk, d_v, float(scale), out.data_ptr(), lse.data_ptr(),
                                     _stream(stream, q.device)), "dsa_grouped_prefill")
    return out, lse


def dsa_topk_to_key_mask(idx, k: int, words: int, cu_seqlens_q=None, cu_seqlens_kv=None, out=None, stream=None):
    """Packed key mask [T, words] uint32 (viewed as int32 in torch)."""
    import torch
    _need(idx, torch.int32, "idx", 2)
    T, ld = idx.shape
    if out is None:
        out = torch.empty((T, words), dtype=torch.int32, device=idx.device)
    aq, pq = _host_i32(cu_seqlens_q)
    ak, pk = _host_i32(cu_seqlens_kv)
    nreq = 0 if aq is None else len(aq) - 1
    _check(lib().dsa_topk_to_key_mask(idx.data_ptr(), T, k, ld, pq, pk, nreq, out.data_ptr(), words,
                                      _stream(stream, idx.device)), "dsa_topk_to_key_mask")
    return out


def dsa_local_to_global(idx_local, k: int, kv_lens, block_table, block_size: int, N: int, cu_seqlens_q=None,
                        out=None, stream=None):
    """Request-local KV positions [T, ld] -> physical rows of a paged KV cache
    through block_table [num_req, max_blocks] (device int32).  kv_lens: host
    KV length per request.  Returns idx_global [T, ld] (may be ``out`` =
    ``idx_local`` for in place)."""
    import torch
    _need(idx_local, torch.int32, "idx_local", 2)
    _need(block_table, torch.int32, "block_table", 2)
    T, ld = idx_local.shape
    if out is None:
        out = torch.empty_like(idx_local)
    aq, pq = _host_i32(cu_seqlens_q)
    al, pl = _host_i32(kv_lens)
    nreq = 0 if aq is None else len(aq) - 1
    _check(lib().dsa_local_to_global(idx_local.data_ptr(), T, k, ld, pq, pl, nreq, block_table.data_ptr(),
                                     block_table.shape[1], block_size, N, out.data_ptr(),
                                     _stream(stream, idx_local.device)), "dsa_local_to_global")
    return out


def dsa_masked_mha_prefill(q, k, v, key_mask, scale: float, cu_seqlens_q=None, cu_seqlens_kv=None, out=None,
                           lse=None, stream=None):
    """Masked dense MHA.  q [T, H, d_qk], k [Nk, H, d_qk], v [Nk, H, d_v] bf16;
    key_mask [T, words] (int32/uint32 bits).  Returns (out [T, H, d_v], lse [T, H])."""
    import torch
    _need(q, torch.bfloat16, "q", 3)
    _need(k, torch.bfloat16, "k", 3)
    _need(v, torch.bfloat16, "v", 3)
    if key_mask.dtype not in (torch.int32,):
        raise TypeError("key_mask must be int32 (bit pattern of uint32 words)")
    _need(key_mask, key_mask.dtype, "key_mask", 2)
    T, H, d_qk = q.shape
    d_v = v.shape[2]
    if out is None:
        out = torch.empty((T, H, d_v), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((T, H), dtype=torch.float32, device=q.device)
    aq, pq = _host_i32(cu_seqlens_q)
    ak, pk = _host_i32(cu_seqlens_kv)
    nreq = 0 if aq is None else len(aq) - 1
    _check(lib().dsa_masked_mha_prefill(q.data_ptr(), k.data_ptr(), v.data_ptr(), key_mask.data_ptr(),
                                        key_mask.shape[1], pq, pk, nreq, T, H, d_qk, d_v, float(scale),
                                        out.data_ptr(), lse.data_ptr(), _stream(stream, q.device)),
           "dsa_masked_mha_prefill")
    return out, lse


def dsa_masked_mha_prefill_strided(q, k, v, key_mask, scale: float, k_pe=None, cu_seqlens_q=None,
                                   cu_seqlens_kv=None, out=None, lse=None, stream=None):
    """Masked dense MHA on strided views.  q [T, H, d_qk], k [Nk, H, d_qk - d_rope] and
    v [Nk, H, d_v] bf16 with unit stride in the last dimension (e.g. k = kv[..., :256] and
    v = kv[..., 256:] of one [Nk, H, 512] projection output, no copies); k_pe [Nk, d_rope]
    (d_rope = 64) holds the RoPE key columns shared by all heads, or None (d_rope = 0).
    Returns (out [T, H, d_v], lse [T, H])."""
    import torch
    for name, x in (("q", q), ("k", k), ("v", v)):
        if x.dtype != torch.bfloat16 or x.dim() != 3 or x.stride(2) != 1:
            raise TypeError(f"{name} must be a 3-D bf16 tensor with unit stride in its last dimension")
    if key_mask.dtype != torch.int32 or key_mask.dim() != 2 or not key_mask.is_contiguous():
        raise TypeError("key_mask must be a contiguous 2-D int32 tensor (bit pattern of uint32 words)")
    d_rope, pe_ptr, pe_stride = 0, None, 0
    if k_pe is not None:
        if k_pe.dtype != torch.bfloat16 or k_pe.dim() != 2 or k_pe.stride(1) != 1:
            raise TypeError("k_pe must be a 2-D bf16 tensor with unit stride in its last dimension")
        d_rope, pe_ptr, pe_stride = k_pe.shape[1], k_pe.data_ptr(), k_pe.stride(0)
    T, H, d_qk = q.shape
    d_v = v.shape[2]
    if k.shape[2] + d_rope != d_qk:
        raise ValueError("k columns + k_pe columns must equal q's head dim")
    if out is None:
        out = torch.empty((T, H, d_v), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((T, H), dtype=torch.float32, device=q.device)
    aq, pq = _host_i32(cu_seqlens_q)
    ak, pk = _host_i32(cu_seqlens_kv)
    nreq = 0 if aq is None else len(aq) - 1
    _check(lib().dsa_masked_mha_prefill_strided(
        q.data_ptr(), q.stride(0), q.stride(1), k.data_ptr(), k.stride(0), k.stride(1), pe_ptr, pe_stride,
        v.data_ptr(), v.stride(0), v.stride(1), key_mask.data_ptr(), key_mask.shape[1], pq, pk, nreq, T, H,
        d_qk, d_rope, d_v, float(scale), out.data_ptr(), lse.data_ptr(), _stream(stream, q.device)),
        "dsa_masked_mha_prefill_strided")
    return out, lse


def dsa_kv_fp8_row_bytes(d_rope: int) -> int:
    n = int(lib().dsa_kv_fp8_row_bytes(int(d_rope)))
    if n < 0:
        raise DSAError(DSA_ERR_UNSUPPORTED, "dsa_kv_fp8_row_bytes")
    return n


def dsa_kv_fp8_quantize(kv, d_rope: int = 64, out=None, stream=None):
    """bf16 latent rows kv [N, ld_kv] (CUDA) to FP8 rows [N, dsa_kv_fp8_row_bytes(d_rope)] uint8."""
    import torch
    _need(kv, torch.bfloat16, "kv", 2)
    N, ld = kv.shape
    if out is None:
        out = torch.empty((N, dsa_kv_fp8_row_bytes(d_rope)), dtype=torch.uint8, device=kv.device)
    _need(out, torch.uint8, "out", 2)
    _check(lib().dsa_kv_fp8_quantize(kv.data_ptr(), N, ld, int(d_rope), out.data_ptr(), _stream(stream, kv.device)),
           "dsa_kv_fp8_quantize")
    return out


def dsa_kv_fp8_dequantize(fp8, d_rope: int = 64, out=None, stream=None):
    """FP8 rows [N, row_bytes] uint8 (CUDA) to bf16 latent rows [N, 512 + d_rope] (or into out [N, ld_kv])."""
    import torch
    _need(fp8, torch.uint8, "fp8", 2)
    N = fp8.shape[0]
    if fp8.shape[1] != dsa_kv_fp8_row_bytes(d_rope):
        raise ValueError("fp8 rows must be dsa_kv_fp8_row_bytes(d_rope) bytes wide")
    if out is None:
        out = torch.empty((N, 512 + d_rope), dtype=torch.bfloat16, device=fp8.device)
    _need(out, torch.bfloat16, "out", 2)
    _check(lib().dsa_kv_fp8_dequantize(fp8.data_ptr(), N, int(d_rope), out.data_ptr(), out.shape[1],
                                       _stream(stream, fp8.device)), "dsa_kv_fp8_dequantize")
    return out


def dsa_form_calibration_default() -> FormCalibration:
    """The GB300 calibration of the form model (fields as in include/dsa.h)."""
    c = FormCalibration()
    _check(lib().dsa_form_calibration_default(ctypes.byref(c)), "dsa_form_calibration_default")
    return c


def dsa_choose_form(q_lens, kv_lens, H: int, k: int, d_qk: int = 576, masked_dims=None, union_rows=None,
                    calibration: FormCalibration = None):
    """Predicted ms of each form and the fastest applicable one (host only).  q_lens / kv_lens
    per request (queries are the last q_len positions); masked_dims = (d_qk, d_v) of the per-head
    tensors when the masked form can run; union_rows = sum of union_len after dsa_union_build
    (else estimated).  Returns (form name, {form name: ms or None}, union rows used)."""
    ql = np.ascontiguousarray(q_lens, dtype=np.int32)
    kl = np.ascontiguousarray(kv_lens, dtype=np.int32)
    if ql.shape != kl.shape or ql.ndim != 1:
        raise ValueError("q_lens and kv_lens must be 1-D of the same length")
    md = (0, 0) if masked_dims is None else tuple(int(x) for x in masked_dims)
    q = FormQuery(len(ql), ql.ctypes.data_as(_I32P), kl.ctypes.data_as(_I32P), int(H), int(k), int(d_qk), md[0],
                  md[1], -1.0 if union_rows is None else float(union_rows))
    e = FormEstimate()
    _check(lib().dsa_choose_form(ctypes.byref(q), None if calibration is None else ctypes.byref(calibration),
                                 ctypes.byref(e)), "dsa_choose_form")
    ms = {name: (e.ms[i] if e.ms[i] >= 0 else None) for i, name in enumerate(FORMS)}
    return FORMS[e.form], ms, e.union_rows


def dsa_debug_wait_timeout(stream=None, device=None):
    """Queues the failure-path check: one CTA whose bounded wait runs out (about 2 s)."""
    import torch
    dev = device if device is not None else torch.device("cuda", torch.cuda.current_device())
    _check(lib().dsa_debug_wait_timeout(_stream(stream, dev)), "dsa_debug_wait_timeout")


def dsa_last_device_error(stream=None, device=None):
    """Synchronizes the stream and returns (status, [bad_index, timeout, union_overflow, reserved]),
    clearing the device counters."""
    import torch
    dev = device if device is not None else torch.device("cuda", torch.cuda.current_device())
    counts = (ctypes.c_uint32 * 4)()
    st = lib().dsa_last_device_error(_stream(stream, dev), counts)
    return st, [int(c) for c in counts]


def dsa_debug_trace(buffer=None, capacity: int = 0):
    """Diagnostic timeline: record per-tile clock64 stamps of CTAs 0 and 1 into
    ``buffer`` (an int64 CUDA tensor of >= 2 * capacity * 8 elements); call with
    no buffer to switch recording off."""
    if buffer is None:
        _check(lib().dsa_debug_trace(None, 0), "dsa_debug_trace")
        return
    if buffer.numel() < 2 * capacity * 8 or not buffer.is_cuda:
        raise ValueError("trace buffer too small or not on the GPU")
    _check(lib().dsa_debug_trace(buffer.data_ptr(), capacity), "dsa_debug_trace")


def dsa_sparse_prefill_fp8(q, kv_fp8, idx, k: int, scale: float, d_rope: int = 64, d_v: int = 512, out=None,
                           lse=None, stream=None):
    """Per-token sparse prefill over FP8 latent rows kv_fp8 [N, dsa_kv_fp8_row_bytes(d_rope)] uint8, read
    and dequantized inside the kernel.  q [T, H, 512 + d_rope] bf16, idx [T, ld] int32 global rows.
    Returns (out [T, H, d_v] bf16, lse [T, H] fp32), bit-equal to dsa_kv_fp8_dequantize followed by
    dsa_sparse_prefill."""
    import torch
    _need(q, torch.bfloat16, "q", 3)
    _need(kv_fp8, torch.uint8, "kv_fp8", 2)
    _need(idx, torch.int32, "idx", 2)
    T, H, d_qk = q.shape
    N, rb = kv_fp8.shape
    if rb != dsa_kv_fp8_row_bytes(d_rope):
        raise ValueError("kv_fp8 rows must be dsa_kv_fp8_row_bytes(d_rope) bytes")
    if idx.shape[0] != T:
        raise ValueError("idx rows must match q tokens")
    if out is None:
        out = torch.empty((T, H, d_v), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((T, H), dtype=torch.float32, device=q.device)
    _check(lib().dsa_sparse_prefill_fp8(q.data_ptr(), kv_fp8.data_ptr(), N, int(d_rope), idx.data_ptr(), T, H, d_qk,
                                        d_v, k, idx.shape[1], float(scale), out.data_ptr(), lse.data_ptr(),
                                        _stream(stream, q.device)), "dsa_sparse_prefill_fp8")
    return out, lse
