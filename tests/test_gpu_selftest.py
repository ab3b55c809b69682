"""tcgen05 building blocks (instruction/shared-memory descriptors, 128B
swizzle, K-major and MN-major operands, TMEM 32x32b loads) on one
128 x N x K product, against a plain PyTorch fp32 matmul."""
import ctypes
import os

import numpy as np
import pytest

from gpu_util import need_gpu, torch

pytestmark = pytest.mark.gpu

CASES = [(0, 0, 16, 64), (0, 0, 32, 128), (0, 0, 32, 576), (0, 0, 64, 192), (0, 0, 128, 192), (0, 0, 256, 64),
         (1, 0, 16, 128), (1, 0, 32, 128), (1, 0, 128, 64), (0, 1, 64, 64), (0, 1, 128, 128), (0, 1, 256, 64),
         # a_mn = 2: A read from tensor memory (the P operand of P.V)
         (2, 1, 128, 128), (2, 1, 64, 64), (2, 0, 128, 128), (2, 0, 128, 256)]


@pytest.fixture(scope="module")
def selftest():
    need_gpu()
    import dsa_sparse_mla_prefill_gb300 as dsa
    lib = ctypes.CDLL(os.path.join(os.path.dirname(dsa.__file__), "libdsa_selftest.so"))
    fn = lib.dsa_selftest_mma
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int] * 4 + [ctypes.c_void_p, ctypes.c_void_p]
    return fn


@pytest.mark.parametrize("a_mn,b_mn,N,K", CASES)
def test_mma_layouts(selftest, a_mn, b_mn, N, K):
    g = torch.Generator().manual_seed(N * 1000 + K + 7 * a_mn + 13 * b_mn)
    A = torch.randn(128, K, generator=g).to(torch.bfloat16)
    B = torch.randn(N, K, generator=g).to(torch.bfloat16)
    ref = A.float() @ B.float().T
    Ad, Bd = A.cuda(), B.cuda()
    D = torch.full((128, N), float("nan"), device="cuda")
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    rc = selftest(Ad.data_ptr(), Bd.data_ptr(), D.data_ptr(), N, K, a_mn, b_mn, status.data_ptr(),
                  torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    torch.cuda.synchronize()
    assert int(status[1]) == 0, "bounded wait ran out"
    err = (D.cpu() - ref).abs().max().item()
    assert err < 1e-3 * (1 + ref.abs().max().item()), err


@pytest.mark.parametrize("col", [0, 64, 512])
def test_tma_gather4_swizzled_layout(selftest, col):
    """TMA tile::gather4 of 128 listed latent rows (64 columns starting at
    `col`) lands in the 128B-swizzled layout the MMA descriptors assume: row r
    at r*128 bytes, 16-byte piece p at (p ^ (r & 7)) * 16; rows outside the
    table read as zeros."""
    import dsa_sparse_mla_prefill_gb300 as dsa
    lib = ctypes.CDLL(os.path.join(os.path.dirname(dsa.__file__), "libdsa_selftest.so"))
    fn = lib.dsa_selftest_gather4
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p,
                   ctypes.c_void_p, ctypes.c_void_p]
    N, ld = 700, 576
    g = torch.Generator().manual_seed(col + 3)
    kv = torch.randn(N, ld, generator=g).to(torch.bfloat16)
    rows = torch.randint(0, N, (128,), generator=g, dtype=torch.int32)
    rows[5] = -1
    rows[77] = N          # past the end
    rows[126] = N - 1
    out = torch.zeros(128 * 64, dtype=torch.int16, device="cuda")
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    rc = fn(kv.cuda().data_ptr(), N, ld, rows.cuda().data_ptr(), col, out.data_ptr(), status.data_ptr(),
            torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    torch.cuda.synchronize()
    assert int(status[1]) == 0
    img = out.cpu().numpy().view(np.uint16).reshape(128, 8, 8)      # [row][physical piece][element]
    bits = kv.view(torch.int16).numpy().view(np.uint16)
    for r in range(128):
        src = int(rows[r])
        for p in range(8):
            want = bits[src, col + 8 * p: col + 8 * p + 8] if 0 <= src < N else np.zeros(8, np.uint16)
            assert np.array_equal(img[r, p ^ (r & 7)], want), (r, p)


# a_mn, b_mn, N, K, gather: the shapes the pair kernels use (QK: K-major A of
# 128 slots per CTA, K-major q halves, K = 576 through tile::gather4 loads that
# complete on the even CTA's barrier; P.V: MN-major V^T and MN-major P)
PAIR_CASES = [(0, 0, 128, 64, 0), (0, 0, 128, 576, 0), (0, 0, 256, 64, 0), (0, 0, 64, 128, 0), (0, 0, 32, 64, 0),
              (1, 1, 128, 128, 0), (1, 0, 128, 128, 0), (0, 1, 256, 128, 0), (0, 0, 128, 576, 1),
              (0, 0, 128, 128, 1)]


def _lib():
    import dsa_sparse_mla_prefill_gb300 as dsa
    return ctypes.CDLL(os.path.join(os.path.dirname(dsa.__file__), "libdsa_selftest.so"))


@pytest.mark.parametrize("a_mn,b_mn,N,K,gather", PAIR_CASES)
def test_pair_mma_layouts(selftest, a_mn, b_mn, N, K, gather):
    """cta_group::2: one M = 256 product of a 2-CTA cluster, A rows and B
    columns split between the two CTAs' shared memory, D rows split between
    their tensor memories; against a plain PyTorch fp32 matmul."""
    fn = _lib().dsa_selftest_mma_pair
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int] * 5 + [ctypes.c_void_p, ctypes.c_void_p]
    g = torch.Generator().manual_seed(N * 1000 + K + 7 * a_mn + 13 * b_mn + 101 * gather)
    A = torch.randn(256, K, generator=g).to(torch.bfloat16)
    B = torch.randn(N, K, generator=g).to(torch.bfloat16)
    ref = A.float() @ B.float().T
    Ad, Bd = A.cuda(), B.cuda()
    D = torch.full((256, N), float("nan"), device="cuda")
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    rc = fn(Ad.data_ptr(), Bd.data_ptr(), D.data_ptr(), N, K, a_mn, b_mn, gather, status.data_ptr(),
            torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    torch.cuda.synchronize()
    assert int(status[1]) == 0, "bounded wait ran out"
    err = (D.cpu() - ref).abs().max().item()
    assert err < 1e-3 * (1 + ref.abs().max().item()), err
