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


@pytest.mark.gpu
def test_tma_gather4_multicast_cluster(selftest):
    """tile::gather4 with cluster multicast: each CTA of a 2-CTA cluster
    issues half of the 128 row gathers for both; both CTAs end up with the
    same 128B-swizzled image of all 128 rows (rows outside the table read as
    zeros)."""
    import dsa_sparse_mla_prefill_gb300 as dsa
    lib = ctypes.CDLL(os.path.join(os.path.dirname(dsa.__file__), "libdsa_selftest.so"))
    fn = lib.dsa_selftest_gather4_mc
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p,
                   ctypes.c_void_p, ctypes.c_void_p]
    N, ld, col = 900, 576, 512
    g = torch.Generator().manual_seed(11)
    kv = torch.randn(N, ld, generator=g).to(torch.bfloat16)
    rows = torch.randint(0, N, (128,), generator=g, dtype=torch.int32)
    rows[3] = -1
    rows[100] = N
    out = torch.zeros(2 * 128 * 64, dtype=torch.int16, device="cuda")
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    rc = fn(kv.cuda().data_ptr(), N, ld, rows.cuda().data_ptr(), col, out.data_ptr(), status.data_ptr(),
            torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    torch.cuda.synchronize()
    assert int(status[1]) == 0
    imgs = out.cpu().numpy().view(np.uint16).reshape(2, 128, 8, 8)
    bits = kv.view(torch.int16).numpy().view(np.uint16)
    for rank in range(2):
        for r in range(128):
            src = int(rows[r])
            for p in range(8):
                want = bits[src, col + 8 * p: col + 8 * p + 8] if 0 <= src < N else np.zeros(8, np.uint16)
                assert np.array_equal(imgs[rank, r, p ^ (r & 7)], want), (rank, r, p)


# ---------------------------------------------------------------------------
# Timing probes of the self-test library (the measurements behind the
# kernels' issue structure).  Cycle counts depend on the GPU and on what else
# runs, so these check only that every probe completes with no bounded wait
# running out and reports positive, self-consistent counts.
# ---------------------------------------------------------------------------
def _lib():
    import dsa_sparse_mla_prefill_gb300 as dsa
    return ctypes.CDLL(os.path.join(os.path.dirname(dsa.__file__), "libdsa_selftest.so"))


@pytest.mark.parametrize("mode", [3, 8, 9, 10, 11, 12, 13, 14, 15, 16, 17, 18, 19, 20, 21, 22, 23, 24, 25, 26, 27, 28])
def test_mma_issue_timing_modes(selftest, mode):
    fn = _lib().dsa_selftest_mma_timing
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.c_int] * 3 + [ctypes.c_void_p] * 3
    out = torch.zeros(2, dtype=torch.int64, device="cuda")
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    rc = fn(64, 144, mode, out.data_ptr(), status.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    torch.cuda.synchronize()
    assert int(status[1]) == 0, "bounded wait ran out"
    total = int(out[1])
    # at least the 36 MMAs one issuing warp ends with, at ~20 cycles or more each
    assert 36 * 20 < total < 10_000_000, total


@pytest.mark.parametrize("mc", [0, 1])
def test_gather4_rate_probe(selftest, mc):
    fn = _lib().dsa_selftest_gather4_rate
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                   ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                   ctypes.c_void_p]
    N, ld, grid, per = 4096, 576, 8, 256
    g = torch.Generator().manual_seed(3)
    kv = torch.randn(N, ld, generator=g).to(torch.bfloat16).cuda()
    rows = torch.randint(0, N, (grid * per * 4,), generator=g, dtype=torch.int32).cuda()
    out = torch.zeros(grid, dtype=torch.int64, device="cuda")
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    for flags in (0, 3, 4, 8):
        rc = fn(kv.data_ptr(), N, ld, rows.data_ptr(), grid, per, 8, 4, mc, flags, out.data_ptr(), status.data_ptr(),
                torch.cuda.current_stream().cuda_stream)
        assert rc == 0
        torch.cuda.synchronize()
        assert int(status[1]) == 0
        assert (out > 0).all()


@pytest.mark.parametrize("mc,flags,warps,lanes", [(0, 0, 8, 4), (1, 0, 6, 3), (0, 32, 6, 32), (1, 32, 6, 16),
                                                  (0, 16, 8, 4), (0, 64 | 128 | 4, 8, 4)])
def test_ring_turnaround_probe(selftest, mc, flags, warps, lanes):
    fn = _lib().dsa_selftest_ring_rate
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_void_p] + [ctypes.c_int] * 9 + \
        [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    N, ld, grid, ntiles = 4096, 576, 4, 4
    stages = warps if flags & 32 else 6
    g = torch.Generator().manual_seed(5)
    kv = torch.randn(N, ld, generator=g).to(torch.bfloat16).cuda()
    rows = torch.sort(torch.randint(0, N, (grid // 2 * ntiles, 128), generator=g, dtype=torch.int32), dim=1)
    rows = rows.values.reshape(-1).cuda()
    out = torch.zeros(grid, dtype=torch.int64, device="cuda")
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    rc = fn(kv.data_ptr(), N, ld, rows.data_ptr(), ntiles, grid, 9 * ntiles, stages, warps, lanes, mc, 100, flags,
            out.data_ptr(), status.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    torch.cuda.synchronize()
    assert int(status[1]) == 0
    # every stage is held 100 cycles by the consumer
    assert (out >= 9 * ntiles * 100).all(), out
