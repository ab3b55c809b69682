"""Union list / head-group mask and top-k key mask on the GPU against the
oracle: bit-exact over the whole buffers (padding included)."""
import numpy as np
import pytest

import oracle.dsa_oracle as O
from gpu_util import i32, need_gpu, torch
from synth import WORKLOADS, make_indices, scaled_down

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


def _rows(rng, T, N, k, ld, bad=False):
    idx = np.full((T, ld), -1, dtype=np.int32)
    for t in range(T):
        n = int(rng.integers(0, min(k, N) + 1))
        idx[t, rng.choice(k, size=n, replace=False)] = rng.choice(N, size=n, replace=False)
        if ld > k:
            idx[t, k:] = rng.integers(-1, N, size=ld - k)
    return idx


def _check_union(idx, k, G, N, cu, union_block=128):
    import dsa_sparse_mla_prefill_gb300 as dsa
    upad = O.union_pad(G, k, union_block)
    u, ul, m = dsa.dsa_union_build(i32(idx), k, G, N, cu_seqlens_q=cu, union_pad=upad)
    torch.cuda.synchronize()
    ru, rl, rm = O.union_build(idx, k, G, N, cu, upad)
    assert np.array_equal(ul.cpu().numpy(), rl)
    assert np.array_equal(u.cpu().numpy(), ru)
    assert np.array_equal(m.cpu().numpy(), rm)


@pytest.mark.parametrize("G", [1, 2, 4, 8])
def test_union_random_ragged(G):
    rng = np.random.default_rng(G)
    q_lens = [13, 1, 40, 7]
    cu = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    idx = _rows(rng, int(cu[-1]), 3000, 200, 211)
    _check_union(idx, 200, G, 3000, cu, union_block=16)


@pytest.mark.parametrize("G,N", [(8, 200_000), (2, 200_000), (8, 60_000)])
def test_union_large_tables(G, N):
    """Tables large enough that G per-token bitmaps no longer fit the builder's shared-memory
    budget (G = 8, N = 200k: the single-bitmap variant), and ones where they still do."""
    rng = np.random.default_rng(N + G)
    q_lens = [37, 27]
    cu = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    idx = _rows(rng, int(cu[-1]), N, 384, 392)
    _check_union(idx, 384, G, N, cu)


def test_union_tiny_uniform_config():
    w = WORKLOADS["tiny_uniform_512"]
    idx = make_indices(w, np.random.default_rng(w.seed))
    _check_union(idx, w.k, 8, w.N, w.cu_seqlens_q())


def test_union_nope_two_requests_wide_buffer():
    w = scaled_down(WORKLOADS["nope_2x8192"], (1200, 1100), (1200, 1100), k=512, ld=544)
    idx = make_indices(w, np.random.default_rng(3))
    _check_union(idx, w.k, 8, w.N, w.cu_seqlens_q())


def test_union_full_grouped_config():
    """Every group of the 21504-query / 32768-row workload, bit-exact."""
    w = WORKLOADS["grouped_21k_of_32k"]
    idx = make_indices(w, np.random.default_rng(w.seed))
    _check_union(idx, w.k, w.G, w.N, w.cu_seqlens_q())


def test_union_bad_indices_are_ignored_and_counted():
    import dsa_sparse_mla_prefill_gb300 as dsa
    dsa.dsa_last_device_error()
    rng = np.random.default_rng(5)
    idx = _rows(rng, 16, 500, 64, 64)
    clean = idx.copy()
    idx[3, 5] = 500       # == N
    idx[7, 0] = -7        # < -1
    idx[9, 63] = 10 ** 6
    for t, c in [(3, 5), (7, 0), (9, 63)]:
        clean[t, c] = -1
    upad = O.union_pad(8, 64, 128)
    u, ul, m = dsa.dsa_union_build(i32(idx), 64, 8, 500, union_pad=upad)
    st, counts = dsa.dsa_last_device_error()
    assert st == 0 and counts[0] == 3
    ru, rl, rm = O.union_build(clean, 64, 8, 500, [0, 16], upad)
    assert np.array_equal(u.cpu().numpy(), ru) and np.array_equal(m.cpu().numpy(), rm)


def test_union_empty_tokens_and_empty_group():
    idx = np.full((10, 8), -1, dtype=np.int32)
    idx[9, 2] = 4
    _check_union(idx, 8, 4, 50, np.array([0, 10], np.int32), union_block=16)


def _check_key_mask(idx, k, cq, ck, words):
    import dsa_sparse_mla_prefill_gb300 as dsa
    km = dsa.dsa_topk_to_key_mask(i32(idx), k, words, cu_seqlens_q=cq, cu_seqlens_kv=ck)
    torch.cuda.synchronize()
    ref = O.topk_to_key_mask(idx, k, cq, ck, words)
    assert np.array_equal(km.cpu().numpy().view(np.uint32), ref)


def test_key_mask_two_requests_random():
    rng = np.random.default_rng(9)
    kv_lens, q_lens, k = [300, 517], [120, 77], 64
    cq = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    ck = np.concatenate([[0], np.cumsum(kv_lens)]).astype(np.int32)
    idx = np.full((sum(q_lens), 70), -1, dtype=np.int32)
    for r in range(2):
        for t in range(cq[r], cq[r + 1]):
            n = int(rng.integers(0, k + 1))
            idx[t, rng.choice(k, size=n, replace=False)] = rng.choice(kv_lens[r], size=n, replace=False) + ck[r]
    _check_key_mask(idx, k, cq, ck, 20)


def test_key_mask_full_masked_config():
    w = WORKLOADS["masked_2x8192"]
    idx = make_indices(w, np.random.default_rng(w.seed))
    words = (max(w.kv_lens) + 31) // 32
    import dsa_sparse_mla_prefill_gb300 as dsa
    km = dsa.dsa_topk_to_key_mask(i32(idx), w.k, words, cu_seqlens_q=w.cu_seqlens_q(),
                                  cu_seqlens_kv=w.cu_seqlens_kv()).cpu().numpy().view(np.uint32)
    rng = np.random.default_rng(0)
    rows = sorted(set(rng.integers(0, w.T, 300).tolist()) | {0, 1, 2047, 2048, 8191, 8192, 16383})
    n0 = sum(1 for t in rows if t < 8192)
    ref = O.topk_to_key_mask(idx[rows], w.k, [0, n0, len(rows)], w.cu_seqlens_kv(), words)
    assert np.array_equal(km[rows], ref)
    # popcount of every row equals its number of valid selections
    pc = np.unpackbits(km.view(np.uint8), axis=1).sum(1)
    assert np.array_equal(pc, (idx[:, :w.k] >= 0).sum(1))
