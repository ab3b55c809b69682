"""Request-local -> physical row conversion on the GPU (through the C ABI)
against the oracle: bit-exact rows, the same count of ignored entries, in
place, and the per-token prefill over a paged KV table equal to the one over
the contiguous table."""
import numpy as np
import pytest

import oracle.dsa_oracle as O
from gpu_util import bf, f32, i32, need_gpu, torch
from synth import normal_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


def paged_case(seed, kv_lens, q_lens, B, k, ld, n_bad=3):
    """Shuffled physical blocks (plus spare ones), request-local indices with
    -1 anywhere and some invalid entries."""
    rng = np.random.default_rng(seed)
    nb = [-(-n // B) for n in kv_lens]
    max_blocks = max(nb) + 2
    total = sum(nb) + 5
    ids = rng.permutation(total)
    bt = np.full((len(kv_lens), max_blocks), -1, dtype=np.int32)
    p = 0
    for r, n in enumerate(nb):
        bt[r, :n] = ids[p:p + n]
        p += n
    cq = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    T = int(cq[-1])
    idx = np.full((T, ld), -1, dtype=np.int32)
    for r in range(len(kv_lens)):
        for t in range(cq[r], cq[r + 1]):
            n = min(kv_lens[r], int(rng.integers(0, k + 1)))
            cols = rng.choice(k, size=n, replace=False)
            idx[t, cols] = rng.choice(kv_lens[r], size=n, replace=False)
            for _ in range(n_bad if kv_lens[r] else 0):
                c = int(rng.integers(0, ld))
                idx[t, c] = int(rng.choice([kv_lens[r] + int(rng.integers(0, 5)), -2 - int(rng.integers(0, 9))]))
    return idx, cq, np.asarray(kv_lens, dtype=np.int32), bt, total * B


@pytest.mark.parametrize("ld,k,B", [(72, 64, 16), (70, 64, 16), (128, 100, 64), (33, 33, 1)])
def test_convert_bit_exact(ld, k, B):
    import dsa_sparse_mla_prefill_gb300 as dsa
    idx, cq, kl, bt, N = paged_case(1 + ld, [300, 17, 0, 129], [40, 9, 3, 60], B, k, ld)
    want, bad = O.local_to_global(idx, k, cq, kl, bt, B, N)
    dsa.dsa_last_device_error()
    out = torch.full(idx.shape, 12345, dtype=torch.int32, device="cuda")
    dsa.dsa_local_to_global(i32(idx), k, kl, i32(bt), B, N, cu_seqlens_q=cq, out=out)
    torch.cuda.synchronize()
    st, counts = dsa.dsa_last_device_error()
    assert np.array_equal(out.cpu().numpy(), want)
    assert counts[0] == bad and counts[1] == 0


def test_convert_in_place_and_rows_past_table():
    """In place; a table smaller than the blocks it names (rows >= N) gives -1."""
    import dsa_sparse_mla_prefill_gb300 as dsa
    idx, cq, kl, bt, N = paged_case(7, [64, 100], [20, 30], 8, 48, 48)
    N_small = N - 16   # the two highest physical blocks fall outside the table
    want, bad = O.local_to_global(idx, 48, cq, kl, bt, 8, N_small)
    dsa.dsa_last_device_error()
    buf = i32(idx)
    dsa.dsa_local_to_global(buf, 48, kl, i32(bt), 8, N_small, cu_seqlens_q=cq, out=buf)
    torch.cuda.synchronize()
    st, counts = dsa.dsa_last_device_error()
    assert np.array_equal(buf.cpu().numpy(), want)
    assert counts[0] == bad


def test_per_token_prefill_over_paged_kv():
    """Converted indices over a paged KV table give the same per-token result,
    bit for bit, as global indices over the contiguous table."""
    import dsa_sparse_mla_prefill_gb300 as dsa
    rng = np.random.default_rng(21)
    H, d_qk, B, k = 16, 576, 16, 96
    kv_lens, q_lens = [200, 131], [37, 50]
    cq = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    ck = np.concatenate([[0], np.cumsum(kv_lens)])
    T, Ncont = int(cq[-1]), int(ck[-1])
    kv_cont = normal_bf16(rng, (Ncont, d_qk))
    q = normal_bf16(rng, (T, H, d_qk))
    nb = [-(-n // B) for n in kv_lens]
    total = sum(nb) + 3
    ids = rng.permutation(total)
    bt = np.full((2, max(nb)), -1, dtype=np.int32)
    bt[0, :nb[0]] = ids[:nb[0]]
    bt[1, :nb[1]] = ids[nb[0]:nb[0] + nb[1]]
    kv_phys = normal_bf16(rng, (total * B, d_qk))   # unused rows stay random
    for r in range(2):
        for x in range(kv_lens[r]):
            kv_phys[bt[r, x // B] * B + x % B] = kv_cont[ck[r] + x]
    local = np.full((T, k), -1, dtype=np.int32)
    for r in range(2):
        for t in range(cq[r], cq[r + 1]):
            n = min(k, kv_lens[r])
            local[t, :n] = rng.choice(kv_lens[r], size=n, replace=False)
    glob_cont = np.where(local >= 0, local + np.repeat(ck[:-1], q_lens)[:, None], -1).astype(np.int32)
    rows = dsa.dsa_local_to_global(i32(local), k, np.asarray(kv_lens, np.int32), i32(bt), B, total * B,
                                   cu_seqlens_q=cq)
    o1, l1 = dsa.dsa_sparse_prefill(bf(q), bf(kv_phys), rows, k, 0.07)
    o2, l2 = dsa.dsa_sparse_prefill(bf(q), bf(kv_cont), i32(glob_cont), k, 0.07)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_grouped_prefill_over_paged_kv():
    """Converted indices feed the union build (sorted by physical row) and the grouped
    form over the paged table: union and mask bit-exact against the oracle on the same
    converted rows, and the output equal to the per-token oracle on the contiguous table."""
    import dsa_sparse_mla_prefill_gb300 as dsa
    rng = np.random.default_rng(22)
    H, d_qk, B, k, G = 16, 576, 16, 96, 8
    kv_lens, q_lens = [260, 190], [45, 30]
    cq = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    ck = np.concatenate([[0], np.cumsum(kv_lens)])
    T, Ncont = int(cq[-1]), int(ck[-1])
    kv_cont = normal_bf16(rng, (Ncont, d_qk))
    q = normal_bf16(rng, (T, H, d_qk))
    nb = [-(-n // B) for n in kv_lens]
    total = sum(nb) + 4
    ids = rng.permutation(total)
    bt = np.full((2, max(nb)), -1, dtype=np.int32)
    bt[0, :nb[0]] = ids[:nb[0]]
    bt[1, :nb[1]] = ids[nb[0]:nb[0] + nb[1]]
    kv_phys = normal_bf16(rng, (total * B, d_qk))
    for r in range(2):
        for x in range(kv_lens[r]):
            kv_phys[bt[r, x // B] * B + x % B] = kv_cont[ck[r] + x]
    local = np.full((T, k), -1, dtype=np.int32)
    for r in range(2):
        for t in range(cq[r], cq[r + 1]):
            # causal, with the neighbouring tokens sharing most of their rows
            pos = kv_lens[r] - q_lens[r] + (t - cq[r])
            n = min(k, pos + 1)
            local[t, :n] = rng.choice(pos + 1, size=n, replace=False)
    glob_cont = np.where(local >= 0, local + np.repeat(ck[:-1], q_lens)[:, None], -1).astype(np.int32)
    N = total * B
    rows = dsa.dsa_local_to_global(i32(local), k, np.asarray(kv_lens, np.int32), i32(bt), B, N, cu_seqlens_q=cq)
    upad = dsa.dsa_union_pad(G, k, 128)
    u, ul, m = dsa.dsa_union_build(rows, k, G, N, cu_seqlens_q=cq, union_pad=upad)
    o, l = dsa.dsa_grouped_prefill(bf(q), bf(kv_phys), u, ul, m, G, 0.07, cu_seqlens_q=cq)
    torch.cuda.synchronize()
    st, counts = dsa.dsa_last_device_error()
    assert st == 0, counts
    rows_h = rows.cpu().numpy()
    ru, rl, rm = O.union_build(rows_h, k, G, N, cq, upad)
    assert np.array_equal(u.cpu().numpy(), ru) and np.array_equal(ul.cpu().numpy(), rl)
    assert np.array_equal(m.cpu().numpy(), rm)
    ro, rlse = O.sparse_prefill(q, kv_cont, glob_cont, k, 0.07, d_qk, 512)
    res = O.compare(f32(o), l.cpu().numpy().astype(np.float64), ro, rlse)
    assert res["ok"], res


def test_convert_full_size_sampled():
    """The headline index shape (16384 x 2048) through a shuffled 64-row block
    table; sampled tokens against the oracle, and every valid entry mapped."""
    import dsa_sparse_mla_prefill_gb300 as dsa
    rng = np.random.default_rng(5)
    T, k, B = 16384, 2048, 64
    N = T
    nbk = N // B
    bt = rng.permutation(nbk + 8)[:nbk].astype(np.int32)[None, :]
    idx = np.full((T, k), -1, dtype=np.int32)
    for t in range(0, T, 1):
        n = min(k, t + 1)
        if n == t + 1:
            idx[t, :n] = rng.permutation(n)
        else:
            idx[t] = rng.choice(t + 1, size=k, replace=False)
    out = dsa.dsa_local_to_global(i32(idx), k, np.array([N], np.int32), i32(bt), B, (nbk + 8) * B)
    torch.cuda.synchronize()
    st, counts = dsa.dsa_last_device_error()
    assert counts[0] == 0
    got = out.cpu().numpy()
    assert np.array_equal(got >= 0, idx >= 0)
    toks = np.sort(rng.choice(T, size=24, replace=False))
    want, _ = O.local_to_global(idx[toks], k, None, [N], bt, B, (nbk + 8) * B)
    assert np.array_equal(got[toks], want)
