"""Pins for the fp64 oracle: checks against facts that do not come from the
oracle itself (brute force written separately, closed forms, invariants, an
independent library routine).  Each ``pin_*`` returns True when it holds, so
that ``test_oracle_pins.py`` can also plant mistakes in the oracle and show
that some pin catches each of them.

All pins look the oracle up through the module at call time (``O.xxx``),
so a monkeypatched oracle function is what they exercise.
"""
from __future__ import annotations

import math
import struct

import numpy as np

import oracle.dsa_oracle as O
from synth import normal_bf16, f32_to_bf16_bits

TOL = 1e-12


# ----------------------------------------------------------------------------
# a separately written decoder and brute-force dense attention (pure Python)
# ----------------------------------------------------------------------------
def _bf16_bits_to_float(b: int) -> float:
    return struct.unpack("<f", struct.pack("<I", (int(b) & 0xFFFF) << 16))[0]


def brute_dense_attention(q_bits, kv_bits, idx, k, scale, d_qk, d_v):
    """Full N-length scores with -inf where the key is not selected, then a
    dense softmax.  Plain Python floats and loops."""
    T, H, _ = q_bits.shape
    N = kv_bits.shape[0]
    kvf = [[_bf16_bits_to_float(kv_bits[n, d]) for d in range(kv_bits.shape[1])] for n in range(N)]
    out = np.zeros((T, H, d_v))
    lse = np.zeros((T, H))
    for t in range(T):
        chosen = set(int(x) for x in idx[t][:k] if 0 <= int(x) < N)
        for h in range(H):
            qv = [_bf16_bits_to_float(q_bits[t, h, d]) for d in range(d_qk)]
            scores = []
            for n in range(N):
                if n in chosen:
                    scores.append(scale * math.fsum(qv[d] * kvf[n][d] for d in range(d_qk)))
                else:
                    scores.append(-math.inf)
            mx = max(scores)
            if mx == -math.inf:
                lse[t, h] = -math.inf
                continue
            w = [math.exp(s - mx) if s != -math.inf else 0.0 for s in scores]
            z = math.fsum(w)
            lse[t, h] = mx + math.log(z)
            for d in range(d_v):
                out[t, h, d] = math.fsum(w[n] * kvf[n][d] for n in range(N)) / z
    return out, lse


def _close(a, b, tol=TOL):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    if a.shape != b.shape:
        return False
    if not np.array_equal(np.isinf(a), np.isinf(b)):
        return False
    f = np.isfinite(b)
    return bool(np.all(np.abs(a[f] - b[f]) <= tol * (1.0 + np.abs(b[f]))))


def _random_rows(rng, T, N, k, ld, p_dense=0.0):
    """Index rows with -1 anywhere in the first k columns, junk-free beyond."""
    idx = np.full((T, ld), -1, dtype=np.int32)
    for t in range(T):
        n = int(rng.integers(0, min(k, N) + 1))
        sel = rng.choice(N, size=n, replace=False)
        row = np.full(k, -1, dtype=np.int64)
        pos = rng.choice(k, size=n, replace=False)
        row[pos] = sel
        idx[t, :k] = row
        if ld > k:  # columns beyond k may hold anything valid; they must be ignored
            idx[t, k:] = rng.integers(-1, N, size=ld - k)
    return idx


# ----------------------------------------------------------------------------
# per-token pins
# ----------------------------------------------------------------------------
def pin_bruteforce(seed=0) -> bool:
    """Oracle == brute-force dense attention with a -inf mask (tiny sizes,
    RoPE-like extra K columns so d_qk > d_v, -1 anywhere, ld > k)."""
    rng = np.random.default_rng(seed)
    ok = True
    for (T, N, H, d_qk, d_v, k, ld) in [(6, 20, 3, 24, 16, 7, 9), (5, 33, 2, 32, 32, 40, 40),
                                        (4, 9, 4, 12, 8, 3, 5)]:
        q = normal_bf16(rng, (T, H, d_qk))
        kv = normal_bf16(rng, (N, d_qk))
        idx = _random_rows(rng, T, N, k, ld)
        scale = 1.0 / math.sqrt(float(d_qk) * 0.75)
        o_ref, l_ref = brute_dense_attention(q, kv, idx, k, scale, d_qk, d_v)
        o, l = O.sparse_prefill(q, kv, idx, k, scale, d_qk, d_v)
        ok &= _close(o, o_ref) and _close(l, l_ref)
    return ok


def pin_single_key(seed=1) -> bool:
    """|S_t| = 1: out = that row's V, lse = its scaled score."""
    rng = np.random.default_rng(seed)
    T, N, H, d_qk, d_v = 4, 10, 3, 16, 8
    q = normal_bf16(rng, (T, H, d_qk))
    kv = normal_bf16(rng, (N, d_qk))
    idx = np.full((T, 5), -1, dtype=np.int32)
    rows = [3, 0, 9, 5]
    for t, r in enumerate(rows):
        idx[t, t % 5] = r
    scale = 0.37
    o, l = O.sparse_prefill(q, kv, idx, 5, scale, d_qk, d_v)
    ok = True
    for t, r in enumerate(rows):
        v = [_bf16_bits_to_float(kv[r, d]) for d in range(d_v)]
        for h in range(H):
            s = scale * math.fsum(_bf16_bits_to_float(q[t, h, d]) * _bf16_bits_to_float(kv[r, d])
                                  for d in range(d_qk))
            ok &= abs(l[t, h] - s) <= TOL * (1 + abs(s))
            ok &= bool(np.all(np.abs(o[t, h] - np.asarray(v)) <= TOL))
    return ok


def pin_zero_query(seed=2) -> bool:
    """q = 0: uniform weights, out = mean of the selected V rows, lse = ln n."""
    rng = np.random.default_rng(seed)
    T, N, H, d_qk, d_v, k = 3, 30, 2, 16, 12, 11
    q = np.zeros((T, H, d_qk), dtype=np.uint16)
    kv = normal_bf16(rng, (N, d_qk))
    idx = _random_rows(rng, T, N, k, k)
    idx[0, :] = -1
    idx[0, 2] = 7
    o, l = O.sparse_prefill(q, kv, idx, k, 0.5, d_qk, d_v)
    ok = True
    for t in range(T):
        sel = [int(x) for x in idx[t] if x >= 0]
        if not sel:
            ok &= bool(np.all(o[t] == 0)) and bool(np.all(np.isneginf(l[t])))
            continue
        mean = [math.fsum(_bf16_bits_to_float(kv[n, d]) for n in sel) / len(sel) for d in range(d_v)]
        for h in range(H):
            ok &= abs(l[t, h] - math.log(len(sel))) <= TOL
            ok &= bool(np.all(np.abs(o[t, h] - np.asarray(mean)) <= TOL))
    return ok


def pin_equal_keys(seed=3) -> bool:
    """All selected K rows equal (V rows differ): uniform weights; lse = s + ln n."""
    rng = np.random.default_rng(seed)
    N, H, d_qk, d_v, k = 12, 3, 20, 8, 6
    kv = normal_bf16(rng, (N, d_qk))
    shared = normal_bf16(rng, (d_qk - d_v,))
    kv[:, d_v:] = shared[None, :]
    kv[:, :d_v] = normal_bf16(rng, (N, d_v))
    q = normal_bf16(rng, (1, H, d_qk))
    q[0, :, :d_v] = 0  # score depends only on the shared (RoPE-like) columns
    idx = np.array([[1, 4, -1, 9, 10, 2]], dtype=np.int32)
    sel = [1, 4, 9, 10, 2]
    o, l = O.sparse_prefill(q, kv, idx, k, 0.25, d_qk, d_v)
    ok = True
    for h in range(H):
        s = 0.25 * math.fsum(_bf16_bits_to_float(q[0, h, d]) * _bf16_bits_to_float(shared[d - d_v])
                             for d in range(d_v, d_qk))
        ok &= abs(l[0, h] - (s + math.log(len(sel)))) <= TOL * (1 + abs(s))
        mean = [math.fsum(_bf16_bits_to_float(kv[n, d]) for n in sel) / len(sel) for d in range(d_v)]
        ok &= bool(np.all(np.abs(o[0, h] - np.asarray(mean)) <= TOL))
    return ok


def pin_two_keys_closed_form() -> bool:
    """Hand-worked case: q = (1, 0), rows r0 = (0, 0), r1 = (1, 1), scale 1,
    D_QK = D_V = 2.  Scores 0 and 1, so weights 1/(1+e), e/(1+e);
    out = (e/(1+e)) * (1, 1); lse = ln(1 + e)."""
    one = f32_to_bf16_bits(np.array([1.0], np.float32))[0]
    q = np.array([[[one, 0]]], dtype=np.uint16)
    kv = np.array([[0, 0], [one, one]], dtype=np.uint16)
    idx = np.array([[1, -1, 0]], dtype=np.int32)
    o, l = O.sparse_prefill(q, kv, idx, 3, 1.0, 2, 2)
    w1 = math.e / (1.0 + math.e)
    return abs(l[0, 0] - math.log(1.0 + math.e)) <= TOL and \
        bool(np.all(np.abs(o[0, 0] - w1) <= TOL))


def pin_order_and_padding_invariance(seed=4) -> bool:
    """Permuting a row's first k entries, moving -1s around and changing the
    columns beyond k leave the result unchanged (to rounding)."""
    rng = np.random.default_rng(seed)
    T, N, H, d_qk, d_v, k, ld = 5, 40, 2, 24, 16, 12, 16
    q = normal_bf16(rng, (T, H, d_qk))
    kv = normal_bf16(rng, (N, d_qk))
    idx = _random_rows(rng, T, N, k, ld)
    o1, l1 = O.sparse_prefill(q, kv, idx, k, 0.3, d_qk, d_v)
    idx2 = idx.copy()
    for t in range(T):
        idx2[t, :k] = rng.permutation(idx2[t, :k])
        idx2[t, k:] = rng.integers(-1, N, size=ld - k)
    o2, l2 = O.sparse_prefill(q, kv, idx2, k, 0.3, d_qk, d_v)
    return _close(o1, o2, 1e-13) and _close(l1, l2, 1e-13)


def pin_dense_causal_sdpa(seed=5) -> bool:
    """k >= t+1 with every position selected equals dense causal attention,
    checked against torch's scaled_dot_product_attention in float64 (CPU)."""
    import torch
    import torch.nn.functional as F
    rng = np.random.default_rng(seed)
    T, H, d_qk, d_v = 23, 4, 40, 32
    q = normal_bf16(rng, (T, H, d_qk))
    kv = normal_bf16(rng, (T, d_qk))
    k = T + 3
    idx = np.full((T, k), -1, dtype=np.int32)
    for t in range(T):
        idx[t, :t + 1] = rng.permutation(t + 1)
    scale = 1.0 / math.sqrt(17.0)
    o, _ = O.sparse_prefill(q, kv, idx, k, scale, d_qk, d_v)

    def dec(b):
        return torch.from_numpy((b.astype(np.uint32) << 16).view(np.float32).astype(np.float64))
    qt = dec(q).permute(1, 0, 2).unsqueeze(0)                 # [1, H, T, D]
    kt = dec(kv).unsqueeze(0).unsqueeze(0).expand(1, H, T, d_qk)
    vt = dec(kv[:, :d_v]).unsqueeze(0).unsqueeze(0).expand(1, H, T, d_v)
    ref = F.scaled_dot_product_attention(qt, kt, vt, is_causal=True, scale=scale)
    ref = ref[0].permute(1, 0, 2).numpy()
    return bool(np.max(np.abs(o - ref)) <= 1e-12)


# ----------------------------------------------------------------------------
# union / mask pins
# ----------------------------------------------------------------------------
def brute_union(idx, k, G, N, cu):
    """Union and mask from Python sets (independent of np.unique/searchsorted)."""
    res = []
    cu = [int(x) for x in cu]
    for r in range(len(cu) - 1):
        for s in range(cu[r], cu[r + 1], G):
            n = min(G, cu[r + 1] - s)
            sets = [set(int(x) for x in idx[s + j][:k] if 0 <= int(x) < N) for j in range(n)]
            u = sorted(set().union(*sets))
            m = [sum((1 << j) for j in range(n) if x in sets[j]) for x in u]
            res.append((u, m))
    return res


def pin_union_worked_example() -> bool:
    """Hand-worked: G = 2, k = 4; token 0 selects {5, 2, 9}, token 1 {9, 3, 5}.
    Union (ascending) = [2, 3, 5, 9]; membership bits = [01, 10, 11, 11];
    union_pad = ceil(2*4 / 4) * 4 = 8 with a union block of 4."""
    idx = np.array([[5, 2, -1, 9], [9, 3, 5, -1]], dtype=np.int32)
    upad = O.union_pad(2, 4, 4)
    u, ul, m = O.union_build(idx, 4, 2, 16, [0, 2], upad)
    return upad == 8 and ul.tolist() == [4] and \
        u.tolist() == [[2, 3, 5, 9, -1, -1, -1, -1]] and m.tolist() == [[1, 2, 3, 3, 0, 0, 0, 0]]


def pin_union_bruteforce(seed=6) -> bool:
    """Union/mask equal the Python-set construction over ragged requests and
    every G in 1..8, and satisfy the structural invariants."""
    rng = np.random.default_rng(seed)
    ok = True
    for G in range(1, 9):
        q_lens = [int(x) for x in rng.integers(1, 3 * G + 2, size=3)]
        T = sum(q_lens)
        N, k, ld = 70, 9, 11
        idx = _random_rows(rng, T, N, k, ld)
        cu = np.concatenate([[0], np.cumsum(q_lens)])
        upad = O.union_pad(G, k, 8)
        u, ul, m = O.union_build(idx, k, G, N, cu, upad)
        ref = brute_union(idx, k, G, N, cu)
        ok &= len(ref) == u.shape[0]
        for g, (ru, rm) in enumerate(ref):
            U = int(ul[g])
            ok &= U == len(ru)
            ok &= u[g, :U].tolist() == ru and m[g, :U].tolist() == rm
            ok &= bool(np.all(u[g, U:] == -1)) and bool(np.all(m[g, U:] == 0))
            ok &= bool(np.all(np.diff(u[g, :U]) > 0))
    return ok


def pin_union_popcounts(seed=7) -> bool:
    """For every token j of a group, the number of union slots with bit j set
    equals the size of its own valid top-k set."""
    rng = np.random.default_rng(seed)
    T, N, k, G = 37, 200, 25, 8
    idx = _random_rows(rng, T, N, k, k)
    cu = [0, 20, 37]
    upad = O.union_pad(G, k, 16)
    u, ul, m = O.union_build(idx, k, G, N, cu, upad)
    ok = True
    for g, (t0, n) in enumerate(O.groups(cu, G)):
        for j in range(n):
            cnt = int(((m[g].astype(np.int64) >> j) & 1).sum())
            ok &= cnt == int(((idx[t0 + j][:k] >= 0)).sum())
        ok &= int(ul[g]) <= min(n * k, N)
    return ok


def pin_grouped_equals_per_token(seed=8) -> bool:
    """Grouped attention over (union, mask) equals per-token attention for
    ragged requests, several H / G and empty tokens."""
    rng = np.random.default_rng(seed)
    ok = True
    for (H, G, q_lens) in [(4, 2, [5, 3]), (2, 8, [13]), (1, 8, [9, 1, 8]), (8, 1, [4])]:
        T = sum(q_lens)
        N, d_qk, d_v, k = 50, 24, 16, 10
        q = normal_bf16(rng, (T, H, d_qk))
        kv = normal_bf16(rng, (N, d_qk))
        idx = _random_rows(rng, T, N, k, k)
        idx[0, :] = -1  # one token with no selection at all
        cu = np.concatenate([[0], np.cumsum(q_lens)])
        o1, l1 = O.sparse_prefill(q, kv, idx, k, 0.2, d_qk, d_v)
        upad = O.union_pad(G, k, 8)
        u, ul, m = O.union_build(idx, k, G, N, cu, upad)
        o2, l2 = O.grouped_prefill(q, kv, u, ul, m, G, cu, 0.2, d_qk, d_v)
        ok &= _close(o1, o2, 1e-12) and _close(l1, l2, 1e-12)
    return ok


def pin_key_mask_bruteforce(seed=9) -> bool:
    """Key-mask bits equal the request-local positions of the valid top-k."""
    rng = np.random.default_rng(seed)
    kv_lens = [40, 70]
    q_lens = [6, 5]
    cq = np.concatenate([[0], np.cumsum(q_lens)])
    ck = np.concatenate([[0], np.cumsum(kv_lens)])
    k = 9
    idx = np.full((sum(q_lens), k), -1, dtype=np.int32)
    for r in range(2):
        for t in range(cq[r], cq[r + 1]):
            n = int(rng.integers(0, k + 1))
            sel = rng.choice(kv_lens[r], size=n, replace=False) + ck[r]
            idx[t, rng.choice(k, size=n, replace=False)] = sel
    words = 3
    km = O.topk_to_key_mask(idx, k, cq, ck, words)
    ok = True
    for r in range(2):
        for t in range(cq[r], cq[r + 1]):
            want = set(int(x) - int(ck[r]) for x in idx[t] if x >= 0)
            got = set(n for n in range(32 * words) if (int(km[t, n // 32]) >> (n % 32)) & 1)
            ok &= want == got
    return ok


def pin_masked_equals_sparse(seed=10) -> bool:
    """Masked MHA over per-head K/V equals sparse attention when every head's
    K/V is the shared latent row (k[n, h] = kv[n, :d_qk], v[n, h] = kv[n, :d_v]),
    across two requests (key offsets matter)."""
    rng = np.random.default_rng(seed)
    kv_lens, q_lens = [17, 23], [6, 9]
    H, d_qk, d_v, k = 3, 24, 16, 8
    cq = np.concatenate([[0], np.cumsum(q_lens)])
    ck = np.concatenate([[0], np.cumsum(kv_lens)])
    N, T = sum(kv_lens), sum(q_lens)
    kv = normal_bf16(rng, (N, d_qk))
    q = normal_bf16(rng, (T, H, d_qk))
    idx = np.full((T, k), -1, dtype=np.int32)
    for r in range(2):
        for t in range(cq[r], cq[r + 1]):
            n = int(rng.integers(0, k + 1))
            idx[t, :n] = rng.choice(kv_lens[r], size=n, replace=False) + ck[r]
    km = O.topk_to_key_mask(idx, k, cq, ck, 1)
    kh = np.repeat(kv[:, None, :], H, axis=1)
    vh = np.repeat(kv[:, None, :d_v], H, axis=1)
    o1, l1 = O.masked_mha_prefill(q, kh, vh, km, cq, ck, 0.3)
    o2, l2 = O.sparse_prefill(q, kv, idx, k, 0.3, d_qk, d_v)
    return _close(o1, o2, 1e-12) and _close(l1, l2, 1e-12)


def pin_masked_dense_causal_sdpa(seed=11) -> bool:
    """A causal full mask makes masked MHA equal to dense causal SDPA (float64,
    per-head K/V, one request)."""
    import torch
    import torch.nn.functional as F
    rng = np.random.default_rng(seed)
    T, H, d_qk, d_v = 19, 3, 24, 8
    q = normal_bf16(rng, (T, H, d_qk))
    kh = normal_bf16(rng, (T, H, d_qk))
    vh = normal_bf16(rng, (T, H, d_v))
    km = np.zeros((T, 1), dtype=np.uint32)
    for t in range(T):
        km[t, 0] = np.uint32((1 << (t + 1)) - 1)
    o, _ = O.masked_mha_prefill(q, kh, vh, km, [0, T], [0, T], 0.4)

    def dec(b):
        return torch.from_numpy((b.astype(np.uint32) << 16).view(np.float32).astype(np.float64))
    ref = F.scaled_dot_product_attention(dec(q).permute(1, 0, 2)[None], dec(kh).permute(1, 0, 2)[None],
                                         dec(vh).permute(1, 0, 2)[None], is_causal=True, scale=0.4)
    ref = ref[0].permute(1, 0, 2).numpy()
    return bool(np.max(np.abs(o - ref)) <= 1e-12)


def pin_local_to_global_paged_round_trip(seed=12) -> bool:
    """Paged storage round trip: each request's KV rows are copied block by
    block into a shuffled physical table through its block table; the row the
    oracle returns for position x must hold the request's row x.  Invalid
    entries (past the request, unmapped block, below -1) come back -1 and are
    counted; -1 and columns at or past k come back -1 uncounted."""
    rng = np.random.default_rng(seed)
    B = 4
    kv_lens = [13, 7, 0, 21]
    nb = [-(-n // B) for n in kv_lens]
    max_blocks = max(nb) + 1
    total_blocks = sum(nb) + 3
    phys_ids = rng.permutation(total_blocks)
    bt = np.full((len(kv_lens), max_blocks), -1, dtype=np.int32)
    pos = 0
    for r, n in enumerate(nb):
        bt[r, :n] = phys_ids[pos:pos + n]
        pos += n
    N = total_blocks * B
    local = [rng.integers(0, 1 << 30, size=n) for n in kv_lens]
    phys = np.full(N, -7, dtype=np.int64)
    for r in range(len(kv_lens)):
        for b in range(nb[r]):
            seg = local[r][b * B:(b + 1) * B]
            phys[bt[r, b] * B: bt[r, b] * B + len(seg)] = seg
    q_lens = [3, 2, 2, 4]
    cq = np.concatenate([[0], np.cumsum(q_lens)])
    k, ld = 6, 8
    T = int(cq[-1])
    idx = np.full((T, ld), -1, dtype=np.int32)
    want_bad = 0
    for r in range(len(kv_lens)):
        for t in range(cq[r], cq[r + 1]):
            n = min(kv_lens[r], 4)
            idx[t, :n] = rng.choice(kv_lens[r], size=n, replace=False) if n else []
            idx[t, 4] = kv_lens[r] + 2          # past the request
            idx[t, 5] = -3                      # below -1
            idx[t, 6] = 0 if kv_lens[r] else -1  # column >= k: ignored
            want_bad += 2
    out, bad = O.local_to_global(idx, k, cq, kv_lens, bt, B, N)
    ok = bad == want_bad
    for r in range(len(kv_lens)):
        for t in range(cq[r], cq[r + 1]):
            for j in range(ld):
                x = int(idx[t, j])
                if j < k and 0 <= x < kv_lens[r]:
                    ok &= int(out[t, j]) >= 0 and phys[int(out[t, j])] == local[r][x]
                else:
                    ok &= int(out[t, j]) == -1
    return bool(ok)


def pin_local_to_global_contiguous(seed=13) -> bool:
    """Closed form: requests laid out back to back in whole blocks (block ids
    consecutive from the request's first block) map position x to
    first_row + x."""
    rng = np.random.default_rng(seed)
    B, kv_lens = 8, [20, 5, 33]
    nb = [-(-n // B) for n in kv_lens]
    first = np.concatenate([[0], np.cumsum(nb)])[:-1]
    bt = np.full((3, max(nb)), -1, dtype=np.int32)
    for r in range(3):
        bt[r, :nb[r]] = first[r] + np.arange(nb[r])
    cq = [0, 2, 3, 6]
    idx = np.full((6, 5), -1, dtype=np.int32)
    for r in range(3):
        for t in range(cq[r], cq[r + 1]):
            idx[t] = rng.integers(0, kv_lens[r], size=5)
    out, bad = O.local_to_global(idx, 5, cq, kv_lens, bt, B, int(sum(nb)) * B)
    want = np.empty_like(idx)
    for r in range(3):
        want[cq[r]:cq[r + 1]] = idx[cq[r]:cq[r + 1]] + first[r] * B
    return bad == 0 and bool(np.array_equal(out, want))


def pin_e4m3_decode_closed_forms() -> bool:
    """float8 e4m3 codes whose values follow from the format by hand: 1 =
    0.0111.000, the largest finite 448 = 0.1111.110 (2^8 x 1.75), the smallest
    normal 2^-6 = 0.0001.000, the smallest subnormal 2^-9 = 0.0000.001,
    7 x 2^-9 = 0.0000.111, -1, NaN = 0.1111.111, +0 and -0."""
    codes = [0x38, 0x7E, 0x08, 0x01, 0x07, 0xB8, 0x00, 0x80]
    want = [1.0, 448.0, 2.0 ** -6, 2.0 ** -9, 7 * 2.0 ** -9, -1.0, 0.0, -0.0]
    got = O.e4m3_decode(codes)
    return bool(np.array_equal(got, want) and np.isnan(O.e4m3_decode([0x7F, 0xFF])).all()
                and np.signbit(got[-1]))


def pin_e4m3_encode_library() -> bool:
    """Rounding to e4m3 equals torch's float8_e4m3fn conversion (a library
    routine) on random magnitudes over the whole range and on every midpoint
    between neighbouring values (ties to even), both signs."""
    import torch
    rng = np.random.default_rng(13)
    x = (rng.standard_normal(50000) * np.exp2(rng.integers(-12, 9, 50000))).astype(np.float32)
    x = x[np.abs(x) <= 448.0]
    grid = O.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    mid = ((grid[:-1] + grid[1:]) / 2).astype(np.float32)
    x = np.concatenate([x, mid, -mid])
    lib = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    return bool(np.array_equal(O.e4m3_encode(x), lib))


def pin_kv_fp8_round_trip(seed=14) -> bool:
    """FP8 rows: a block whose values are e4m3 values times a power of two
    (its amax 448 times that power) comes back exactly; random blocks come
    back within half an e4m3 step (2^-4 relative, 2^-10 of the scale for
    subnormal codes) plus bf16 rounding; the scale is amax / 448; an all-zero
    block has scale 1 and codes 0; the RoPE columns pass through."""
    rng = np.random.default_rng(seed)
    N, d_rope = 6, 64
    grid = O.e4m3_decode(rng.integers(0, 0x7F, size=(N, 512)).astype(np.uint8))
    grid[:, ::128] = 448.0
    sgn = np.where(rng.random((N, 512)) < 0.5, -1.0, 1.0)
    exact = (sgn * grid * np.exp2(rng.integers(-20, 10, size=(N, 1)))).astype(np.float32)
    def bits(f):
        return (np.asarray(f, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)
    rope = rng.integers(0, 1 << 16, size=(N, d_rope)).astype(np.uint16)
    rope = np.where(((rope >> 7) & 0xFF) == 0xFF, rope & 0x807F, rope)   # finite bf16 patterns
    kv = np.concatenate([bits(exact), rope], axis=1)
    rows = O.kv_fp8_quantize(kv, d_rope)
    ok = np.array_equal(O.kv_fp8_dequantize(rows, d_rope), kv)
    r = (rng.standard_normal((N, 512)) * np.exp2(rng.integers(-8, 8, size=(N, 1)))).astype(np.float32)
    r[2, 128:256] = 0.0
    kv2 = np.concatenate([bits(r), rope], axis=1)
    x = (kv2[:, :512].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    rows2 = O.kv_fp8_quantize(kv2, d_rope)
    back = (O.kv_fp8_dequantize(rows2, d_rope)[:, :512].astype(np.uint32) << 16).view(np.float32)
    scale = np.ascontiguousarray(rows2[:, 512:528]).view("<f4").reshape(N, 4).astype(np.float64)
    amax = np.abs(x.reshape(N, 4, 128)).max(axis=2)
    ok &= bool(np.allclose(scale, np.where(amax > 0, amax / 448.0, 1.0), rtol=2 ** -23, atol=0))
    s = np.repeat(scale, 128, axis=1)
    tol = np.maximum(np.abs(x) * 2.0 ** -4, s * 2.0 ** -10) * (1 + 2.0 ** -7) + np.abs(x) * 2.0 ** -8
    ok &= bool(np.all(np.abs(back - x) <= tol))
    ok &= bool(np.all(rows2[2, 128:256] == 0) and scale[2, 1] == 1.0)
    ok &= bool(np.array_equal(O.kv_fp8_dequantize(rows2, d_rope)[:, 512:], rope))
    return ok


# ----------------------------------------------------------------------------
# the tolerance checker every parity test relies on
# ----------------------------------------------------------------------------
def _accepts(got_out, got_lse, ref_out, ref_lse):
    return bool(O.compare(got_out, got_lse, ref_out, ref_lse)["ok"])


def pin_compare_statistics() -> bool:
    """Hand-worked statistics: out ref = (3, 4) (norm 5) against (3, 4.01):
    max-abs 0.01, relative L2 0.01 / 5 = 0.002; lse ref (2, -inf, +inf) with
    got (2.004, -inf, +inf): max-abs 0.004, relative L2 0.004 / 2 = 0.002."""
    r = O.compare(np.array([3.0, 4.01]), np.array([2.004, -np.inf, np.inf]),
                  np.array([3.0, 4.0]), np.array([2.0, -np.inf, np.inf]))
    ok = bool(r["ok"]) and abs(r["out_max_abs"] - 0.01) < 1e-12 and abs(r["out_rel_l2"] - 0.002) < 1e-12
    ok &= abs(r["lse_max_abs"] - 0.004) < 1e-12 and abs(r["lse_rel_l2"] - 0.002) < 1e-12
    ok &= bool(r["lse_inf_match"]) and not r["nan"]
    # identical inputs: every statistic zero
    z = O.compare(np.ones((2, 3)), np.zeros(2), np.ones((2, 3)), np.zeros(2))
    ok &= bool(z["ok"]) and z["out_max_abs"] == 0 and z["out_rel_l2"] == 0 and z["lse_max_abs"] == 0
    # empty tensors pass
    ok &= _accepts(np.zeros((0, 4, 8)), np.zeros((0, 4)), np.zeros((0, 4, 8)), np.zeros((0, 4)))
    return ok


def pin_compare_out_bounds() -> bool:
    """Each out bound on its own, just inside and just outside.
    rel-L2: ref = ones(10000) and got = ref (1 + e) give exactly e (the
    difference over the norm of ref, not of got: at e = 0.00502 the ratio to
    the norm of got would be 0.004995 and pass).  max-abs: one entry off by
    0.019 / 0.021 in a 10^4-vector of ones (relative L2 0.0002)."""
    n = 10000
    ref = np.ones(n)
    lse = np.zeros(4)
    ok = _accepts(ref * (1 + 0.0049), lse, ref, lse)
    ok &= not _accepts(ref * (1 + 0.00502), lse, ref, lse)
    one = ref.copy()
    one[123] += 0.019
    ok &= _accepts(one, lse, ref, lse)
    one[123] += 0.002
    ok &= not _accepts(one, lse, ref, lse)
    # all-zero reference: the plain norm of the difference is the measure
    ok &= _accepts(np.full(4, 1e-3), lse, np.zeros(4), lse)
    ok &= not _accepts(np.full(4, 3e-3), lse, np.zeros(4), lse)
    return ok


def pin_compare_lse_bounds() -> bool:
    """The two lse bounds on their own, on the finite entries: ref 0.1 with
    got 0.11 everywhere is within max-abs (0.01) but 10 % off in relative L2;
    ref 100 with one of 1000 entries off by 0.03 is far within relative L2
    (1e-5) but beyond max-abs.  A finite mismatch of 5 beside agreeing
    infinities must fail."""
    out = np.ones(8)
    n = 1000
    ok = not _accepts(out, np.full(n, 0.11), out, np.full(n, 0.1))
    ok &= _accepts(out, np.full(n, 0.1 + 1e-4), out, np.full(n, 0.1))
    big = np.full(n, 100.0)
    g = big.copy()
    g[7] += 0.03
    ok &= not _accepts(out, g, out, big)
    g[7] = 100.0 + 0.015
    ok &= _accepts(out, g, out, big)
    ref = np.array([-np.inf, 1.0, 2.0])
    ok &= not _accepts(out, np.array([-np.inf, 6.0, 2.0]), out, ref)
    return ok


def pin_compare_infinities_and_nan() -> bool:
    """lse infinities must coincide with their signs; a NaN anywhere, on
    either side, fails; tensors of different shapes are an error, not a
    broadcast."""
    out = np.ones(4)
    ref = np.array([-np.inf, 1.0])
    ok = _accepts(out, np.array([-np.inf, 1.0]), out, ref)
    ok &= not _accepts(out, np.array([0.0, 1.0]), out, ref)            # finite where ref is -inf
    ok &= not _accepts(out, np.array([np.inf, 1.0]), out, ref)         # wrong sign
    ok &= not _accepts(out, np.array([-np.inf, -np.inf]), out, ref)    # -inf where ref is finite
    # NaN beside zeros: read as zero it would pass, so only NaN detection fails it
    zo = np.zeros(4)
    bad = zo.copy()
    bad[2] = np.nan
    zl = np.array([-np.inf, 0.0])
    nl = np.array([-np.inf, np.nan])
    ok &= _accepts(zo, zl, zo, zl)
    ok &= not _accepts(bad, zl, zo, zl)
    ok &= not _accepts(zo, nl, zo, zl)
    ok &= not _accepts(zo, zl, bad, zl)
    ok &= not _accepts(zo, zl, zo, nl)
    try:
        O.compare(np.ones((5, 1, 8)), np.zeros((5, 1)), np.ones((5, 3, 8)), np.zeros((5, 3)))
        ok = False
    except ValueError:
        pass
    return ok


ALL_PINS = [pin_bruteforce, pin_single_key, pin_zero_query, pin_equal_keys, pin_two_keys_closed_form,
            pin_order_and_padding_invariance, pin_dense_causal_sdpa, pin_union_worked_example,
            pin_union_bruteforce, pin_union_popcounts, pin_grouped_equals_per_token,
            pin_key_mask_bruteforce, pin_masked_equals_sparse, pin_masked_dense_causal_sdpa,
            pin_local_to_global_paged_round_trip, pin_local_to_global_contiguous,
            pin_e4m3_decode_closed_forms, pin_e4m3_encode_library, pin_kv_fp8_round_trip,
            pin_compare_statistics, pin_compare_out_bounds, pin_compare_lse_bounds,
            pin_compare_infinities_and_nan]


def run_all_pins():
    res = {}
    for p in ALL_PINS:
        try:
            res[p.__name__] = bool(p())
        except Exception:  # a mutated oracle may also crash: that counts as caught
            res[p.__name__] = False
    return res
