"""fp64 CPU oracle for DSA sparse-MLA prefill.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports, calls or
links this module: only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline leg use it.  It shares no code with the CUDA
path (no kernels, headers, helpers, tables or constants); the only thing the
two sides have in common is the seeded input generator in ``synth/``.

Every function is the plain definition of what the method computes, written
in numpy float64 with bf16 inputs widened exactly.  Library primitives
(matrix product, ``np.unique``, ``np.searchsorted``) serve as single steps;
there is no blocking, fusion or reordering.

Sources (page title, section):

* [P3] "[Perf][DSA] Grouped sparse prefill with the FlashMLA head-group-mask
  kernel": commit message (per-token gather of 2048 x 1152 B; grouping G = 128
  // num_heads consecutive tokens of a request into 128 pseudo-heads over the
  union of their top-k rows, with a head-group mask restoring each token's own
  top-k, with an exact result); How (sorted union via bitmap -> prefix-sum compaction,
  per-token membership bitmask, request-local positions mapped to physical
  rows of the paged KV cache, q gathered into [groups, 128, 576], padding
  rows dropped); review snippet (union_pad / words sizing, the grouped gate).
* [P2] "[Perf][GLM-5.3-Flash] Dense/masked-MHA sparse prefill for the NoPE
  (256, 0, 256) layout + skip the NoPE K concat": Purpose (masked MHA over
  the same top-k semantics; NoPE K is k_nope itself).
* [P1] "[2/N][Attention] Enable masked MHA for sparse MLA prefills": Purpose
  (masked MHA simulating DSA; dense MHA when every key is selected).

Readings where the pages are silent (each listed in the design notes):

* lse is the natural-log log-sum-exp of the scaled scores;
* a token with no valid key gets out = 0 and lse = -inf;
* -1 may appear anywhere in an index row; only the first k columns count;
* any other index outside [0, N) and any duplicate valid index is invalid
  input here (ValueError);
* causality is carried entirely by the indices (sparse) or the mask (masked);
* pseudo-head p = j*H + h for token j of a group and head h;
* the head-group mask is one uint8 per union slot, bit j = token j of the group;
* the union list is strictly ascending, padded with -1 (mask 0) to union_pad;
* a paged KV cache maps position x of request r to physical row
  block_table[r][x // block_size] * block_size + x % block_size; positions
  outside the request, unmapped blocks (negative ids) and rows outside the
  table map to -1 and are counted (this reading of the conversion the pages
  name without printing it);
* an FP8 KV row (the pages keep bf16 KV and refuse quantized caches; this is
  the plainest layout for the latent row): 512 float8 e4m3 NoPE values with
  one fp32 scale (block amax / 448) per 128 of them, the RoPE columns bf16.
"""
from __future__ import annotations

import math

import numpy as np

# ----------------------------------------------------------------------------
# bf16 decoding (exact widening)
# ----------------------------------------------------------------------------


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns (uint16) exactly to float64."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


# ----------------------------------------------------------------------------
# index sets
# ----------------------------------------------------------------------------


def selected_rows(row: np.ndarray, k: int, N: int) -> np.ndarray:
    """The valid selections of one token: the entries of the first k columns
    that lie in [0, N).  -1 means "no selection" wherever it appears [P3, GLM
    comment: -1 padded top-k buffer wider than k].  Any other out-of-range or
    repeated index is invalid input for the oracle."""
    sel = np.asarray(row[:k], dtype=np.int64)
    bad = sel[(sel < -1) | (sel >= N)]
    if bad.size:
        raise ValueError(f"index out of range: {bad[:4]}")
    v = sel[sel >= 0]
    if np.unique(v).size != v.size:
        raise ValueError("duplicate index in one token's top-k row")
    return v


# ----------------------------------------------------------------------------
# per-token sparse attention: the definition
# ----------------------------------------------------------------------------


def attend(qf: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float):
    """softmax(scale * q K^T) V and the log-sum-exp, for one token, all heads.

    qf: [H, D_QK], K: [n, D_QK], V: [n, D_V] (float64).  Returns out [H, D_V]
    and lse [H] (natural log).  n = 0 gives out = 0, lse = -inf."""
    H = qf.shape[0]
    if K.shape[0] == 0:
        return np.zeros((H, V.shape[1])), np.full(H, -np.inf)
    s = scale * (qf @ K.T)                       # [H, n]
    m = s.max(axis=1, keepdims=True)
    e = np.exp(s - m)
    l = e.sum(axis=1)
    lse = m[:, 0] + np.log(l)
    out = (e @ V) / l[:, None]
    return out, lse


def sparse_prefill(q_bits, kv_bits, idx, k: int, scale: float, d_qk: int, d_v: int,
                   tokens=None):
    """Per-token sparse MLA prefill [P3 commit message: the per-token definition].

    For token t and head h, with S_t the valid rows of idx[t, :k]:
      s_j = scale * sum_{d < D_QK} q[t,h,d] * kv[S_t[j], d]
      lse = log sum_j exp(s_j)
      out = sum_j exp(s_j - lse) * kv[S_t[j], 0:D_V]      (V = first D_V columns)

    q_bits [T, H, D_QK] bf16 bits; kv_bits [N, >= D_QK] bf16 bits; idx [T, ld]
    int32.  ``tokens`` restricts the computation to a subset (returned in
    that order).  Returns out [len(tokens), H, D_V] and lse [len(tokens), H]
    in float64."""
    N = kv_bits.shape[0]
    kvf = bf16_to_f64(kv_bits[:, :d_qk])
    tokens = range(q_bits.shape[0]) if tokens is None else tokens
    tokens = list(tokens)
    H = q_bits.shape[1]
    out = np.zeros((len(tokens), H, d_v))
    lse = np.zeros((len(tokens), H))
    for i, t in enumerate(tokens):
        S = selected_rows(idx[t], k, N)
        qf = bf16_to_f64(q_bits[t, :, :d_qk])
        K = kvf[S, :d_qk]
        V = kvf[S, :d_v]
        out[i], lse[i] = attend(qf, K, V, scale)
    return out, lse


# ----------------------------------------------------------------------------
# grouping: union list and head-group membership mask
# ----------------------------------------------------------------------------


def groups(cu_seqlens_q, G: int):
    """Groups of G consecutive tokens of one request (P3 commit message: the
    group size is 128 divided by the head count, and groups never span two
    requests).  A request's last group may be short.  Returns a list of
    (first token, token count)."""
    cu = [int(x) for x in cu_seqlens_q]
    out = []
    for r in range(len(cu) - 1):
        for s in range(cu[r], cu[r + 1], G):
            out.append((s, min(G, cu[r + 1] - s)))
    return out


def union_pad(G: int, k: int, union_block: int) -> int:
    """Per-group union capacity: G*k rounded up to a multiple of the union
    block [P3, review snippet of the union builder's sizes]."""
    return -(-G * k // union_block) * union_block


def union_build(idx, k: int, G: int, N: int, cu_seqlens_q, upad: int):
    """Sorted union of each group's top-k sets and the per-token membership
    mask (P3 How: the builder emits an ascending union list per group and one
    membership bit per token of the group for every union slot).

    union[g, :U_g] = the distinct valid rows of the group's tokens, ascending;
    union[g, U_g:] = -1.  mask[g, u] has bit j set iff union[g, u] is in the
    top-k set of token j of the group (0 in the padding).
    Returns (union int32 [groups, upad], union_len int32 [groups],
    mask uint8 [groups, upad])."""
    if G < 1 or G > 8:
        raise ValueError("G must be in [1, 8]: one mask bit per token of a group")
    grp = groups(cu_seqlens_q, G)
    union = np.full((len(grp), upad), -1, dtype=np.int32)
    ulen = np.zeros(len(grp), dtype=np.int32)
    mask = np.zeros((len(grp), upad), dtype=np.uint8)
    for g, (t0, n) in enumerate(grp):
        sets = [selected_rows(idx[t0 + j], k, N) for j in range(n)]
        u = np.unique(np.concatenate(sets)) if n else np.empty(0, np.int64)
        if u.size > upad:
            raise ValueError("union longer than union_pad")
        union[g, :u.size] = u
        ulen[g] = u.size
        for j, s in enumerate(sets):
            pos = np.searchsorted(u, s)
            mask[g, pos] |= np.uint8(1 << j)
    return union, ulen, mask


def grouped_prefill(q_bits, kv_bits, union, ulen, mask, G: int, cu_seqlens_q,
                    scale: float, d_qk: int, d_v: int, group_ids=None):
    """Grouped sparse prefill [P3 commit message and How].

    The G tokens of group g act as G*H pseudo-heads p = j*H + h over the
    group's union list; pseudo-head p sees union slot u iff bit j of
    mask[g, u] is set (other slots score -inf).  Written as a dense softmax
    over the union with a -inf mask, independently of ``sparse_prefill``;
    the two must agree, because the pages state that the grouped form gives
    the per-token result exactly.  Pseudo-heads beyond the group's tokens are
    padding and are dropped.  Returns out [T, H, D_V] and lse [T, H] for the tokens of the
    chosen groups (zeros elsewhere)."""
    T, H = q_bits.shape[0], q_bits.shape[1]
    kvf_all = kv_bits
    grp = groups(cu_seqlens_q, G)
    out = np.zeros((T, H, d_v))
    lse = np.zeros((T, H))
    gids = range(len(grp)) if group_ids is None else group_ids
    for g in gids:
        t0, n = grp[g]
        U = int(ulen[g])
        rows = union[g, :U].astype(np.int64)
        Kf = bf16_to_f64(kvf_all[rows, :d_qk])                     # [U, D_QK]
        Vf = Kf[:, :d_v]
        Qp = bf16_to_f64(q_bits[t0:t0 + n, :, :d_qk]).reshape(n * H, d_qk)   # p = j*H + h
        member = ((mask[g, :U][None, :].astype(np.int64) >> (np.arange(n * H) // H)[:, None]) & 1) == 1
        s = scale * (Qp @ Kf.T)                                     # [n*H, U]
        s = np.where(member, s, -np.inf)
        m = s.max(axis=1, keepdims=True) if U else np.full((n * H, 1), -np.inf)
        has = np.isfinite(m[:, 0])
        m_safe = np.where(has[:, None], m, 0.0)
        e = np.where(member, np.exp(s - m_safe), 0.0)
        l = e.sum(axis=1)
        o = np.where(has[:, None], (e @ Vf) / np.where(has, l, 1.0)[:, None], 0.0)
        ls = np.where(has, m[:, 0] + np.log(np.where(has, l, 1.0)), -np.inf)
        out[t0:t0 + n] = o.reshape(n, H, d_v)
        lse[t0:t0 + n] = ls.reshape(n, H)
    return out, lse


# ----------------------------------------------------------------------------
# masked dense MHA
# ----------------------------------------------------------------------------


def topk_to_key_mask(idx, k: int, cu_seqlens_q, cu_seqlens_kv, words: int):
    """Per-token key mask [P1 commit log: scatter top-k into the mask, zeroed
    in the kernel].  Token t of request r: bit n of row t (word n >> 5, bit
    n & 31, LSB first) is set iff global row cu_seqlens_kv[r] + n is among
    its valid top-k.  Returns uint32 [T, words]."""
    cq = [int(x) for x in cu_seqlens_q]
    ck = [int(x) for x in cu_seqlens_kv]
    T = cq[-1]
    N = ck[-1]
    km = np.zeros((T, words), dtype=np.uint32)
    for r in range(len(cq) - 1):
        for t in range(cq[r], cq[r + 1]):
            S = selected_rows(idx[t], k, N)
            n = S - ck[r]
            if np.any((n < 0) | (n >= ck[r + 1] - ck[r])):
                raise ValueError("index outside its request's KV range")
            if np.any(n >= 32 * words):
                raise ValueError("key mask too narrow")
            for x in n:
                km[t, x >> 5] |= np.uint32(1 << (int(x) & 31))
    return km


def local_to_global(idx_local, k: int, cu_seqlens_q, kv_lens, block_table, block_size: int, N: int):
    """Request-local positions -> physical rows [P3 How: positions mapped to
    physical rows of the paged KV cache].  Token t of request r, entry j < k
    with position x: row = block_table[r][x // block_size] * block_size +
    x % block_size when 0 <= x < kv_lens[r], the block id is >= 0 and the row
    lies in [0, N); -1 stays -1; columns j >= k and every other entry give
    -1.  Returns (int32 [T, ld], number of entries that were neither -1 nor
    mapped among the first k columns)."""
    idx_local = np.asarray(idx_local, dtype=np.int64)
    bt = np.asarray(block_table, dtype=np.int64)
    T, ld = idx_local.shape
    cq = [0, T] if cu_seqlens_q is None else [int(x) for x in cu_seqlens_q]
    out = np.full((T, ld), -1, dtype=np.int32)
    bad = 0
    for r in range(len(cq) - 1):
        kv_len = int(kv_lens[r])
        for t in range(cq[r], cq[r + 1]):
            for j in range(min(k, ld)):
                x = int(idx_local[t, j])
                if x == -1:
                    continue
                if x < 0 or x >= kv_len:
                    bad += 1
                    continue
                blk = int(bt[r, x // block_size])
                row = blk * block_size + x % block_size
                if blk < 0 or row >= N:
                    bad += 1
                    continue
                out[t, j] = row
    return out, bad


def masked_mha_prefill(q_bits, k_bits, v_bits, key_mask, cu_seqlens_q, cu_seqlens_kv,
                       scale: float, tokens=None):
    """Masked dense MHA simulating DSA [P1 Purpose; P2 Purpose].

    Token t of request r, head h: softmax over the keys n whose mask bit is
    set of scale * q[t,h] . k[c_r + n, h], weighting v[c_r + n, h]
    (c_r = cu_seqlens_kv[r]).  Per-head q/k/v, no key sharing across heads.
    Returns out [len(tokens), H, D_V] and lse [len(tokens), H]."""
    cq = [int(x) for x in cu_seqlens_q]
    ck = [int(x) for x in cu_seqlens_kv]
    T, H, _ = q_bits.shape
    d_v = v_bits.shape[2]
    tokens = list(range(T)) if tokens is None else list(tokens)
    req_of = np.searchsorted(np.asarray(cq[1:]), np.asarray(tokens), side="right")
    out = np.zeros((len(tokens), H, d_v))
    lse = np.zeros((len(tokens), H))
    for i, t in enumerate(tokens):
        r = int(req_of[i])
        nk = ck[r + 1] - ck[r]
        bits = key_mask[t]
        n = np.array([x for x in range(nk) if (int(bits[x >> 5]) >> (x & 31)) & 1], dtype=np.int64)
        rows = ck[r] + n
        for h in range(H):
            qf = bf16_to_f64(q_bits[t, h][None, :])
            K = bf16_to_f64(k_bits[rows, h])
            V = bf16_to_f64(v_bits[rows, h])
            o, l = attend(qf, K, V, scale)
            out[i, h] = o[0]
            lse[i, h] = l[0]
    return out, lse


# ----------------------------------------------------------------------------
# FP8 latent rows (a storage format for the KV cache; the pages keep bf16 KV,
# so this is the plainest reading of the "FP8 KV cache" step: the 512 NoPE
# columns as float8 e4m3 with one fp32 scale per 128 of them, the RoPE
# columns kept bf16; row = 512 codes | 4 scales | 2 * d_rope bytes)
# ----------------------------------------------------------------------------
E4M3_MAX = 448.0


def e4m3_decode(codes) -> np.ndarray:
    """float8 e4m3 (1 sign, 4 exponent bits with bias 7, 3 mantissa bits, no
    infinities, S.1111.111 = NaN) to float64, from its definition."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    val = np.where(e == 0, (m / 8.0) * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    val = sign * val
    return np.where((e == 15) & (m == 7), np.nan, val)


def e4m3_encode(x) -> np.ndarray:
    """float32 values to e4m3 codes: the nearest finite e4m3 value, ties to the
    even code, magnitudes beyond 448 saturated to 448; the sign is kept (also
    for values that round to zero).  Written as a search over the 127
    non-negative finite codes."""
    x = np.asarray(x, dtype=np.float32).astype(np.float64)
    grid = e4m3_decode(np.arange(0x7F, dtype=np.uint8))       # codes 0x00..0x7E, ascending
    a = np.minimum(np.abs(x), E4M3_MAX)
    hi = np.clip(np.searchsorted(grid, a, side="left"), 0, 0x7E)
    lo = np.maximum(hi - 1, 0)
    dlo = a - grid[lo]
    dhi = grid[hi] - a
    pick = np.where(dlo < dhi, lo, np.where(dhi < dlo, hi, np.where(lo % 2 == 0, lo, hi)))
    pick = np.where(grid[hi] == a, hi, pick)
    return (pick | np.where(np.signbit(x), 0x80, 0)).astype(np.uint8)


def _f32_to_bf16_bits(x) -> np.ndarray:
    """float32 to bf16 bits, round to nearest even (finite inputs)."""
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return r.astype(np.uint16)


def kv_fp8_row_bytes(d_rope: int) -> int:
    return 512 + 16 + 2 * d_rope


def kv_fp8_quantize(kv_bits, d_rope: int) -> np.ndarray:
    """bf16 latent rows [N, >= 512 + d_rope] to FP8 rows [N, row_bytes] uint8.
    Block b (columns 128b .. 128b+127): scale = amax / 448 in float32 (1 when
    the block is all zero), codes = e4m3(x / scale) with the division in
    float32; the RoPE columns are copied."""
    kv_bits = np.asarray(kv_bits, dtype=np.uint16)
    N = kv_bits.shape[0]
    x = (kv_bits[:, :512].astype(np.uint32) << 16).view(np.float32).reshape(N, 4, 128)
    amax = np.abs(x).max(axis=2)
    scale = np.where(amax > 0, (amax / np.float32(E4M3_MAX)).astype(np.float32), np.float32(1.0))
    codes = e4m3_encode((x / scale[:, :, None]).astype(np.float32)).reshape(N, 512)
    out = np.zeros((N, kv_fp8_row_bytes(d_rope)), dtype=np.uint8)
    out[:, :512] = codes
    out[:, 512:528] = scale.astype("<f4").view(np.uint8).reshape(N, 16)
    if d_rope:
        out[:, 528:] = np.ascontiguousarray(kv_bits[:, 512:512 + d_rope]).astype("<u2").view(np.uint8)
    return out


def kv_fp8_dequantize(rows, d_rope: int) -> np.ndarray:
    """FP8 rows to bf16 latent rows [N, 512 + d_rope]: e4m3 value times its
    block's scale in float32, rounded to bf16; RoPE columns copied."""
    rows = np.asarray(rows, dtype=np.uint8)
    N = rows.shape[0]
    vals = e4m3_decode(rows[:, :512]).astype(np.float32).reshape(N, 4, 128)
    scale = np.ascontiguousarray(rows[:, 512:528]).view("<f4").reshape(N, 4)
    prod = (vals * scale[:, :, None]).astype(np.float32).reshape(N, 512)
    out = np.zeros((N, 512 + d_rope), dtype=np.uint16)
    out[:, :512] = _f32_to_bf16_bits(prod)
    if d_rope:
        out[:, 512:] = np.ascontiguousarray(rows[:, 528:528 + 2 * d_rope]).view("<u2")
    return out


# ----------------------------------------------------------------------------
# comparison used by the parity tests
# ----------------------------------------------------------------------------


def compare(got_out, got_lse, ref_out, ref_lse, max_abs=2e-2, rel_l2=5e-3):
    """Tolerance check of a result against the oracle's: max-abs 2e-2 and
    relative-L2 5e-3, the bound this library states for bf16 inputs with fp32
    accumulation (the pages saw a relative error of 2e-3, "[Perf][DSA] Grouped
    sparse prefill with the FlashMLA head-group-mask kernel", commit message).

    * out: max |got - ref| <= max_abs and ||got - ref||_2 / ||ref||_2 <= rel_l2
      over the whole tensor (when ||ref|| = 0 the plain norm of the
      difference is compared instead);
    * lse: the same two bounds over the entries finite on both sides, and the
      infinite entries (with their signs) must be the same on both sides;
    * a NaN on either side fails; so do shapes that differ (no broadcasting).

    Returns a dict of the statistics and ``ok``."""
    go = np.asarray(got_out, dtype=np.float64)
    ro = np.asarray(ref_out, dtype=np.float64)
    gl = np.asarray(got_lse, dtype=np.float64)
    rl = np.asarray(ref_lse, dtype=np.float64)
    if go.shape != ro.shape or gl.shape != rl.shape:
        raise ValueError(f"compare: shapes differ: out {go.shape} vs {ro.shape}, lse {gl.shape} vs {rl.shape}")
    nan = bool(np.isnan(go).any() or np.isnan(gl).any() or np.isnan(ro).any() or np.isnan(rl).any())
    d = np.abs(go - ro)
    d = np.where(np.isnan(d), np.inf, d)
    out_max = float(d.max()) if d.size else 0.0
    den = float(np.sqrt((ro ** 2).sum()))
    out_rel = float(np.sqrt((d ** 2).sum()) / den) if den > 0 else float(np.sqrt((d ** 2).sum()))
    inf_same = bool(np.array_equal(np.isinf(gl), np.isinf(rl)) and
                    np.array_equal(np.sign(gl[np.isinf(gl)]), np.sign(rl[np.isinf(rl)])))
    fin = np.isfinite(rl) & np.isfinite(gl)
    dl = np.abs(gl[fin] - rl[fin])
    lse_max = float(dl.max()) if dl.size else 0.0
    lden = float(np.sqrt((rl[fin] ** 2).sum()))
    lse_rel = float(np.sqrt((dl ** 2).sum()) / lden) if lden > 0 else float(np.sqrt((dl ** 2).sum()))
    ok = (not nan) and inf_same and out_max <= max_abs and out_rel <= rel_l2 and \
        lse_max <= max_abs and lse_rel <= rel_l2
    return dict(ok=ok, out_max_abs=out_max, out_rel_l2=out_rel, lse_max_abs=lse_max,
                lse_rel_l2=lse_rel, lse_inf_match=inf_same, nan=nan)
