"""Seeded synthetic workloads for DSA sparse-MLA prefill.

This module is the only code shared by the CUDA path's tests/bench and the
CPU oracle.  It draws inputs and nothing else: it holds none of the attention,
union or mask arithmetic.  Everything is driven by ``numpy.random.default_rng``
so the oracle and the GPU see byte-identical inputs.

Shapes and structure follow the workloads the pages measure:

* per-token sparse prefill over a 576-wide latent KV row (512 NoPE + 64 RoPE),
  top-2048 indices ("[Perf][DSA] Grouped sparse prefill with the FlashMLA
  head-group-mask kernel", commit message and Why: 2048 x 1152 B per token);
* locality of the top-k sets: the union of 8 adjacent tokens' top-2048 is
  about 2.4k keys on real prompts (same page, Why).  Real prompts are not
  available, so a block-shared generator reproduces that union size;
* the NoPE layout (512 + 0) with a 2176-column index buffer padded with -1
  (same page, GLM comment);
* masked dense MHA with per-head q/k/v of 192/128 dims and 128 heads
  ("[2/N][Attention] Enable masked MHA for sparse MLA prefills", Purpose),
  and of 256/256 dims with 64 heads, with or without 64 shared RoPE key
  columns ("[Perf][GLM-5.3-Flash] ...", commit messages: the GLM-5 and
  GLM-5.3-Flash NoPE layouts).

Values are N(0, 1) rounded to bfloat16 (round-to-nearest-even), returned as
raw uint16 bit patterns.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np


# ----------------------------------------------------------------------------
# bf16 encoding of random draws (input preparation only)
# ----------------------------------------------------------------------------
def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest-even) and return the bits."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounded = (b + np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return rounded.astype(np.uint16)


def normal_bf16(rng: np.random.Generator, shape, chunk: int = 1 << 24) -> np.ndarray:
    """N(0,1) draws rounded to bf16, as uint16 bits (chunked to bound memory)."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        out[s:e] = f32_to_bf16_bits(rng.standard_normal(e - s, dtype=np.float32))
    return out.reshape(shape)


# ----------------------------------------------------------------------------
# top-k index generators
# ----------------------------------------------------------------------------
def uniform_topk(rng: np.random.Generator, positions: np.ndarray, k: int, ld: int,
                 kv_offset: int = 0) -> np.ndarray:
    """Token at request position p takes all of [0, p] when p+1 <= k, else k
    distinct uniform draws from [0, p].  Rows are shuffled, then -1 padded to
    ``ld`` columns.  ``kv_offset`` turns request positions into global rows."""
    T = len(positions)
    out = np.full((T, ld), -1, dtype=np.int32)
    for i, p in enumerate(positions):
        p = int(p)
        if p + 1 <= k:
            sel = np.arange(p + 1, dtype=np.int64)
        else:
            sel = rng.choice(p + 1, size=k, replace=False)
        sel = rng.permutation(sel)
        out[i, :len(sel)] = sel + kv_offset
    return out


def _choice_excluding(rng, hi: int, excluded: np.ndarray, size: int) -> np.ndarray:
    """``size`` distinct uniform draws from [0, hi) minus ``excluded``."""
    avail = np.ones(hi, dtype=bool)
    avail[excluded] = False
    cand = np.flatnonzero(avail)
    size = min(size, len(cand))
    return rng.choice(cand, size=size, replace=False)


def locality_topk(rng: np.random.Generator, positions: np.ndarray, k: int, ld: int,
                  kv_offset: int = 0, block: int = 8, recent: int = None,
                  pool: int = None, swap: int = None, wide: bool = False) -> np.ndarray:
    """Block-local top-k sets with the overlap the pages measure.

    Tokens are blocked by ``block`` on request position (t0 = block*floor(p/block)).
    Each block draws a base set of k positions from [0, t0]: the ``recent``
    newest positions plus uniform distinct draws from the rest.  Each token
    replaces ``swap`` (15%) of the base with picks from a block-shared pool of
    ``pool`` fresh positions, so 8 tokens' union is about k + pool = 2400.
    A token with p+1 <= k takes every position of [0, p] (dense).
    ``wide=True`` draws each token's replacements independently from [0, p]
    instead (a wider-union stress variant).
    Rows are shuffled, then -1 padded to ``ld`` columns.  The defaults scale
    with k: recent = k/2, swap = 15% of k, pool = 11k/64 (1024 / 307 / 352 at
    k = 2048).
    """
    recent = k // 2 if recent is None else recent
    swap = int(0.15 * k) if swap is None else swap
    pool = (11 * k) // 64 if pool is None else pool
    T = len(positions)
    out = np.full((T, ld), -1, dtype=np.int32)
    positions = np.asarray(positions, dtype=np.int64)
    i = 0
    while i < T:
        t0 = block * (int(positions[i]) // block)
        j = i
        while j < T and block * (int(positions[j]) // block) == t0:
            j += 1
        base = pool_pos = None
        if t0 + 1 > k:
            lo = max(0, t0 - recent + 1)
            rec = np.arange(lo, t0 + 1, dtype=np.int64)
            rest = rng.choice(lo, size=k - len(rec), replace=False) if k > len(rec) else np.empty(0, np.int64)
            base = np.concatenate([rec, rest.astype(np.int64)])
            if not wide:
                pool_pos = _choice_excluding(rng, t0 + 1, base, pool)
        for r in range(i, j):
            p = int(positions[r])
            if p + 1 <= k:
                sel = np.arange(p + 1, dtype=np.int64)
            else:
                if wide:
                    nswap = swap
                    drop = rng.choice(len(base), size=nswap, replace=False)
                    keep = np.delete(base, drop)
                    add = _choice_excluding(rng, p + 1, keep, nswap)
                else:
                    nswap = min(swap, len(pool_pos))
                    drop = rng.choice(len(base), size=nswap, replace=False)
                    keep = np.delete(base, drop)
                    add = rng.choice(pool_pos, size=nswap, replace=False)
                sel = np.concatenate([keep, add.astype(np.int64)])
            sel = rng.permutation(sel)
            out[r, :len(sel)] = sel + kv_offset
        i = j
    return out


# ----------------------------------------------------------------------------
# workload configurations
# ----------------------------------------------------------------------------
@dataclass(frozen=True)
class Workload:
    """One synthetic workload.  Sizes only; drawing happens in ``make_*``."""
    name: str
    mode: str                      # "sparse" (latent MLA) or "masked" (per-head MHA)
    q_lens: tuple                  # query tokens per request
    kv_lens: tuple                 # KV rows per request
    H: int
    d_qk: int
    d_v: int
    k: int
    ld: int
    scale: float
    index_gen: str                 # "uniform" | "locality" | "locality_wide"
    G: int = 0                     # grouped-mode tokens per group (0 = per-token only)
    seed: int = 0
    notes: str = ""
    d_rope: int = 0                # masked: key columns shared by all heads (the RoPE part)
    split_kv: bool = False         # masked: k and v drawn as one [N, H, d_qk - d_rope + d_v] projection

    @property
    def T(self) -> int:
        return int(sum(self.q_lens))

    @property
    def N(self) -> int:
        return int(sum(self.kv_lens))

    def cu_seqlens_q(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.q_lens)]).astype(np.int32)

    def cu_seqlens_kv(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.kv_lens)]).astype(np.int32)

    def positions(self) -> list:
        """Request-local query positions (queries are the last q_len rows of each request)."""
        return [np.arange(kv - q, kv, dtype=np.int64) for q, kv in zip(self.q_lens, self.kv_lens)]


WORKLOADS = {
    # 512 causal tokens over a 512-row latent cache, uniform top-128.
    "tiny_uniform_512": Workload(
        name="tiny_uniform_512", mode="sparse", q_lens=(512,), kv_lens=(512,), H=16,
        d_qk=576, d_v=512, k=128, ld=128, scale=1.0 / math.sqrt(192.0),
        index_gen="uniform", G=8, seed=0,
        notes="1 request, uniform top-128 without replacement from [0,t]"),
    # DeepSeek-V3.2 shard (128 heads / 4): one 16k-token chunk, top-2048.
    "v32_h32_16k": Workload(
        name="v32_h32_16k", mode="sparse", q_lens=(16384,), kv_lens=(16384,), H=32,
        d_qk=576, d_v=512, k=2048, ld=2048, scale=1.0 / math.sqrt(192.0),
        index_gen="locality", G=4, seed=1,
        notes="1 request, 16384 causal tokens, locality top-2048"),
    # The same shard at the tail of a 131072-row context: 16384 queries at
    # positions 114688..131071, so the latent table (151 MB) exceeds the L2.
    "v32_h32_16k_of_128k": Workload(
        name="v32_h32_16k_of_128k", mode="sparse", q_lens=(16384,), kv_lens=(131072,), H=32,
        d_qk=576, d_v=512, k=2048, ld=2048, scale=1.0 / math.sqrt(192.0),
        index_gen="locality", G=4, seed=7,
        notes="16384 queries after 114688 cached rows, locality top-2048; table larger than the L2"),
    # 21504 queries appended after 11264 cached rows (32768-row prompt), H=16, G=8.
    "grouped_21k_of_32k": Workload(
        name="grouped_21k_of_32k", mode="sparse", q_lens=(21504,), kv_lens=(32768,), H=16,
        d_qk=576, d_v=512, k=2048, ld=2048, scale=1.0 / math.sqrt(192.0),
        index_gen="locality", G=8, seed=2,
        notes="queries at positions 11264..32767, every token has 2048 valid keys"),
    # GLM NoPE layout: 2 x 8192 causal, D_QK = 512, 2176-column index buffer.
    "nope_2x8192": Workload(
        name="nope_2x8192", mode="sparse", q_lens=(8192, 8192), kv_lens=(8192, 8192), H=16,
        d_qk=512, d_v=512, k=2048, ld=2176, scale=1.0 / 16.0,
        index_gen="locality", G=8, seed=3,
        notes="2 requests, top-2048 in a 2176-column buffer padded with -1"),
    # Masked dense MHA simulating DSA: 128 heads, qk 192 / v 128.
    "masked_2x8192": Workload(
        name="masked_2x8192", mode="masked", q_lens=(8192, 8192), kv_lens=(8192, 8192), H=128,
        d_qk=192, d_v=128, k=2048, ld=2048, scale=1.0 / math.sqrt(192.0),
        index_gen="locality", G=0, seed=4,
        notes="per-token key mask = locality top-2048 (dense when t < 2048)"),
    # GLM-5.3-Flash NoPE layout (64 heads, qk 256 + rope 0, v 256): k and v
    # are the two halves of one per-head projection output.
    "masked_nope_2x8192": Workload(
        name="masked_nope_2x8192", mode="masked", q_lens=(8192, 8192), kv_lens=(8192, 8192), H=64,
        d_qk=256, d_v=256, k=2048, ld=2048, scale=1.0 / 16.0,
        index_gen="locality", G=0, seed=5, d_rope=0, split_kv=True,
        notes="per-token key mask = locality top-2048; k = kv[..., :256], v = kv[..., 256:]"),
    # GLM-5 layout (64 heads, qk 192 + rope 64, v 256): the RoPE key columns
    # are one [N, 64] block shared by all heads.
    "masked_glm5_2x8192": Workload(
        name="masked_glm5_2x8192", mode="masked", q_lens=(8192, 8192), kv_lens=(8192, 8192), H=64,
        d_qk=256, d_v=256, k=2048, ld=2048, scale=1.0 / 16.0,
        index_gen="locality", G=0, seed=6, d_rope=64, split_kv=True,
        notes="per-token key mask = locality top-2048; k = [kv[..., :192], k_pe], v = kv[..., 192:]"),
}


def scaled_down(w: Workload, q_lens, kv_lens, k=None, ld=None, H=None, name=None, seed=None,
                index_gen=None, G=None) -> Workload:
    """A smaller workload with the same structure (used for oracle-sized tests)."""
    k = w.k if k is None else k
    return Workload(
        name=name or (w.name + "_small"), mode=w.mode, q_lens=tuple(q_lens), kv_lens=tuple(kv_lens),
        H=w.H if H is None else H, d_qk=w.d_qk, d_v=w.d_v, k=k,
        ld=(k if ld is None else ld), scale=w.scale,
        index_gen=w.index_gen if index_gen is None else index_gen,
        G=w.G if G is None else G, seed=w.seed if seed is None else seed, notes="scaled",
        d_rope=w.d_rope, split_kv=w.split_kv)


def make_indices(w: Workload, rng: np.random.Generator, locality_block: int = 8) -> np.ndarray:
    """Global-row top-k indices ``[T, ld]`` int32, -1 padded."""
    rows = []
    kv_off = w.cu_seqlens_kv()
    for r, pos in enumerate(w.positions()):
        if w.index_gen == "uniform":
            rows.append(uniform_topk(rng, pos, w.k, w.ld, int(kv_off[r])))
        elif w.index_gen in ("locality", "locality_wide"):
            rows.append(locality_topk(rng, pos, w.k, w.ld, int(kv_off[r]), block=locality_block,
                                      wide=(w.index_gen == "locality_wide")))
        else:
            raise ValueError(w.index_gen)
    return np.concatenate(rows, axis=0) if rows else np.zeros((0, w.ld), np.int32)


@dataclass
class SparseInputs:
    w: Workload
    q: np.ndarray          # [T, H, d_qk] bf16 bits
    kv: np.ndarray         # [N, d_qk] bf16 bits (V = first d_v columns)
    idx: np.ndarray        # [T, ld] int32 global rows, -1 padded
    cu_seqlens_q: np.ndarray
    cu_seqlens_kv: np.ndarray


@dataclass
class MaskedInputs:
    w: Workload
    q: np.ndarray          # [T, H, d_qk] bf16 bits
    k: np.ndarray          # [N, H, d_qk] bf16 bits (every head's whole key row)
    v: np.ndarray          # [N, H, d_v] bf16 bits
    idx: np.ndarray        # [T, ld] int32 global rows (source of the key mask)
    cu_seqlens_q: np.ndarray
    cu_seqlens_kv: np.ndarray
    kvp: np.ndarray = None   # split_kv: [N, H, d_qk - d_rope + d_v], k = kvp[..., :d_qk - d_rope], v = the rest
    k_pe: np.ndarray = None  # d_rope > 0: [N, d_rope], the last d_rope columns of every head's key row


def make_sparse_inputs(w: Workload, with_values: bool = True) -> SparseInputs:
    assert w.mode == "sparse"
    rng = np.random.default_rng(w.seed)
    idx = make_indices(w, rng)
    vrng = np.random.default_rng([w.seed, 1])
    if with_values:
        kv = normal_bf16(vrng, (w.N, w.d_qk))
        q = normal_bf16(vrng, (w.T, w.H, w.d_qk))
    else:
        kv = q = None
    return SparseInputs(w, q, kv, idx, w.cu_seqlens_q(), w.cu_seqlens_kv())


def make_masked_inputs(w: Workload, with_values: bool = True) -> MaskedInputs:
    assert w.mode == "masked"
    rng = np.random.default_rng(w.seed)
    idx = make_indices(w, rng)
    vrng = np.random.default_rng([w.seed, 1])
    kvp = k_pe = None
    if with_values and w.split_kv:
        dn = w.d_qk - w.d_rope
        q = normal_bf16(vrng, (w.T, w.H, w.d_qk))
        kvp = normal_bf16(vrng, (w.N, w.H, dn + w.d_v))
        k = np.empty((w.N, w.H, w.d_qk), dtype=np.uint16)
        k[..., :dn] = kvp[..., :dn]
        if w.d_rope:
            k_pe = normal_bf16(vrng, (w.N, w.d_rope))
            k[..., dn:] = k_pe[:, None, :]
        v = np.ascontiguousarray(kvp[..., dn:])
    elif with_values:
        q = normal_bf16(vrng, (w.T, w.H, w.d_qk))
        k = normal_bf16(vrng, (w.N, w.H, w.d_qk))
        v = normal_bf16(vrng, (w.N, w.H, w.d_v))
    else:
        q = k = v = None
    return MaskedInputs(w, q, k, v, idx, w.cu_seqlens_q(), w.cu_seqlens_kv(), kvp, k_pe)
