"""Masked dense MHA (and its key mask) on the GPU against the fp64 oracle.
Tolerance as for the sparse forms: out/lse max-abs <= 2e-2, rel-L2 <= 5e-3,
lse infinities equal."""
import numpy as np
import pytest

import oracle.dsa_oracle as O
from gpu_util import bf, f32, i32, need_gpu, stratified_tokens, torch
from synth import WORKLOADS, locality_topk, make_masked_inputs, normal_bf16, scaled_down

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


def words_for(kv_lens):
    w = (max(kv_lens) + 31) // 32
    return (w + 3) // 4 * 4


def run_masked(q, k, v, idx, kk, cq, ck, scale, words):
    import dsa_sparse_mla_prefill_gb300 as dsa
    T, H, _ = q.shape
    ix = i32(idx)
    km = dsa.dsa_topk_to_key_mask(ix, kk, words, cu_seqlens_q=cq, cu_seqlens_kv=ck)
    out = torch.full((T, H, v.shape[2]), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((T, H), float("nan"), dtype=torch.float32, device="cuda")
    dsa.dsa_masked_mha_prefill(bf(q), bf(k), bf(v), km, scale, cu_seqlens_q=cq, cu_seqlens_kv=ck, out=out, lse=lse)
    torch.cuda.synchronize()
    st, counts = dsa.dsa_last_device_error()
    assert st == 0, counts
    return km.cpu().numpy().view(np.uint32), f32(out), lse.cpu().numpy().astype(np.float64)


def causal_inputs(seed, q_lens, kv_lens, H, k, d_qk=192, d_v=128):
    rng = np.random.default_rng(seed)
    cq = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    ck = np.concatenate([[0], np.cumsum(kv_lens)]).astype(np.int32)
    rows = []
    for r, (nq, nk) in enumerate(zip(q_lens, kv_lens)):
        pos = np.arange(nk - nq, nk)
        rows.append(locality_topk(rng, pos, k, k, kv_offset=int(ck[r])))
    idx = np.concatenate(rows)
    q = normal_bf16(rng, (int(cq[-1]), H, d_qk))
    kk = normal_bf16(rng, (int(ck[-1]), H, d_qk))
    vv = normal_bf16(rng, (int(ck[-1]), H, d_v))
    return q, kk, vv, idx, cq, ck


@pytest.mark.parametrize("q_lens,kv_lens,H,k", [
    ([150, 200], [150, 200], 4, 64),          # two causal requests, partial query tiles
    ([300], [300], 2, 300),                    # k >= t+1 everywhere: dense causal
    ([97, 130], [400, 130], 3, 96),            # chunked context: queries after 303 cached rows
])
def test_masked_all_tokens(q_lens, kv_lens, H, k):
    q, kk, vv, idx, cq, ck = causal_inputs(len(q_lens) * 7 + H, q_lens, kv_lens, H, k)
    words = words_for(kv_lens)
    km, o, l = run_masked(q, kk, vv, idx, k, cq, ck, 1.0 / np.sqrt(192.0), words)
    ref_km = O.topk_to_key_mask(idx, k, cq, ck, words)
    assert np.array_equal(km, ref_km)
    ro, rl = O.masked_mha_prefill(q, kk, vv, ref_km, cq, ck, 1.0 / np.sqrt(192.0))
    res = O.compare(o, l, ro, rl)
    assert res["ok"], res


def test_masked_empty_rows_and_sparse_equivalence():
    """Tokens with an empty mask get out = 0, lse = -inf.  With every head's
    k/v equal to one shared latent row the masked form equals the per-token
    sparse form of the same indices (spec invariant)."""
    rng = np.random.default_rng(3)
    T, N, H, k = 140, 260, 4, 40
    kv = normal_bf16(rng, (N, 192))
    q = normal_bf16(rng, (T, H, 192))
    idx = np.full((T, k), -1, dtype=np.int32)
    for t in range(T):
        n = int(rng.integers(0, k + 1))
        idx[t, :n] = rng.choice(N, size=n, replace=False)
    idx[5, :] = -1
    kh = np.ascontiguousarray(np.repeat(kv[:, None, :], H, axis=1))
    vh = np.ascontiguousarray(np.repeat(kv[:, None, :128], H, axis=1))
    km, o, l = run_masked(q, kh, vh, idx, k, np.array([0, T], np.int32), np.array([0, N], np.int32), 0.1,
                          words_for([N]))
    ro, rl = O.sparse_prefill(q, kv, idx, k, 0.1, 192, 128)
    res = O.compare(o, l, ro, rl)
    assert res["ok"], res
    assert np.all(o[5] == 0) and np.all(np.isneginf(l[5]))


def test_masked_full_size_sampled():
    w = WORKLOADS["masked_2x8192"]
    x = make_masked_inputs(w)
    words = words_for(w.kv_lens)
    km, o, l = run_masked(x.q, x.k, x.v, x.idx, w.k, x.cu_seqlens_q, x.cu_seqlens_kv, w.scale, words)
    assert np.isfinite(o).all() and np.isfinite(l).all()
    rng = np.random.default_rng(5)
    toks = stratified_tokens(w.T, 24, rng, must=[0, 127, 128, 2047, 2048, 8191, 8192, 8193, 16383])
    n0 = sum(1 for t in toks if t < 8192)
    ref_km = O.topk_to_key_mask(x.idx[toks], w.k, [0, n0, len(toks)], x.cu_seqlens_kv, words)
    assert np.array_equal(km[toks], ref_km)
    ro, rl = O.masked_mha_prefill(x.q, x.k, x.v, km, x.cu_seqlens_q, x.cu_seqlens_kv, w.scale, tokens=toks)
    res = O.compare(o[toks], l[toks], ro, rl)
    assert res["ok"], res
