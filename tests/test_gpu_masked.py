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
    sparse form of the same indices (the masked form must reproduce the sparse gather semantics)."""
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


# ----------------------------------------------------------------------------
# strided operands and the shared RoPE key columns (the GLM-5 and GLM-5.3-Flash
# NoPE geometries, d_qk = d_v = 256, and DeepSeek-V3.2's 192/128)
# ----------------------------------------------------------------------------
def split_inputs(seed, q_lens, kv_lens, H, k, d_qk, d_rope, d_v, q_pad=0):
    """idx, q, one per-head projection kvp [Nk, H, d_qk - d_rope + d_v] (k = its first
    columns, v the rest), the shared RoPE block k_pe [Nk, d_rope], and the whole key rows
    k [Nk, H, d_qk] and v for the oracle.  q is returned inside a wider [T, H, d_qk + q_pad]
    buffer when q_pad > 0, so the kernel reads it through a head stride."""
    rng = np.random.default_rng(seed)
    cq = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    ck = np.concatenate([[0], np.cumsum(kv_lens)]).astype(np.int32)
    rows = []
    for r, (nq, nk) in enumerate(zip(q_lens, kv_lens)):
        rows.append(locality_topk(rng, np.arange(nk - nq, nk), k, k, kv_offset=int(ck[r])))
    idx = np.concatenate(rows)
    T, N, dn = int(cq[-1]), int(ck[-1]), d_qk - d_rope
    qbuf = normal_bf16(rng, (T, H, d_qk + q_pad))
    kvp = normal_bf16(rng, (N, H, dn + d_v))
    k_pe = normal_bf16(rng, (N, d_rope)) if d_rope else None
    kfull = np.empty((N, H, d_qk), dtype=np.uint16)
    kfull[..., :dn] = kvp[..., :dn]
    if d_rope:
        kfull[..., dn:] = k_pe[:, None, :]
    return dict(idx=idx, cq=cq, ck=ck, qbuf=qbuf, q=np.ascontiguousarray(qbuf[..., :d_qk]), kvp=kvp, k_pe=k_pe,
                k=kfull, v=np.ascontiguousarray(kvp[..., dn:]), dn=dn)


def run_strided(x, kk, scale, words):
    """The strided call on device views: k = kvp[..., :dn], v = kvp[..., dn:], q a view of
    its (possibly wider) buffer, k_pe shared.  Returns key mask bits, out, lse."""
    import dsa_sparse_mla_prefill_gb300 as dsa
    d_qk = x["q"].shape[2]
    km = dsa.dsa_topk_to_key_mask(i32(x["idx"]), kk, words, cu_seqlens_q=x["cq"], cu_seqlens_kv=x["ck"])
    kvp = bf(x["kvp"])
    k, v = kvp[..., :x["dn"]], kvp[..., x["dn"]:]
    assert not k.is_contiguous() and not v.is_contiguous()
    q = bf(x["qbuf"])[..., :d_qk]
    k_pe = bf(x["k_pe"]) if x["k_pe"] is not None else None
    T, H = q.shape[:2]
    out = torch.full((T, H, v.shape[2]), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((T, H), float("nan"), dtype=torch.float32, device="cuda")
    dsa.dsa_masked_mha_prefill_strided(q, k, v, km, scale, k_pe=k_pe, cu_seqlens_q=x["cq"],
                                       cu_seqlens_kv=x["ck"], out=out, lse=lse)
    torch.cuda.synchronize()
    st, counts = dsa.dsa_last_device_error()
    assert st == 0, counts
    return km, out, lse


@pytest.mark.parametrize("d_qk,d_rope,d_v", [(256, 0, 256), (256, 64, 256), (192, 64, 128)])
@pytest.mark.parametrize("q_lens,kv_lens,H,k,q_pad", [
    ([150, 200], [150, 200], 3, 64, 0),        # two causal requests, partial query tiles
    ([97, 130], [400, 130], 2, 96, 8),         # chunked context, q read through a head stride
    ([300], [300], 2, 300, 0),                 # dense causal
])
def test_masked_strided_geometries(d_qk, d_rope, d_v, q_lens, kv_lens, H, k, q_pad):
    x = split_inputs(d_qk + d_rope + len(q_lens), q_lens, kv_lens, H, k, d_qk, d_rope, d_v, q_pad)
    words = words_for(kv_lens)
    scale = 1.0 / np.sqrt(d_qk)
    km, o, l = run_strided(x, k, scale, words)
    ref_km = O.topk_to_key_mask(x["idx"], k, x["cq"], x["ck"], words)
    assert np.array_equal(km.cpu().numpy().view(np.uint32), ref_km)
    ro, rl = O.masked_mha_prefill(x["q"], x["k"], x["v"], ref_km, x["cq"], x["ck"], scale)
    res = O.compare(f32(o), l.cpu().numpy().astype(np.float64), ro, rl)
    assert res["ok"], res


@pytest.mark.parametrize("d_qk,d_rope,d_v", [(256, 0, 256), (256, 64, 256), (192, 64, 128)])
def test_masked_strided_equals_contiguous(d_qk, d_rope, d_v):
    """Reading k and v through strides (and the RoPE columns from their own block) gives
    bit for bit what the contiguous call gives on the concatenated copies."""
    import dsa_sparse_mla_prefill_gb300 as dsa
    x = split_inputs(11, [260, 140], [300, 140], 3, 80, d_qk, d_rope, d_v)
    words = words_for([300, 140])
    km, o1, l1 = run_strided(x, 80, 0.07, words)
    o2, l2 = dsa.dsa_masked_mha_prefill(bf(x["q"]), bf(x["k"]), bf(x["v"]), km, 0.07, cu_seqlens_q=x["cq"],
                                        cu_seqlens_kv=x["ck"])
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("name", ["masked_nope_2x8192", "masked_glm5_2x8192"])
def test_masked_256_full_size_sampled(name):
    import dsa_sparse_mla_prefill_gb300 as dsa
    w = WORKLOADS[name]
    x = make_masked_inputs(w)
    words = words_for(w.kv_lens)
    km = dsa.dsa_topk_to_key_mask(i32(x.idx), w.k, words, cu_seqlens_q=x.cu_seqlens_q,
                                  cu_seqlens_kv=x.cu_seqlens_kv)
    dn = w.d_qk - w.d_rope
    kvp = bf(x.kvp)
    k_pe = bf(x.k_pe) if x.k_pe is not None else None
    o, l = dsa.dsa_masked_mha_prefill_strided(bf(x.q), kvp[..., :dn], kvp[..., dn:], km, w.scale, k_pe=k_pe,
                                              cu_seqlens_q=x.cu_seqlens_q, cu_seqlens_kv=x.cu_seqlens_kv)
    torch.cuda.synchronize()
    st, counts = dsa.dsa_last_device_error()
    assert st == 0, counts
    of, lf = f32(o), l.cpu().numpy().astype(np.float64)
    assert np.isfinite(of).all() and np.isfinite(lf).all()
    rng = np.random.default_rng(6)
    toks = stratified_tokens(w.T, 16, rng, must=[0, 127, 128, 2047, 2048, 8191, 8192, 8193, 16383])
    kmh = km.cpu().numpy().view(np.uint32)
    ro, rl = O.masked_mha_prefill(x.q, x.k, x.v, kmh, x.cu_seqlens_q, x.cu_seqlens_kv, w.scale, tokens=toks)
    res = O.compare(of[toks], lf[toks], ro, rl)
    assert res["ok"], res
