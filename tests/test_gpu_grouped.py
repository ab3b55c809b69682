"""Grouped sparse prefill on the GPU (union build + grouped kernel, through
the C ABI) against the fp64 oracle.  The grouped result must equal the
per-token one, so it is checked both against the oracle's grouped form and
against its per-token form.  Same tolerance as the per-token tests."""
import dataclasses
import math

import numpy as np
import pytest

import oracle.dsa_oracle as O
from gpu_util import bf, f32, i32, need_gpu, stratified_tokens, torch
from synth import WORKLOADS, make_sparse_inputs, normal_bf16, scaled_down

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


def run_grouped(q_bits, kv_bits, idx, k, G, N, cu, scale, union_block=128):
    import dsa_sparse_mla_prefill_gb300 as dsa
    T, H, _ = q_bits.shape
    ix = i32(idx)
    upad = dsa.dsa_union_pad(G, k, union_block)
    u, ul, m = dsa.dsa_union_build(ix, k, G, N, cu_seqlens_q=cu, union_pad=upad)
    out = torch.full((T, H, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((T, H), float("nan"), dtype=torch.float32, device="cuda")
    dsa.dsa_grouped_prefill(bf(q_bits), bf(kv_bits), u, ul, m, G, scale, cu_seqlens_q=cu, out=out, lse=lse)
    torch.cuda.synchronize()
    st, counts = dsa.dsa_last_device_error()
    assert st == 0, counts
    return (u.cpu().numpy(), ul.cpu().numpy(), m.cpu().numpy()), f32(out), lse.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("d_qk", [576, 512])
@pytest.mark.parametrize("H,G", [(16, 8), (32, 4)])
def test_grouped_ragged_two_requests(d_qk, H, G):
    """Two requests whose lengths are not multiples of G (short last groups,
    padding pseudo-heads), unions spanning several 64-slot tiles."""
    base = WORKLOADS["grouped_21k_of_32k"]
    w = scaled_down(base, (61, 45), (400, 300), k=160, ld=170, H=H, G=G, seed=31 + H + d_qk)
    w = dataclasses.replace(w, d_qk=d_qk, scale=1.0 / math.sqrt(192.0 if d_qk == 576 else 256.0))
    x = make_sparse_inputs(w)
    (u, ul, m), o, l = run_grouped(x.q, x.kv, x.idx, w.k, G, w.N, x.cu_seqlens_q, w.scale)
    upad = O.union_pad(G, w.k, 128)
    ru, rl, rm = O.union_build(x.idx, w.k, G, w.N, x.cu_seqlens_q, upad)
    assert np.array_equal(ul, rl) and np.array_equal(u, ru) and np.array_equal(m, rm)
    go, gl = O.grouped_prefill(x.q, x.kv, ru, rl, rm, G, x.cu_seqlens_q, w.scale, d_qk, 512)
    res = O.compare(o, l, go, gl)
    assert res["ok"], res
    po, pl = O.sparse_prefill(x.q, x.kv, x.idx, w.k, w.scale, d_qk, 512)
    res = O.compare(o, l, po, pl)
    assert res["ok"], res


def test_grouped_empty_tokens_and_groups():
    """A group whose tokens select nothing (empty union), tokens with no
    selection inside a non-empty group, and a single-token request."""
    rng = np.random.default_rng(17)
    H, G, k, N = 16, 8, 48, 300
    q_lens = [16, 1, 11]
    T = sum(q_lens)
    cu = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    q = normal_bf16(rng, (T, H, 576))
    kv = normal_bf16(rng, (N, 576))
    idx = np.full((T, k), -1, dtype=np.int32)
    for t in range(T):
        n = int(rng.integers(1, k + 1))
        idx[t, rng.choice(k, size=n, replace=False)] = rng.choice(N, size=n, replace=False)
    idx[0:8, :] = -1        # first group: empty union
    idx[10, :] = -1         # a token without selection in group 2
    _, o, l = run_grouped(q, kv, idx, k, G, N, cu, 0.07)
    po, pl = O.sparse_prefill(q, kv, idx, k, 0.07, 576, 512)
    res = O.compare(o, l, po, pl)
    assert res["ok"], res
    assert np.all(o[0:8] == 0) and np.all(np.isneginf(l[0:8]))


@pytest.mark.parametrize("name", ["grouped_21k_of_32k", "nope_2x8192"])
def test_grouped_full_size_sampled(name):
    """Full-size workload in the bench's launch configuration; sampled tokens
    against the per-token oracle, every output finite."""
    w = WORKLOADS[name]
    x = make_sparse_inputs(w)
    _, o, l = run_grouped(x.q, x.kv, x.idx, w.k, w.G, w.N, x.cu_seqlens_q, w.scale)
    assert np.isfinite(o).all() and np.isfinite(l).all()
    rng = np.random.default_rng(77)
    toks = stratified_tokens(w.T, 40, rng, must=[1, 7, 8, 2047, 2048, 8191, 8192, w.T - 8])
    ro, rl = O.sparse_prefill(x.q, x.kv, x.idx, w.k, w.scale, w.d_qk, w.d_v, tokens=toks)
    res = O.compare(o[toks], l[toks], ro, rl)
    assert res["ok"], res


@pytest.mark.parametrize("name,index_gen", [("v32_h32_16k", None), ("grouped_21k_of_32k", "locality_wide")])
def test_grouped_full_size_bench_launches(name, index_gen):
    """The grouped launches the bench times beyond the two above: the 16384-token
    H = 32 chunk as groups of G = 4 (union ~2.2k per group), and the wide-union
    stress variant of the 21504-token workload (every token draws its own
    replacements, union ~4.3k per group).  Union list, lengths and mask bit-exact
    over the whole buffers; sampled tokens against the per-token oracle."""
    w = WORKLOADS[name]
    if index_gen is not None:
        w = dataclasses.replace(w, name=name + "_wide", index_gen=index_gen)
    x = make_sparse_inputs(w)
    (u, ul, m), o, l = run_grouped(x.q, x.kv, x.idx, w.k, w.G, w.N, x.cu_seqlens_q, w.scale)
    upad = O.union_pad(w.G, w.k, 128)
    ru, rl, rm = O.union_build(x.idx, w.k, w.G, w.N, x.cu_seqlens_q, upad)
    assert np.array_equal(ul, rl) and np.array_equal(u, ru) and np.array_equal(m, rm)
    if index_gen is not None:
        assert float(rl.mean()) > 3000   # the wide variant really widens the union
    assert np.isfinite(o).all() and np.isfinite(l).all()
    rng = np.random.default_rng(78)
    toks = stratified_tokens(w.T, 40, rng, must=[1, 3, 4, 7, 8, 2047, 2048, 8191, 8192, w.T - 4, w.T - 8])
    ro, rl2 = O.sparse_prefill(x.q, x.kv, x.idx, w.k, w.scale, w.d_qk, w.d_v, tokens=toks)
    res = O.compare(o[toks], l[toks], ro, rl2)
    assert res["ok"], res


@pytest.mark.parametrize("H,G", [(16, 8), (32, 4)])
def test_grouped_contiguous_runs(H, G):
    """Unions made of long runs of consecutive rows: dense sliding windows in
    the first request, and in the second a run that ends at the table's last
    row next to scattered rows.  Whole 64-slot halves of a tile are then one
    contiguous block (fetched as one tiled load) beside gathered halves, with
    runs that start and end inside a half and ragged union tails."""
    rng = np.random.default_rng(5 + H)
    k, N = 320, 700
    q_lens = [300, 37]
    T = sum(q_lens)
    cu = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    q = normal_bf16(rng, (T, H, 576))
    kv = normal_bf16(rng, (N, 576))
    idx = np.full((T, k), -1, dtype=np.int32)
    for t in range(q_lens[0]):
        rows = np.arange(max(0, t - k + 1), t + 1, dtype=np.int32)
        idx[t, :len(rows)] = rng.permutation(rows)
    for i in range(q_lens[1]):
        sel = np.concatenate([np.arange(N - 150, N), rng.choice(N - 150, size=100 + i, replace=False)])
        idx[q_lens[0] + i, :len(sel)] = rng.permutation(sel).astype(np.int32)
    (u, ul, m), o, l = run_grouped(q, kv, idx, k, G, N, cu, 0.07)
    upad = O.union_pad(G, k, 128)
    ru, rl, rm = O.union_build(idx, k, G, N, cu, upad)
    assert np.array_equal(ul, rl) and np.array_equal(u, ru) and np.array_equal(m, rm)
    po, pl = O.sparse_prefill(q, kv, idx, k, 0.07, 576, 512)
    res = O.compare(o, l, po, pl)
    assert res["ok"], res


def test_grouped_equals_per_token_kernel():
    """The two GPU forms agree with each other on a mid-size workload."""
    import dsa_sparse_mla_prefill_gb300 as dsa
    w = scaled_down(WORKLOADS["grouped_21k_of_32k"], (1024,), (3000,), k=512, ld=512, seed=41)
    x = make_sparse_inputs(w)
    _, og, lg = run_grouped(x.q, x.kv, x.idx, w.k, 8, w.N, x.cu_seqlens_q, w.scale)
    op, lp = dsa.dsa_sparse_prefill(bf(x.q), bf(x.kv), i32(x.idx), w.k, w.scale)
    torch.cuda.synchronize()
    res = O.compare(og, lg, f32(op), lp.cpu().numpy().astype(np.float64))
    assert res["ok"], res


def test_grouped_empty_kv_table():
    """N = 0: every union is empty; zero output and lse = -inf for every
    pseudo-head (the kv pointer may be null)."""
    import dsa_sparse_mla_prefill_gb300 as dsa
    H, G, k, T = 16, 8, 8, 13
    q = bf(normal_bf16(np.random.default_rng(5), (T, H, 576)))
    kv = torch.empty((0, 576), dtype=torch.bfloat16, device="cuda")
    idx = torch.full((T, k), -1, dtype=torch.int32, device="cuda")
    upad = dsa.dsa_union_pad(G, k, 128)
    u, ul, m = dsa.dsa_union_build(idx, k, G, 0, union_pad=upad)
    out = torch.full((T, H, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((T, H), float("nan"), dtype=torch.float32, device="cuda")
    out, lse = dsa.dsa_grouped_prefill(q, kv, u, ul, m, G, 0.125, out=out, lse=lse)
    torch.cuda.synchronize()
    assert int(ul.sum()) == 0
    assert torch.all(out == 0).item()
    assert torch.all(torch.isneginf(lse)).item()
