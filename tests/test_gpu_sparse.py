"""Per-token sparse prefill on the GPU (through the C ABI) against the fp64
oracle: every token at oracle-sized shapes spanning several 128-key tiles and
a ragged tail, edge cases, and sampled tokens of the full-size workloads in
the launch configuration the bench times.  Tolerance (from the method's
bf16-in / fp32-accumulate arithmetic): out and lse max-abs <= 2e-2 and
relative-L2 <= 5e-3; lse infinities must match exactly."""
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


def run_gpu(q_bits, kv_bits, idx, k, scale, poison=True):
    import dsa_sparse_mla_prefill_gb300 as dsa
    T, H, _ = q_bits.shape
    q, kv, ix = bf(q_bits), bf(kv_bits), i32(idx)
    out = torch.full((T, H, 512), float("nan"), dtype=torch.bfloat16, device="cuda") if poison else None
    lse = torch.full((T, H), float("nan"), dtype=torch.float32, device="cuda") if poison else None
    out, lse = dsa.dsa_sparse_prefill(q, kv, ix, k, scale, out=out, lse=lse)
    torch.cuda.synchronize()
    return f32(out), lse.cpu().numpy().astype(np.float64)


def check(q_bits, kv_bits, idx, k, scale, d_qk, tokens=None):
    o, l = run_gpu(q_bits, kv_bits, idx, k, scale)
    ro, rl = O.sparse_prefill(q_bits, kv_bits, idx, k, scale, d_qk, 512, tokens=tokens)
    if tokens is not None:
        o, l = o[tokens], l[tokens]
    res = O.compare(o, l, ro, rl)
    assert res["ok"], res
    return res


def test_tiny_uniform_config_all_tokens():
    w = WORKLOADS["tiny_uniform_512"]
    x = make_sparse_inputs(w)
    check(x.q, x.kv, x.idx, w.k, w.scale, w.d_qk)


@pytest.mark.parametrize("H", [16, 32])
@pytest.mark.parametrize("d_qk", [576, 512])
def test_ragged_tiles_locality(H, d_qk):
    """k = 300: two full 128-key tiles and a 44-key tail; tokens below k are dense."""
    base = WORKLOADS["v32_h32_16k"]
    w = scaled_down(base, (333,), (700,), k=300, ld=310, H=H, seed=11 + H + d_qk)
    w = dataclasses.replace(w, d_qk=d_qk, scale=1.0 / math.sqrt(192.0 if d_qk == 576 else 256.0))
    x = make_sparse_inputs(w)
    check(x.q, x.kv, x.idx, w.k, w.scale, d_qk)


def test_two_requests_nope_wide_index_buffer():
    w = scaled_down(WORKLOADS["nope_2x8192"], (150, 170), (150, 170), k=260, ld=280)
    x = make_sparse_inputs(w)
    check(x.q, x.kv, x.idx, w.k, w.scale, w.d_qk)


def test_edge_rows_empty_scattered_bad_and_single():
    """Rows that are all -1, rows with -1 anywhere, bad entries (ignored and
    counted), a single selection, k not a multiple of 128, and more tokens
    per CTA than one (T > SM count is not needed for that: the grid is
    min(T, SMs))."""
    import dsa_sparse_mla_prefill_gb300 as dsa
    dsa.dsa_last_device_error()
    rng = np.random.default_rng(21)
    T, N, H, k, ld = 40, 900, 16, 200, 205
    q = normal_bf16(rng, (T, H, 576))
    kv = normal_bf16(rng, (N, 576))
    idx = np.full((T, ld), -1, dtype=np.int32)
    for t in range(T):
        n = int(rng.integers(1, k + 1))
        idx[t, rng.choice(k, size=n, replace=False)] = rng.choice(N, size=n, replace=False)
        idx[t, k:] = rng.integers(-5, 2 * N, size=ld - k)   # ignored columns, junk allowed
    idx[0, :] = -1
    idx[1, :k] = -1
    idx[1, 17] = 5
    idx[2, :k] = -1
    idx[2, 199] = N - 1
    clean = idx.copy()
    bad = [(5, 3, N), (6, 0, -2), (7, 100, 10 ** 7)]
    for t, c, v in bad:
        idx[t, c] = v
        clean[t, c] = -1
    o, l = run_gpu(q, kv, idx, k, 0.07)
    st, counts = dsa.dsa_last_device_error()
    assert st == 0 and counts[0] == len(bad)
    ro, rl = O.sparse_prefill(q, kv, clean, k, 0.07, 576, 512)
    res = O.compare(o, l, ro, rl)
    assert res["ok"], res
    assert np.all(o[0] == 0) and np.all(np.isneginf(l[0]))


@pytest.mark.parametrize("T", [1, 3])
def test_fewer_tokens_than_sms(T):
    rng = np.random.default_rng(T)
    N, H, k = 400, 32, 256
    q = normal_bf16(rng, (T, H, 576))
    kv = normal_bf16(rng, (N, 576))
    idx = np.stack([rng.choice(N, size=k, replace=False) for _ in range(T)]).astype(np.int32)
    check(q, kv, idx, k, 1.0 / math.sqrt(192.0), 576)


def test_many_tokens_per_cta_small_k():
    """T well above the SM count so every CTA runs several tokens (pipeline
    phases across tokens), with k = 64 < one tile."""
    rng = np.random.default_rng(4)
    T, N, H, k = 700, 256, 16, 64
    q = normal_bf16(rng, (T, H, 512))
    kv = normal_bf16(rng, (N, 512))
    idx = np.stack([rng.choice(N, size=k, replace=False) for _ in range(T)]).astype(np.int32)
    idx[::7, ::3] = -1
    check(q, kv, idx, k, 1.0 / 16.0, 512)


@pytest.mark.parametrize("name", ["v32_h32_16k", "nope_2x8192", "grouped_21k_of_32k", "v32_h32_16k_of_128k"])
def test_full_size_sampled(name):
    """Full-size workload, launched exactly as the bench does; the oracle
    checks a stratified sample of tokens (both ends, dense early tokens,
    uniform strata); every output must be finite."""
    w = WORKLOADS[name]
    x = make_sparse_inputs(w)
    o, l = run_gpu(x.q, x.kv, x.idx, w.k, w.scale)
    assert np.isfinite(o).all() and np.isfinite(l).all()
    rng = np.random.default_rng(123)
    toks = stratified_tokens(w.T, 40, rng, must=[1, 2047, 2048, 8191, 8192, w.T // 2, w.T - 1])
    ro, rl = O.sparse_prefill(x.q, x.kv, x.idx, w.k, w.scale, w.d_qk, w.d_v, tokens=toks)
    res = O.compare(o[toks], l[toks], ro, rl)
    assert res["ok"], res


def test_empty_kv_table():
    """N = 0: every index is out of range, so every token has no keys: zero
    output and lse = -inf (the kv pointer may be null)."""
    import dsa_sparse_mla_prefill_gb300 as dsa
    T, H, k = 5, 16, 8
    q = bf(normal_bf16(np.random.default_rng(3), (T, H, 576)))
    kv = torch.empty((0, 576), dtype=torch.bfloat16, device="cuda")
    idx = torch.full((T, k), -1, dtype=torch.int32, device="cuda")
    out = torch.full((T, H, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((T, H), float("nan"), dtype=torch.float32, device="cuda")
    out, lse = dsa.dsa_sparse_prefill(q, kv, idx, k, 0.125, out=out, lse=lse)
    torch.cuda.synchronize()
    assert torch.all(out == 0).item()
    assert torch.all(torch.isneginf(lse)).item()
