"""Per-token sparse prefill reading FP8 latent rows directly
(dsa_sparse_prefill_fp8) against the oracle's per-token result on the oracle's
dequantized rows, and bit for bit against dsa_kv_fp8_dequantize followed by
dsa_sparse_prefill (the kernel dequantizes on chip with the same arithmetic,
so the two must agree in every bit of out and lse)."""
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


def bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def run_both(q_bits, rows, idx, k, scale, d_rope):
    """The FP8 kernel and the dequantize + bf16 per-token pair on the same inputs."""
    import dsa_sparse_mla_prefill_gb300 as dsa
    T, H, _ = q_bits.shape
    q, ix = bf(q_bits), i32(idx)
    f8 = torch.from_numpy(np.ascontiguousarray(rows)).cuda()
    out = torch.full((T, H, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((T, H), float("nan"), dtype=torch.float32, device="cuda")
    dsa.dsa_sparse_prefill_fp8(q, f8, ix, k, scale, d_rope=d_rope, out=out, lse=lse)
    torch.cuda.synchronize()
    st, counts = dsa.dsa_last_device_error()
    assert st == 0, counts
    kv_deq = dsa.dsa_kv_fp8_dequantize(f8, d_rope) if rows.shape[0] > 0 else \
        torch.empty((0, 512 + d_rope), dtype=torch.bfloat16, device="cuda")
    o2, l2 = dsa.dsa_sparse_prefill(q, kv_deq, ix, k, scale)
    torch.cuda.synchronize()
    return out, lse, o2, l2


def check(q_bits, rows, idx, k, scale, d_rope, tokens=None):
    out, lse, o2, l2 = run_both(q_bits, rows, idx, k, scale, d_rope)
    # bit for bit against dequantize + per-token
    assert np.array_equal(bits(out), bits(o2))
    assert np.array_equal(lse.cpu().numpy().view(np.uint32), l2.cpu().numpy().view(np.uint32))
    # the oracle on the oracle's own dequantized rows
    kv_ref = O.kv_fp8_dequantize(rows, d_rope)
    d_qk = 512 + d_rope
    o, l = f32(out), lse.cpu().numpy().astype(np.float64)
    if tokens is None:
        ro, rl = O.sparse_prefill(q_bits, kv_ref, idx, k, scale, d_qk, 512)
        res = O.compare(o, l, ro, rl)
    else:
        ro, rl = O.sparse_prefill(q_bits, kv_ref, idx, k, scale, d_qk, 512, tokens=tokens)
        res = O.compare(o[tokens], l[tokens], ro, rl)
    assert res["ok"], res
    return o, l


@pytest.mark.parametrize("d_rope", [64, 0])
@pytest.mark.parametrize("H", [16, 32])
def test_fp8_ragged(d_rope, H):
    """Several tokens per CTA, k = 300 with 5 % of the entries -1 holes (about
    285 valid rows: three tiles, the last ragged), both layouts."""
    base = WORKLOADS["v32_h32_16k"]
    w = scaled_down(base, (173, 29), (700, 330), k=300, ld=308, H=H, seed=11 + H + d_rope, index_gen="uniform")
    w = dataclasses.replace(w, d_qk=512 + d_rope, scale=1.0 / math.sqrt(192.0 if d_rope else 256.0))
    x = make_sparse_inputs(w)
    idx = x.idx.copy()
    rng = np.random.default_rng(5)
    holes = rng.random(idx.shape) < 0.05
    idx[holes] = -1
    rows = O.kv_fp8_quantize(x.kv, d_rope)
    check(x.q, rows, idx, w.k, w.scale, d_rope)


def test_fp8_awkward_rows_and_scales():
    """Rows scaled by 2^-60 .. 2^0 (block scales down to the float32
    subnormal range), all-zero blocks and negative zeros: the on-chip
    dequantize keeps subnormal products exactly."""
    rng = np.random.default_rng(7)
    H, k, N, T = 32, 256, 500, 40
    kv = normal_bf16(rng, (N, 576))
    kv[3, 128:256] = 0
    kv[4, 0:128] = 0x8000
    sc = np.exp2(rng.integers(-60, 1, size=(N, 1))).astype(np.float32)
    vals = ((kv.astype(np.uint32) << 16).view(np.float32) * sc).astype(np.float32)
    kv = (vals.view(np.uint32) >> 16).astype(np.uint16)
    rows = O.kv_fp8_quantize(kv, 64)
    q = normal_bf16(rng, (T, H, 576))
    idx = np.full((T, k), -1, dtype=np.int32)
    for t in range(T):
        n = int(rng.integers(1, k + 1))
        idx[t, :n] = rng.choice(N, size=n, replace=False)
    idx[5, :] = -1                      # a token without selection
    idx[6, :] = -1
    idx[6, 200:202] = [3, 4]            # only the all-zero and the negative-zero blocks' rows
    check(q, rows, idx, k, 0.05, 64)


def test_fp8_empty_table_and_tokens():
    """N = 0 (kv may be null): zero output and lse = -inf for every head."""
    import dsa_sparse_mla_prefill_gb300 as dsa
    H, k, T = 16, 8, 9
    q = bf(normal_bf16(np.random.default_rng(1), (T, H, 576)))
    f8 = torch.empty((0, 656), dtype=torch.uint8, device="cuda")
    idx = torch.full((T, k), -1, dtype=torch.int32, device="cuda")
    out, lse = dsa.dsa_sparse_prefill_fp8(q, f8, idx, k, 0.1)
    torch.cuda.synchronize()
    assert torch.all(out == 0).item() and torch.all(torch.isneginf(lse)).item()


@pytest.mark.parametrize("name", ["v32_h32_16k", "v32_h32_16k_of_128k"])
def test_fp8_full_size_sampled(name):
    """The bench's FP8 launch: the whole output bit-equal to dequantize +
    per-token, sampled tokens (every tile count, the ends) against the oracle."""
    w = WORKLOADS[name]
    x = make_sparse_inputs(w)
    rows = O.kv_fp8_quantize(x.kv, 64)
    rng = np.random.default_rng(79)
    toks = stratified_tokens(w.T, 24, rng, must=[0, 1, 127, 128, 2047, 2048, w.T - 1])
    o, l = check(x.q, rows, x.idx, w.k, w.scale, 64, tokens=toks)
    assert np.isfinite(o).all() and np.isfinite(l).all()
