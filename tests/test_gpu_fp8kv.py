"""FP8 latent rows on the GPU against the oracle: quantize and dequantize bit for
bit (codes, scales, RoPE bytes, bf16 values), and the attention forms over the
dequantized cache against the oracle's per-token result on the oracle's own
dequantized rows."""
import numpy as np
import pytest

import oracle.dsa_oracle as O
from gpu_util import bf, f32, i32, need_gpu, torch
from synth import WORKLOADS, make_sparse_inputs, normal_bf16, scaled_down

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


def bits(t):
    """bf16 tensor -> its uint16 bit patterns (host numpy)."""
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def awkward_rows(rng, N, width):
    """bf16 rows with mixed magnitudes, an all-zero block, negative zeros and values far
    below their block's maximum (they round to zero or to subnormal codes)."""
    x = normal_bf16(rng, (N, width))
    # the special blocks sit in rows 0, 1, 2 (as many of them as there are rows)
    x[0, 128:256] = 0
    x[min(1, N - 1), 0:128] = 0x8000          # -0.0
    r = min(2, N - 1)
    x[r, 256:384] = normal_bf16(rng, (128,)) & 0x80FF   # tiny values (exponent field 1)
    x[r, 300] = 0x4300                        # 128.0 in the same block
    scale = np.exp2(rng.integers(-30, 30, size=(N, 1))).astype(np.float32)
    vals = ((x.astype(np.uint32) << 16).view(np.float32) * scale).astype(np.float32)
    return (vals.view(np.uint32) >> 16).astype(np.uint16)


@pytest.mark.parametrize("d_rope,ld,N", [(64, 576, 300), (64, 584, 300), (0, 512, 300),
                                         (64, 576, 1), (64, 576, 13), (0, 512, 8)])
def test_quantize_dequantize_bit_exact(d_rope, ld, N):
    """Row counts below, at and off the kernel's eight-row step (ragged tails)."""
    import dsa_sparse_mla_prefill_gb300 as dsa
    rng = np.random.default_rng(ld + d_rope + N)
    kv = awkward_rows(rng, N, ld)
    want = O.kv_fp8_quantize(kv, d_rope)
    got = dsa.dsa_kv_fp8_quantize(bf(kv), d_rope)
    torch.cuda.synchronize()
    assert np.array_equal(got.cpu().numpy(), want)
    # dequantize the oracle's rows (independent of the GPU quantizer)
    back = dsa.dsa_kv_fp8_dequantize(torch.from_numpy(want).cuda(), d_rope)
    torch.cuda.synchronize()
    assert np.array_equal(bits(back), O.kv_fp8_dequantize(want, d_rope))


def test_dequantize_every_code():
    """Rows holding every finite code under assorted positive scales."""
    import dsa_sparse_mla_prefill_gb300 as dsa
    rng = np.random.default_rng(3)
    N = 64
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    rows = np.zeros((N, O.kv_fp8_row_bytes(64)), dtype=np.uint8)
    rows[:, :512] = rng.choice(codes, size=(N, 512))
    rows[:, :254] = codes
    scales = np.exp2(rng.uniform(-40, 40, size=(N, 4))).astype("<f4")
    rows[:, 512:528] = scales.view(np.uint8).reshape(N, 16)
    rows[:, 528:] = (normal_bf16(rng, (N, 64)).astype("<u2")).view(np.uint8).reshape(N, 128)
    back = dsa.dsa_kv_fp8_dequantize(torch.from_numpy(rows).cuda(), 64)
    torch.cuda.synchronize()
    assert np.array_equal(bits(back), O.kv_fp8_dequantize(rows, 64))


def test_attention_over_fp8_cache():
    """Per-token and grouped forms over the dequantized cache equal the oracle's
    per-token result on the oracle's dequantized rows."""
    import dsa_sparse_mla_prefill_gb300 as dsa
    w = scaled_down(WORKLOADS["grouped_21k_of_32k"], (640,), (2000,), k=256, ld=256, seed=31)
    x = make_sparse_inputs(w)
    rows = O.kv_fp8_quantize(x.kv, 64)
    kv_deq_ref = O.kv_fp8_dequantize(rows, 64)
    fp8 = dsa.dsa_kv_fp8_quantize(bf(x.kv), 64)
    kv_deq = dsa.dsa_kv_fp8_dequantize(fp8, 64)
    q, idx = bf(x.q), i32(x.idx)
    o1, l1 = dsa.dsa_sparse_prefill(q, kv_deq, idx, w.k, w.scale)
    u, ul, m = dsa.dsa_union_build(idx, w.k, w.G, w.N, cu_seqlens_q=x.cu_seqlens_q)
    o2, l2 = dsa.dsa_grouped_prefill(q, kv_deq, u, ul, m, w.G, w.scale, cu_seqlens_q=x.cu_seqlens_q)
    torch.cuda.synchronize()
    st, counts = dsa.dsa_last_device_error()
    assert st == 0, counts
    assert np.array_equal(bits(kv_deq), kv_deq_ref)
    ro, rl = O.sparse_prefill(x.q, kv_deq_ref, x.idx, w.k, w.scale, w.d_qk, w.d_v)
    for o, l in ((o1, l1), (o2, l2)):
        res = O.compare(f32(o), l.cpu().numpy().astype(np.float64), ro, rl)
        assert res["ok"], res


def test_full_headline_table_bit_exact():
    import dsa_sparse_mla_prefill_gb300 as dsa
    w = WORKLOADS["v32_h32_16k"]
    x = make_sparse_inputs(w)
    want = O.kv_fp8_quantize(x.kv, 64)
    got = dsa.dsa_kv_fp8_quantize(bf(x.kv), 64)
    back = dsa.dsa_kv_fp8_dequantize(got, 64)
    torch.cuda.synchronize()
    assert np.array_equal(got.cpu().numpy(), want)
    assert np.array_equal(bits(back), O.kv_fp8_dequantize(want, 64))
