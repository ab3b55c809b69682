"""The oracle against its pins, and planted mistakes that the pins must catch.

Mistakes are planted in the oracle (on the CPU, through monkeypatch); the
pins are the functions of ``oracle_pins.py``.
"""
import math

import numpy as np
import pytest

import oracle.dsa_oracle as O
import oracle_pins as P


@pytest.mark.parametrize("pin", P.ALL_PINS, ids=lambda p: p.__name__)
def test_pin_holds(pin):
    assert pin()


# ----------------------------------------------------------------------------
# planted mistakes
# ----------------------------------------------------------------------------
_orig_sparse = O.sparse_prefill
_orig_attend = O.attend
_orig_union = O.union_build
_orig_grouped = O.grouped_prefill
_orig_keymask = O.topk_to_key_mask
_orig_masked = O.masked_mha_prefill
_orig_l2g = O.local_to_global


def _attend_lse_base2(qf, K, V, scale):
    out, lse = _orig_attend(qf, K, V, scale)
    return out, lse / math.log(2.0)


def _attend_sign(qf, K, V, scale):
    return _orig_attend(qf, K, V, -scale)


def _attend_no_max_shift_wrong_norm(qf, K, V, scale):
    out, lse = _orig_attend(qf, K, V, scale)
    n = max(K.shape[0], 1)
    return out * (1.0 + 1.0 / n), lse


def _attend_transposed_values(qf, K, V, scale):
    # weights applied to K's first D_V columns reversed: a transposed/wrong operand
    return _orig_attend(qf, K, V[::-1].copy(), scale)


def _sparse_drop_rope(q, kv, idx, k, scale, d_qk, d_v, tokens=None):
    return _orig_sparse(q[..., :d_v], kv[:, :d_v], idx, k, scale, d_v, d_v, tokens)


def _sparse_wrong_scale(q, kv, idx, k, scale, d_qk, d_v, tokens=None):
    return _orig_sparse(q, kv, idx, k, 1.0 / math.sqrt(d_qk), d_qk, d_v, tokens)


def _sparse_v_from_tail(q, kv, idx, k, scale, d_qk, d_v, tokens=None):
    o, l = _orig_sparse(q, kv, idx, k, scale, d_qk, d_qk, tokens)
    return o[..., d_qk - d_v:], l


def _sparse_ignore_k(q, kv, idx, k, scale, d_qk, d_v, tokens=None):
    return _orig_sparse(q, kv, idx, idx.shape[1], scale, d_qk, d_v, tokens)


def _union_mask_shifted(idx, k, G, N, cu, upad):
    u, ul, m = _orig_union(idx, k, G, N, cu, upad)
    return u, ul, (m.astype(np.uint16) << 1).astype(np.uint8)


def _union_descending(idx, k, G, N, cu, upad):
    u, ul, m = _orig_union(idx, k, G, N, cu, upad)
    for g in range(u.shape[0]):
        U = int(ul[g])
        u[g, :U] = u[g, :U][::-1]
        m[g, :U] = m[g, :U][::-1]
    return u, ul, m


def _union_pad_zero(idx, k, G, N, cu, upad):
    u, ul, m = _orig_union(idx, k, G, N, cu, upad)
    for g in range(u.shape[0]):
        u[g, int(ul[g]):] = 0
    return u, ul, m


def _grouped_head_major(q, kv, u, ul, m, G, cu, scale, d_qk, d_v, group_ids=None):
    # pseudo-head order h*G + j instead of j*H + h
    T, H = q.shape[:2]
    q2 = q.copy()
    for (t0, n) in O.groups(cu, G):
        blk = q[t0:t0 + n].reshape(n * H, -1)
        perm = np.array([(p % n) * H + p // n for p in range(n * H)])
        q2[t0:t0 + n] = blk[perm].reshape(n, H, -1)
    return _orig_grouped(q2, kv, u, ul, m, G, cu, scale, d_qk, d_v, group_ids)


def _keymask_no_offset(idx, k, cq, ck, words):
    km = np.zeros((int(cq[-1]), words), dtype=np.uint32)
    for t in range(int(cq[-1])):
        for x in idx[t][:k]:
            if x >= 0 and x < 32 * words:
                km[t, x >> 5] |= np.uint32(1 << (int(x) & 31))
    return km


def _masked_shared_head(q, k, v, km, cq, ck, scale, tokens=None):
    return _orig_masked(q, np.repeat(k[:, :1], k.shape[1], axis=1), v, km, cq, ck, scale, tokens)


def _l2g_div_mod_swapped(idx, k, cq, kv_lens, bt, B, N):
    idx = np.asarray(idx)
    out = np.full(idx.shape, -1, dtype=np.int32)
    cqq = [0, idx.shape[0]] if cq is None else list(cq)
    for r in range(len(cqq) - 1):
        for t in range(cqq[r], cqq[r + 1]):
            for j in range(min(k, idx.shape[1])):
                x = int(idx[t, j])
                if 0 <= x < kv_lens[r] and x % B < bt.shape[1] and bt[r, x % B] >= 0:
                    out[t, j] = int(bt[r, x % B]) * B + x // B
    return out, 0


def _l2g_first_request_table(idx, k, cq, kv_lens, bt, B, N):
    return _orig_l2g(idx, k, cq, kv_lens, np.repeat(np.asarray(bt)[:1], len(bt), axis=0), B, N)


def _l2g_no_range_check(idx, k, cq, kv_lens, bt, B, N):
    return _orig_l2g(idx, k, cq, [np.asarray(bt).shape[1] * B] * len(kv_lens), bt, B, N)


_orig_e4m3_decode = O.e4m3_decode
_orig_e4m3_encode = O.e4m3_encode


def _e4m3_bias8(codes):
    return _orig_e4m3_decode(codes) / 2.0


def _e4m3_ties_away(x):
    x32 = np.asarray(x, dtype=np.float32)
    c = _orig_e4m3_encode(x32)
    grid = _orig_e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    a = np.abs(x32.astype(np.float64))
    lo = c & 0x7F
    up = np.minimum(lo + 1, 0x7E)
    tie = (lo < 0x7E) & (a == (grid[lo] + grid[up]) / 2)
    return np.where(tie, up | (c & 0x80), c).astype(np.uint8)


def _fp8_scale_per_64(kv_bits, d_rope):
    kv_bits = np.asarray(kv_bits, dtype=np.uint16)
    N = kv_bits.shape[0]
    x = (kv_bits[:, :512].astype(np.uint32) << 16).view(np.float32).reshape(N, 8, 64)
    amax = np.abs(x).max(axis=2)
    scale = np.where(amax > 0, (amax / np.float32(448.0)).astype(np.float32), np.float32(1.0))
    codes = O.e4m3_encode((x / scale[:, :, None]).astype(np.float32)).reshape(N, 512)
    out = np.zeros((N, O.kv_fp8_row_bytes(d_rope)), dtype=np.uint8)
    out[:, :512] = codes
    out[:, 512:528] = scale[:, ::2].astype("<f4").view(np.uint8).reshape(N, 16)
    if d_rope:
        out[:, 528:] = np.ascontiguousarray(kv_bits[:, 512:512 + d_rope]).astype("<u2").view(np.uint8)
    return out


_orig_compare = O.compare


def _compare_rel_over_got(got_out, got_lse, ref_out, ref_lse, max_abs=2e-2, rel_l2=5e-3):
    # relative L2 against the norm of the result instead of the reference
    r = _orig_compare(got_out, got_lse, ref_out, ref_lse, max_abs, rel_l2)
    go = np.asarray(got_out, dtype=np.float64)
    d = np.abs(go - np.asarray(ref_out, dtype=np.float64))
    den = float(np.sqrt((go ** 2).sum()))
    r["out_rel_l2"] = float(np.sqrt((d ** 2).sum()) / den) if den > 0 else 0.0
    r["ok"] = (not r["nan"]) and r["lse_inf_match"] and r["out_max_abs"] <= max_abs and \
        r["out_rel_l2"] <= rel_l2 and r["lse_max_abs"] <= max_abs and r["lse_rel_l2"] <= rel_l2
    return r


def _compare_inf_always_same(got_out, got_lse, ref_out, ref_lse, max_abs=2e-2, rel_l2=5e-3):
    gl = np.nan_to_num(np.asarray(got_lse, dtype=np.float64), posinf=0.0, neginf=0.0)
    rl = np.nan_to_num(np.asarray(ref_lse, dtype=np.float64), posinf=0.0, neginf=0.0)
    r = _orig_compare(got_out, np.where(np.isinf(got_lse), rl, gl), ref_out, rl, max_abs, rel_l2)
    return r


def _compare_ignores_lse_rel(got_out, got_lse, ref_out, ref_lse, max_abs=2e-2, rel_l2=5e-3):
    r = _orig_compare(got_out, got_lse, ref_out, ref_lse, max_abs, rel_l2)
    r["ok"] = (not r["nan"]) and r["lse_inf_match"] and r["out_max_abs"] <= max_abs and \
        r["out_rel_l2"] <= rel_l2 and r["lse_max_abs"] <= max_abs
    return r


def _compare_ignores_out_max(got_out, got_lse, ref_out, ref_lse, max_abs=2e-2, rel_l2=5e-3):
    r = _orig_compare(got_out, got_lse, ref_out, ref_lse, max_abs, rel_l2)
    r["ok"] = (not r["nan"]) and r["lse_inf_match"] and r["out_rel_l2"] <= rel_l2 and \
        r["lse_max_abs"] <= max_abs and r["lse_rel_l2"] <= rel_l2
    return r


def _compare_nan_blind(got_out, got_lse, ref_out, ref_lse, max_abs=2e-2, rel_l2=5e-3):
    f = lambda a: np.nan_to_num(np.asarray(a, dtype=np.float64), nan=0.0, posinf=np.inf, neginf=-np.inf)
    return _orig_compare(f(got_out), f(got_lse), f(ref_out), f(ref_lse), max_abs, rel_l2)


def _compare_fin_masks_large(got_out, got_lse, ref_out, ref_lse, max_abs=2e-2, rel_l2=5e-3):
    # finite lse entries that differ by more than 1 are dropped from the check
    gl = np.asarray(got_lse, dtype=np.float64).copy()
    rl = np.asarray(ref_lse, dtype=np.float64)
    far = np.isfinite(gl) & np.isfinite(rl) & (np.abs(gl - rl) > 1.0)
    gl[far] = rl[far]
    return _orig_compare(got_out, gl, ref_out, rl, max_abs, rel_l2)


def _compare_broadcasts(got_out, got_lse, ref_out, ref_lse, max_abs=2e-2, rel_l2=5e-3):
    go, ro = np.broadcast_arrays(np.asarray(got_out, dtype=np.float64), np.asarray(ref_out, dtype=np.float64))
    gl, rl = np.broadcast_arrays(np.asarray(got_lse, dtype=np.float64), np.asarray(ref_lse, dtype=np.float64))
    return _orig_compare(go, gl, ro, rl, max_abs, rel_l2)


MUTATIONS = [
    ("attend", _attend_lse_base2),
    ("attend", _attend_sign),
    ("attend", _attend_no_max_shift_wrong_norm),
    ("attend", _attend_transposed_values),
    ("sparse_prefill", _sparse_drop_rope),
    ("sparse_prefill", _sparse_wrong_scale),
    ("sparse_prefill", _sparse_v_from_tail),
    ("sparse_prefill", _sparse_ignore_k),
    ("union_build", _union_mask_shifted),
    ("union_build", _union_descending),
    ("union_build", _union_pad_zero),
    ("grouped_prefill", _grouped_head_major),
    ("topk_to_key_mask", _keymask_no_offset),
    ("masked_mha_prefill", _masked_shared_head),
    ("local_to_global", _l2g_div_mod_swapped),
    ("local_to_global", _l2g_first_request_table),
    ("local_to_global", _l2g_no_range_check),
    ("e4m3_decode", _e4m3_bias8),
    ("e4m3_encode", _e4m3_ties_away),
    ("kv_fp8_quantize", _fp8_scale_per_64),
    ("compare", _compare_rel_over_got),
    ("compare", _compare_inf_always_same),
    ("compare", _compare_ignores_lse_rel),
    ("compare", _compare_ignores_out_max),
    ("compare", _compare_nan_blind),
    ("compare", _compare_fin_masks_large),
    ("compare", _compare_broadcasts),
]


@pytest.mark.parametrize("name,fn", MUTATIONS, ids=[f.__name__ for _, f in MUTATIONS])
def test_planted_mistake_is_caught(monkeypatch, name, fn):
    monkeypatch.setattr(O, name, fn)
    res = P.run_all_pins()
    failed = [k for k, v in res.items() if not v]
    assert failed, f"no pin caught the planted mistake {fn.__name__}"
