"""The form dispatcher (dsa_choose_form, host only): its predicted times against
a brute-force recomputation of the model token by token and group by group,
the applicability rules, argument checks, and the crossovers its GB300
calibration encodes."""
import math

import pytest

import dsa_sparse_mla_prefill_gb300 as dsa


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from dsa_sparse_mla_prefill_gb300 import build as b
    b.build()


def brute(q_lens, kv_lens, H, k, d_qk, mdims, c, union_rows=None):
    """The model with every sum taken token by token (no closed forms)."""
    hbm, tc = c.hbm_gbs * 1e6, c.bf16_tflops * 1e9
    T = sum(q_lens)
    pairs = 0
    causal = 0
    union = 0.0
    G = 128 // H if 128 % H == 0 else 0
    for nq, nk in zip(q_lens, kv_lens):
        pos = list(range(nk - nq, nk))
        for p in pos:
            pairs += min(k, p + 1)
            causal += p + 1                      # keys 0..p of the request
        if 1 <= G <= 8:
            for g0 in range(0, nq, G):
                last = pos[min(g0 + G, nq) - 1]
                union += min(last + 1, math.ceil(min(k, last + 1) * (1 + c.union_growth)))
    ms = {}
    ms["per_token"] = (pairs * 2 * d_qk + T * H * (d_qk + 512) * 2 + T * k * 4 + T * H * 4) / (c.per_token_frac * hbm) \
        + c.per_token_ms0
    U = union if union_rows is None else union_rows
    if 1 <= G <= 8:
        frac = c.grouped_frac_576 if d_qk == 576 else c.grouped_frac_512
        ms["grouped"] = 2 * 128 * U * (d_qk + 512) / (frac * tc) + c.grouped_ms0 + T * k * 4 / (c.union_frac * hbm) \
            + c.union_ms0
    else:
        ms["grouped"] = None
    if mdims in ((192, 128), (256, 256)):
        frac = c.masked_frac_256 if mdims[0] == 256 else c.masked_frac_192
        words = ((max(kv_lens) + 31) // 32 + 3) // 4 * 4
        ms["masked"] = 2 * H * causal * sum(mdims) / (frac * tc) + c.masked_ms0 \
            + T * (k * 4 + words * 4) / (c.key_mask_frac * hbm) + c.key_mask_ms0
    else:
        ms["masked"] = None
    return ms, U


@pytest.mark.parametrize("q_lens,kv_lens,H,k,d_qk,mdims", [
    ([300], [300], 32, 64, 576, (192, 128)),            # causal, ragged last group
    ([97, 130], [400, 130], 16, 96, 576, (256, 256)),   # chunked context, G = 8
    ([5, 1, 70], [5, 33, 70], 64, 8, 512, None),        # tiny requests, G = 2, no masked form
    ([50], [50], 3, 16, 576, (192, 128)),               # H = 3: no grouped form
])
def test_model_matches_brute_force(q_lens, kv_lens, H, k, d_qk, mdims):
    c = dsa.dsa_form_calibration_default()
    form, ms, U = dsa.dsa_choose_form(q_lens, kv_lens, H, k, d_qk, mdims)
    ref, refU = brute(q_lens, kv_lens, H, k, d_qk, mdims, c)
    assert U == pytest.approx(refU, rel=1e-12)
    for f in dsa.FORMS:
        if ref[f] is None:
            assert ms[f] is None
        else:
            assert ms[f] == pytest.approx(ref[f], rel=1e-12)
    avail = {f: v for f, v in ms.items() if v is not None}
    assert form == min(avail, key=avail.get)


def test_given_union_rows_and_custom_calibration():
    c = dsa.dsa_form_calibration_default()
    c.grouped_frac_576 = 0.9
    c.union_growth = 0.0
    form, ms, U = dsa.dsa_choose_form([1000], [3000], 16, 128, 576, None, union_rows=123456.0, calibration=c)
    ref, _ = brute([1000], [3000], 16, 128, 576, None, c, union_rows=123456.0)
    assert U == 123456.0
    assert ms["grouped"] == pytest.approx(ref["grouped"], rel=1e-12)
    assert ms["masked"] is None


def test_applicability_and_errors():
    for H, ok in ((16, True), (32, True), (128, True), (8, False), (3, False), (256, False)):
        _, ms, _ = dsa.dsa_choose_form([64], [64], H, 32, 576, None)
        assert (ms["grouped"] is not None) == ok, H
    for md, ok in (((192, 128), True), ((256, 256), True), ((256, 128), False), ((576, 512), False)):
        _, ms, _ = dsa.dsa_choose_form([64], [64], 16, 32, 576, md)
        assert (ms["masked"] is not None) == ok, md
    with pytest.raises(dsa.DSAError) as e:
        dsa.dsa_choose_form([10], [5], 16, 32)            # more queries than KV positions
    assert e.value.status == dsa.DSA_ERR_INVALID_ARG
    with pytest.raises(dsa.DSAError) as e:
        dsa.dsa_choose_form([10], [10], 16, 32, d_qk=192)  # not a latent width
    assert e.value.status == dsa.DSA_ERR_UNSUPPORTED
    c = dsa.dsa_form_calibration_default()
    c.masked_frac_192 = 0.0
    with pytest.raises(dsa.DSAError):
        dsa.dsa_choose_form([10], [10], 16, 32, calibration=c)


def test_gb300_crossovers():
    """What the GB300 calibration encodes for one causal prompt at H = 32 (DeepSeek-V3.2 at
    TP4): masked while the causal triangle is small, grouped beyond ~20k tokens, and masked
    overtaking per-token near 36k tokens (the threshold the pages give for TP4)."""
    pick = {L: dsa.dsa_choose_form([L], [L], 32, 2048, 576, (192, 128))[0] for L in (2048, 8192, 16384, 32768, 65536)}
    assert pick == {2048: "masked", 8192: "masked", 16384: "masked", 32768: "grouped", 65536: "grouped"}
    # without the grouped form: masked up to the per-token crossover
    c = dsa.dsa_form_calibration_default()
    lo, hi = 20000, 60000
    while hi - lo > 256:
        mid = (lo + hi) // 2
        _, ms, _ = dsa.dsa_choose_form([mid], [mid], 32, 2048, 576, (192, 128), calibration=c)
        lo, hi = (mid, hi) if ms["masked"] < ms["per_token"] else (lo, mid)
    assert 30000 < lo < 42000
