// Choice between the three exact forms of DSA prefill (host code only).
//
// "[Perf][GLM-5.3-Flash] ...", commit messages: prompts within the top-k
// budget take dense MHA, longer ones masked MHA up to a length threshold (36k
// tokens at TP4, 64k at TP8) and the per-token kernel beyond;  "[Perf][DSA]
// Grouped sparse prefill ...", How: the grouped form can replace masked MHA
// for everything longer than the top-k budget.  The thresholds on the pages
// belong to their kernels; here each form's time is predicted from the work
// it does (the roofline quantity of its dominant kernel) and the fraction of
// the measured peak that form reaches on this GPU, and the fastest applicable
// form is taken:
//   per-token  logical gather bytes sum_t n_t * 2 d_qk + q, out, indices, lse
//              at per_token_frac of HBM;
//   grouped    2 * 128 * sum_g U_g * (d_qk + 512) FLOPs at grouped_frac of bf16,
//              plus the union build (index bytes at union_frac of HBM);
//   masked     2 * H * sum_r (q_r (q_r + 1) / 2 + q_r c_r) * (d_qk + d_v) FLOPs
//              (the causal triangle with its context) at masked_frac of bf16,
//              plus the key mask (index and mask bytes at key_mask_frac of HBM);
// each plus a fixed cost.  n_t = min(k, position + 1); U_g is the union of
// group g's rows: given by the caller after dsa_union_build, else estimated as
// min(last position + 1, n_last (1 + union_growth)).
#include <cmath>
#include <cstdint>

#include "../../include/dsa.h"

namespace {

// sum over m = a..b of min(k, m) for 1 <= a <= b.
double clamped_sum(int64_t a, int64_t b, int64_t k) {
  if (b < a) return 0.0;
  if (b <= k) return 0.5 * (double)(a + b) * (double)(b - a + 1);
  if (a > k) return (double)k * (double)(b - a + 1);
  return 0.5 * (double)(a + k) * (double)(k - a + 1) + (double)k * (double)(b - k);
}

bool masked_dims_ok(int d_qk, int d_v) { return (d_qk == 192 && d_v == 128) || (d_qk == 256 && d_v == 256); }

}  // namespace

extern "C" {

int dsa_form_calibration_default(dsa_form_calibration* c) {
  if (!c) return DSA_ERR_INVALID_ARG;
  // GB300 (one GPU, SM clock 2070 MHz): the measured copy bandwidth and
  // cuBLAS bf16 rate, and per-form fractions fitted to causal prompts of
  // 2k-32k tokens at H = 32 (top-2048, locality indices) and to the 64-head
  // 256/256 masked workload.
  c->hbm_gbs = 6690.5;
  c->bf16_tflops = 1940.6;
  c->per_token_frac = 0.977;
  c->per_token_ms0 = 0.07;
  c->union_frac = 0.32;   // the byte-map builder at G = 4 (16384 queries: 0.072 ms)
  c->union_ms0 = 0.009;
  c->grouped_frac_576 = 0.515;
  c->grouped_frac_512 = 0.504;
  c->grouped_ms0 = 0.033;
  c->masked_frac_192 = 0.568;
  c->masked_frac_256 = 0.65;
  c->masked_ms0 = 0.045;
  c->key_mask_frac = 0.66;
  c->key_mask_ms0 = 0.021;
  c->union_growth = 0.17;
  return DSA_OK;
}

int dsa_choose_form(const dsa_form_query* q, const dsa_form_calibration* calib, dsa_form_estimate* out) {
  if (!q || !out || q->num_req < 1 || !q->q_lens || !q->kv_lens || q->H < 1 || q->k < 1) return DSA_ERR_INVALID_ARG;
  if (q->d_qk != 512 && q->d_qk != 576) return DSA_ERR_UNSUPPORTED;
  dsa_form_calibration c;
  if (calib) {
    c = *calib;
  } else {
    dsa_form_calibration_default(&c);
  }
  if (!(c.hbm_gbs > 0) || !(c.bf16_tflops > 0) || !(c.per_token_frac > 0) || !(c.union_frac > 0) ||
      !(c.grouped_frac_576 > 0) || !(c.grouped_frac_512 > 0) || !(c.masked_frac_192 > 0) ||
      !(c.masked_frac_256 > 0) || !(c.key_mask_frac > 0) || c.union_growth < 0)
    return DSA_ERR_INVALID_ARG;
  const int64_t k = q->k;
  const int H = q->H;
  const int G = 128 / H;
  const bool grouped_ok = (128 % H) == 0 && G >= 1 && G <= 8;
  const bool masked_ok = masked_dims_ok(q->masked_d_qk, q->masked_d_v);
  int64_t T = 0, kv_max = 0;
  double pairs = 0.0, causal = 0.0, union_est = 0.0;
  for (int r = 0; r < q->num_req; ++r) {
    const int64_t nq = q->q_lens[r], nk = q->kv_lens[r];
    if (nq < 0 || nk < nq) return DSA_ERR_INVALID_ARG;
    const int64_t ctx = nk - nq;   // queries are the last nq positions
    T += nq;
    if (nk > kv_max) kv_max = nk;
    pairs += clamped_sum(ctx + 1, nk, k);
    causal += 0.5 * (double)nq * (double)(nq + 1) + (double)nq * (double)ctx;
    if (grouped_ok)
      for (int64_t g0 = 0; g0 < nq; g0 += G) {
        const int64_t last = ctx + (g0 + G < nq ? g0 + G : nq) - 1;   // position of the group's last token
        const double n_last = (double)(last + 1 < k ? last + 1 : k);
        union_est += std::fmin((double)(last + 1), std::ceil(n_last * (1.0 + c.union_growth)));
      }
  }
  const double hbm = c.hbm_gbs * 1e6;       // bytes per ms
  const double tc = c.bf16_tflops * 1e9;    // FLOPs per ms
  // per-token
  const double pt_bytes = pairs * 2.0 * q->d_qk + (double)T * H * (q->d_qk + 512) * 2.0 + (double)T * k * 4.0 +
                          (double)T * H * 4.0;
  out->ms[DSA_FORM_PER_TOKEN] = T == 0 ? 0.0 : pt_bytes / (c.per_token_frac * hbm) + c.per_token_ms0;
  // grouped (with its union build)
  out->union_rows = q->union_rows >= 0 ? q->union_rows : union_est;
  if (grouped_ok) {
    const double frac = q->d_qk == 576 ? c.grouped_frac_576 : c.grouped_frac_512;
    const double flops = 2.0 * 128.0 * out->union_rows * (q->d_qk + 512);
    const double ub = (double)T * k * 4.0;
    out->ms[DSA_FORM_GROUPED] =
        T == 0 ? 0.0 : flops / (frac * tc) + c.grouped_ms0 + ub / (c.union_frac * hbm) + c.union_ms0;
  } else {
    out->ms[DSA_FORM_GROUPED] = -1.0;
  }
  // masked (with its key mask)
  if (masked_ok) {
    const double frac = q->masked_d_qk == 256 ? c.masked_frac_256 : c.masked_frac_192;
    const double flops = 2.0 * H * causal * (q->masked_d_qk + q->masked_d_v);
    const double words = (double)(((kv_max + 31) / 32 + 3) / 4 * 4);
    const double kb = (double)T * (k * 4.0 + words * 4.0);
    out->ms[DSA_FORM_MASKED] =
        T == 0 ? 0.0 : flops / (frac * tc) + c.masked_ms0 + kb / (c.key_mask_frac * hbm) + c.key_mask_ms0;
  } else {
    out->ms[DSA_FORM_MASKED] = -1.0;
  }
  int best = DSA_FORM_PER_TOKEN;
  for (int f = 1; f < 3; ++f)
    if (out->ms[f] >= 0 && out->ms[f] < out->ms[best]) best = f;
  out->form = best;
  return DSA_OK;
}

}  // extern "C"
