// Masked dense MHA simulating DSA for sm_103a.
//
// "[2/N][Attention] Enable masked MHA for sparse MLA prefills", Purpose: for
// short prefills a dense MHA with a per-token key mask (the token's top-k
// set) replaces the sparse MQA kernel; "[Perf][GLM-5.3-Flash] ...", Purpose,
// runs the same path on the decompressed per-head q/k/v.  Per head h and
// query t of request r:
//     out[t,h,:] = softmax_{n : bit n of key_mask[t]}( scale * q[t,h,:] . k[c_r+n,h,:] ) . v[c_r+n,h,:]
//
// One CTA per (128-query tile, head), FlashAttention-style over 128-key
// tiles of the request:
//   warps 5-8   cp.async loads of the q tile and of each k/v tile (128B
//               swizzled); before a key tile they read its 4 mask words per
//               query row and skip tiles where every bit is zero (the whole
//               upper causal triangle, and any empty tile).
//   warp 4      one thread: S = Q K^T (M = 128 queries, N = 128 keys) into a
//               double-buffered TMEM S, then O += P V with P read from TMEM.
//   warps 0-3   thread i owns query row i: mask, online softmax (base 2, lazy
//               rescale), P packed bf16 into the S columns it came from, and
//               the epilogue.
#include "dsa_device.cuh"
#include "dsa_kernels.h"

namespace dsa {
namespace masked {

constexpr int BQ = 128;
constexpr int BKV = 128;
constexpr int NTHREADS = 288;
constexpr int LAG = 2;
constexpr float kTau = 8.0f;

template <int DQK, int DV>
struct Cfg {
  static constexpr int QC = DQK / 64;   // swizzle columns of q / k
  static constexpr int VC = DV / 64;    // swizzle columns of v
  static constexpr uint32_t Q_BYTES = QC * BQ * 128u;
  static constexpr uint32_t K_BYTES = QC * BKV * 128u;
  static constexpr uint32_t V_BYTES = VC * BKV * 128u;
  static constexpr uint32_t OFF_Q = 0;
  static constexpr uint32_t OFF_K = OFF_Q + Q_BYTES;             // [2]
  static constexpr uint32_t OFF_V = OFF_K + 2 * K_BYTES;         // [2]
  static constexpr uint32_t OFF_MASK = OFF_V + 2 * V_BYTES;      // [2][128] x uint4
  static constexpr uint32_t OFF_INFO = OFF_MASK + 2 * BQ * 16u;  // tile index per stage [2], votes [2]
  static constexpr uint32_t OFF_BAR = OFF_INFO + 64u;
  static constexpr int NBAR = 16;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8u;
  static constexpr uint32_t SMEM_BYTES = OFF_MISC + 64u + 1024u;
  static constexpr uint32_t COL_S = 0;      // [2] x 128 columns
  static constexpr uint32_t COL_O = 256;    // DV columns
  static constexpr uint32_t TMEM_COLS = 512;
};

enum {
  B_Q_FULL = 0,
  B_ST_FULL = 1,   // [2]
  B_ST_EMPTY = 3,  // [2]
  B_S_FULL = 5,    // [2]
  B_S_EMPTY = 7,   // [2]
  B_P_FULL = 9,
  B_PV_DONE = 10,
  B_PROD_SYNC = 11,
  B_DRAIN = 12,
};

template <int DQK, int DV>
__global__ void __launch_bounds__(NTHREADS, 1) masked_mha_kernel(MaskedArgs a) {
  using C = Cfg<DQK, DV>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_u32 + 1023u) & ~1023u) - raw_u32);
  const uint32_t sbase = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile uint32_t* tmem_base_ptr = misc;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 1);
  volatile int* stage_tile = reinterpret_cast<volatile int*>(smem + C::OFF_INFO);      // [2]
  int* votes = reinterpret_cast<int*>(smem + C::OFF_INFO + 16);                        // [4] ring
  unsigned int* err = a.err;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---- work item: (head, query tile) ----
  const int nqt = a.num_qtiles;
  const int h = blockIdx.x / nqt;
  const int qt = nqt - 1 - (blockIdx.x % nqt);
  int r = 0;
  while (r + 1 < a.req.num_req && a.req.cu_g[r + 1] <= qt) ++r;
  const int q0 = a.req.cu_q[r] + (qt - a.req.cu_g[r]) * BQ;
  const int nq = min(BQ, a.req.cu_q[r + 1] - q0);
  const int kv0 = a.req.cu_kv[r];
  const int nkv = a.req.cu_kv[r + 1] - kv0;
  const int ntk = (nkv + BKV - 1) / BKV;
  const int H = a.H;

  if (threadIdx.x == 0) {
    mbar_init(&bars[B_Q_FULL], 128);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars[B_ST_FULL + i], 128);
      mbar_init(&bars[B_ST_EMPTY + i], 1);
      mbar_init(&bars[B_S_FULL + i], 1);
      mbar_init(&bars[B_S_EMPTY + i], 1);
    }
    mbar_init(&bars[B_P_FULL], 128);
    mbar_init(&bars[B_PV_DONE], 1);
    mbar_init(&bars[B_PROD_SYNC], 128);
    mbar_init(&bars[B_DRAIN], 1);
    votes[0] = votes[1] = votes[2] = votes[3] = 0;
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 4) {
    tmem_alloc(const_cast<uint32_t*>(tmem_base_ptr), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_base_ptr;

  if (warp >= 5) {
    // ------------------------------------------------------------------
    // producers
    // ------------------------------------------------------------------
    const int ptid = threadIdx.x - 160;
    const int p8 = ptid & 7;
    const int rsub = ptid >> 3;  // 0..15
    uint64_t* pend[LAG + 2];
    int npend = 0;
    auto flush = [&]() {
      cp_async_wait_all();
      fence_proxy_async_smem();
      for (int i = 0; i < npend; ++i) mbar_arrive(pend[i]);
      npend = 0;
    };
    auto push = [&](uint64_t* bar) {
      cp_async_commit();
      pend[npend++] = bar;
      if (npend > LAG) {
        cp_async_wait<LAG>();
        fence_proxy_async_smem();
        mbar_arrive(pend[0]);
        for (int i = 1; i < npend; ++i) pend[i - 1] = pend[i];
        --npend;
      }
    };
    auto wait_free = [&](uint64_t* bar, uint32_t parity) -> bool {
      if (mbar_ready(bar, parity)) return true;
      flush();
      return mbar_wait(bar, parity, abort_flag, err);
    };
    // q tile: rows q0 .. q0+127 of head h
    {
      const uint32_t qs = sbase + C::OFF_Q;
      for (int pass = 0; pass < (BQ / 16) * C::QC; ++pass) {
        const int row = (pass % (BQ / 16)) * 16 + rsub;
        const int c = pass / (BQ / 16);
        const bool valid = row < nq;
        const uint16_t* src = a.q + ((size_t)(valid ? q0 + row : 0) * H + h) * DQK + c * 64 + p8 * 8;
        cp_async16(qs + c * (BQ * 128) + row * 128 + ((p8 ^ (row & 7)) << 4), src, valid ? 16u : 0u);
      }
      push(&bars[B_Q_FULL]);
    }
    const uint32_t* km_row = reinterpret_cast<const uint32_t*>(a.key_mask) +
                             (size_t)(q0 + (ptid < nq ? ptid : 0)) * a.words;
    uint32_t sync_phase = 0;
    uint32_t st = 0;  // stages used
    bool ok = true;
    for (int j = 0; j < ntk && ok; ++j) {
      uint4 w = make_uint4(0, 0, 0, 0);
      if (ptid < nq) w = __ldg(reinterpret_cast<const uint4*>(km_row + 4 * j));
      const bool any = (w.x | w.y | w.z | w.w) != 0u;
      // one vote slot per key tile, 4-slot ring: slot (j-1)&3 was read by
      // every thread before the barrier below and is next written at j+3,
      // which no thread reaches before thread 0 has passed barrier j+1
      if (__any_sync(0xffffffffu, any) && lane == 0) atomicOr(&votes[j & 3], 1);
      if (!group_sync(&bars[B_PROD_SYNC], sync_phase, abort_flag, err)) { ok = false; break; }
      const int v = *reinterpret_cast<volatile int*>(&votes[j & 3]);
      if (ptid == 0) votes[(j + 3) & 3] = 0;
      if (v == 0) continue;
      const int s = st & 1;
      if (!wait_free(&bars[B_ST_EMPTY + s], ((st >> 1) & 1) ^ 1)) { ok = false; break; }
      reinterpret_cast<uint4*>(smem + C::OFF_MASK + s * BQ * 16)[ptid] = w;
      if (ptid == 0) stage_tile[s] = j;
      const uint32_t ks = sbase + C::OFF_K + s * C::K_BYTES;
      const uint32_t vs = sbase + C::OFF_V + s * C::V_BYTES;
      for (int pass = 0; pass < (BKV / 16) * C::QC; ++pass) {
        const int row = (pass % (BKV / 16)) * 16 + rsub;
        const int c = pass / (BKV / 16);
        const int key = j * BKV + row;
        const bool valid = key < nkv;
        const uint16_t* src = a.k + ((size_t)(kv0 + (valid ? key : 0)) * H + h) * DQK + c * 64 + p8 * 8;
        cp_async16(ks + c * (BKV * 128) + row * 128 + ((p8 ^ (row & 7)) << 4), src, valid ? 16u : 0u);
      }
      for (int pass = 0; pass < (BKV / 16) * C::VC; ++pass) {
        const int row = (pass % (BKV / 16)) * 16 + rsub;
        const int c = pass / (BKV / 16);
        const int key = j * BKV + row;
        const bool valid = key < nkv;
        const uint16_t* src = a.v + ((size_t)(kv0 + (valid ? key : 0)) * H + h) * DV + c * 64 + p8 * 8;
        cp_async16(vs + c * (BKV * 128) + row * 128 + ((p8 ^ (row & 7)) << 4), src, valid ? 16u : 0u);
      }
      push(&bars[B_ST_FULL + s]);
      ++st;
    }
    if (ok) {
      // end marker
      const int s = st & 1;
      if (wait_free(&bars[B_ST_EMPTY + s], ((st >> 1) & 1) ^ 1)) {
        if (ptid == 0) stage_tile[s] = -1;
        push(&bars[B_ST_FULL + s]);
      }
    }
    flush();
  } else if (warp == 4) {
    // ------------------------------------------------------------------
    // tcgen05 issuer
    // ------------------------------------------------------------------
    if (lane == 0) {
      constexpr uint32_t IDESC_QK = idesc_bf16_f32(128, BKV, false, false);
      constexpr uint32_t IDESC_PV = idesc_bf16_f32(128, DV, false, true);
      const uint32_t qs = sbase + C::OFF_Q;
      bool ok = mbar_wait(&bars[B_Q_FULL], 0, abort_flag, err);
      tc_fence_after();
      uint32_t n = 0;  // tiles consumed (stage sequence)
      auto issue_qk = [&](uint32_t i) -> bool {
        const int s = i & 1, sb = i & 1;
        if (!mbar_wait(&bars[B_S_EMPTY + sb], ((i >> 1) & 1) ^ 1, abort_flag, err)) return false;
        tc_fence_after();
        const uint32_t ks = sbase + C::OFF_K + s * C::K_BYTES;
#pragma unroll
        for (int c = 0; c < C::QC; ++c)
          mma_bf16_ss_x4(tmem + C::COL_S + sb * 128, sdesc_sw128(qs + c * (BQ * 128), 16, 1024),
                         sdesc_sw128(ks + c * (BKV * 128), 16, 1024), 2u, 2u, IDESC_QK, c > 0 ? 1u : 0u);
        mma_commit(&bars[B_S_FULL + sb]);
        return true;
      };
      int cur_tile = -1;
      if (ok) {
        ok = mbar_wait(&bars[B_ST_FULL + 0], 0, abort_flag, err);
        if (ok) {
          tc_fence_after();
          cur_tile = stage_tile[0];
          if (cur_tile >= 0) ok = issue_qk(0);
        }
      }
      while (ok && cur_tile >= 0) {
        const uint32_t nx = n + 1;
        // next stage: its QK overlaps this tile's softmax
        if (!mbar_wait(&bars[B_ST_FULL + (nx & 1)], (nx >> 1) & 1, abort_flag, err)) { ok = false; break; }
        tc_fence_after();
        const int nx_tile = stage_tile[nx & 1];
        if (nx_tile >= 0 && !issue_qk(nx)) { ok = false; break; }
        // O += P V for the current tile
        if (!mbar_wait(&bars[B_P_FULL], n & 1, abort_flag, err)) { ok = false; break; }
        tc_fence_after();
        const int s = n & 1;
        const uint32_t vs = sbase + C::OFF_V + s * C::V_BYTES;
#pragma unroll
        for (int half = 0; half < 2; ++half)
          mma_bf16_ts_x4(tmem + C::COL_O, tmem + C::COL_S + s * 128 + half * 32,
                         sdesc_sw128(vs + half * 4 * 2048, BKV * 128, 1024), 8u, 128u, IDESC_PV,
                         (n > 0 || half > 0) ? 1u : 0u);
        mma_commit(&bars[B_PV_DONE]);
        mma_commit(&bars[B_ST_EMPTY + s]);
        mma_commit(&bars[B_S_EMPTY + s]);
        n = nx;
        cur_tile = nx_tile;
      }
      mma_commit(&bars[B_DRAIN]);
      mbar_wait(&bars[B_DRAIN], 0, abort_flag, err);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------
    // softmax + epilogue: thread i <-> query row i <-> TMEM lane i
    // ------------------------------------------------------------------
    const int row = threadIdx.x;
    const float sl2 = a.scale * 1.4426950408889634f;
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    float m_run = -INFINITY, l_run = 0.f;
    uint32_t n = 0;
    bool ok = true;
    while (true) {
      const int s = n & 1;
      if (!mbar_wait_warp(&bars[B_ST_FULL + s], (n >> 1) & 1, abort_flag, err)) { ok = false; break; }
      const int tile = stage_tile[s];
      if (tile < 0) break;
      const uint4 mw = reinterpret_cast<const uint4*>(smem + C::OFF_MASK + s * BQ * 16)[row];
      if (!mbar_wait_warp(&bars[B_S_FULL + s], (n >> 1) & 1, abort_flag, err)) { ok = false; break; }
      tc_fence_after();
      float sv[BKV];
#pragma unroll
      for (int c = 0; c < BKV; c += 16) tmem_ld16(tmem + lane_off + C::COL_S + s * 128 + c, sv + c);
      tmem_ld_wait();
      const uint32_t mwords[4] = {mw.x, mw.y, mw.z, mw.w};
      float tmax = -INFINITY;
#pragma unroll
      for (int c = 0; c < BKV; ++c) {
        const bool on = (mwords[c >> 5] >> (c & 31)) & 1u;
        sv[c] = on ? sv[c] * sl2 : -INFINITY;
        tmax = fmaxf(tmax, sv[c]);
      }
      const bool need = tmax > m_run + kTau;
      float alpha = 1.f;
      if (need) {
        const float mn = fmaxf(m_run, tmax);
        alpha = (m_run == -INFINITY) ? 0.f : exp2f(m_run - mn);
        m_run = mn;
        l_run *= alpha;
      }
      // O rows that need rescaling: the previous P.V must be finished first
      if (__any_sync(0xffffffffu, need && n > 0)) {
        if (!mbar_wait_warp(&bars[B_PV_DONE], (n - 1) & 1, abort_flag, err)) { ok = false; break; }
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < DV; c += 16) {
          float o[16];
          tmem_ld16(tmem + lane_off + C::COL_O + c, o);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i) o[i] *= alpha;
          tmem_st16(tmem + lane_off + C::COL_O + c, o);
        }
        tmem_st_wait();
      }
      const float mref = (m_run == -INFINITY) ? 0.f : m_run;
#pragma unroll
      for (int c = 0; c < BKV; c += 32) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const uint16_t b0 = f32_to_bf16_rn(exp2f(sv[c + 2 * i] - mref));
          const uint16_t b1 = f32_to_bf16_rn(exp2f(sv[c + 2 * i + 1] - mref));
          l_run += bf16_to_f32(b0) + bf16_to_f32(b1);
          pk[i] = (uint32_t)b0 | ((uint32_t)b1 << 16);
        }
        tmem_st16_u32(tmem + lane_off + C::COL_S + s * 128 + c / 2, pk);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bars[B_P_FULL]);
      ++n;
    }
    // epilogue
    if (ok) {
      const int t = q0 + row;
      if (n > 0) {
        const bool got = mbar_wait_warp(&bars[B_PV_DONE], (n - 1) & 1, abort_flag, err);
        tc_fence_after();
        if (got) {
          const float inv_l = (l_run > 0.f) ? 1.f / l_run : 0.f;
#pragma unroll 1
          for (int c = 0; c < DV; c += 16) {
            float o[16];
            tmem_ld16(tmem + lane_off + C::COL_O + c, o);
            tmem_ld_wait();
            if (row < nq) {
              uint32_t pk[8];
#pragma unroll
              for (int i = 0; i < 8; ++i)
                pk[i] = (uint32_t)f32_to_bf16_rn(o[2 * i] * inv_l) |
                        ((uint32_t)f32_to_bf16_rn(o[2 * i + 1] * inv_l) << 16);
              uint4* dst = reinterpret_cast<uint4*>(a.out + ((size_t)t * H + h) * DV + c);
              dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
              dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
            }
          }
        }
      } else if (row < nq) {
        uint4* dst = reinterpret_cast<uint4*>(a.out + ((size_t)t * H + h) * DV);
        for (int c = 0; c < DV / 8; ++c) dst[c] = make_uint4(0, 0, 0, 0);
      }
      if (row < nq)
        a.lse[(size_t)t * H + h] = (l_run > 0.f) ? (m_run + log2f(l_run)) * 0.6931471805599453f : -INFINITY;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 4) tmem_dealloc(tmem, C::TMEM_COLS);
}

template <int DQK, int DV>
static int launch_t(const MaskedArgs& a, cudaStream_t stream) {
  using C = Cfg<DQK, DV>;
  static int attr_set[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set[dev]) {
    if (cudaFuncSetAttribute(masked_mha_kernel<DQK, DV>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::SMEM_BYTES) != cudaSuccess)
      return -1;
    attr_set[dev] = 1;
  }
  const long long grid = (long long)a.num_qtiles * a.H;
  if (grid == 0) return 0;
  masked_mha_kernel<DQK, DV><<<(unsigned)grid, NTHREADS, C::SMEM_BYTES, stream>>>(a);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace masked

int launch_masked_mha(const MaskedArgs& a, int /*num_sms*/, cudaStream_t stream) {
  if (a.d_qk == 192 && a.d_v == 128) return masked::launch_t<192, 128>(a, stream);
  return -2;
}

}  // namespace dsa
