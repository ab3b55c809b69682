// Masked dense MHA simulating DSA for sm_103a.
//
// "[2/N][Attention] Enable masked MHA for sparse MLA prefills", Purpose: for
// short prefills a dense MHA with a per-token key mask (the token's top-k
// set) replaces the sparse MQA kernel; "[Perf][GLM-5.3-Flash] ...", Purpose,
// runs the same path on the decompressed per-head q/k/v.  Per head h and
// query t of request r:
//     out[t,h,:] = softmax_{n : bit n of key_mask[t]}( scale * q[t,h,:] . k[c_r+n,h,:] ) . v[c_r+n,h,:]
//
// Geometries ("[Perf][GLM-5.3-Flash] ...", Purpose and review snippets: the
// masked-MHA allow-list): (d_qk, d_v) = (192, 128) for DeepSeek-V3.2 and
// (256, 256) for GLM-5 (192 + 64 RoPE columns) and GLM-5.3-Flash (NoPE, 256
// + 0).  q, k and v are read through strided 3-D tensor maps, so k and v may
// be views into the per-head kv projection (no copy); when the RoPE columns
// are shared by all heads they come from their own [Nk, 64] buffer and the
// concatenated K is never formed ("skip the NoPE K concat", and the same for
// the RoPE part).
//
// One CTA per (128-query tile, head), FlashAttention-style over 128-key
// tiles of the request:
//   warp 9      TMA: the q tile and each k tile as 3-D boxes of one head
//               (64 columns x 1 head x rows, 128B-swizzled; the shared RoPE
//               columns as 2-D boxes); before a key tile it reads the tile's
//               4 mask words of every query row and skips tiles where every
//               bit is zero (the whole upper causal triangle, and any empty
//               tile).  K and V have their own 2-stage rings: a K stage
//               returns after its QK, a V stage after its PV, so the next
//               tiles' K loads are not held up by this tile's softmax.  At
//               d_qk = 192 a K stage is the whole 128-key tile and a V stage
//               too; at 256 (64 KB per tile) a K stage is half the columns
//               and a V stage half the keys, so both rings fit next to q.
//   warp 8      one thread: S = Q K^T (M = 128 queries, N = 128 keys) into a
//               double-buffered TMEM S.
//   warp 10     one thread: O += P V with P read from TMEM (two issuing
//               threads: one thread's per-tile waits, fences and commits
//               were the longer loop).
//   warp 11     TMA: the v tiles, following the tile sequence that warp 9
//               posts, so K loads never wait behind a V stage.
//   warps 0-7   two threads per query row (TMEM lane): warp w holds row
//               32(w%4) + lane and keys 64(w/4) .. +63 of each tile; mask,
//               online softmax (base 2, lazy rescale) with the row max
//               agreed through a per-tile pair exchange, P packed bf16 into
//               the S columns it came from, and the epilogue.
#include "dsa_device.cuh"
#include "dsa_kernels.h"

namespace dsa {
namespace masked {

constexpr int BQ = 128;
constexpr int BKV = 128;
constexpr int HK = BKV / 2;     // keys per softmax thread
constexpr int NTHREADS = 384;   // 12 warps
constexpr float kTau = 8.0f;

template <int DQK, int DV>
struct Cfg {
  static constexpr int QC = DQK / 64;   // swizzle columns of q / k
  static constexpr int VC = DV / 64;    // swizzle columns of v
  static constexpr int KSC = DQK > 192 ? 2 : QC;   // swizzle columns per K stage (all 128 keys)
  static constexpr int KPT = QC / KSC;             // K stages per key tile
  static constexpr int VR = DV > 128 ? 64 : BKV;   // keys per V stage (all DV columns)
  static constexpr int VPT = BKV / VR;             // V stages per key tile
  static_assert(QC % KSC == 0 && BKV % VR == 0 && VR % 64 == 0, "stage split");
  static constexpr uint32_t Q_BYTES = QC * BQ * 128u;
  static constexpr uint32_t K_BYTES = KSC * BKV * 128u;   // one K stage
  static constexpr uint32_t V_BYTES = VC * VR * 128u;     // one V stage
  static constexpr uint32_t OFF_Q = 0;
  static constexpr uint32_t OFF_K = OFF_Q + Q_BYTES;             // [2]
  static constexpr uint32_t OFF_V = OFF_K + 2 * K_BYTES;         // [2]
  static constexpr uint32_t OFF_MASK = OFF_V + 2 * V_BYTES;      // [4][128] x uint4 (tile info ring)
  static constexpr uint32_t OFF_PAIR = OFF_MASK + 4 * BQ * 16u;  // [2][2][128] floats
  static constexpr uint32_t OFF_INFO = OFF_PAIR + 2 * 2 * BQ * 4u;  // key-tile index per info slot [4]
  static constexpr uint32_t OFF_BAR = OFF_INFO + 64u;
  static constexpr int NBAR = 26;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8u;
  static constexpr uint32_t SMEM_BYTES = OFF_MISC + 64u + 1024u;
  static_assert(SMEM_BYTES <= 227u * 1024u, "shared memory budget");
  static constexpr uint32_t COL_S = 0;      // [2] x 128 columns; P (bf16 pairs) in the first 64
  static constexpr uint32_t COL_O = 256;    // DV columns
  static constexpr uint32_t TMEM_COLS = 512;
};

enum {
  B_Q_FULL = 0,
  B_K_FULL = 1,    // [2] k tile landed (or the end marker, no bytes)
  B_K_EMPTY = 3,   // [2] QK of the stage's tile completed
  B_V_FULL = 5,    // [2] v tile landed
  B_V_EMPTY = 7,   // [2] P.V of the stage's tile completed
  B_INFO = 9,      // [4] the tile's index and mask words are written (or the end marker)
  B_S_FULL = 13,   // [2]
  B_S_EMPTY = 15,  // [2] P.V completed (P aliases S)
  B_P_FULL = 17,   // 256 arrivals
  B_PV_DONE = 18,
  B_DRAIN = 19,     // [2] QK issuer, PV issuer
  B_PAIR = 21,     // [4] the two softmax warps of a TMEM lane quarter (64 arrivals)
};

template <int DQK, int DV>
__global__ void __launch_bounds__(NTHREADS, 1) masked_mha_kernel(const __grid_constant__ MaskedArgs a) {
  using C = Cfg<DQK, DV>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_u32 + 1023u) & ~1023u) - raw_u32);
  const uint32_t sbase = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile uint32_t* tmem_base_ptr = misc;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 1);
  volatile int* stage_tile = reinterpret_cast<volatile int*>(smem + C::OFF_INFO);      // [4]
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

  if (threadIdx.x == 0) {
    mbar_init(&bars[B_Q_FULL], 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars[B_K_FULL + i], 1);
      mbar_init(&bars[B_K_EMPTY + i], 1);
      mbar_init(&bars[B_V_FULL + i], 1);
      mbar_init(&bars[B_V_EMPTY + i], 1);
      mbar_init(&bars[B_S_FULL + i], 1);
      mbar_init(&bars[B_S_EMPTY + i], 1);
    }
    for (int i = 0; i < 4; ++i) mbar_init(&bars[B_INFO + i], 1);
    mbar_init(&bars[B_P_FULL], 256);
    mbar_init(&bars[B_PV_DONE], 1);
    mbar_init(&bars[B_DRAIN + 0], 1);
    mbar_init(&bars[B_DRAIN + 1], 1);
    for (int i = 0; i < 4; ++i) mbar_init(&bars[B_PAIR + i], 64);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 8) {
    tmem_alloc(const_cast<uint32_t*>(tmem_base_ptr), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_base_ptr;

  if (warp == 9) {
    // ------------------------------------------------------------------
    // TMA producer: q tile, then each key tile with any mask bit set
    // ------------------------------------------------------------------
    if (lane == 0) {
      mbar_arrive_expect_tx(&bars[B_Q_FULL], C::Q_BYTES);
      for (int c = 0; c < C::QC; ++c)
        tma_load_3d(sbase + C::OFF_Q + c * (BQ * 128), &a.tmap_q, c * 64, h, q0, &bars[B_Q_FULL]);
    }
    const uint32_t* km = a.key_mask;
    uint32_t st = 0;    // key tiles posted
    uint32_t nku = 0;   // K stage uses issued
    bool ok = true;
    for (int j = 0; j < ntk && ok; ++j) {
      // the tile's 4 mask words of query rows lane, lane+32, lane+64, lane+96
      uint4 w[4];
      uint32_t any = 0;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int row = lane + 32 * i;
        w[i] = make_uint4(0, 0, 0, 0);
        if (row < nq) w[i] = __ldg(reinterpret_cast<const uint4*>(km + (size_t)(q0 + row) * a.words) + j);
        any |= w[i].x | w[i].y | w[i].z | w[i].w;
      }
      if (!__any_sync(0xffffffffu, any != 0)) continue;
      // K stage use u = st * KPT + i goes to stage u % 2.  Info slot st % 4
      // is rewritten only after the QK of the tile before completed its
      // first K stage; that QK waited for the P.V of tile st-3, which
      // followed the softmax and the P.V of tile st-4 that read the slot.
      const int is = st & 3;
      const int kr = kv0 + j * BKV;   // first key row of the tile
      // keys past the request read the next request's rows (their mask bits
      // are zero) or, past the table, zeros
#pragma unroll
      for (int i = 0; i < C::KPT && ok; ++i) {
        const uint32_t u = nku;   // == st * KPT + i
        const int s = u & 1;
        if (!mbar_wait_warp(&bars[B_K_EMPTY + s], ((u >> 1) & 1) ^ 1, abort_flag, err)) { ok = false; break; }
        if (i == 0) {
#pragma unroll
          for (int m = 0; m < 4; ++m)
            reinterpret_cast<uint4*>(smem + C::OFF_MASK + is * BQ * 16)[lane + 32 * m] = w[m];
          if (lane == 0) stage_tile[is] = j;
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars[B_INFO + is]);
        }
        if (lane == 0) {
          mbar_arrive_expect_tx(&bars[B_K_FULL + s], C::K_BYTES);
          for (int c = 0; c < C::KSC; ++c) {
            const int cg = i * C::KSC + c;   // swizzle column of the head's key row
            const uint32_t dst = sbase + C::OFF_K + s * C::K_BYTES + c * (BKV * 128);
            if (cg < a.k_chunks)
              tma_load_3d(dst, &a.tmap_k, cg * 64, h, kr, &bars[B_K_FULL + s]);
            else   // shared RoPE columns
              tma_load_2d(dst, &a.tmap_kpe, (cg - a.k_chunks) * 64, kr, &bars[B_K_FULL + s]);
          }
        }
        ++nku;
      }
      if (!ok) break;
      ++st;
    }
    bool marked = false;
    if (ok) {
      // end marker (to the softmax through the info ring, to the MMA issuer
      // through a K stage without bytes)
      const int s = nku & 1;
      marked = mbar_wait_warp(&bars[B_K_EMPTY + s], ((nku >> 1) & 1) ^ 1, abort_flag, err);
      if (marked && lane == 0) {
        stage_tile[st & 3] = -1;
        mbar_arrive(&bars[B_INFO + (st & 3)]);
        mbar_arrive(&bars[B_K_FULL + s]);
      }
    }
    // Let copies still in flight land before the CTA can exit: q, and the
    // last data phase of each K stage barrier (counted by the uses issued,
    // so a tile whose loads stopped half way is covered too).  Once the end
    // marker is posted on K stage use nku, that barrier's data phase nku-2
    // was consumed already (and its parity now names the marker's successor
    // phase).
    if (lane == 0) {
      mbar_wait_drain(&bars[B_Q_FULL], 0, err);
      for (uint32_t i = (nku > 2 ? nku - 2 : 0); i < nku; ++i)
        if (!(marked && i + 2 == nku)) mbar_wait_drain(&bars[B_K_FULL + (i & 1)], (i >> 1) & 1, err);
    }
    __syncwarp();
  } else if (warp == 11) {
    // ------------------------------------------------------------------
    // V producer: the tile sequence comes through the info ring, so the K
    // stream (warp 9) runs ahead of the V stream.  It reads info slot n
    // before it can load V of tile n+1, which the P.V of tile n+1 needs
    // before slot n is rewritten for tile n+4.
    // ------------------------------------------------------------------
    uint32_t nvu = 0;   // V stage uses issued
    bool ok = true;
    for (uint32_t n = 0; ok; ++n) {
      const int is = n & 3;
      if (!mbar_wait_warp(&bars[B_INFO + is], (n >> 2) & 1, abort_flag, err)) break;
      const int tile = stage_tile[is];
      if (tile < 0) break;
      const int kr = kv0 + tile * BKV;
#pragma unroll
      for (int i = 0; i < C::VPT; ++i) {
        const uint32_t u = nvu;   // == n * VPT + i: keys i*VR .. of the tile
        const int s = u & 1;
        if (!mbar_wait_warp(&bars[B_V_EMPTY + s], ((u >> 1) & 1) ^ 1, abort_flag, err)) { ok = false; break; }
        if (lane == 0) {
          mbar_arrive_expect_tx(&bars[B_V_FULL + s], C::V_BYTES);
          for (int c = 0; c < C::VC; ++c)
            tma_load_3d(sbase + C::OFF_V + s * C::V_BYTES + c * (C::VR * 128), &a.tmap_v, c * 64, h, kr + i * C::VR,
                        &bars[B_V_FULL + s]);
        }
        ++nvu;
      }
    }
    if (lane == 0)
      for (uint32_t i = (nvu > 2 ? nvu - 2 : 0); i < nvu; ++i)
        mbar_wait_drain(&bars[B_V_FULL + (i & 1)], (i >> 1) & 1, err);
    __syncwarp();
  } else if (warp == 8) {
    // ------------------------------------------------------------------
    // QK issuer: S = Q K^T for each key tile as soon as its K stage landed
    // and its S buffer is free (the P.V of the tile two back completed)
    // ------------------------------------------------------------------
    if (lane == 0) {
      constexpr uint32_t IDESC_QK = idesc_bf16_f32(128, BKV, false, false);
      const uint32_t qs = sbase + C::OFF_Q;
      bool ok = mbar_wait(&bars[B_Q_FULL], 0, abort_flag, err);
      tc_fence_after();
      for (uint32_t n = 0; ok; ++n) {
        const int sb = n & 1;   // S buffer
        bool end = false;
#pragma unroll
        for (int i = 0; i < C::KPT; ++i) {
          const uint32_t u = n * C::KPT + i;   // K stage use
          const int s = u & 1;
          if (!mbar_wait(&bars[B_K_FULL + s], (u >> 1) & 1, abort_flag, err)) { ok = false; break; }
          tc_fence_after();
          if (i == 0) {
            if (stage_tile[n & 3] < 0) { end = true; break; }   // end marker
            if (!mbar_wait(&bars[B_S_EMPTY + sb], ((n >> 1) & 1) ^ 1, abort_flag, err)) { ok = false; break; }
            tc_fence_after();
          }
          const uint32_t ks = sbase + C::OFF_K + s * C::K_BYTES;
#pragma unroll
          for (int c = 0; c < C::KSC; ++c) {
            const int cq = i * C::KSC + c;
            mma_bf16_ss_x4(tmem + C::COL_S + sb * 128, sdesc_sw128(qs + cq * (BQ * 128), 16, 1024),
                           sdesc_sw128(ks + c * (BKV * 128), 16, 1024), 2u, 2u, IDESC_QK, cq > 0 ? 1u : 0u);
          }
          mma_commit(&bars[B_K_EMPTY + s]);
        }
        if (!ok || end) break;
        mma_commit(&bars[B_S_FULL + sb]);
      }
      mma_commit(&bars[B_DRAIN + 0]);
      mbar_wait(&bars[B_DRAIN + 0], 0, abort_flag, err);
    }
    __syncwarp();
  } else if (warp == 10) {
    // ------------------------------------------------------------------
    // P.V issuer: O += P V once the softmax packed P (bf16, in the S
    // columns) and the V stage landed; the tile sequence and its end come
    // through the info ring.  A thread of its own, so that the next tiles'
    // QK is never queued behind a wait for the softmax.
    // ------------------------------------------------------------------
    if (lane == 0) {
      constexpr uint32_t IDESC_PV = idesc_bf16_f32(128, DV, false, true);
      bool ok = true;
      for (uint32_t n = 0; ok; ++n) {
        const int sb = n & 1;   // S buffer holding P
        const int is = n & 3;
        if (!mbar_wait(&bars[B_INFO + is], (n >> 2) & 1, abort_flag, err)) break;
        if (stage_tile[is] < 0) break;   // end marker
        if (!mbar_wait(&bars[B_P_FULL], n & 1, abort_flag, err)) break;
#pragma unroll
        for (int i = 0; i < C::VPT; ++i) {
          const uint32_t u = n * C::VPT + i;   // V stage use: keys i*VR .. of the tile
          const int s = u & 1;
          if (!mbar_wait(&bars[B_V_FULL + s], (u >> 1) & 1, abort_flag, err)) { ok = false; break; }
          tc_fence_after();
          const uint32_t vs = sbase + C::OFF_V + s * C::V_BYTES;
          // 64 keys per x4 batch: P columns (bf16 pairs) of those keys, V rows of those keys
#pragma unroll
          for (int g = 0; g < C::VR / 64; ++g)
            mma_bf16_ts_x4(tmem + C::COL_O, tmem + C::COL_S + sb * 128 + (i * C::VR + g * 64) / 2,
                           sdesc_sw128(vs + g * 64 * 128, C::VR * 128, 1024), 8u, 128u, IDESC_PV,
                           (n > 0 || i > 0 || g > 0) ? 1u : 0u);
          mma_commit(&bars[B_V_EMPTY + s]);
        }
        if (!ok) break;
        mma_commit(&bars[B_PV_DONE]);
        mma_commit(&bars[B_S_EMPTY + sb]);
      }
      mma_commit(&bars[B_DRAIN + 1]);
      mbar_wait(&bars[B_DRAIN + 1], 0, abort_flag, err);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------
    // softmax + epilogue: two threads per query row (TMEM lane); this one
    // holds keys 64*half .. 64*half+63 of every tile and output columns
    // (DV/2)*half .. of the row
    // ------------------------------------------------------------------
    const int half = warp >> 2;
    const int row = (warp & 3) * 32 + lane;
    const float sl2 = a.scale * 1.4426950408889634f;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    float* pair = reinterpret_cast<float*>(smem + C::OFF_PAIR);   // [parity][half][row]
    uint64_t* pair_bar = &bars[B_PAIR + (warp & 3)];
    uint32_t pair_phase = 0;
    float m_run = -INFINITY, l_run = 0.f;
    uint32_t n = 0;
    bool ok = true;
    while (true) {
      const int s = n & 1;
      const int is = n & 3;
      if (!mbar_wait_warp(&bars[B_INFO + is], (n >> 2) & 1, abort_flag, err)) { ok = false; break; }
      const int tile = stage_tile[is];
      if (tile < 0) break;
      const uint4 mw = reinterpret_cast<const uint4*>(smem + C::OFF_MASK + is * BQ * 16)[row];
      const uint32_t mwords[2] = {half ? mw.z : mw.x, half ? mw.w : mw.y};
      if (!mbar_wait_warp(&bars[B_S_FULL + s], (n >> 1) & 1, abort_flag, err)) { ok = false; break; }
      tc_fence_after();
      float sv[HK];
#pragma unroll
      for (int c = 0; c < HK; c += 16) tmem_ld16(tmem + lane_off + C::COL_S + s * 128 + HK * half + c, sv + c);
      tmem_ld_wait();
      float hmax = -INFINITY;
#pragma unroll
      for (int c = 0; c < HK; ++c) {
        const bool on = (mwords[c >> 5] >> (c & 31)) & 1u;
        sv[c] = on ? sv[c] : -INFINITY;
        hmax = fmaxf(hmax, sv[c]);
      }
      // the row max of both halves (raw scores; the scale is applied in the exponent)
      pair[((n & 1) * 2 + half) * BQ + row] = hmax;
      if (!group_sync(pair_bar, pair_phase, abort_flag, err)) { ok = false; break; }
      const float omax = pair[((n & 1) * 2 + (half ^ 1)) * BQ + row];
      const float tmax = (half == 0 ? fmaxf(hmax, omax) : fmaxf(omax, hmax)) * sl2;
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
        for (int c = (DV / 2) * half; c < (DV / 2) * (half + 1); c += 16) {
          float o[16];
          tmem_ld16(tmem + lane_off + C::COL_O + c, o);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i) o[i] *= alpha;
          tmem_st16(tmem + lane_off + C::COL_O + c, o);
        }
      }
      const float mref = (m_run == -INFINITY) ? 0.f : m_run;
#pragma unroll
      for (int c = 0; c < HK; c += 32) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          pk[i] = pack_bf16x2(exp2f(fmaf(sv[c + 2 * i], sl2, -mref)), exp2f(fmaf(sv[c + 2 * i + 1], sl2, -mref)));
          l_run += __uint_as_float(pk[i] << 16) + __uint_as_float(pk[i] & 0xffff0000u);
        }
        tmem_st16_u32(tmem + lane_off + C::COL_S + s * 128 + (HK * half + c) / 2, pk);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bars[B_P_FULL]);
      ++n;
    }
    // epilogue
    if (ok) {
      const int t = q0 + row;
      // the row sum of both halves (pair slot of parity n: last read before barrier n-1)
      pair[((n & 1) * 2 + half) * BQ + row] = l_run;
      const bool synced = group_sync(pair_bar, pair_phase, abort_flag, err);
      const float lsum = pair[(n & 1) * 2 * BQ + row] + pair[((n & 1) * 2 + 1) * BQ + row];
      if (synced && n > 0) {
        const bool got = mbar_wait_warp(&bars[B_PV_DONE], (n - 1) & 1, abort_flag, err);
        tc_fence_after();
        if (got) {
          const float inv_l = (lsum > 0.f) ? 1.f / lsum : 0.f;
#pragma unroll 1
          for (int c = (DV / 2) * half; c < (DV / 2) * (half + 1); c += 16) {
            float o[16];
            tmem_ld16(tmem + lane_off + C::COL_O + c, o);
            tmem_ld_wait();
            if (row < nq) {
              uint32_t pk[8];
#pragma unroll
              for (int i = 0; i < 8; ++i) pk[i] = pack_bf16x2(o[2 * i] * inv_l, o[2 * i + 1] * inv_l);
              uint4* dst = reinterpret_cast<uint4*>(a.out + ((size_t)t * a.H + h) * DV + c);
              dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
              dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
            }
          }
        }
      } else if (synced && row < nq) {
        uint4* dst = reinterpret_cast<uint4*>(a.out + ((size_t)t * a.H + h) * DV + (DV / 2) * half);
        for (int c = 0; c < DV / 16; ++c) dst[c] = make_uint4(0, 0, 0, 0);
      }
      if (synced && half == 0 && row < nq)
        a.lse[(size_t)t * a.H + h] = (lsum > 0.f) ? (m_run + log2f(lsum)) * 0.6931471805599453f : -INFINITY;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 8) tmem_dealloc(tmem, C::TMEM_COLS);
}

template <int DQK, int DV>
static int launch_t(const MaskedArgs& a, cudaStream_t stream) {
  static_assert(Cfg<DQK, DV>::SMEM_BYTES <= 227u * 1024u, "shared memory budget");
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
  if (a.d_qk == 256 && a.d_v == 256) return masked::launch_t<256, 256>(a, stream);
  return -2;
}

}  // namespace dsa
