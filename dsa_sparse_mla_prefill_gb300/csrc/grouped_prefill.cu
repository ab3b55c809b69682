// Grouped sparse MLA prefill for sm_103a.
//
// "[Perf][DSA] Grouped sparse prefill with the FlashMLA head-group-mask
// kernel", commit message and How: the G = 128/H consecutive tokens of a
// group of one request act as 128 pseudo-heads p = j*H + h that attend over
// the sorted union of their top-k rows; the per-token membership mask keeps
// pseudo-head p on the union slots whose bit j is set, so every token sees
// exactly its own top-k and the result equals the per-token form while each
// union row is gathered once per group instead of once per token.
//
// Sizing on one SM does not fit: q for 128 pseudo-heads is 147 KB and the
// 128 x 512 fp32 accumulator alone fills the 512 TMEM columns.  So a group is
// processed by a cluster of two CTAs that split the latent columns:
//   CTA 0 owns NoPE columns 0-255 (+ the 64 RoPE columns), CTA 1 owns NoPE
//   columns 256-511.  Each gathers only its columns of every union row (no
//   row is fetched twice), holds its q columns in shared memory, computes a
//   partial S = q_own . K_own^T (M = 128 pseudo-heads, N = 64 union slots)
//   and keeps its half of O (128 x 256 fp32 = 256 TMEM columns).
//   Partial scores are exchanged over distributed shared memory: CTA r
//   finishes pseudo-heads [64r, 64r+64), receiving the peer's partial rows
//   for them; it applies the mask byte, runs the online softmax (base 2,
//   lazy rescale), writes the bf16 P rows into both CTAs' P tiles and sends
//   the rescale factors, so both halves of O are updated with the same P.
//   Then each CTA issues O_own += P . V_own (N = 256) from its own V columns.
// Warp roles per CTA: warps 0-3 softmax (thread i <-> pseudo-head i <-> TMEM
// lane i; "owner" warps hold this CTA's rows, the others relay the peer's
// rows), warp 4 the tcgen05 issuer, warps 5-6 cp.async gathers.
#include "dsa_device.cuh"
#include "dsa_kernels.h"

namespace dsa {
namespace grouped {

constexpr int BK = 64;          // union slots per tile (the MMA's N for S)
constexpr int NTHREADS = 224;   // 7 warps (keeps the full 255-register budget)
constexpr int NPROD = 64;       // producer threads (warps 5-6)
constexpr int LAG = 2;
constexpr float kTau = 8.0f;

template <int NC>
struct Cfg {
  static constexpr int OWN0 = (NC == 9) ? 5 : 4;   // swizzle columns held by rank 0
  static constexpr int OWNMAX = OWN0;
  static constexpr uint32_t Q_BYTES = OWNMAX * 128u * 128u;
  static constexpr uint32_t KV_CHUNK = BK * 128u;            // 64 keys x 64 cols
  static constexpr uint32_t KV_BYTES = OWNMAX * KV_CHUNK;
  static constexpr uint32_t P_BYTES = 128u * BK * 2u;        // 128 rows x 64 keys, one swizzle column
  static constexpr uint32_t SX_BYTES = 64u * BK * 4u;        // 64 rows x 64 fp32
  static constexpr uint32_t OFF_Q = 0;
  static constexpr uint32_t OFF_KV = OFF_Q + Q_BYTES;        // [2]
  static constexpr uint32_t OFF_P = OFF_KV + 2 * KV_BYTES;   // [2]
  static constexpr uint32_t OFF_SX = OFF_P + 2 * P_BYTES;    // [2]
  static constexpr uint32_t OFF_MASKB = OFF_SX + 2 * SX_BYTES;   // [2][64] bytes
  static constexpr uint32_t OFF_ALPHA = OFF_MASKB + 128u;        // [2][64] floats
  static constexpr uint32_t OFF_FIN = OFF_ALPHA + 512u;          // [64] floats
  static constexpr uint32_t OFF_BAR = OFF_FIN + 256u;
  static constexpr int NBAR = 24;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8u;
  static constexpr uint32_t SMEM_BYTES = OFF_MISC + 64u + 1024u;
  static constexpr uint32_t COL_O = 0;       // 256 columns
  static constexpr uint32_t COL_S = 256;     // [2] x 64 columns
  static constexpr uint32_t TMEM_COLS = 512;
};

enum {
  B_Q_FULL = 0,
  B_Q_EMPTY = 1,
  B_KV_FULL = 2,     // [2]
  B_KV_EMPTY = 4,    // [2]
  B_S_FULL = 6,      // [2]
  B_S_EMPTY = 8,     // [2]
  B_SX_FULL = 10,    // [2] peer relays wrote my rows' partial scores
  B_SX_EMPTY = 12,   // [2] peer owners consumed what I wrote into their buffer
  B_ALPHA_FULL = 14, // [2] peer owners wrote rescale factors for the rows I relay
  B_P_FULL = 16,     // [2] own P rows + peer P rows + relayed rescale done
  B_PV_DONE = 18,
  B_O_EMPTY = 19,
  B_FIN_FULL = 20,
  B_DRAIN = 21,
};

// latent swizzle column held at position c by CTA `rank`
__device__ __forceinline__ int latent_chunk(int rank, int c) { return rank == 0 ? (c < 4 ? c : 8) : 4 + c; }

__device__ __forceinline__ void group_of(const ReqTable& rq, int G, int g, int& t0, int& n) {
  int r = 0;
  while (r + 1 < rq.num_req && rq.cu_g[r + 1] <= g) ++r;
  t0 = rq.cu_q[r] + (g - rq.cu_g[r]) * G;
  n = min(G, rq.cu_q[r + 1] - t0);
}

template <int NC>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NTHREADS, 1) grouped_prefill_kernel(GroupedArgs a) {
  using C = Cfg<NC>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_u32 + 1023u) & ~1023u) - raw_u32);
  const uint32_t sbase = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile uint32_t* tmem_base_ptr = misc;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 1);
  unsigned int* err = a.err;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int rank = (int)cluster_ctarank();
  const int peer = rank ^ 1;
  const int nown = (rank == 0) ? C::OWN0 : 4;
  const int H = a.H;
  const int G = a.G;
  const int d_qk = a.d_qk;
  const int cid = (int)cluster_id_x();
  const int ncl = (int)nclusters_x();

  if (threadIdx.x == 0) {
    mbar_init(&bars[B_Q_FULL], NPROD);
    mbar_init(&bars[B_Q_EMPTY], 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars[B_KV_FULL + i], NPROD);
      mbar_init(&bars[B_KV_EMPTY + i], 1);
      mbar_init(&bars[B_S_FULL + i], 1);
      mbar_init(&bars[B_S_EMPTY + i], 128);
      mbar_init(&bars[B_SX_FULL + i], 64);
      mbar_init(&bars[B_SX_EMPTY + i], 64);
      mbar_init(&bars[B_ALPHA_FULL + i], 64);
      mbar_init(&bars[B_P_FULL + i], 192);
    }
    mbar_init(&bars[B_PV_DONE], 1);
    mbar_init(&bars[B_O_EMPTY], 128);
    mbar_init(&bars[B_FIN_FULL], 64);
    mbar_init(&bars[B_DRAIN], 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 4) {
    tmem_alloc(const_cast<uint32_t*>(tmem_base_ptr), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // the peer's barriers exist before anyone arrives on them
  tc_fence_after();
  const uint32_t tmem = *tmem_base_ptr;

  if (warp >= 5) {
    // ------------------------------------------------------------------
    // producers: own columns of q and of every union row
    // ------------------------------------------------------------------
    const int ptid = threadIdx.x - 160;
    const int p8 = ptid & 7;
    const int rsub = ptid >> 3;
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
    uint32_t gt = 0, lgq = 0;
    bool ok = true;
    for (int g = cid; g < a.num_groups && ok; g += ncl) {
      int t0, n;
      group_of(a.req, G, g, t0, n);
      const int U = min(__ldg(a.union_len + g), a.union_pad);
      const int ntiles = (U + BK - 1) / BK;
      if (ntiles == 0) continue;
      const int nrows = n * H;
      if (!wait_free(&bars[B_Q_EMPTY], (lgq & 1) ^ 1)) { ok = false; break; }
      {
        const uint32_t qs = sbase + C::OFF_Q;
        for (int pass = 0; pass < 16 * nown; ++pass) {
          const int row = (pass & 15) * 8 + rsub;
          const int c = pass >> 4;
          const bool valid = row < nrows;
          const uint16_t* src = a.q + (size_t)(valid ? t0 * H + row : 0) * d_qk + latent_chunk(rank, c) * 64 + p8 * 8;
          cp_async16(qs + c * (128 * 128) + row * 128 + ((p8 ^ (row & 7)) << 4), src, valid ? 16u : 0u);
        }
        push(&bars[B_Q_FULL]);
      }
      const int32_t* urow = a.union_idx + (size_t)g * a.union_pad;
      const uint8_t* mrow = a.mask + (size_t)g * a.union_pad;
      for (int j = 0; j < ntiles; ++j, ++gt) {
        const int s = gt & 1;
        if (!wait_free(&bars[B_KV_EMPTY + s], ((gt >> 1) & 1) ^ 1)) { ok = false; break; }
        if (ptid == 0) DSA_TRACE(a.tr, gt, 0);
        if (ptid < BK) {
          const int u = j * BK + ptid;
          smem[C::OFF_MASKB + s * 64 + ptid] = (u < U) ? __ldg(mrow + u) : (uint8_t)0;
        }
        int kr[8];
        bool kv_ok[8];
#pragma unroll
        for (int rb = 0; rb < 8; ++rb) {
          const int u = j * BK + rb * 8 + rsub;
          const int x = (u < U) ? __ldg(urow + u) : -1;
          kv_ok[rb] = (x >= 0) && (x < a.N);
          kr[rb] = kv_ok[rb] ? x : 0;
        }
        const uint32_t kvs = sbase + C::OFF_KV + s * C::KV_BYTES;
        for (int c = 0; c < nown; ++c) {
          const int lc = latent_chunk(rank, c);
#pragma unroll
          for (int rb = 0; rb < 8; ++rb) {
            const int row = rb * 8 + rsub;
            const uint16_t* src = a.kv + (size_t)kr[rb] * a.ld_kv + lc * 64 + p8 * 8;
            cp_async16(kvs + c * C::KV_CHUNK + row * 128 + ((p8 ^ (row & 7)) << 4), src, kv_ok[rb] ? 16u : 0u);
          }
        }
        push(&bars[B_KV_FULL + s]);
      }
      ++lgq;
    }
    flush();
  } else if (warp == 4) {
    // ------------------------------------------------------------------
    // tcgen05 issuer
    // ------------------------------------------------------------------
    if (lane == 0) {
      constexpr uint32_t IDESC_QK = idesc_bf16_f32(128, BK, false, false);
      constexpr uint32_t IDESC_PV = idesc_bf16_f32(128, 256, false, true);
      const uint32_t qs = sbase + C::OFF_Q;
      uint32_t gt = 0, lgq = 0;
      bool ok = true;
      auto qk_ready = [&](uint32_t i) -> bool {
        const int s = i & 1;
        return mbar_ready(&bars[B_KV_FULL + s], (i >> 1) & 1) && mbar_ready(&bars[B_S_EMPTY + s], ((i >> 1) & 1) ^ 1);
      };
      auto issue_qk = [&](uint32_t i, bool last) {
        const int s = i & 1;
        DSA_TRACE(a.tr, i, 2);
        tc_fence_after();
        const uint32_t kvs = sbase + C::OFF_KV + s * C::KV_BYTES;
        for (int c = 0; c < nown; ++c)
          mma_bf16_ss_x4(tmem + C::COL_S + s * BK, sdesc_sw128(qs + c * (128 * 128), 16, 1024),
                         sdesc_sw128(kvs + c * C::KV_CHUNK, 16, 1024), 2u, 2u, IDESC_QK, c > 0 ? 1u : 0u);
        mma_commit(&bars[B_S_FULL + s]);
        if (last) mma_commit(&bars[B_Q_EMPTY]);
        DSA_TRACE(a.tr, i, 1);
      };
      auto issue_pv = [&](uint32_t i, int j) {
        DSA_TRACE(a.tr, i, 7);
        tc_fence_after();
        const uint32_t ps = sbase + C::OFF_P + (i & 1) * C::P_BYTES;
        const uint32_t kvs = sbase + C::OFF_KV + (i & 1) * C::KV_BYTES;
        // 64 union slots = 4 MMAs of 16: P advances 32 B, V (MN-major) 2048 B
        mma_bf16_ss_x4(tmem + C::COL_O, sdesc_sw128(ps, 16, 1024), sdesc_sw128(kvs, C::KV_CHUNK, 1024), 2u, 128u,
                       IDESC_PV, j > 0 ? 1u : 0u);
        mma_commit(&bars[B_PV_DONE]);
        mma_commit(&bars[B_KV_EMPTY + (i & 1)]);
      };
      for (int g = cid; g < a.num_groups && ok; g += ncl) {
        const int U = min(__ldg(a.union_len + g), a.union_pad);
        const int ntiles = (U + BK - 1) / BK;
        if (ntiles == 0) continue;
        if (!mbar_wait(&bars[B_Q_FULL], lgq & 1, abort_flag, err)) { ok = false; break; }
        tc_fence_after();
        // issue whichever of QK(next) / PV(oldest) is ready first; QK runs at
        // most one tile ahead, which keeps every P buffer's previous P.V ahead
        // of the QK whose scores allow that buffer to be written again
        int nq = 0, np = 0;
        uint64_t t_last = globaltimer();
        while (np < ntiles) {
          bool progressed = false;
          if (nq < ntiles && nq <= np + 1 && qk_ready(gt + nq)) {
            issue_qk(gt + nq, nq == ntiles - 1);
            ++nq;
            progressed = true;
          }
          // P rows arrive from both CTAs: acquire at cluster scope
          if (np < nq && mbar_ready_cluster(&bars[B_P_FULL + ((gt + np) & 1)], ((gt + np) >> 1) & 1) &&
              (np > 0 || mbar_ready(&bars[B_O_EMPTY], (lgq & 1) ^ 1))) {
            issue_pv(gt + np, np);
            ++np;
            progressed = true;
          }
          if (progressed) {
            t_last = globaltimer();
          } else if (*abort_flag) {
            ok = false;
            break;
          } else if (globaltimer() - t_last > kWaitTimeoutNs) {
            *abort_flag = 1;
            atomicAdd(err + ERR_TIMEOUT, 1u);
            ok = false;
            break;
          }
        }
        if (!ok) break;
        gt += ntiles;
        ++lgq;
      }
      mma_commit(&bars[B_DRAIN]);
      mbar_wait(&bars[B_DRAIN], 0, abort_flag, err);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------
    // softmax warps: owners finish their pseudo-heads, relays serve the peer
    // ------------------------------------------------------------------
    const int row = threadIdx.x;             // pseudo-head = TMEM lane
    const bool owner = (warp >> 1) == rank;
    const int lrow = row & 63;               // row inside its owner's block
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    const float sl2 = a.scale * 1.4426950408889634f;
    const int tok = row / H;                 // token of the group this pseudo-head belongs to
    const uint32_t sx_local = sbase + C::OFF_SX;
    const uint32_t sx_peer = map_peer(sx_local, peer);
    const uint32_t p_local = sbase + C::OFF_P;
    const uint32_t p_peer = map_peer(p_local, peer);
    const uint32_t alpha_peer = map_peer(sbase + C::OFF_ALPHA, peer);
    const uint32_t fin_peer = map_peer(sbase + C::OFF_FIN, peer);
    const uint32_t bar_base = smem_u32(bars);
    auto peer_bar = [&](int idx) { return map_peer(bar_base + idx * 8, peer); };
    uint32_t gt = 0, lgq = 0;
    bool ok = true;
    for (int g = cid; g < a.num_groups && ok; g += ncl) {
      int t0, n;
      group_of(a.req, G, g, t0, n);
      const int U = min(__ldg(a.union_len + g), a.union_pad);
      const int ntiles = (U + BK - 1) / BK;
      const int nrows = n * H;
      uint16_t* out_row = a.out + (size_t)(t0 * H + row) * 512 + 256 * rank;
      if (ntiles == 0) {
        if (row < nrows) {
          for (int c = 0; c < 32; ++c) reinterpret_cast<uint4*>(out_row)[c] = make_uint4(0, 0, 0, 0);
          if (owner) a.lse[(size_t)t0 * H + row] = -INFINITY;
        }
        continue;
      }
      float m_run = -INFINITY, l_run = 0.f;
      for (int j = 0; j < ntiles; ++j) {
        const uint32_t i = gt + j;
        const int sb = i & 1;
        const uint32_t ph = (i >> 1) & 1;
        if (!mbar_wait_warp(&bars[B_S_FULL + sb], ph, abort_flag, err)) { ok = false; break; }
        if (row == 0) DSA_TRACE(a.tr, i, 3);
        tc_fence_after();
        float sv[BK];
#pragma unroll
        for (int c = 0; c < BK; c += 16) tmem_ld16(tmem + lane_off + C::COL_S + sb * BK + c, sv + c);
        tmem_ld_wait();
        tc_fence_before();
        mbar_arrive(&bars[B_S_EMPTY + sb]);
        if (!owner) {
          // relay: partial scores of the peer's row to the peer
          if (!mbar_wait_cluster_warp(&bars[B_SX_EMPTY + sb], ph ^ 1, abort_flag, err)) { ok = false; break; }
          const uint32_t dst = sx_peer + sb * C::SX_BYTES + lrow * (BK * 4);
#pragma unroll
          for (int c = 0; c < 16; ++c)
            st_cluster_v4(dst + ((c ^ (lrow & 15)) << 4), __float_as_uint(sv[4 * c]), __float_as_uint(sv[4 * c + 1]),
                          __float_as_uint(sv[4 * c + 2]), __float_as_uint(sv[4 * c + 3]));
          mbar_arrive_remote(peer_bar(B_SX_FULL + sb));
          // the owner's rescale factor for this row, applied to my half of O
          if (!mbar_wait_cluster_warp(&bars[B_ALPHA_FULL + sb], ph, abort_flag, err)) { ok = false; break; }
          if (row == 0) DSA_TRACE(a.tr, i, 4);
          const float alpha = reinterpret_cast<volatile float*>(smem + C::OFF_ALPHA)[sb * 64 + lrow];
          if (j > 0 && __any_sync(0xffffffffu, alpha != 1.0f)) {
            if (!mbar_wait_warp(&bars[B_PV_DONE], (i - 1) & 1, abort_flag, err)) { ok = false; break; }
            tc_fence_after();
#pragma unroll 1
            for (int c = 0; c < 256; c += 16) {
              float o[16];
              tmem_ld16(tmem + lane_off + C::COL_O + c, o);
              tmem_ld_wait();
#pragma unroll
              for (int e = 0; e < 16; ++e) o[e] *= alpha;
              tmem_st16(tmem + lane_off + C::COL_O + c, o);
            }
            tmem_st_wait();
          }
          tc_fence_before();
          mbar_arrive(&bars[B_P_FULL + sb]);
          if (row == 0) DSA_TRACE(a.tr, i, 5);
          if (row == 0) DSA_TRACE(a.tr, i, 6);
        } else {
          // owner: complete the scores with the peer's partial row
          if (!mbar_wait_cluster_warp(&bars[B_SX_FULL + sb], ph, abort_flag, err)) { ok = false; break; }
          if (row == 0) DSA_TRACE(a.tr, i, 4);
          const uint8_t* sxr = smem + C::OFF_SX + sb * C::SX_BYTES + lrow * (BK * 4);
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            const float4 x = *reinterpret_cast<const float4*>(sxr + ((c ^ (lrow & 15)) << 4));
            sv[4 * c] += x.x;
            sv[4 * c + 1] += x.y;
            sv[4 * c + 2] += x.z;
            sv[4 * c + 3] += x.w;
          }
          mbar_arrive_remote(peer_bar(B_SX_EMPTY + sb));
          // the producers' mask bytes of this stage (the phase cannot have moved on:
          // the stage is only released after this tile's P.V)
          if (!mbar_wait_warp(&bars[B_KV_FULL + sb], ph, abort_flag, err)) { ok = false; break; }
          if (row == 0) DSA_TRACE(a.tr, i, 5);
          const uint8_t* mb = smem + C::OFF_MASKB + sb * 64;
          float tmax = -INFINITY;
#pragma unroll
          for (int c = 0; c < BK; ++c) {
            const bool on = (mb[c] >> tok) & 1;
            sv[c] = on ? sv[c] * sl2 : -INFINITY;
            tmax = fmaxf(tmax, sv[c]);
          }
          float alpha = 1.f;
          const bool need = tmax > m_run + kTau;
          if (need) {
            const float mn = fmaxf(m_run, tmax);
            alpha = (m_run == -INFINITY) ? 0.f : exp2f(m_run - mn);
            m_run = mn;
            l_run *= alpha;
          }
          st_cluster_f32(alpha_peer + (sb * 64 + lrow) * 4, alpha);
          mbar_arrive_remote(peer_bar(B_ALPHA_FULL + sb));
          if (j > 0 && __any_sync(0xffffffffu, need)) {
            if (!mbar_wait_warp(&bars[B_PV_DONE], (i - 1) & 1, abort_flag, err)) { ok = false; break; }
            tc_fence_after();
#pragma unroll 1
            for (int c = 0; c < 256; c += 16) {
              float o[16];
              tmem_ld16(tmem + lane_off + C::COL_O + c, o);
              tmem_ld_wait();
#pragma unroll
              for (int e = 0; e < 16; ++e) o[e] *= alpha;
              tmem_st16(tmem + lane_off + C::COL_O + c, o);
            }
            tmem_st_wait();
          }
          const float mref = (m_run == -INFINITY) ? 0.f : m_run;
          const uint32_t prow_off = sb * C::P_BYTES + row * 128;
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            uint32_t pk[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const uint16_t b0 = f32_to_bf16_rn(exp2f(sv[8 * c + 2 * e] - mref));
              const uint16_t b1 = f32_to_bf16_rn(exp2f(sv[8 * c + 2 * e + 1] - mref));
              l_run += bf16_to_f32(b0) + bf16_to_f32(b1);
              pk[e] = (uint32_t)b0 | ((uint32_t)b1 << 16);
            }
            const uint32_t off = prow_off + ((c ^ (row & 7)) << 4);
            *reinterpret_cast<uint4*>(smem + C::OFF_P + off) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            st_cluster_v4(p_peer + off, pk[0], pk[1], pk[2], pk[3]);
          }
          fence_proxy_async_smem();
          fence_proxy_async_cluster();
          tc_fence_before();
          mbar_arrive(&bars[B_P_FULL + sb]);
          mbar_arrive_remote(peer_bar(B_P_FULL + sb));
          if (row == 0) DSA_TRACE(a.tr, i, 6);
        }
      }
      if (!ok) break;
      // ---- epilogue: normalise this CTA's half of O for all 128 rows ----
      float inv_l;
      if (owner) {
        inv_l = (l_run > 0.f) ? 1.f / l_run : 0.f;
        if (row < nrows)
          a.lse[(size_t)t0 * H + row] = (l_run > 0.f) ? (m_run + log2f(l_run)) * 0.6931471805599453f : -INFINITY;
        st_cluster_f32(fin_peer + lrow * 4, inv_l);
        mbar_arrive_remote(peer_bar(B_FIN_FULL));
      } else {
        if (!mbar_wait_cluster_warp(&bars[B_FIN_FULL], lgq & 1, abort_flag, err)) { ok = false; break; }
        inv_l = reinterpret_cast<volatile float*>(smem + C::OFF_FIN)[lrow];
      }
      if (!mbar_wait_warp(&bars[B_PV_DONE], (gt + ntiles - 1) & 1, abort_flag, err)) { ok = false; break; }
      tc_fence_after();
#pragma unroll 1
      for (int c = 0; c < 256; c += 16) {
        float o[16];
        tmem_ld16(tmem + lane_off + C::COL_O + c, o);
        tmem_ld_wait();
        if (row < nrows) {
          uint32_t pk[8];
#pragma unroll
          for (int e = 0; e < 8; ++e)
            pk[e] = (uint32_t)f32_to_bf16_rn(o[2 * e] * inv_l) | ((uint32_t)f32_to_bf16_rn(o[2 * e + 1] * inv_l) << 16);
          uint4* dst = reinterpret_cast<uint4*>(out_row + c);
          dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
          dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
        }
      }
      tc_fence_before();
      mbar_arrive(&bars[B_O_EMPTY]);
      gt += ntiles;
      ++lgq;
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // no CTA leaves while its peer may still write into it
  tc_fence_after();
  if (warp == 4) tmem_dealloc(tmem, C::TMEM_COLS);
}

template <int NC>
static int launch_t(const GroupedArgs& a, int num_sms, cudaStream_t stream) {
  using C = Cfg<NC>;
  static int attr_set[64] = {0};
  static int max_clusters[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set[dev]) {
    if (cudaFuncSetAttribute(grouped_prefill_kernel<NC>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::SMEM_BYTES) != cudaSuccess)
      return -1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * (num_sms / 2), 1, 1);
    cfg.blockDim = dim3(NTHREADS, 1, 1);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = 2;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, grouped_prefill_kernel<NC>, &cfg) != cudaSuccess || n < 1) {
      cudaGetLastError();
      n = num_sms / 2;
    }
    max_clusters[dev] = n;
    attr_set[dev] = 1;
  }
  if (a.num_groups == 0) return 0;
  int ncl = dev < 64 ? max_clusters[dev] : num_sms / 2;
  if (ncl > a.num_groups) ncl = a.num_groups;
  grouped_prefill_kernel<NC><<<2 * ncl, NTHREADS, C::SMEM_BYTES, stream>>>(a);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace grouped

int launch_grouped_prefill(const GroupedArgs& a, int num_sms, cudaStream_t stream) {
  if (a.d_qk == 576) return grouped::launch_t<9>(a, num_sms, stream);
  if (a.d_qk == 512) return grouped::launch_t<8>(a, num_sms, stream);
  return -2;
}

}  // namespace dsa
