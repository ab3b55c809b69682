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
// One SM cannot hold it: q for 128 pseudo-heads is 147 KB and the 128 x 512
// fp32 accumulator alone fills the 512 TMEM columns.  So a group is processed
// by a cluster of two CTAs that split the latent columns:
//   CTA 0 owns NoPE columns 0-255 (+ the 64 RoPE columns), CTA 1 owns NoPE
//   columns 256-511.  Each gathers only its columns of every union row (no
//   row is fetched twice), holds its q columns in tensor memory, computes a
//   partial S_r = q_own . K_own^T (M = 128 pseudo-heads, N = 64 union slots,
//   A read from TMEM) and keeps its half of O (128 x 256 fp32).
// TMEM per CTA: O 256 columns, q 160 (bf16 pairs), S 64, P 32 = 512.
// Per tile the two CTAs swap their partial scores once over distributed
// shared memory (thread p sends row p, 256 bytes, with st.async counting the
// bytes on the peer's barrier) and both add them in the same order, so both
// hold the same full S and run the same online softmax (base 2, lazy
// rescale) on all 128 rows: P, the running max and the running sum agree bit
// for bit without further exchange.  Each CTA then issues O_own += P . V_own
// with P (bf16) read from tensor memory (N = 256).  The softmax threads send
// the scores of tile j+1 before finishing tile j, so the exchange latency
// overlaps the softmax.
// Warp roles per CTA (16 warps): warps 0-7 softmax, two threads per
// pseudo-head: warp w holds TMEM lanes 32(w%4) .. +31 (pseudo-head p =
// lane) and slots 32(w/4) .. +31 of each 64-slot tile; the two halves of a
// row agree on the running max through a per-tile pair exchange (in the
// already consumed half of the row's SX buffer).  They also load q per group into TMEM.  Warp 8 issues QK, warp 9
// issues PV, warps 10-15 issue the TMA row gathers (tile::gather4, 4 rows x
// 128 bytes each) into a 4-stage ring.  Warps 0-7 run at 168 registers, the
// others at 88.
#include "dsa_device.cuh"
#include "dsa_kernels.h"

namespace dsa {
namespace grouped {

constexpr int BK = 64;          // union slots per tile (the MMA's N for S)
constexpr int NTHREADS = 512;   // 16 warps, launched at 128 registers each
constexpr int REGS_SOFTMAX = 168;
constexpr int REGS_OTHER = 88;  // 8*32*168 + 8*32*88 = 512*128
constexpr int NSTAGE = 4;       // gather ring depth
constexpr int NPROD_WARPS = 6;
constexpr float kTau = 8.0f;    // lazy-rescale threshold (log2 units)

template <int NC>
struct Cfg {
  static constexpr int OWN0 = (NC == 9) ? 5 : 4;   // swizzle columns held by rank 0
  static constexpr int OWNMAX = OWN0;
  static constexpr uint32_t KV_CHUNK = BK * 128u;            // 64 keys x 64 cols
  static constexpr uint32_t KV_BYTES = OWNMAX * KV_CHUNK;
  static constexpr uint32_t SX_BYTES = 128u * BK * 4u;       // 128 rows x 64 fp32 (the peer's partial S)
  static constexpr uint32_t OFF_KV = 0;                      // [NSTAGE]
  static constexpr uint32_t OFF_SX = OFF_KV + NSTAGE * KV_BYTES;  // [2]
  static constexpr uint32_t OFF_MASKB = OFF_SX + 2 * SX_BYTES;    // [NSTAGE][64] bytes
  static constexpr uint32_t OFF_BAR = OFF_MASKB + NSTAGE * 64u;
  static constexpr int NBAR = 24;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8u;
  static constexpr uint32_t SMEM_BYTES = OFF_MISC + 64u + 1024u;
  static_assert(SMEM_BYTES <= 227u * 1024u, "shared memory budget");
  static constexpr uint32_t COL_O = 0;       // 256 columns
  static constexpr uint32_t COL_Q = 256;     // OWNMAX * 32 columns (bf16 pairs)
  static constexpr uint32_t COL_S = 416;     // 64 columns
  static constexpr uint32_t COL_P = 480;     // 32 columns (bf16 pairs)
  static constexpr uint32_t TMEM_COLS = 512;
};

enum {
  B_Q_FULL = 0,      // q of the group in TMEM (256 arrivals)
  B_KV_FULL = 1,     // [NSTAGE] union rows + mask bytes of the stage landed
  B_KV_EMPTY = 5,    // [NSTAGE] P.V of the stage's tile completed
  B_S_FULL = 9,      // partial S in TMEM
  B_S_EMPTY = 10,    // the softmax threads read S
  B_SX_FULL = 11,    // [2] the peer's partial S landed in my SX buffer (byte count)
  B_SX_FREE = 13,    // [2] the peer read what I wrote into its SX buffer
  B_P_FULL = 15,     // P rows in TMEM (and any O rescale done)
  B_PV_DONE = 16,    // P.V completed (P columns free, O up to date)
  B_O_EMPTY = 17,
  B_DRAIN = 18,      // [2] one per MMA issuer
  B_PAIR = 20,       // [4] the two softmax warps of a TMEM lane quarter (64 arrivals)
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
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NTHREADS, 1)
grouped_prefill_kernel(const __grid_constant__ GroupedArgs a) {
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
  const int cid = (int)cluster_id_x();
  const int ncl = (int)nclusters_x();

  if (threadIdx.x == 0) {
    mbar_init(&bars[B_Q_FULL], 256);
    for (int i = 0; i < NSTAGE; ++i) {
      mbar_init(&bars[B_KV_FULL + i], 1);
      mbar_init(&bars[B_KV_EMPTY + i], 1);
    }
    mbar_init(&bars[B_S_FULL], 1);
    mbar_init(&bars[B_S_EMPTY], 256);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars[B_SX_FULL + i], 1);
      mbar_init(&bars[B_SX_FREE + i], 256);
      mbar_init(&bars[B_DRAIN + i], 1);
    }
    mbar_init(&bars[B_P_FULL], 256);
    mbar_init(&bars[B_PV_DONE], 1);
    mbar_init(&bars[B_O_EMPTY], 256);
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
  cluster_sync();  // the peer's barriers exist before anyone arrives on them
  tc_fence_after();
  const uint32_t tmem = *tmem_base_ptr;

  if (warp >= 8) {
    regs_dec<REGS_OTHER>();
    if (warp >= 10) {
      // ----------------------------------------------------------------
      // TMA producers (warps 10-15, lanes 0-7 issue: 48 issuers).  A tile's
      // 16 * nown gather4 (rows 4g .. 4g+3 of own swizzle column c) are
      // dealt to the issuers, rotating from tile to tile so each gets the
      // same share; warp 10 also stores the tile's mask bytes.  Warp 10 lane 0
      // (the leader) arms each stage's byte count after the mask bytes are
      // stored; copies from the other issuers may complete first, which
      // only drives the transaction count negative until then.
      // ----------------------------------------------------------------
      constexpr int NI = NPROD_WARPS * 8;
      const int pw = warp - 10;
      const int iss = pw * 8 + lane;
      const bool issuer = lane < 8;
      const bool leader = (pw == 0) && (lane == 0);
      const int ng = 16 * nown;
      uint32_t gt = 0;
      bool ok = true;
      for (int g = cid; g < a.num_groups && ok; g += ncl) {
        const int U = min(__ldg(a.union_len + g), a.union_pad);
        const int ntiles = (U + BK - 1) / BK;
        if (ntiles == 0) continue;
        const int32_t* urow = a.union_idx + (size_t)g * a.union_pad;
        const uint8_t* mrow = a.mask + (size_t)g * a.union_pad;
        for (int j = 0; j < ntiles && ok; ++j, ++gt) {
          const int s = gt % NSTAGE;
          if (!mbar_wait_warp(&bars[B_KV_EMPTY + s], ((gt / NSTAGE) & 1) ^ 1, abort_flag, err)) { ok = false; break; }
          if (leader) DSA_TRACE(a.tr, gt, 0);
          if (pw == 0) {
            if (lane < 16) {
              // mask bytes of union slots j*64 .. j*64+63 (zero past the union)
              const int u0 = j * BK + 4 * lane;
              uint32_t w = 0;
              if (u0 + 3 < U) {
                w = __ldg(reinterpret_cast<const uint32_t*>(mrow + u0));
              } else {
                for (int e = 0; e < 4; ++e)
                  if (u0 + e < U) w |= (uint32_t)__ldg(mrow + u0 + e) << (8 * e);
              }
              *reinterpret_cast<uint32_t*>(smem + C::OFF_MASKB + s * 64 + 4 * lane) = w;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive_expect_tx(&bars[B_KV_FULL + s], (uint32_t)nown * C::KV_CHUNK);
          }
          if (issuer) {
            const uint32_t kvs = sbase + C::OFF_KV + s * C::KV_BYTES;
            const int b = (int)((iss + gt * (uint32_t)(ng % NI)) % NI);
            for (int e = b; e < ng; e += NI) {
              const int rg = e & 15;
              const int c = e >> 4;
              // union rows of the row group; nothing at or past U is read
              // (a tile may run past the padded row)
              const int u = j * BK + 4 * rg;
              int4 r = make_int4(-1, -1, -1, -1);
              if (u + 3 < U) {
                r = __ldg(reinterpret_cast<const int4*>(urow + u));
              } else {
                if (u + 0 < U) r.x = __ldg(urow + u + 0);
                if (u + 1 < U) r.y = __ldg(urow + u + 1);
                if (u + 2 < U) r.z = __ldg(urow + u + 2);
              }
              if (r.x < 0 || r.x >= a.N) r.x = -1;
              if (r.y < 0 || r.y >= a.N) r.y = -1;
              if (r.z < 0 || r.z >= a.N) r.z = -1;
              if (r.w < 0 || r.w >= a.N) r.w = -1;
              tma_gather4(kvs + c * C::KV_CHUNK + rg * 512, &a.tmap_kv, latent_chunk(rank, c) * 64, r.x, r.y, r.z,
                          r.w, &bars[B_KV_FULL + s]);
            }
          }
        }
      }
      // Let copies still in flight land before the CTA can exit: wait for
      // the last phase each stage was used in (an older phase's parity can
      // alias).
      if (leader) {
        for (uint32_t i = (gt > NSTAGE ? gt - NSTAGE : 0); i < gt; ++i)
          mbar_wait_drain(&bars[B_KV_FULL + (i % NSTAGE)], (i / NSTAGE) & 1);
      }
      __syncwarp();
    } else if (warp == 8) {
      // ----------------------------------------------------------------
      // QK issuer: partial S = q_own . K_own^T, q (A) from TMEM
      // ----------------------------------------------------------------
      if (lane == 0) {
        constexpr uint32_t IDESC_QK = idesc_bf16_f32(128, BK, false, false);
        uint32_t gt = 0, lgq = 0;
        bool ok = true;
        for (int g = cid; g < a.num_groups && ok; g += ncl) {
          const int U = min(__ldg(a.union_len + g), a.union_pad);
          const int ntiles = (U + BK - 1) / BK;
          if (ntiles == 0) continue;
          if (!mbar_wait(&bars[B_Q_FULL], lgq & 1, abort_flag, err)) { ok = false; break; }
          tc_fence_after();
          for (int j = 0; j < ntiles && ok; ++j, ++gt) {
            const int s = gt % NSTAGE;
            if (!mbar_wait(&bars[B_S_EMPTY], (gt & 1) ^ 1, abort_flag, err)) { ok = false; break; }
            if (!mbar_wait(&bars[B_KV_FULL + s], (gt / NSTAGE) & 1, abort_flag, err)) { ok = false; break; }
            DSA_TRACE(a.tr, gt, 2);
            tc_fence_after();
            const uint32_t kvs = sbase + C::OFF_KV + s * C::KV_BYTES;
            // per swizzle column: 4 MMAs of K = 16, A advances 8 TMEM columns, B 32 bytes
            for (int c = 0; c < nown; ++c)
              mma_bf16_ts_x4(tmem + C::COL_S, tmem + C::COL_Q + 32 * c, sdesc_sw128(kvs + c * C::KV_CHUNK, 16, 1024),
                             8u, 2u, IDESC_QK, c > 0 ? 1u : 0u);
            mma_commit(&bars[B_S_FULL]);
            DSA_TRACE(a.tr, gt, 1);
          }
          ++lgq;
        }
        mma_commit(&bars[B_DRAIN + 0]);
        mbar_wait(&bars[B_DRAIN + 0], 0, abort_flag, err);
      }
      __syncwarp();
    } else if (warp == 9) {
      // ----------------------------------------------------------------
      // PV issuer: O_own += P . V_own, P (bf16) read from tensor memory
      // ----------------------------------------------------------------
      if (lane == 0) {
        constexpr uint32_t IDESC_PV = idesc_bf16_f32(128, 256, false, true);
        uint32_t gt = 0, lgq = 0;
        bool ok = true;
        for (int g = cid; g < a.num_groups && ok; g += ncl) {
          const int U = min(__ldg(a.union_len + g), a.union_pad);
          const int ntiles = (U + BK - 1) / BK;
          if (ntiles == 0) continue;
          for (int j = 0; j < ntiles && ok; ++j, ++gt) {
            const int s = gt % NSTAGE;
            if (!mbar_wait(&bars[B_P_FULL], gt & 1, abort_flag, err)) { ok = false; break; }
            if (j == 0 && !mbar_wait(&bars[B_O_EMPTY], (lgq & 1) ^ 1, abort_flag, err)) { ok = false; break; }
            DSA_TRACE(a.tr, gt, 6);
            tc_fence_after();
            // 64 union slots = 4 MMAs of 16: P advances 8 TMEM columns, V (MN-major) 2048 B
            const uint32_t kvs = sbase + C::OFF_KV + s * C::KV_BYTES;
            mma_bf16_ts_x4(tmem + C::COL_O, tmem + C::COL_P, sdesc_sw128(kvs, C::KV_CHUNK, 1024), 8u, 128u, IDESC_PV,
                           j > 0 ? 1u : 0u);
            mma_commit(&bars[B_PV_DONE]);
            mma_commit(&bars[B_KV_EMPTY + s]);
          }
          ++lgq;
        }
        mma_commit(&bars[B_DRAIN + 1]);
        mbar_wait(&bars[B_DRAIN + 1], 0, abort_flag, err);
      }
      __syncwarp();
    }
  } else {
    regs_inc<REGS_SOFTMAX>();
    // ------------------------------------------------------------------
    // softmax warps: thread (row, half) <-> pseudo-head row = TMEM lane,
    // slots 32*half .. 32*half+31 of each tile
    // ------------------------------------------------------------------
    constexpr int HK = BK / 2;               // slots per thread
    const int half = warp >> 2;
    const int row = (warp & 3) * 32 + lane;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const float sl2 = a.scale * 1.4426950408889634f;
    const int tok = row / H;  // token of the group this pseudo-head belongs to
    // my row of the SX buffers: 16-byte pieces XOR-swizzled by row; this
    // thread moves pieces 8*half .. 8*half+7
    const uint32_t sx_row = C::OFF_SX + row * (BK * 4);
    const uint32_t sx_peer = map_peer(sbase + sx_row, peer);
    const uint32_t bar_base = smem_u32(bars);
    auto peer_bar = [&](int idx) { return map_peer(bar_base + idx * 8, peer); };
    auto piece = [&](int c) { return (uint32_t)(((8 * half + c) ^ (row & 15)) << 4); };
    uint64_t* pair_bar = &bars[B_PAIR + (warp & 3)];
    uint32_t pair_phase = 0;
    uint32_t gt = 0, lgq = 0;
    bool ok = true;

    // Step A of tile i: this thread's half of the partial S row from TMEM,
    // S freed for the next QK, the half sent to the peer once it has read
    // what we sent two tiles ago.
    auto step_a = [&](uint32_t i, float* v) -> bool {
      if (!mbar_wait_warp(&bars[B_S_FULL], i & 1, abort_flag, err)) return false;
      if (row == 0 && half == 0) DSA_TRACE(a.tr, i, 3);
      tc_fence_after();
      tmem_ld16(tmem + lane_off + C::COL_S + HK * half, v);
      tmem_ld16(tmem + lane_off + C::COL_S + HK * half + 16, v + 16);
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(&bars[B_S_EMPTY]);
      const int sb = i & 1;
      if (!mbar_wait_cluster_warp(&bars[B_SX_FREE + sb], ((i >> 1) & 1) ^ 1, abort_flag, err)) return false;
      // (my own receive buffer for tile i: armed after tile i-2's completed)
      if (threadIdx.x == 0) mbar_arrive_expect_tx(&bars[B_SX_FULL + sb], C::SX_BYTES);
      const uint32_t dst = sx_peer + sb * C::SX_BYTES;
      const uint32_t rbar = peer_bar(B_SX_FULL + sb);
#pragma unroll
      for (int c = 0; c < 8; ++c)
        st_async_v4(dst + piece(c), __float_as_uint(v[4 * c]), __float_as_uint(v[4 * c + 1]),
                    __float_as_uint(v[4 * c + 2]), __float_as_uint(v[4 * c + 3]), rbar);
      if (row == 0 && half == 0) DSA_TRACE(a.tr, i, 7);
      return true;
    };

    // Step B of tile i (j-th of its group): add the peer's partial half row,
    // mask, agree on the running max with the other half, P (bf16 pairs)
    // into TMEM.
    // For the last tile of a group the SX_FREE arrival is left to the
    // epilogue, which still uses the buffer to add the two halves' row sums.
    auto step_b = [&](uint32_t i, int j, bool last, float* v, float& m_run, float& l_run) -> bool {
      const int sb = i & 1;
      if (!mbar_wait_cluster_warp(&bars[B_SX_FULL + sb], (i >> 1) & 1, abort_flag, err)) return false;
      if (row == 0 && half == 0) DSA_TRACE(a.tr, i, 4);
      uint8_t* sxr = smem + sx_row + sb * C::SX_BYTES;
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const float4 x = *reinterpret_cast<const float4*>(sxr + piece(c));
        // S = S_0 + S_1 with the operands in rank order on both CTAs
        if (rank == 0) {
          v[4 * c] = v[4 * c] + x.x;
          v[4 * c + 1] = v[4 * c + 1] + x.y;
          v[4 * c + 2] = v[4 * c + 2] + x.z;
          v[4 * c + 3] = v[4 * c + 3] + x.w;
        } else {
          v[4 * c] = x.x + v[4 * c];
          v[4 * c + 1] = x.y + v[4 * c + 1];
          v[4 * c + 2] = x.z + v[4 * c + 2];
          v[4 * c + 3] = x.w + v[4 * c + 3];
        }
      }
      // the stage's mask bytes (its phase cannot have moved on: the stage is
      // released only after this tile's P.V); raw scores are kept, masked
      // slots become -inf, the scale is applied in the exponent
      const int s = i % NSTAGE;
      if (!mbar_wait_warp(&bars[B_KV_FULL + s], (i / NSTAGE) & 1, abort_flag, err)) return false;
      float hmax = -INFINITY;
      {
        const uint4* mb4 = reinterpret_cast<const uint4*>(smem + C::OFF_MASKB + s * 64 + HK * half);
#pragma unroll
        for (int q4 = 0; q4 < 2; ++q4) {
          const uint4 m4 = mb4[q4];
          const uint32_t mw[4] = {m4.x, m4.y, m4.z, m4.w};
#pragma unroll
          for (int w = 0; w < 4; ++w) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int c = 16 * q4 + 4 * w + e;
              const bool on = (mw[w] >> (8 * e + tok)) & 1u;
              v[c] = on ? v[c] : -INFINITY;
              hmax = fmaxf(hmax, v[c]);
            }
          }
        }
      }
      // the other half's max, through a fixed slot of the consumed half of
      // my SX row (the peer may refill the row only after both halves
      // arrived below)
      reinterpret_cast<volatile float*>(sxr + piece(0))[0] = hmax;
      if (!group_sync(pair_bar, pair_phase, abort_flag, err)) return false;
      const float omax = reinterpret_cast<volatile float*>(smem + sx_row + sb * C::SX_BYTES +
                                                           ((((8 * (half ^ 1)) ^ (row & 15))) << 4))[0];
      // (every loaded value was consumed above, so the loads have completed)
      const float tmax = (half == 0 ? fmaxf(hmax, omax) : fmaxf(omax, hmax)) * sl2;
      if (!last) mbar_arrive_remote_relaxed(peer_bar(B_SX_FREE + sb));
      // lazy rescale: move the reference only when the max grows by more than kTau
      const bool need = tmax > m_run + kTau;
      float alpha = 1.f;
      if (need) {
        const float mn = fmaxf(m_run, tmax);
        alpha = (m_run == -INFINITY) ? 0.f : exp2f(m_run - mn);
        m_run = mn;
        l_run *= alpha;
      }
      // P.V of the previous tile must be complete before P is overwritten or O rescaled
      if (!mbar_wait_warp(&bars[B_PV_DONE], (i - 1) & 1, abort_flag, err)) return false;
      tc_fence_after();
      if (j > 0 && __any_sync(0xffffffffu, need)) {
#pragma unroll 1
        for (int c = 128 * half; c < 128 * half + 128; c += 16) {
          float o[16];
          tmem_ld16(tmem + lane_off + C::COL_O + c, o);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 16; ++e) o[e] *= alpha;
          tmem_st16(tmem + lane_off + C::COL_O + c, o);
        }
      }
      const float mref = (m_run == -INFINITY) ? 0.f : m_run;
      uint32_t pk[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        pk[e] = pack_bf16x2(exp2f(fmaf(v[2 * e], sl2, -mref)), exp2f(fmaf(v[2 * e + 1], sl2, -mref)));
        l_run += __uint_as_float(pk[e] << 16) + __uint_as_float(pk[e] & 0xffff0000u);
      }
      tmem_st16_u32(tmem + lane_off + C::COL_P + 16 * half, pk);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bars[B_P_FULL]);
      if (row == 0 && half == 0) DSA_TRACE(a.tr, i, 5);
      return true;
    };

    for (int g = cid; g < a.num_groups && ok; g += ncl) {
      int t0, n;
      group_of(a.req, G, g, t0, n);
      const int U = min(__ldg(a.union_len + g), a.union_pad);
      const int ntiles = (U + BK - 1) / BK;
      const int nrows = n * H;
      uint16_t* out_row = a.out + (size_t)(t0 * H + row) * 512 + 256 * rank + 128 * half;
      if (ntiles == 0) {
        if (row < nrows) {
          for (int c = 0; c < 16; ++c) reinterpret_cast<uint4*>(out_row)[c] = make_uint4(0, 0, 0, 0);
          if (rank == 0 && half == 0) a.lse[(size_t)t0 * H + row] = -INFINITY;
        }
        continue;
      }
      // q row t0*H + row, own columns, into TMEM as bf16 pairs: this thread
      // writes the 32 columns 32*half .. +31 of every own swizzle column (the
      // previous group's QK MMAs completed before its last scores were read)
      {
        const int64_t qrow = (int64_t)t0 * H + row;
        const bool qvalid = qrow < (int64_t)a.T * H;
        const uint16_t* src = a.q + (qvalid ? qrow : 0) * a.d_qk + HK * half;
        uint4 qv[C::OWNMAX][4];
#pragma unroll
        for (int c = 0; c < C::OWNMAX; ++c)
#pragma unroll
          for (int e = 0; e < 4; ++e)
            qv[c][e] = (c < nown && qvalid)
                           ? __ldg(reinterpret_cast<const uint4*>(src + latent_chunk(rank, c) * 64) + e)
                           : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int c = 0; c < C::OWNMAX; ++c)
          if (c < nown)
            tmem_st16_u32(tmem + lane_off + C::COL_Q + 32 * c + 16 * half, reinterpret_cast<const uint32_t*>(qv[c]));
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&bars[B_Q_FULL]);
      }
      float m_run = -INFINITY, l_run = 0.f;
      float va[HK], vb[HK];
      if (!step_a(gt, va)) { ok = false; break; }
      for (int j = 0; j < ntiles;) {
        if (j + 1 < ntiles && !step_a(gt + j + 1, vb)) { ok = false; break; }
        if (!step_b(gt + j, j, j + 1 == ntiles, va, m_run, l_run)) { ok = false; break; }
        if (++j == ntiles) break;
        if (j + 1 < ntiles && !step_a(gt + j + 1, va)) { ok = false; break; }
        if (!step_b(gt + j, j, j + 1 == ntiles, vb, m_run, l_run)) { ok = false; break; }
        ++j;
      }
      if (!ok) break;
      // ---- epilogue: row sum of both halves, normalise this CTA's half of O ----
      // (through the row's slot in the last tile's SX buffer, which the peer
      // cannot refill before both halves' deferred SX_FREE arrivals below)
      float lsum;
      {
        const int sb = (gt + ntiles - 1) & 1;
        volatile float* slot = reinterpret_cast<volatile float*>(smem + sx_row + sb * C::SX_BYTES);
        slot[half] = l_run;
        if (!group_sync(pair_bar, pair_phase, abort_flag, err)) { ok = false; break; }
        lsum = slot[0] + slot[1];  // (consumes the loads before the arrival)
        mbar_arrive_remote_relaxed(peer_bar(B_SX_FREE + sb));
      }
      const float inv_l = (lsum > 0.f) ? 1.f / lsum : 0.f;
      if (rank == 0 && half == 0 && row < nrows)
        a.lse[(size_t)t0 * H + row] = (lsum > 0.f) ? (m_run + log2f(lsum)) * 0.6931471805599453f : -INFINITY;
      if (!mbar_wait_warp(&bars[B_PV_DONE], (gt + ntiles - 1) & 1, abort_flag, err)) { ok = false; break; }
      tc_fence_after();
#pragma unroll 1
      for (int c = 0; c < 128; c += 16) {
        float o[16];
        tmem_ld16(tmem + lane_off + C::COL_O + 128 * half + c, o);
        tmem_ld_wait();
        if (row < nrows) {
          uint32_t pk[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) pk[e] = pack_bf16x2(o[2 * e] * inv_l, o[2 * e + 1] * inv_l);
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
  if (warp == 8) tmem_dealloc(tmem, C::TMEM_COLS);
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
