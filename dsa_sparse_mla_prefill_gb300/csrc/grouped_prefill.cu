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
// A group is processed by a pair of CTAs (a 2-CTA cluster) acting as one
// through cta_group::2 tensor-core instructions.  The union is walked in
// pair tiles of 256 slots; CTA r owns slots 128r .. 128r+127 of each.
//   S^T = K q^T      M = 256 pair MMAs, 16 columns each: A = the 256 slots'
//                    key rows (CTA r supplies its own 128, gathered into its
//                    own shared memory), B = q of the 128 pseudo-heads (CTA r
//                    supplies pseudo-heads 64r .. 64r+63); CTA r's tensor
//                    memory receives S^T for its 128 slots x all 128 heads.
//   softmax          in each CTA, thread i <-> slot i (TMEM lane i); the
//                    running max of every pseudo-head is agreed between the
//                    two CTAs once per tile (an 8-warp barrier across the
//                    pair), so P of both halves shares one reference.
//   O^T += V^T P^T   M = 256 pair MMAs over the tile's 256 slots: A = V^T,
//                    CTA r supplying output columns 256b + 128r .. +127 of
//                    M-block b (it gathers those columns of all 256 slots),
//                    B = P^T, CTA r supplying pseudo-heads 64r .. 64r+63 for
//                    all 256 slots (the softmax of each CTA stages its slots'
//                    P of the peer's heads and the copy engine moves it into
//                    the peer's shared memory); O^T of CTA r = its 256 output columns x 128
//                    heads, the whole 512 x 128 output between the pair.
// Each CTA thus gathers per 256 slots its 128 key rows (all D_QK columns)
// and 256 rows x 256 value columns: half the gather of one CTA doing the
// whole group, with no data loaded for the other CTA (no TMA multicast).
// TMA loads of both CTAs complete on the even CTA's barriers
// (cp.async.bulk.tensor .cta_group::2), where the single MMA-issuing thread
// of each stream waits; every MMA completion is committed to both CTAs'
// barriers.
//
// O^T lives in tensor memory once (TMEM holds O^T and two S^T buffers), so a
// group's epilogue (the pair's row sums, lse, out = O / l) is deferred until
// the next group's first tile has stored its P: the group's last P.V then
// runs beside that softmax instead of stalling it, and O is read, scaled and
// packed before it is released to the next group's first P.V.
//
// Warp roles (24 warps): 0-7 softmax (two per TMEM lane quarter: warp w
// holds slots 32(w%4) .. +31 and pseudo-heads 64(w/4) .. +63, as two blocks
// of 32), 8 QK issuer (and tensor-memory allocation), 9 PV issuer (issuers
// run in the even CTA only), 10-16 K-ring producers, 17-23 V-ring producers
// (the warps of a stream share every stage).
#include "dsa_device.cuh"
#include "dsa_kernels.h"

namespace dsa {
namespace grouped {

constexpr int BK = 128;          // slots per CTA per pair tile (the pair MMA's M / 2)
constexpr int PT = 2 * BK;       // slots per pair tile
constexpr int HP = 128;          // pseudo-heads (the pair MMA's N)
constexpr int HC = 64;           // pseudo-heads whose q / P this CTA supplies
constexpr int NTHREADS = 768;    // 24 warps, launched at 80 registers each
constexpr int REGS_SOFTMAX = 160;
constexpr int REGS_OTHER = 40;   // 8*32*160 + 16*32*40 = 768*80
constexpr int KW0 = 10, NKWARP = 7, KLANES = 5;    // K producers: warps 10-16, lanes 0-4 (33 requests)
constexpr int VW0 = 17, NVWARP = 7, VLANES = 10;   // V producers: warps 17-23, lanes 0-9 (64 requests)
constexpr float kTau = 8.0f;     // lazy-rescale threshold (log2 units)
constexpr uint16_t kBoth = 3;    // commit to both CTAs' barriers

struct Cfg {
  static constexpr uint32_t CHUNK_BYTES = BK * 128u;          // 128 slots x 64 columns
  static constexpr uint32_t UNIT_BYTES = 2u * CHUNK_BYTES;    // 128 slots x 128 columns
  static constexpr uint32_t Q_CHUNK = HC * 128u;              // 64 pseudo-heads x 64 columns
  static constexpr uint32_t KSTAGE_BYTES = CHUNK_BYTES + Q_CHUNK;
  static constexpr uint32_t P_BYTES = PT * 128u;              // 256 slots x 64 heads, MN-major
  static constexpr int NKR = 3;    // K stages
  static constexpr int NPB = 2;    // P buffers
  static constexpr int NVR = 2;    // V slots
  // softmax exchange: [parity][head block][block of 32 heads][8 warps of the pair][32]
  static constexpr uint32_t RED_BYTES = 2u * 2u * 2u * 8u * 32u * 4u;
  // each softmax warp's copy of -(running max) of its 64 heads, read back by
  // every lane as broadcast loads
  static constexpr uint32_t NEGM_BYTES = 8u * 64u * 4u;
  static constexpr uint32_t OFF_KR = 0;
  static constexpr uint32_t OFF_VR = OFF_KR + NKR * KSTAGE_BYTES;
  static constexpr uint32_t OFF_P = OFF_VR + NVR * UNIT_BYTES;
  // P of this CTA's slots for the peer's heads, staged for one bulk copy
  // per warp into the peer's P buffer
  static constexpr uint32_t STG_BYTES = BK * 128u;
  static constexpr uint32_t OFF_STG = OFF_P + NPB * P_BYTES;
  static constexpr uint32_t OFF_RED = OFF_STG + STG_BYTES;
  static constexpr uint32_t OFF_NEGM = OFF_RED + RED_BYTES;
  static constexpr uint32_t OFF_BAR = OFF_NEGM + NEGM_BYTES;
  static constexpr int NBAR = 40;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8u;
  static constexpr uint32_t SMEM_BYTES = OFF_MISC + 64u;
  // no alignment slack: the dynamic shared memory must start 1024-aligned
  // (checked at entry)
  static_assert(SMEM_BYTES <= 227u * 1024u, "shared memory budget");
  static_assert(NKWARP * KLANES >= 33 && NVWARP * VLANES >= 64 && VW0 + NVWARP == NTHREADS / 32, "producers");
  static constexpr uint32_t COL_O = 0;     // O^T: 2 M-blocks x 128 heads
  static constexpr uint32_t COL_S = 256;   // S^T: 2 buffers x 128 heads
  static constexpr uint32_t TMEM_COLS = 512;
};

enum {
  B_KF = 0,      // [NKR <= 4] even CTA: one arrive.expect_tx (both CTAs' bytes)
  B_KE = 4,      // [NKR] one commit
  B_VF = 8,      // [NVR <= 4] even CTA: one arrive.expect_tx
  B_VE = 12,     // [NVR] one commit
  B_SF = 16,     // [2] one commit
  B_SE = 18,     // [2] even CTA: the 16 softmax warps of the pair
  B_PF = 20,     // [NPB] even CTA: one relay arrival from the odd CTA (its P_RX completed)
  B_PE = 22,     // [NPB] one commit (the P.V that read P buffer b is done)
  B_OF = 24,     // one commit
  B_OE = 25,     // even CTA: the 16 softmax warps of the pair
  B_XB = 26,     // [parity][head block][block of 32]: 4 local warps + the peer's 4 x 128 bytes
  B_DRAIN = 34,  // [2] one per MMA issuer
  B_PRX = 36,    // [NPB] P buffer b complete: this CTA's 8 softmax warps + 16 KB copied in by the peer
  B_STG = 38,    // the staging rows were copied out: the peer's acknowledgement of the last copy
};

__device__ __forceinline__ void group_of(const ReqTable& rq, int G, int g, int& t0, int& n) {
  int r = 0;
  while (r + 1 < rq.num_req && rq.cu_g[r + 1] <= g) ++r;
  t0 = rq.cu_q[r] + (g - rq.cu_g[r]) * G;
  n = min(G, rq.cu_q[r + 1] - t0);
}

// The four union slots u .. u+3 (row indices; -1 past the union or out of
// range, which TMA reads as zeros).  Nothing at or past U is read.
__device__ __forceinline__ int4 union_rows4(const int32_t* urow, int U, int N, int u) {
  int4 r = make_int4(-1, -1, -1, -1);
  if (u + 3 < U) {
    r = __ldg(reinterpret_cast<const int4*>(urow + u));
  } else {
    if (u + 0 < U) r.x = __ldg(urow + u + 0);
    if (u + 1 < U) r.y = __ldg(urow + u + 1);
    if (u + 2 < U) r.z = __ldg(urow + u + 2);
  }
  if (r.x < 0 || r.x >= N) r.x = -1;
  if (r.y < 0 || r.y >= N) r.y = -1;
  if (r.z < 0 || r.z >= N) r.z = -1;
  if (r.w < 0 || r.w >= N) r.w = -1;
  return r;
}

// The first row of the 64 union slots u0 .. u0+63 when they are one run of
// consecutive rows inside the table (the union is sorted and distinct, so the
// two end slots decide), else -1.
__device__ __forceinline__ int run_start(const int32_t* urow, int U, int N, int u0) {
  if (u0 + 63 >= U) return -1;
  const int first = __ldg(urow + u0);
  const int last = __ldg(urow + u0 + 63);
  return (first >= 0 && last < N && last - first == 63) ? first : -1;
}

// Warp-level transposed max/sum reduction over 32 lanes for 32 values per
// lane: afterwards lane L holds the reduction over the warp of value L.
template <bool IS_MAX>
__device__ __forceinline__ float warp_transpose_reduce32(float* v) {
  const uint32_t lane = lane_id();
  auto op = [](float a, float b) { return IS_MAX ? fmaxf(a, b) : a + b; };
  int n = 32;
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    n >>= 1;
    const bool upper = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      if (i < n) {
        const float send = upper ? v[i] : v[i + n];
        const float keep = upper ? v[i + n] : v[i];
        v[i] = op(keep, __shfl_xor_sync(0xffffffffu, send, o));
      }
    }
  }
  return v[0];
}

// One arrival of the calling warp (lane 0, once every lane of the warp is
// done) on a barrier of the even CTA, given by its offset in this CTA.
__device__ __forceinline__ void warp_arrive_leader(uint64_t* bar) {
  __syncwarp();
  if (lane_id() == 0) mbar_arrive_remote(map_peer(smem_u32(bar), 0));
}

template <int NC>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NTHREADS, 1)
grouped_prefill_kernel(const __grid_constant__ GroupedArgs a) {
  using C = Cfg;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  if ((raw_u32 & 1023u) != 0) {
    // same base in every CTA of the launch: the whole grid stops here
    if (threadIdx.x == 0) atomicAdd(a.err + ERR_TIMEOUT, 1u);
    return;
  }
  uint8_t* smem = smem_raw;
  const uint32_t sbase = raw_u32;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile uint32_t* tmem_base_ptr = misc;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 1);
  unsigned int* err = a.err;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int rank = (int)cluster_ctarank();
  const bool leader = rank == 0;
  const int H = a.H;
  const int G = a.G;
  const int cid = (int)cluster_id_x();
  const int ncl = (int)nclusters_x();

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::NKR; ++i) {
      mbar_init(&bars[B_KF + i], 1);
      mbar_init(&bars[B_KE + i], 1);
    }
    for (int i = 0; i < C::NVR; ++i) {
      mbar_init(&bars[B_VF + i], 1);
      mbar_init(&bars[B_VE + i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars[B_SF + i], 1);
      mbar_init(&bars[B_SE + i], 16);
      mbar_init(&bars[B_DRAIN + i], 1);
    }
    for (int i = 0; i < 8; ++i) mbar_init(&bars[B_XB + i], 4);
    for (int i = 0; i < C::NPB; ++i) {
      mbar_init(&bars[B_PF + i], 1);
      mbar_init(&bars[B_PRX + i], 8);
      mbar_init(&bars[B_PE + i], 1);
    }
    mbar_init(&bars[B_STG], 1);
    mbar_init(&bars[B_OF], 1);
    mbar_init(&bars[B_OE], 16);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 8) {
    tmem_alloc_pair(const_cast<uint32_t*>(tmem_base_ptr), C::TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers exist before any copy, commit or arrival reaches them
  tc_fence_after();
  const uint32_t tmem = *tmem_base_ptr;

  if (warp >= 8) {
    regs_dec<REGS_OTHER>();
    if (warp >= 10) {
      // ----------------------------------------------------------------
      // TMA producers (both CTAs).  Every load lands in this CTA's own
      // shared memory and completes on the even CTA's barrier, where the
      // issuer of the MMAs that read it waits; the even CTA's producer arms
      // the bytes of both CTAs.  A stage is refilled once the MMAs that read
      // it have completed in the pair (commit to both CTAs' EMPTY barriers).
      // A warp issues its TMA requests one after another (the SM's request
      // rate grows with the number of warps issuing), so every stage and
      // unit is shared by the warps of its stream:
      //   K (warps 10-16): chunk c of a pair tile = this CTA's 128 slots x
      //     columns 64c .. 64c+63 (requests 0-31: slots 4e .. 4e+3) + q chunk
      //     c of its 64 pseudo-heads (request 32); lanes 0-4 of each warp.
      //   V (warps 17-23): unit u = 2b + h of a pair tile = the tile's slots
      //     128h .. 128h+127 x this CTA's columns 256b + 128r .. +127, as two
      //     64-column swizzle columns (requests 0-63: slots 4(e % 32) .. +3,
      //     swizzle column e / 32); lanes 0-9 of each warp.
      // A 64-slot half that is one run of consecutive rows is one tiled load
      // (box 64 columns x 64 rows) instead of 16 gathers.
      // ----------------------------------------------------------------
      const bool kstream = warp < VW0;
      const int e = kstream ? (warp - KW0) * KLANES + (lane < KLANES ? lane : 64)   // K request 0..32
                            : (warp - VW0) * VLANES + (lane < VLANES ? lane : 64);  // V request 0..63
      const bool kgather = kstream && e < 32;
      const bool kq = kstream && e == 32;
      const bool vgather = !kstream && e < 64;
      const int rg = e & 31;                                    // row group (4 slots) of 128
      const int vcc = (e >> 5) & 1;                             // V swizzle column
      const bool arm = leader && lane == 0 && (warp == KW0 || warp == VW0);
      uint32_t gt = 0, pos = 0;
      bool ok = true;
      for (int g = cid; g < a.num_groups && ok; g += ncl) {
        int t0, n;
        group_of(a.req, G, g, t0, n);
        const int U = min(__ldg(a.union_len + g), a.union_pad);
        const int ntiles = (U + PT - 1) / PT;
        if (ntiles == 0) continue;
        const int32_t* urow = a.union_idx + (size_t)g * a.union_pad;
        for (int j = 0; j < ntiles && ok; ++j, ++gt) {
          if (kstream) {
            const int u0 = j * PT + BK * rank;             // this CTA's 128 slots
            const int first = kgather ? run_start(urow, U, a.N, u0 + 64 * (rg >> 4)) : -1;
            const int4 r = (kgather && first < 0) ? union_rows4(urow, U, a.N, u0 + 4 * rg)
                                                   : make_int4(-1, -1, -1, -1);
#pragma unroll 1
            for (int c = 0; c < NC; ++c, ++pos) {
              const int ks = (int)(pos % C::NKR);
              if (!mbar_wait_cluster_warp(&bars[B_KE + ks], ((pos / C::NKR) & 1) ^ 1, abort_flag, err)) {
                ok = false;
                break;
              }
              const uint32_t full0 = map_peer(smem_u32(&bars[B_KF + ks]), 0);
              if (arm) mbar_arrive_expect_tx(&bars[B_KF + ks], 2u * C::KSTAGE_BYTES);
              const uint32_t stage = sbase + C::OFF_KR + ks * C::KSTAGE_BYTES;
              if (kgather) {
                if (first >= 0) {
                  if ((rg & 15) == 0)
                    tma_load_2d_pair(stage + (rg >> 4) * (C::CHUNK_BYTES / 2), &a.tmap_kv_blk, c * 64, first, full0);
                } else {
                  tma_gather4_pair(stage + rg * 512, &a.tmap_kv, c * 64, r.x, r.y, r.z, r.w, full0);
                }
              }
              // q rows t0*H + 64 rank .. +63 of q viewed [T*H, D_QK], columns 64c ..
              if (kq) tma_load_2d_pair(stage + C::CHUNK_BYTES, &a.tmap_q, c * 64, t0 * H + HC * rank, full0);
            }
          } else {
            for (int u = 0; u < 4 && ok; ++u, ++pos) {
              const int b = u >> 1, hh = u & 1;
              const int vg = (int)(pos % C::NVR);
              if (!mbar_wait_cluster_warp(&bars[B_VE + vg], ((pos / C::NVR) & 1) ^ 1, abort_flag, err)) {
                ok = false;
                break;
              }
              const uint32_t full0 = map_peer(smem_u32(&bars[B_VF + vg]), 0);
              if (arm) mbar_arrive_expect_tx(&bars[B_VF + vg], 2u * C::UNIT_BYTES);
              if (vgather) {
                const int u0 = j * PT + BK * hh;
                const int first = run_start(urow, U, a.N, u0 + 64 * (rg >> 4));
                const int col = 256 * b + 128 * rank + 64 * vcc;
                const uint32_t vdst = sbase + C::OFF_VR + vg * C::UNIT_BYTES + vcc * C::CHUNK_BYTES;
                if (first >= 0) {
                  if ((rg & 15) == 0)
                    tma_load_2d_pair(vdst + (rg >> 4) * (C::CHUNK_BYTES / 2), &a.tmap_kv_blk, col, first, full0);
                } else {
                  const int4 r = union_rows4(urow, U, a.N, u0 + 4 * rg);
                  tma_gather4_pair(vdst + rg * 512, &a.tmap_kv, col, r.x, r.y, r.z, r.w, full0);
                }
              }
            }
          }
        }
      }
      if (!ok) {
        // a wait ran out: loads already issued land within microseconds;
        // give them that long before this CTA (their target) can leave
        const uint64_t t0 = globaltimer();
        while (globaltimer() - t0 < 20000ull) {
        }
      }
      __syncwarp();
    } else if (warp == 8) {
      // ----------------------------------------------------------------
      // QK issuer (even CTA): S^T = K q^T, chunk by chunk, into the S double
      // buffer; each K stage goes back to both CTAs' producers once its MMAs
      // complete, and S_FULL is committed to both CTAs' softmax.
      // ----------------------------------------------------------------
      if (leader && lane == 0) {
        constexpr uint32_t IDESC_QK = idesc_bf16_f32(256, HP, false, false);
        uint32_t gt = 0, kpos = 0;
        bool ok = true;
        for (int g = cid; g < a.num_groups && ok; g += ncl) {
          const int U = min(__ldg(a.union_len + g), a.union_pad);
          const int ntiles = (U + PT - 1) / PT;
          for (int j = 0; j < ntiles && ok; ++j, ++gt) {
            const int sb = gt & 1;
            const uint32_t d_s = tmem + C::COL_S + sb * HP;
            if (!mbar_wait_cluster(&bars[B_SE + sb], ((gt >> 1) & 1) ^ 1, abort_flag, err)) { ok = false; break; }
            DSA_TRACE(a.tr, gt, 2);
            tc_fence_after();
#pragma unroll 1
            for (int c = 0; c < NC; ++c, ++kpos) {
              const uint32_t slot = kpos % C::NKR;
              if (!mbar_wait_cluster(&bars[B_KF + slot], (kpos / C::NKR) & 1, abort_flag, err)) {
                ok = false;
                break;
              }
              tc_fence_after();
              const uint32_t stage = sbase + C::OFF_KR + slot * C::KSTAGE_BYTES;
              mma_pair_bf16_ss_x4(d_s, sdesc_sw128(stage, 16, 1024), sdesc_sw128(stage + C::CHUNK_BYTES, 16, 1024),
                                  2u, 2u, IDESC_QK, c > 0 ? 1u : 0u);
              mma_pair_commit(&bars[B_KE + slot], kBoth);
            }
            if (!ok) break;
            DSA_TRACE(a.tr, gt, 4);
            mma_pair_commit(&bars[B_SF + sb], kBoth);
          }
        }
        mma_pair_commit(&bars[B_DRAIN + 0], 1);
        mbar_wait(&bars[B_DRAIN + 0], 0, abort_flag, err);
      } else if (!leader && lane == 0) {
        // relay (odd CTA): once this CTA's P buffer is complete (its softmax
        // done, the peer's copy landed), tell the even CTA's P.V issuer, and
        // tell the even CTA that its staging rows may be rewritten
        const uint32_t stg0 = map_peer(smem_u32(&bars[B_STG]), 0);
        uint32_t gt = 0;
        bool ok = true;
        for (int g = cid; g < a.num_groups && ok; g += ncl) {
          const int U = min(__ldg(a.union_len + g), a.union_pad);
          const int ntiles = (U + PT - 1) / PT;
          for (int j = 0; j < ntiles; ++j, ++gt) {
            const int pb = gt & 1;
            if (!mbar_wait_cluster(&bars[B_PRX + pb], (gt >> 1) & 1, abort_flag, err)) { ok = false; break; }
            DSA_TRACE(a.tr, gt, 2);
            mbar_arrive_remote(map_peer(smem_u32(&bars[B_PF + pb]), 0));
            mbar_arrive_remote_relaxed(stg0);
          }
        }
      }
      __syncwarp();
    } else if (warp == 9) {
      // ----------------------------------------------------------------
      // PV issuer (even CTA): O^T += V^T P^T for the tile's four V units
      // (M-block b, slot half h); each unit goes back to both CTAs'
      // producers once its MMAs complete; P_EMPTY and (last tile of a
      // group) O_FULL are committed to both CTAs.
      // ----------------------------------------------------------------
      if (leader && lane == 0) {
        constexpr uint32_t IDESC_PV = idesc_bf16_f32(256, HP, true, true);
        const uint32_t stg1 = map_peer(smem_u32(&bars[B_STG]), 1);
        uint32_t gt = 0, vpos = 0, lgq = 0;
        bool ok = true;
        for (int g = cid; g < a.num_groups && ok; g += ncl) {
          const int U = min(__ldg(a.union_len + g), a.union_pad);
          const int ntiles = (U + PT - 1) / PT;
          if (ntiles == 0) continue;
          for (int j = 0; j < ntiles && ok; ++j, ++gt) {
            // this CTA's P buffer and rescale (then the odd CTA may reuse its
            // staging rows, whose copy has landed here), then the peer's
            // (relayed)
            const int pb = gt & 1;
            const uint32_t pph = (gt >> 1) & 1;
            if (!mbar_wait_cluster(&bars[B_PRX + pb], pph, abort_flag, err)) { ok = false; break; }
            // (a bare "read done" signal: no data of this thread to publish)
            mbar_arrive_remote_relaxed(stg1);
            if (!mbar_wait_cluster(&bars[B_PF + pb], pph, abort_flag, err)) { ok = false; break; }
            DSA_TRACE(a.tr, gt, 7);
            if (j == 0 && !mbar_wait_cluster(&bars[B_OE], (lgq & 1) ^ 1, abort_flag, err)) { ok = false; break; }
            tc_fence_after();
            for (int u = 0; u < 4 && ok; ++u, ++vpos) {
              const int b = u >> 1, hh = u & 1;
              const uint32_t slot = vpos % C::NVR;
              if (!mbar_wait_cluster(&bars[B_VF + slot], (vpos / C::NVR) & 1, abort_flag, err)) {
                ok = false;
                break;
              }
              tc_fence_after();
              const uint32_t ubase = sbase + C::OFF_VR + slot * C::UNIT_BYTES;
              const uint32_t d_o = tmem + C::COL_O + b * HP;
              // 16 slots per MMA: V^T MN-major (the unit's two swizzle columns
              // CHUNK_BYTES apart), P^T MN-major rows 128h + 64hf ..
              uint64_t adesc = sdesc_sw128(ubase, C::CHUNK_BYTES, 1024);
              uint64_t bdesc = sdesc_sw128(sbase + C::OFF_P + pb * C::P_BYTES + BK * hh * 128, C::P_BYTES, 1024);
#pragma unroll 1
              for (int hf = 0; hf < 2; ++hf) {
                mma_pair_bf16_ss_x4(d_o, adesc, bdesc, 128u, 128u, IDESC_PV, (j > 0 || hh > 0 || hf > 0) ? 1u : 0u);
                adesc += 4u * 128u;   // 64 slots = 8 KB, in 16-byte units of the start field
                bdesc += 4u * 128u;
              }
              mma_pair_commit(&bars[B_VE + slot], kBoth);
            }
            if (!ok) break;
            mma_pair_commit(&bars[B_PE + pb], kBoth);
            DSA_TRACE(a.tr, gt, 0);
            if (j == ntiles - 1) mma_pair_commit(&bars[B_OF], kBoth);
          }
          ++lgq;
        }
        mma_pair_commit(&bars[B_DRAIN + 1], 1);
        mbar_wait(&bars[B_DRAIN + 1], 0, abort_flag, err);
      }
      __syncwarp();
    }
  } else {
    regs_inc<REGS_SOFTMAX>();
    // ------------------------------------------------------------------
    // softmax + epilogue: thread (slot i = TMEM lane i, head block hb) holds
    // pseudo-heads 64hb .. 64hb+63 of slot i as two blocks of 32 (sub = 0,
    // 1); lane L keeps the reference (running max) and this warp's running
    // sum of heads 64hb + 32sub + L (scaled scores, base 2).  Every tile, the
    // 8 warps of the pair that hold head block hb exchange their per-head
    // tile maxima, block by block: each posts its 32 values into its own
    // CTA's buffer (and arrives, arming the peer's 128 bytes) and into the
    // peer's with st.async, which completes on the peer's barrier; block 0's
    // exchange is in flight while block 1's maxima are taken, block 1's
    // while block 0's P is made.  All 8 warps compute the same reference.
    // It moves only when the tile max of a head exceeds it by more than
    // kTau (lazy rescale), so O is rarely rescaled and P stays below 2^kTau.
    // ------------------------------------------------------------------
    const int hb = warp >> 2;
    const int qw = warp & 3;
    const int key = qw * 32 + lane;  // 0..127: this CTA's slot of the tile
    const int slot8 = 4 * rank + qw; // this warp among the 8 of head block hb
    const uint32_t lane_off = (uint32_t)(qw * 32) << 16;
    const float c_log2 = a.scale * 1.4426950408889634f;   // scale / ln 2 > 0
    float* red = reinterpret_cast<float*>(smem + C::OFF_RED);
    const uint32_t red_peer = map_peer(smem_u32(red), rank ^ 1);
    float* negm = reinterpret_cast<float*>(smem + C::OFF_NEGM) + warp * 64;
    // this slot's P row: in this CTA's P buffer when it supplies heads of
    // block hb (hb == rank), else in the staging buffer, whose rows of this
    // warp are copied as one block into the peer's P buffer (rows 128 rank
    // + 32 qw ..)
    const bool p_local = hb == rank;
    const uint32_t p_row = p_local ? smem_u32(smem + C::OFF_P) + (uint32_t)(BK * rank + key) * 128u
                                   : smem_u32(smem + C::OFF_STG) + (uint32_t)key * 128u;
    const uint32_t stg_warp = smem_u32(smem + C::OFF_STG) + (uint32_t)(32 * qw) * 128u;
    const uint32_t peer_rows = map_peer(smem_u32(smem + C::OFF_P) + (uint32_t)(BK * rank + 32 * qw) * 128u, rank ^ 1);
    uint32_t gt = 0, lgq = 0;
    uint32_t xph[2] = {0, 0};   // exchanges of block 0 / 1 so far
    bool ok = true;

    // Post this warp's 32 values (lane L: head 64hb + 32sub + L) of an
    // exchange of block `sub`; returns the buffer parity it used.
    auto post = [&](int sub, float v) -> uint32_t {
      const uint32_t par = xph[sub] & 1;
      const uint32_t bidx = (par * 2 + hb) * 2 + sub;
      const uint32_t idx = (bidx * 8 + slot8) * 32 + lane;
      red[idx] = v;
      __syncwarp();
      if (lane == 0) mbar_arrive_expect_tx(&bars[B_XB + bidx], 128u);
      st_async_f32(red_peer + idx * 4u, v, map_peer(smem_u32(&bars[B_XB + bidx]), rank ^ 1));
      return par;
    };
    // Wait for the exchange of block `sub` posted with parity `par`: all 8
    // warps' values are then in red[.. bidx * 256 ..].
    auto wait_x = [&](int sub, uint32_t par) -> bool {
      const uint32_t bidx = (par * 2 + hb) * 2 + sub;
      const bool w_ok = mbar_wait_cluster_warp(&bars[B_XB + bidx], (xph[sub] >> 1) & 1, abort_flag, err);
      ++xph[sub];
      return w_ok;
    };
    auto gathered = [&](int sub, uint32_t par, bool is_max) -> float {
      const uint32_t base = (((par * 2 + hb) * 2 + sub) * 8) * 32 + lane;
      float r = is_max ? -INFINITY : 0.f;
#pragma unroll
      for (int w8 = 0; w8 < 8; ++w8) r = is_max ? fmaxf(r, red[base + 32 * w8]) : r + red[base + 32 * w8];
      return r;
    };

    // Epilogue of a group (et0: its first token, enrows: its pseudo-head
    // rows, em / el: the reference and this warp's running sums): the
    // pair's sums, lse, and out = O / l.  It runs once the next group's
    // first tile has stored its P, so the group's last P.V overlaps that
    // softmax instead of being waited for; O is released to the next
    // group's P.V as soon as it has been read.
    auto epilogue = [&](int et0, int enrows, const float* em, const float* el) -> bool {
      // both blocks' partial sums posted before either is waited for (one round trip)
      uint32_t pp[2];
      pp[0] = post(0, el[0]);
      pp[1] = post(1, el[1]);
      float l[2];
#pragma unroll
      for (int sub = 0; sub < 2; ++sub) {
        if (!wait_x(sub, pp[sub])) return false;
        l[sub] = gathered(sub, pp[sub], false);
      }
      float inv_l[2];
#pragma unroll
      for (int sub = 0; sub < 2; ++sub) {
        inv_l[sub] = (l[sub] > 0.f) ? 1.0f / l[sub] : 0.f;
        const int p = 64 * hb + 32 * sub + lane;
        if (leader && qw == 0 && p < enrows)
          a.lse[(size_t)et0 * H + p] = (l[sub] > 0.f) ? (em[sub] + log2f(l[sub])) * 0.6931471805599453f : -INFINITY;
      }
      // 1/l of the warp's 64 heads, read back as broadcasts (head 64hb + hl at negm[hl])
      negm[lane] = inv_l[0];
      negm[32 + lane] = inv_l[1];
      __syncwarp();
      if (!mbar_wait_cluster_warp(&bars[B_OF], lgq & 1, abort_flag, err)) return false;
      tc_fence_after();
      // O^T lane = output column: lanes 2i and 2i+1 hold adjacent columns; for
      // each pair of heads (hl, hl+1) the even lane takes head hl of both
      // columns and the odd lane head hl+1 (one exchange), so each stores one
      // bf16 pair.  All of O is read, scaled and packed before O is released
      // to the next group's P.V; the stores follow.
      const uint32_t odd = (uint32_t)(lane & 1);
      uint32_t pk[2][32];   // [M-block][head pair]: bf16 x2 of this lane's head of the pair
#pragma unroll
      for (int b = 0; b < 2; ++b) {
#pragma unroll
        for (int q32 = 0; q32 < 2; ++q32) {
          // two 16-column loads in flight per wait
          float o[32];
          tmem_ld16(tmem + lane_off + C::COL_O + b * HP + 64 * hb + 32 * q32, o);
          tmem_ld16(tmem + lane_off + C::COL_O + b * HP + 64 * hb + 32 * q32 + 16, o + 16);
          tmem_ld_wait();
#pragma unroll
          for (int h = 0; h < 32; h += 2) {
            const int hl = 32 * q32 + h;   // heads 64hb + hl (even lane), + hl + 1 (odd lane)
            const float mine = odd ? o[h + 1] : o[h];
            const float x = __shfl_xor_sync(0xffffffffu, odd ? o[h] : o[h + 1], 1);
            const float il = negm[hl + odd];
            pk[b][hl / 2] = odd ? pack_bf16x2(x * il, mine * il) : pack_bf16x2(mine * il, x * il);
          }
        }
      }
      tc_fence_before();
      warp_arrive_leader(&bars[B_OE]);
      ++lgq;
      uint16_t* out_g = a.out + (size_t)(et0 * H + 64 * hb) * 512 + 128 * rank + (key & ~1);
#pragma unroll
      for (int b = 0; b < 2; ++b) {
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int hl = 2 * i + (int)odd;
          if (64 * hb + hl < enrows)
            *reinterpret_cast<uint32_t*>(out_g + (size_t)hl * 512 + 256 * b) = pk[b][i];
        }
      }
      return true;
    };

    bool pend = false;   // a group whose epilogue has not run yet
    int pe_t0 = 0, pe_nrows = 0;
    float pe_m[2] = {0.f, 0.f}, pe_l[2] = {0.f, 0.f};
    for (int g = cid; g < a.num_groups && ok; g += ncl) {
      int t0, n;
      group_of(a.req, G, g, t0, n);
      const int U = min(__ldg(a.union_len + g), a.union_pad);
      const int ntiles = (U + PT - 1) / PT;
      const int nrows = n * H;
      const uint8_t* mrow = a.mask + (size_t)g * a.union_pad;
      if (ntiles == 0) {
        // no union rows: zero output and lse = -inf; CTA r writes columns
        // 256b + 128r + key of the heads of block hb
        for (int h = 0; h < 64; ++h) {
          const int p = 64 * hb + h;
          if (p < nrows) {
            for (int b = 0; b < 2; ++b) a.out[(size_t)(t0 * H + p) * 512 + 256 * b + 128 * rank + key] = 0;
            if (leader && key == 0) a.lse[(size_t)t0 * H + p] = -INFINITY;
          }
        }
        continue;
      }
      // the token (bit of the mask byte) of each head of the two blocks
      int t_lo[2], split[2];
#pragma unroll
      for (int sub = 0; sub < 2; ++sub) {
        const int base = 64 * hb + 32 * sub;
        t_lo[sub] = base / H;
        split[sub] = (t_lo[sub] + 1) * H - base;
      }
      float m_l[2] = {-INFINITY, -INFINITY};   // reference of heads 64hb + 32sub + lane (scaled, base 2)
      float l_l[2] = {0.f, 0.f};               // this warp's running sums of the same heads
      for (int j = 0; j < ntiles; ++j, ++gt) {
        const int sb = gt & 1;
        const int u = j * PT + BK * rank + key;
        const uint32_t mbyte = (u < U) ? (uint32_t)__ldg(mrow + u) : 0u;
        if (!mbar_wait_cluster_warp(&bars[B_SF + sb], (gt >> 1) & 1, abort_flag, err)) { ok = false; break; }
        if (key == 0 && hb == 0) DSA_TRACE(a.tr, gt, 3);
        tc_fence_after();
        float s[2][32];
        const uint32_t s_addr = tmem + lane_off + C::COL_S + sb * HP + 64 * hb;
#pragma unroll
        for (int q16 = 0; q16 < 4; ++q16) tmem_ld16(s_addr + 16 * q16, &s[q16 >> 1][16 * (q16 & 1)]);
        tmem_ld_wait();
        tc_fence_before();
        warp_arrive_leader(&bars[B_SE + sb]);
        // mask (raw scores; the scale is positive, so maxima commute with
        // it) and each block's per-head maxima over this warp's 32 slots,
        // lane h keeping head h's, posted as soon as they are taken
        uint32_t par[2];
#pragma unroll
        for (int sub = 0; sub < 2; ++sub) {
          // the block's 32 heads belong to one token, or (H = 16) to two
          // split at head 16: split is 16 or at least 32 (H = 128 / G)
          const bool on_lo = (mbyte >> t_lo[sub]) & 1u;
          const bool on_hi = split[sub] < 32 ? ((mbyte >> (t_lo[sub] + 1)) & 1u) != 0 : on_lo;
          // (each warp-wide max goes to this warp's negm area, every lane
          // storing the same value to the same word; lane L reads head L's
          // back: cheaper than selecting it lane by lane.  negm is rewritten
          // with the reference only after these are read.)
#pragma unroll
          for (int h = 0; h < 32; ++h) {
            const bool on = (h < 16) ? on_lo : on_hi;
            s[sub][h] = on ? s[sub][h] : -INFINITY;
            float r;
            asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(s[sub][h]));
            negm[32 * sub + h] = r;
          }
          __syncwarp();
          par[sub] = post(sub, negm[32 * sub + lane]);
        }
        // P buffer pb (in both CTAs) is free once the P.V two tiles back is
        // done; the staging rows once the peer acknowledged the last copy
        const int pb = gt & 1;
        if (!mbar_wait_cluster_warp(&bars[B_PE + pb], ((gt >> 1) & 1) ^ 1, abort_flag, err)) { ok = false; break; }
        if (!p_local && !mbar_wait_cluster_warp(&bars[B_STG], (gt & 1) ^ 1, abort_flag, err)) { ok = false; break; }
        if (key == 0 && hb == 0) DSA_TRACE(a.tr, gt, 5);
        const uint32_t p_dst = p_row + (p_local ? (uint32_t)pb * C::P_BYTES : 0u);
        // block by block: the pair's tile max, the reference (the same in
        // both CTAs: the same inputs in the same order), then P = 2^(c s - m)
        // rounded to bf16 (0 for masked slots), stored as it is made: P^T of
        // this slot, heads 64hb .. 64hb+63, row 128 rank + key of CTA hb's
        // P buffer (or of the staging rows), 128 bytes = 8 chunks of 8
        // heads, chunk c at (c ^ (row & 7)) * 16 (128-byte swizzle,
        // MN-major); and the row sums (of P before its rounding to bf16)
        float alpha[2] = {1.f, 1.f};
        const uint32_t sw = (uint32_t)(key & 7);
#pragma unroll
        for (int sub = 0; sub < 2; ++sub) {
          if (!wait_x(sub, par[sub])) { ok = false; break; }
          const float tm = gathered(sub, par[sub], true) * c_log2;
          if (tm > m_l[sub] + kTau) {
            alpha[sub] = (m_l[sub] == -INFINITY) ? 0.f : exp2f(m_l[sub] - tm);
            m_l[sub] = tm;
            l_l[sub] *= alpha[sub];
          }
          negm[32 * sub + lane] = (m_l[sub] == -INFINITY) ? 0.f : -m_l[sub];
          __syncwarp();
#pragma unroll
          for (int h = 0; h < 32; h += 8) {
            const float4 n0 = *reinterpret_cast<const float4*>(negm + 32 * sub + h);
            const float4 n1 = *reinterpret_cast<const float4*>(negm + 32 * sub + h + 4);
            float p[8];
            p[0] = exp2f(fmaf(s[sub][h + 0], c_log2, n0.x));
            p[1] = exp2f(fmaf(s[sub][h + 1], c_log2, n0.y));
            p[2] = exp2f(fmaf(s[sub][h + 2], c_log2, n0.z));
            p[3] = exp2f(fmaf(s[sub][h + 3], c_log2, n0.w));
            p[4] = exp2f(fmaf(s[sub][h + 4], c_log2, n1.x));
            p[5] = exp2f(fmaf(s[sub][h + 5], c_log2, n1.y));
            p[6] = exp2f(fmaf(s[sub][h + 6], c_log2, n1.z));
            p[7] = exp2f(fmaf(s[sub][h + 7], c_log2, n1.w));
            const uint32_t c = (uint32_t)(4 * sub + h / 8);
            const uint32_t addr = p_dst + ((c ^ sw) << 4);
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(pack_bf16x2(p[0], p[1])),
                         "r"(pack_bf16x2(p[2], p[3])), "r"(pack_bf16x2(p[4], p[5])), "r"(pack_bf16x2(p[6], p[7]))
                         : "memory");
#pragma unroll
            for (int i = 0; i < 8; ++i) s[sub][h + i] = p[i];
          }
          l_l[sub] += warp_transpose_reduce32<false>(s[sub]);
        }
        if (!ok) break;
        if (key == 0 && hb == 0) DSA_TRACE(a.tr, gt, 1);
        if (j > 0 && __any_sync(0xffffffffu, alpha[0] != 1.f || alpha[1] != 1.f)) {
          // O must hold the previous tile's P.V before it is rescaled
          if (!mbar_wait_cluster_warp(&bars[B_PE + (pb ^ 1)], ((gt - 1) >> 1) & 1, abort_flag, err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          // O^T lane = this CTA's output column of M-block b, TMEM columns = heads
#pragma unroll 1
          for (int b = 0; b < 2; ++b) {
#pragma unroll 1
            for (int q16 = 0; q16 < 4; ++q16) {
              float o[16];
              const uint32_t ta = tmem + lane_off + C::COL_O + b * HP + 64 * hb + 16 * q16;
              tmem_ld16(ta, o);
              tmem_ld_wait();
              const float av = (q16 >> 1) ? alpha[1] : alpha[0];
#pragma unroll
              for (int h = 0; h < 16; ++h) o[h] *= __shfl_sync(0xffffffffu, av, 16 * (q16 & 1) + h);
              tmem_st16(ta, o);
            }
          }
          tmem_st_wait();
        }
        // P (and the rescale) visible to the tensor core; the peer-bound
        // rows go out as one 4 KB copy; then this warp's arrival on P_RX
        // (the warps holding this CTA's own heads also arm the 16 KB the
        // peer copies in)
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (!p_local)
            bulk_copy_to_peer(peer_rows + (uint32_t)pb * C::P_BYTES, stg_warp, 32u * 128u,
                              map_peer(smem_u32(&bars[B_PRX + pb]), rank ^ 1));
          if (p_local)
            mbar_arrive_expect_tx(&bars[B_PRX + pb], 32u * 128u);
          else
            mbar_arrive(&bars[B_PRX + pb]);
        }
        if (key == 0 && hb == 0) DSA_TRACE(a.tr, gt, 6);
        if (j == 0 && pend) {
          if (!epilogue(pe_t0, pe_nrows, pe_m, pe_l)) {
            ok = false;
            break;
          }
          pend = false;
        }
      }
      if (!ok) break;
      // this group's epilogue waits for the next group's first tile
      pend = true;
      pe_t0 = t0;
      pe_nrows = nrows;
      pe_m[0] = m_l[0];
      pe_m[1] = m_l[1];
      pe_l[0] = l_l[0];
      pe_l[1] = l_l[1];
    }
    if (ok && pend) epilogue(pe_t0, pe_nrows, pe_m, pe_l);
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // neither CTA leaves or frees tensor memory while the pair may still use it
  tc_fence_after();
  if (warp == 8) tmem_dealloc_pair(tmem, C::TMEM_COLS);
}

template <int NC>
static int launch_t(const GroupedArgs& a, int num_sms, cudaStream_t stream) {
  using C = Cfg;
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
