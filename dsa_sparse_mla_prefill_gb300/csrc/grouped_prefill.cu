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
// A group is processed by a cluster of two CTAs that split the pseudo-heads:
// CTA r owns pseudo-heads 64r .. 64r+63 (its q rows: 64 x D_QK) and the
// matching 64 columns of the output.  Each CTA gathers every union row of
// the group into its own shared memory (plain tile::gather4 loads, no
// multicast) and releases each stage with its own MMA commit; the pair shares
// nothing but the group, whose rows the two CTAs read from L2 at the same
// time.  No scores cross the cluster.  Within a CTA the data path is the
// per-token one with 64 heads:
//   S^T = K q^T with the union slots on the M side (M = 128 slots, N = 64),
//   streamed chunk by chunk through a K ring whose stages hold a K chunk
//   (128 slots x 64 columns) and the matching q chunk (64 rows x 64
//   columns, re-read from L2 every tile: q is not kept resident, which
//   leaves room for five stages);
//   O^T += V^T P^T per 128-column V unit (V re-gathered into a V ring, an L2
//   hit), O^T = 4 x 64 TMEM columns, P^T in shared memory (one or two buffers);
//   the online softmax (base 2, lazy rescale) runs with thread i <-> slot i
//   (TMEM lane i) in eight warps, two per lane quarter, each holding 32 of
//   the 64 pseudo-heads.
// Warp roles (24 warps): 0-7 softmax (at REGS_SOFTMAX registers, the others
// at REGS_OTHER), 8 and 11 QK issuers (alternate K chunks, two partial S^T
// sums; warp 11 idle for 8-chunk rows), 9 and 10 PV issuers (units 0/2 and
// 1/3), 12-17 K-ring producers (one per stage for 9-chunk rows, all six on
// every stage for 8-chunk rows), 18-23 V-ring producers (all six on every
// V unit).
#include "dsa_device.cuh"
#include "dsa_kernels.h"

namespace dsa {
namespace grouped {

constexpr int BK = 128;          // union slots per tile (the MMA's M)
constexpr int HC = 64;           // pseudo-heads per CTA (the MMA's N)
constexpr int HW = 32;           // pseudo-heads per softmax warp
constexpr int NTHREADS = 768;    // 24 warps, launched at 80 registers each
constexpr int REGS_SOFTMAX = 144;
constexpr int REGS_OTHER = 48;   // 8*32*144 + 16*32*48 <= 768*80
constexpr int NKW = 6;           // K producer warps (one per K stage)
constexpr int NVR = 2;           // V ring slots: unit m in slot m mod 2, PV issuer m mod 2
constexpr float kTau = 8.0f;     // lazy-rescale threshold (log2 units)

template <int NC>
struct Cfg {
  // QK issuing threads: two for the 9-chunk (NoPE + RoPE) rows, where one
  // thread's per-chunk wait, fence and commit set the tile period; one for
  // 8-chunk rows, where two made the softmax the slower stage (measured)
  static constexpr int NQ = (NC % 2) ? 2 : 1;
  // K ring stages (K chunk + q chunk each); even with two issuers, so that
  // stage s is issuer s & 1's.  With two issuers the softmax keeps ahead of
  // P.V, so one P^T buffer serves and its 16 KB go to the K ring.
  static constexpr int NKR = NQ == 2 ? 6 : 5;
  static constexpr int NPB = NQ == 2 ? 1 : 2;   // P^T buffers
  // slack for aligning the dynamic shared memory to 1024 bytes; the 6-stage
  // layout has no room for it and requires an aligned base (checked at
  // entry: the launch stops and counts an early stop otherwise)
  static constexpr uint32_t ALIGN_SLACK = NQ == 2 ? 0u : 1024u;
  // K producers: with two issuers warp 12+s owns stage s (17 lanes issue a
  // stage); with one, all six warps take part in every stage (3 lanes each).
  // Both measured per layout: each is the faster one where it is used.
  static constexpr bool OWNED = NQ == 2;
  static constexpr uint32_t CHUNK_BYTES = BK * 128u;          // 128 slots x 64 columns
  static constexpr uint32_t UNIT_BYTES = 2u * CHUNK_BYTES;    // 128 slots x 128 columns
  static constexpr uint32_t Q_CHUNK = HC * 128u;              // 64 rows x 64 columns
  static constexpr uint32_t KSTAGE_BYTES = CHUNK_BYTES + Q_CHUNK;
  static constexpr uint32_t P_BYTES = 2u * HC * 128u;         // one buffer: 128 slots = 2 swizzle columns
  static constexpr uint32_t RED_BYTES = 2u * 2u * 4u * HW * 4u;  // [parity][half][warp][head]
  static constexpr uint32_t OFF_KR = 0;
  static constexpr uint32_t OFF_VR = OFF_KR + NKR * KSTAGE_BYTES;
  static_assert(NKR <= NKW && (NQ == 1 || NKR % 2 == 0), "K ring layout: one producer warp per stage");
  static constexpr uint32_t OFF_P = OFF_VR + NVR * UNIT_BYTES;
  static constexpr uint32_t OFF_RED = OFF_P + NPB * P_BYTES;
  static constexpr uint32_t OFF_BAR = OFF_RED + RED_BYTES;
  static constexpr int NBAR = 32;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8u;
  static constexpr uint32_t SMEM_BYTES = OFF_MISC + 128u + ALIGN_SLACK;
  static_assert(SMEM_BYTES <= 227u * 1024u, "shared memory budget");
  static constexpr uint32_t COL_O = 0;       // O^T: 4 units x 64 columns
  static constexpr uint32_t COL_S = 256;     // S^T: 2 buffers x 2 partial sums x 64 columns
  static constexpr uint32_t TMEM_COLS = 512;
};

enum {
  B_S_FULL = 0,      // [2] one commit per QK issuer
  B_S_EMPTY = 2,     // [2]
  B_P_FULL = 4,      // [NPB] 256 arrivals (softmax threads)
  B_P_EMPTY = 6,     // [NPB] one commit per PV issuer
  B_O_FULL = 8,      // one commit per PV issuer
  B_O_EMPTY = 9,     // 256 arrivals
  B_DRAIN = 10,      // [4] one per MMA issuer
  B_SMX_SYNC = 14,   // [2] one per head half (4 warps)
  B_KR_FULL = 16,    // [NKR <= 6]
  B_KR_EMPTY = 22,   // [NKR <= 6] one QK commit
  B_VR_FULL = 28,    // [NVR]
  B_VR_EMPTY = 30,   // [NVR] one PV commit
};
static_assert(NVR <= 2, "barrier layout");


__device__ __forceinline__ void group_of(const ReqTable& rq, int G, int g, int& t0, int& n) {
  int r = 0;
  while (r + 1 < rq.num_req && rq.cu_g[r + 1] <= g) ++r;
  t0 = rq.cu_q[r] + (g - rq.cu_g[r]) * G;
  n = min(G, rq.cu_q[r + 1] - t0);
}

// The four union slots 4rg .. 4rg+3 of tile j (row indices; -1 past the
// union or out of range, which TMA reads as zeros).  Nothing at or past U is
// read: a tile may run past the padded row.
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

template <int NC>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NTHREADS, 1)
grouped_prefill_kernel(const __grid_constant__ GroupedArgs a) {
  using C = Cfg<NC>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  if (C::ALIGN_SLACK == 0 && (raw_u32 & 1023u) != 0) {
    // same base in every CTA of the launch: the whole grid stops here
    if (threadIdx.x == 0) atomicAdd(a.err + ERR_TIMEOUT, 1u);
    return;
  }
  uint8_t* smem = smem_raw + (((raw_u32 + 1023u) & ~1023u) - raw_u32);
  const uint32_t sbase = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile uint32_t* tmem_base_ptr = misc;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 1);
  float* red = reinterpret_cast<float*>(smem + C::OFF_RED);
  unsigned int* err = a.err;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int rank = (int)cluster_ctarank();
  const int H = a.H;
  const int G = a.G;
  const int cid = (int)cluster_id_x();
  const int ncl = (int)nclusters_x();

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars[B_S_FULL + i], C::NQ);
      mbar_init(&bars[B_S_EMPTY + i], 256);
      mbar_init(&bars[B_SMX_SYNC + i], 128);
    }
    for (int i = 0; i < C::NPB; ++i) {
      mbar_init(&bars[B_P_FULL + i], 256);
      mbar_init(&bars[B_P_EMPTY + i], 2);
    }
    mbar_init(&bars[B_O_FULL], 2);
    mbar_init(&bars[B_O_EMPTY], 256);
    for (int i = 0; i < 4; ++i) mbar_init(&bars[B_DRAIN + i], 1);
    for (int i = 0; i < C::NKR; ++i) {
      mbar_init(&bars[B_KR_FULL + i], 1);
      mbar_init(&bars[B_KR_EMPTY + i], 1);
    }
    for (int i = 0; i < NVR; ++i) {
      mbar_init(&bars[B_VR_FULL + i], 1);
      mbar_init(&bars[B_VR_EMPTY + i], 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 8) {
    tmem_alloc(const_cast<uint32_t*>(tmem_base_ptr), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs of the pair start together
  tc_fence_after();
  const uint32_t tmem = *tmem_base_ptr;

  if (warp >= 8) {
    regs_dec<REGS_OTHER>();
    if (warp >= 12) {
      // ----------------------------------------------------------------
      // TMA producers.  K stream (warps 12-17): a stage holds K chunk c of a
      // tile (128 slots x columns 64c .. 64c+63) plus q chunk c of this CTA's
      // 64 pseudo-heads; requests 0-31 gather the tile's 32 row groups of 4
      // slots, request 32 loads the q chunk.  OWNED: warp 12+s fills stage s
      // with every chunk that maps there, lane l gathering row group l and
      // lane 0 also loading q (a warp's per-stage loop of wait, arm and
      // issue costs several hundred cycles, so stages are filled side by
      // side); otherwise all six warps take part in every stage, lanes 0-5
      // of each.  V stream (warps 18-23): the 128-column units m of every
      // tile go to V slot m mod 2; all six warps take part in every unit,
      // lanes 0-10 of each sharing its 64 gathers (32 row groups x 2 swizzle
      // columns; a unit's refill sits on the P.V critical path twice per
      // tile, so its issue time matters).
      // When a 64-slot half of the tile is one contiguous run of rows, the
      // half is one tiled load (box 64 columns x 64 rows) instead of 16
      // gathers.  The union lists distinct rows in ascending order, so the
      // run test needs only the half's two end slots.
      // A stage's leader (lane 0 of its K warp, or of warp 12, and of warp
      // 18 for V) arms the full byte count of the stage.  Every warp of a
      // slot passes through each of its phases in order.
      // ----------------------------------------------------------------
      const bool kstream = warp < 18;
      const int kw = warp - 12;                 // K stage owned (OWNED; none past the ring)
      // K request of this lane: 0-31 gathers, 32 the q chunk (OWNED: lane 0
      // issues its gather and the q chunk)
      const int kreq = C::OWNED ? lane : kw * 6 + (lane < 6 ? lane : 64);
      const bool kq = kstream && (C::OWNED ? lane == 0 : kreq == 32);
      // V: all six warps take part in every unit, lanes 0-10 of each
      const int e = (warp - 18) * 11 + (lane < 11 ? lane : 64);   // V gather index 0..63
      const bool issuer = kstream ? (kreq < 33) : (e < 64);
      const bool kgather = kstream && kreq < 32;
      const int rg = kstream ? (kreq & 31) : (e & 31);   // row group of the tile
      const int hf = rg >> 4;                            // its 64-slot half
      const int vcc = (e >> 5) & 1;             // V swizzle column
      const bool leader = (lane == 0) && (kstream ? (C::OWNED || kw == 0) : warp == 18);
      uint32_t gt = 0, pos = 0;
      int64_t last_armed = -1;
      bool ok = true;
      for (int g = cid; g < a.num_groups && ok; g += ncl) {
        int t0, n;
        group_of(a.req, G, g, t0, n);
        const int U = min(__ldg(a.union_len + g), a.union_pad);
        const int ntiles = (U + BK - 1) / BK;
        if (ntiles == 0) continue;
        const int32_t* urow = a.union_idx + (size_t)g * a.union_pad;
        for (int j = 0; j < ntiles && ok; ++j, ++gt) {
          if (warp == 12 && lane == 0) DSA_TRACE(a.tr, gt, 0);
          const int u0 = j * BK + 64 * hf;     // this lane's 64-slot half of the tile
          int first = -1;
          bool run = false;
          if (u0 + 63 < U) {
            first = __ldg(urow + u0);
            const int last = __ldg(urow + u0 + 63);
            run = first >= 0 && last < a.N && last - first == 63;
          }
          const uint32_t half_off = (uint32_t)hf * (C::CHUNK_BYTES / 2);
          const bool run_lead = (rg & 15) == 0;   // issues the half's tiled load
          if (kstream) {
            const int4 r = (kgather && !run) ? union_rows4(urow, U, a.N, j * BK + 4 * rg) : make_int4(-1, -1, -1, -1);
            for (int c = 0; c < NC; ++c, ++pos) {
              const int ks = (int)(pos % C::NKR);
              if (C::OWNED && ks != kw) continue;
              if (!mbar_wait_warp(&bars[B_KR_EMPTY + ks], ((pos / C::NKR) & 1) ^ 1, abort_flag, err)) {
                ok = false;
                break;
              }
              const uint32_t stage = sbase + C::OFF_KR + ks * C::KSTAGE_BYTES;
              if (leader) mbar_arrive_expect_tx(&bars[B_KR_FULL + ks], C::KSTAGE_BYTES);
              if (kgather) {
                if (run) {
                  if (run_lead) tma_load_2d(stage + half_off, &a.tmap_kv_blk, c * 64, first, &bars[B_KR_FULL + ks]);
                } else {
                  tma_gather4(stage + rg * 512, &a.tmap_kv, c * 64, r.x, r.y, r.z, r.w, &bars[B_KR_FULL + ks]);
                }
              }
              if (kq)
                // q rows t0*H + 64 rank .. +63 of q viewed [T*H, D_QK], columns 64c ..
                tma_load_2d(stage + C::CHUNK_BYTES, &a.tmap_q, c * 64, t0 * H + HC * rank, &bars[B_KR_FULL + ks]);
              last_armed = pos;
            }
          } else {
            const int4 r = (issuer && !run) ? union_rows4(urow, U, a.N, j * BK + 4 * rg) : make_int4(-1, -1, -1, -1);
            for (int m = 0; m < 4; ++m, ++pos) {
              const int vg = (int)(pos % NVR);   // V slot of this unit
              if (!mbar_wait_warp(&bars[B_VR_EMPTY + vg], ((pos / NVR) & 1) ^ 1, abort_flag, err)) {
                ok = false;
                break;
              }
              if (leader) mbar_arrive_expect_tx(&bars[B_VR_FULL + vg], C::UNIT_BYTES);
              const uint32_t vdst = sbase + C::OFF_VR + vg * C::UNIT_BYTES + vcc * C::CHUNK_BYTES;
              if (run) {
                if (issuer && run_lead)
                  tma_load_2d(vdst + half_off, &a.tmap_kv_blk, (2 * m + vcc) * 64, first, &bars[B_VR_FULL + vg]);
              } else if (issuer) {
                tma_gather4(vdst + rg * 512, &a.tmap_kv, (2 * m + vcc) * 64, r.x, r.y, r.z, r.w,
                            &bars[B_VR_FULL + vg]);
              }
              last_armed = pos;
            }
          }
        }
      }
      // Let copies still in flight land before the CTA can exit: the last
      // phase of every stage this warp's leader armed completes only once
      // all of its bytes have landed.
      if (leader && last_armed >= 0) {
        if (kstream) {
          // the last phase of every stage this leader armed
          for (int64_t p = last_armed; p >= 0 && p > last_armed - C::NKR; --p)
            if (!C::OWNED || (int)(p % C::NKR) == kw)
              mbar_wait_drain(&bars[B_KR_FULL + (int)(p % C::NKR)], (uint32_t)(p / C::NKR) & 1, err);
        } else {
          for (int64_t p = last_armed; p >= 0 && p > last_armed - NVR; --p)
            mbar_wait_drain(&bars[B_VR_FULL + (int)(p % NVR)], (uint32_t)(p / NVR) & 1, err);
        }
      }
      __syncwarp();
    } else if (warp == 8 || (warp == 11 && C::NQ == 2)) {
      // ----------------------------------------------------------------
      // QK issuers: S^T = K q^T chunk by chunk.  With two issuing threads
      // the chunks alternate between them (warp 8 takes ring positions of
      // even parity, warp 11 odd ones; with an even ring size each stage
      // belongs to one of them), each summing into its own partial S^T; the
      // softmax adds the two.  One thread issuing every chunk spends most of
      // its time in the per-chunk wait, fence and commit, not in MMAs.
      // Each K chunk is released to the producers once its MMAs complete;
      // S_FULL takes one commit from each issuer.
      // ----------------------------------------------------------------
      const uint32_t qa = warp == 8 ? 0u : 1u;
      if (lane == 0) {
        constexpr uint32_t IDESC_QK = idesc_bf16_f32(128, HC, false, false);
        uint32_t gt = 0, kpos = 0;
        bool ok = true;
        for (int g = cid; g < a.num_groups && ok; g += ncl) {
          const int U = min(__ldg(a.union_len + g), a.union_pad);
          const int ntiles = (U + BK - 1) / BK;
          if (ntiles == 0) continue;
          for (int j = 0; j < ntiles && ok; ++j, ++gt) {
            const int sb = gt & 1;
            const uint32_t d_s = tmem + C::COL_S + (2 * sb + qa) * HC;
            if (!mbar_wait(&bars[B_S_EMPTY + sb], ((gt >> 1) & 1) ^ 1, abort_flag, err)) { ok = false; break; }
            if (qa == 0) DSA_TRACE(a.tr, gt, 2);
            tc_fence_after();
            bool first = true;
            for (int c = 0; c < NC; ++c, ++kpos) {
              if (C::NQ == 2 && (kpos & 1u) != qa) continue;
              const uint32_t slot = kpos % C::NKR;
              if (!mbar_wait(&bars[B_KR_FULL + slot], (kpos / C::NKR) & 1, abort_flag, err)) { ok = false; break; }
              tc_fence_after();
              const uint32_t stage = sbase + C::OFF_KR + slot * C::KSTAGE_BYTES;
              mma_bf16_ss_x4(d_s, sdesc_sw128(stage, 16, 1024), sdesc_sw128(stage + C::CHUNK_BYTES, 16, 1024), 2u, 2u,
                             IDESC_QK, first ? 0u : 1u);
              mma_commit(&bars[B_KR_EMPTY + slot]);
              first = false;
            }
            if (!ok) break;
            if (qa == 0) DSA_TRACE(a.tr, gt, 1);
            mma_commit(&bars[B_S_FULL + sb]);
          }
        }
        mma_commit(&bars[B_DRAIN + 2 + qa]);
        mbar_wait(&bars[B_DRAIN + 2 + qa], 0, abort_flag, err);
      }
      __syncwarp();
    } else if (warp == 9 || warp == 10) {
      // ----------------------------------------------------------------
      // PV issuers: O^T += V^T P^T, warp 9 for units 0 and 2, warp 10 for
      // units 1 and 3 (V slot = unit mod 2); each unit released to the
      // producers once its MMAs complete
      // ----------------------------------------------------------------
      const int pvi = warp - 9;
      if (lane == 0) {
        constexpr uint32_t IDESC_PV = idesc_bf16_f32(128, HC, true, false);
        const uint32_t p_base = sbase + C::OFF_P;
        uint32_t gt = 0, lgq = 0;
        bool ok = true;
        for (int g = cid; g < a.num_groups && ok; g += ncl) {
          const int U = min(__ldg(a.union_len + g), a.union_pad);
          const int ntiles = (U + BK - 1) / BK;
          if (ntiles == 0) continue;
          for (int j = 0; j < ntiles && ok; ++j, ++gt) {
            const int pb = C::NPB == 2 ? (int)(gt & 1) : 0;
            const uint32_t pph = C::NPB == 2 ? (gt >> 1) : gt;   // phase of P buffer pb
            if (!mbar_wait(&bars[B_P_FULL + pb], pph & 1, abort_flag, err)) { ok = false; break; }
            if (pvi == 0) DSA_TRACE(a.tr, gt, 7);
            tc_fence_after();
            if (j == 0) {
              if (!mbar_wait(&bars[B_O_EMPTY], (lgq & 1) ^ 1, abort_flag, err)) { ok = false; break; }
              tc_fence_after();
            }
            for (int m = pvi; m < 4 && ok; m += 2) {
              const uint32_t vp = gt * 4 + m;
              if (!mbar_wait(&bars[B_VR_FULL + pvi], (vp / NVR) & 1, abort_flag, err)) { ok = false; break; }
              tc_fence_after();
              const uint32_t ubase = sbase + C::OFF_VR + pvi * C::UNIT_BYTES;
              const uint32_t d_o = tmem + C::COL_O + m * HC;
#pragma unroll
              for (int hf = 0; hf < 2; ++hf) {
                // 16 slots (2048 B of V^T, MN-major; the unit's two swizzle
                // columns CHUNK_BYTES apart) per MMA; P^T one 64-slot
                // swizzle column per half
                const uint64_t adesc = sdesc_sw128(ubase + hf * 4 * 2048, C::CHUNK_BYTES, 1024);
                const uint64_t bdesc = sdesc_sw128(p_base + pb * C::P_BYTES + hf * (HC * 128), 16, 1024);
                mma_bf16_ss_x4(d_o, adesc, bdesc, 128u, 2u, IDESC_PV, (j > 0 || hf > 0) ? 1u : 0u);
              }
              mma_commit(&bars[B_VR_EMPTY + pvi]);
            }
            if (!ok) break;
            mma_commit(&bars[B_P_EMPTY + pb]);
            if (j == ntiles - 1) mma_commit(&bars[B_O_FULL]);
          }
          ++lgq;
        }
        mma_commit(&bars[B_DRAIN + pvi]);
        mbar_wait(&bars[B_DRAIN + pvi], 0, abort_flag, err);
      }
      __syncwarp();
    }
  } else {
    regs_inc<REGS_SOFTMAX>();
    // ------------------------------------------------------------------
    // softmax + epilogue: thread (key i = TMEM lane i, head half hh) holds
    // the 32 local pseudo-heads 32hh .. 32hh+31 of union slot i of the tile.
    // The running max and sum are per head and the same for every thread,
    // so lane L keeps them for head L only and shuffles them out.
    // ------------------------------------------------------------------
    const int hh = warp >> 2;
    const int key = (warp & 3) * 32 + lane;  // 0..127
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const float scale_log2 = a.scale * 1.4426950408889634f;
    uint64_t* smx = &bars[B_SMX_SYNC + hh];
    // token of local pseudo-head h: t_lo for h < split, t_lo + 1 after
    const int base = HC * rank + HW * hh;
    const int t_lo = base / H;
    const int split = (t_lo + 1) * H - base;
    uint32_t gt = 0, lgq = 0, sync_phase = 0;
    bool ok = true;
    for (int g = cid; g < a.num_groups && ok; g += ncl) {
      int t0, n;
      group_of(a.req, G, g, t0, n);
      const int U = min(__ldg(a.union_len + g), a.union_pad);
      const int ntiles = (U + BK - 1) / BK;
      const int nrows = n * H;
      const uint8_t* mrow = a.mask + (size_t)g * a.union_pad;
      if (ntiles == 0) {
        // no union rows: zero output, lse = -inf for this CTA's pseudo-heads
        for (int h = 0; h < HW; ++h) {
          const int p = base + h;
          if (p < nrows) {
            for (int c = key; c < 512; c += 128) a.out[(size_t)(t0 * H + p) * 512 + c] = 0;
            if (key == 0) a.lse[(size_t)t0 * H + p] = -INFINITY;
          }
        }
        continue;
      }
      float m_l = -INFINITY;  // running max of head `lane` (base 2, scaled)
      float l_l = 0.f;        // this warp's running sum of head `lane`
      for (int j = 0; j < ntiles; ++j, ++gt) {
        const int sb = gt & 1;
        const int pb = C::NPB == 2 ? (int)(gt & 1) : 0;
        const uint32_t pph = C::NPB == 2 ? (gt >> 1) : gt;   // phase of P buffer pb
        // this slot's membership byte (zero past the union)
        const int u = j * BK + key;
        const uint32_t mbyte = (u < U) ? (uint32_t)__ldg(mrow + u) : 0u;
        const bool on_lo = (mbyte >> t_lo) & 1u;
        const bool on_hi = (mbyte >> (t_lo + 1)) & 1u;
        if (!mbar_wait_warp(&bars[B_S_FULL + sb], (gt >> 1) & 1, abort_flag, err)) { ok = false; break; }
        if (key == 0 && hh == 0) DSA_TRACE(a.tr, gt, 3);
        tc_fence_after();
        // S^T = the QK issuers' partial sums
        float s[HW];
        const uint32_t s_addr = tmem + lane_off + C::COL_S + 2 * sb * HC + HW * hh;
        if constexpr (C::NQ == 2) {
#pragma unroll
          for (int q16 = 0; q16 < HW / 16; ++q16) {
            float t[16];
            tmem_ld16(s_addr + 16 * q16, s + 16 * q16);
            tmem_ld16(s_addr + HC + 16 * q16, t);
            tmem_ld_wait();
#pragma unroll
            for (int h = 0; h < 16; ++h) s[16 * q16 + h] += t[h];
          }
        } else {
#pragma unroll
          for (int q16 = 0; q16 < HW / 16; ++q16) tmem_ld16(s_addr + 16 * q16, s + 16 * q16);
          tmem_ld_wait();
        }
        tc_fence_before();
        mbar_arrive(&bars[B_S_EMPTY + sb]);
        if (key == 0 && hh == 0) DSA_TRACE(a.tr, gt, 5);
        bool mine = false;
#pragma unroll
        for (int h = 0; h < HW; ++h) {
          const bool on = (h < split) ? on_lo : on_hi;
          s[h] = on ? s[h] * scale_log2 : -INFINITY;
          mine |= (s[h] > __shfl_sync(0xffffffffu, m_l, h) + kTau);
        }
        // Lazy rescale: the tile max matters only when some score exceeds
        // the running max by more than kTau.  Each warp of the head half
        // votes; a warp that votes yes publishes its per-head max.  The new
        // reference is the max over those warps, which bounds every score of
        // the tile (the others lie within kTau of the old reference).
        const bool wneed = __any_sync(0xffffffffu, mine);
        float* redb = red + ((gt & 1) * 2 + hh) * (4 * HW);
        volatile uint32_t* vote = misc + 4 + ((gt & 1) * 2 + hh) * 4;
        if (wneed) {
          float r[HW];
#pragma unroll
          for (int h = 0; h < HW; ++h) r[h] = s[h];
          redb[(warp & 3) * HW + lane] = warp_transpose_reduce32<true>(r);
        }
        if (lane == 0) vote[warp & 3] = wneed ? 1u : 0u;
        if (!group_sync(smx, sync_phase, abort_flag, err)) { ok = false; break; }
        uint32_t vw[4];
#pragma unroll
        for (int w = 0; w < 4; ++w) vw[w] = vote[w];
        const bool need = (vw[0] | vw[1] | vw[2] | vw[3]) != 0;
        if (key == 0 && hh == 0) DSA_TRACE(a.tr, gt, 4);
        float alpha_l = 1.f;
        if (need) {
          float tm = -INFINITY;
#pragma unroll
          for (int w = 0; w < 4; ++w)
            if (vw[w]) tm = fmaxf(tm, redb[w * HW + lane]);
          const float mn = fmaxf(m_l, tm);
          alpha_l = (m_l == -INFINITY) ? 0.f : exp2f(m_l - mn);
          m_l = mn;
          l_l *= alpha_l;
        }
        // P (bf16) and its row sums first, in registers: only the stores
        // into the P^T buffer wait for the P.V that last read it (NPB tiles
        // ago); s[] becomes the bf16-rounded P for the row sums
        uint32_t pk[HW / 2];
#pragma unroll
        for (int h = 0; h < HW; h += 2) {
          const float m0 = __shfl_sync(0xffffffffu, m_l, h);
          const float m1 = __shfl_sync(0xffffffffu, m_l, h + 1);
          const uint16_t b0 = f32_to_bf16_rn(exp2f(s[h] - ((m0 == -INFINITY) ? 0.f : m0)));
          const uint16_t b1 = f32_to_bf16_rn(exp2f(s[h + 1] - ((m1 == -INFINITY) ? 0.f : m1)));
          s[h] = bf16_to_f32(b0);
          s[h + 1] = bf16_to_f32(b1);
          pk[h / 2] = (uint32_t)b0 | ((uint32_t)b1 << 16);
        }
        l_l += warp_transpose_reduce32<false>(s);
        if (!mbar_wait_warp(&bars[B_P_EMPTY + pb], (pph & 1) ^ 1, abort_flag, err)) { ok = false; break; }
        // P^T[head][slot] (K-major swizzled, 2 columns of 64 slots)
        {
          const uint32_t kcol = key & 63;
          uint8_t* pcol = smem + C::OFF_P + pb * C::P_BYTES + (key >> 6) * (HC * 128);
#pragma unroll
          for (int h = 0; h < HW; ++h)
            *reinterpret_cast<uint16_t*>(pcol + sw128_offset(HW * hh + h, kcol)) =
                (uint16_t)((h & 1) ? (pk[h / 2] >> 16) : (pk[h / 2] & 0xffffu));
        }
        if (need && j > 0) {
          // O must hold the previous tile's P.V before it is rescaled
          const int pbp = C::NPB == 2 ? (int)((gt - 1) & 1) : 0;
          const uint32_t pphp = C::NPB == 2 ? ((gt - 1) >> 1) : (gt - 1);
          if (!mbar_wait_warp(&bars[B_P_EMPTY + pbp], pphp & 1, abort_flag, err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          // O^T lane = output column 128m + key, TMEM columns = heads
#pragma unroll 1
          for (int m = 0; m < 4; ++m) {
#pragma unroll
            for (int q16 = 0; q16 < 2; ++q16) {
              float o[16];
              const uint32_t ta = tmem + lane_off + C::COL_O + m * HC + HW * hh + 16 * q16;
              tmem_ld16(ta, o);
              tmem_ld_wait();
#pragma unroll
              for (int h = 0; h < 16; ++h) o[h] *= __shfl_sync(0xffffffffu, alpha_l, 16 * q16 + h);
              tmem_st16(ta, o);
            }
          }
          tmem_st_wait();
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(&bars[B_P_FULL + pb]);
        if (key == 0 && hh == 0) DSA_TRACE(a.tr, gt, 6);
      }
      if (!ok) break;
      // -------- epilogue --------
      float* redb = red + ((gt & 1) * 2 + hh) * (4 * HW);  // not in use by the tile path now
      if (!group_sync(smx, sync_phase, abort_flag, err)) { ok = false; break; }
      redb[(warp & 3) * HW + lane] = l_l;
      if (!group_sync(smx, sync_phase, abort_flag, err)) { ok = false; break; }
      const float l = redb[0 * HW + lane] + redb[1 * HW + lane] + redb[2 * HW + lane] + redb[3 * HW + lane];
      const float inv_l_l = (l > 0.f) ? 1.0f / l : 0.f;
      if (warp == 4 * hh && base + lane < nrows)
        a.lse[(size_t)t0 * H + base + lane] = (l > 0.f) ? (m_l + log2f(l)) * 0.6931471805599453f : -INFINITY;
      if (!group_sync(smx, sync_phase, abort_flag, err)) { ok = false; break; }
      if (!mbar_wait_warp(&bars[B_O_FULL], lgq & 1, abort_flag, err)) { ok = false; break; }
      tc_fence_after();
      uint16_t* out_g = a.out + (size_t)(t0 * H + base) * 512;
#pragma unroll 1
      for (int m = 0; m < 4; ++m) {
#pragma unroll
        for (int q16 = 0; q16 < 2; ++q16) {
          float o[16];
          tmem_ld16(tmem + lane_off + C::COL_O + m * HC + HW * hh + 16 * q16, o);
          tmem_ld_wait();
#pragma unroll
          for (int h = 0; h < 16; ++h) {
            const float il = __shfl_sync(0xffffffffu, inv_l_l, 16 * q16 + h);
            if (base + 16 * q16 + h < nrows) out_g[(16 * q16 + h) * 512 + m * 128 + key] = f32_to_bf16_rn(o[h] * il);
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&bars[B_O_EMPTY]);
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
