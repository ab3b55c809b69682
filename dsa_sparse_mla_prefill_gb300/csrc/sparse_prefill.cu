// Per-token sparse MLA prefill for sm_103a.
//
// What it computes ("[Perf][DSA] Grouped sparse prefill with the FlashMLA
// head-group-mask kernel", commit message and Why): every query token t with
// H heads attends to its own top-k latent KV rows,
//     out[t,h,:] = softmax_j(scale * q[t,h,:] . kv[idx_j, 0:D_QK]) . kv[idx_j, 0:D_V]
// plus the natural-log log-sum-exp.  Each selected row is re-gathered for
// every token (2048 x 1152 B per token at top-2048, D_QK = 576), so the form
// is bound by the gather.
//
// Design (one persistent CTA per SM, tokens round-robin over CTAs; the key
// rows of a tile are gathered twice, once for QK and once for PV, so the
// QK of the next tile can stream while this tile's softmax runs; the
// second gather hits L2):
//   warp 6      compacts the token's index row (valid entries only, order
//               kept) into shared memory; out-of-range entries are counted.
//   warps 8-19  issue TMA loads: q per token (tiled boxes) and the key
//               rows as tile::gather4 (4 rows x 128 bytes per instruction)
//               straight into 128B-swizzled tiles of 128 keys.  Warps 8-13
//               stream the D_QK/64 key chunks (128 keys x 64 columns) of
//               every tile into the K ring, warps 14-19 the four 128-column
//               V units into the V ring; copies complete on the stage's
//               mbarrier by byte count.
//   warps 4,5,7 one thread each issues tcgen05.mma with the keys on the M
//               side (M = 128 keys, N = H): warp 4 S^T = K q^T chunk by
//               chunk into a double-buffered S, warps 5 and 7 O^T += V^T P^T
//               for alternate V units, V^T read MN-major.  Issue cost is
//               serial per warp, so the streams overlap; every chunk and
//               unit returns to the producers as soon as its MMAs complete.
//   warps 0-3   thread i owns key i of the tile (TMEM lane i): online softmax
//               in base 2 with a lazy rescale (only when a head's running
//               max grows by more than 2^8), P written bf16 to shared
//               memory, and the epilogue (O^T lane = output column).
//   Warps 0-3 run at 192 registers, warps 4-19 at 72.
#include "dsa_device.cuh"
#include "dsa_kernels.h"

namespace dsa {
namespace sparse {

constexpr int BK = 128;         // keys per tile (the MMA's M)
constexpr int KMAX = 2048;      // longest index row the kernel compacts
constexpr int NTHREADS = 640;   // 20 warps, launched at 96 registers each
constexpr int REGS_SOFTMAX = 192; // warpgroup 0 after rebalancing
constexpr int REGS_OTHER = 72;    // warpgroups 1-4 (4*32*192 + 16*32*72 = 640*96)
constexpr float kTau = 8.0f;    // lazy-rescale threshold (log2 units)

template <int H, int NC>
struct Cfg {
  static constexpr uint32_t CHUNK_BYTES = BK * 128u;            // 128 keys x 64 columns: one swizzle column
  static constexpr uint32_t UNIT_BYTES = 2u * CHUNK_BYTES;      // 128 keys x 128 columns: one PV M-block
  static constexpr uint32_t Q_BYTES = NC * H * 128u;
  static constexpr uint32_t P_BYTES = 2u * H * 128u;            // 128 keys = 2 swizzle columns
  static constexpr uint32_t KIDX_BYTES = 2u * KMAX * 4u;
  static constexpr uint32_t RED_BYTES = 2u * 4u * H * 4u;
  static constexpr int NBAR = 44;
  static constexpr uint32_t TAIL = NBAR * 8u + 64u + 1024u;     // barriers, misc words, alignment slack
  static constexpr uint32_t SMEM_LIMIT = 227u * 1024u;
  // V ring: 128-column units for PV; K ring: 64-column chunks for QK.
  // Every thread that waits on a ring barrier must pass through each of
  // its phases in order (a phase two ahead has the parity of one that
  // already completed).  With two V slots, unit m of every tile sits in
  // slot m mod 2, filled by V producer group m mod 2 and consumed by PV
  // issuer m mod 2; K slot s is filled by K producer warp s and consumed
  // by the QK issuer, which takes every chunk.
  static constexpr int NVR = 2;
  static constexpr int NKR_FIT =
      (int)((SMEM_LIMIT - TAIL - Q_BYTES - P_BYTES - KIDX_BYTES - RED_BYTES - NVR * UNIT_BYTES) / CHUNK_BYTES);
  static constexpr int NKR = 6;   // one slot per K-stream warp
  static_assert(NKR_FIT >= NKR, "shared memory budget");
  static_assert(NVR == 2, "V slot = unit mod 2 = PV issuer");
  static constexpr uint32_t OFF_KR = 0;
  static constexpr uint32_t OFF_VR = OFF_KR + NKR * CHUNK_BYTES;
  static constexpr uint32_t OFF_Q = OFF_VR + NVR * UNIT_BYTES;
  static constexpr uint32_t OFF_P = OFF_Q + Q_BYTES;
  static constexpr uint32_t OFF_KIDX = OFF_P + P_BYTES;
  static constexpr uint32_t OFF_RED = OFF_KIDX + KIDX_BYTES;
  static constexpr uint32_t OFF_BAR = OFF_RED + RED_BYTES;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8u;
  static constexpr uint32_t SMEM_BYTES = OFF_MISC + 64u + 1024u;
  static_assert(SMEM_BYTES <= SMEM_LIMIT, "shared memory budget");
  // TMEM columns: O^T double buffer (2 x 4H) + S^T double buffer (2 x H)
  static constexpr uint32_t TMEM_COLS = (10 * H <= 256) ? 256u : 512u;
  static constexpr uint32_t COL_O = 0;
  static constexpr uint32_t COL_S = 8u * H;
};

// barrier slots
enum {
  B_IDX_FULL = 0,    // [2]
  B_IDX_EMPTY = 2,   // [2]
  B_Q_FULL = 4,
  B_Q_EMPTY = 5,
  B_S_FULL = 6,      // [2]
  B_S_EMPTY = 8,     // [2]
  B_P_FULL = 10,
  B_P_EMPTY = 11,
  B_O_FULL = 12,     // [2]
  B_O_EMPTY = 14,    // [2]
  B_DRAIN = 16,      // [3] one per MMA issuer
  B_SMX_SYNC = 19,   // softmax warpgroup barrier (128)
  B_KR_FULL = 20,    // [NKR <= 8]
  B_KR_EMPTY = 28,   // [NKR <= 8]
  B_VR_FULL = 36,    // [NVR <= 4]
  B_VR_EMPTY = 40,   // [NVR <= 4]
};

// Warp-level transposed max/sum reduction: every lane holds H values (one
// per head); afterwards lane L holds the reduction over the 32 lanes of head
// (L mod H).  Uses 31 shuffles for H = 32 instead of 5*H.
template <int H, bool IS_MAX>
__device__ __forceinline__ float warp_transpose_reduce(float* v) {
  const uint32_t lane = lane_id();
  auto op = [](float a, float b) { return IS_MAX ? fmaxf(a, b) : a + b; };
  if constexpr (H == 16) {
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = op(v[i], __shfl_xor_sync(0xffffffffu, v[i], 16));
  }
  constexpr int START = (H == 32) ? 16 : 8;
  int n = H;
#pragma unroll
  for (int o = START; o >= 1; o >>= 1) {
    n >>= 1;  // values kept after this step
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

template <int H, int NC>
__global__ void __launch_bounds__(NTHREADS, 1)
sparse_prefill_kernel(const __grid_constant__ SparseArgs a) {
  using C = Cfg<H, NC>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_u32 + 1023u) & ~1023u) - raw_u32);
  const uint32_t sbase = smem_u32(smem);

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile uint32_t* tmem_base_ptr = misc + 0;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 1);
  volatile int* meta = reinterpret_cast<volatile int*>(misc + 2);  // [2] valid count per idx buffer
  int32_t* kidx = reinterpret_cast<int32_t*>(smem + C::OFF_KIDX);
  float* red = reinterpret_cast<float*>(smem + C::OFF_RED);
  unsigned int* err = a.err;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(&bars[B_IDX_FULL + 0], 1);
    mbar_init(&bars[B_IDX_FULL + 1], 1);
    mbar_init(&bars[B_IDX_EMPTY + 0], 16);  // 3 MMA, softmax, 12 producer warps
    mbar_init(&bars[B_IDX_EMPTY + 1], 16);
    mbar_init(&bars[B_Q_FULL], 1);
    mbar_init(&bars[B_Q_EMPTY], 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars[B_S_FULL + i], 1);
      mbar_init(&bars[B_S_EMPTY + i], 128);
      mbar_init(&bars[B_O_FULL + i], 2);   // one commit per PV issuer
      mbar_init(&bars[B_O_EMPTY + i], 128);
    }
    mbar_init(&bars[B_P_FULL], 128);
    mbar_init(&bars[B_P_EMPTY], 2);
    for (int i = 0; i < 3; ++i) mbar_init(&bars[B_DRAIN + i], 1);
    mbar_init(&bars[B_SMX_SYNC], 128);
    for (int i = 0; i < C::NKR; ++i) {
      mbar_init(&bars[B_KR_FULL + i], 1);
      mbar_init(&bars[B_KR_EMPTY + i], 1);
    }
    for (int i = 0; i < C::NVR; ++i) {
      mbar_init(&bars[B_VR_FULL + i], 1);
      mbar_init(&bars[B_VR_EMPTY + i], 1);
    }
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

  const int T = a.T;
  const int stride_t = gridDim.x;

  if (warp >= 4) {
    // warpgroups 1-4 give registers back
    regs_dec<REGS_OTHER>();
    if (warp == 6) {
      // ------------------------------------------------------------------
      // index compaction
      // ------------------------------------------------------------------
      int lt = 0;
      for (int t = blockIdx.x; t < T; t += stride_t, ++lt) {
        const int buf = lt & 1;
        if (!mbar_wait_warp(&bars[B_IDX_EMPTY + buf], ((lt >> 1) & 1) ^ 1, abort_flag, err)) break;
        const int32_t* row = a.idx + (size_t)t * a.ld;
        int32_t* dst = kidx + buf * KMAX;
        int cnt = 0, bad = 0;
        const bool vec = ((a.ld & 3) == 0) && ((reinterpret_cast<uintptr_t>(a.idx) & 15) == 0);
        if (vec) {
          for (int base = 0; base < a.k; base += 512) {
            int4 v[4];
#pragma unroll
            for (int qd = 0; qd < 4; ++qd) {
              const int e0 = base + qd * 128 + lane * 4;
              if (e0 + 3 < a.k) {
                v[qd] = __ldg(reinterpret_cast<const int4*>(row + e0));
              } else {
                v[qd].x = (e0 + 0 < a.k) ? __ldg(row + e0 + 0) : -1;
                v[qd].y = (e0 + 1 < a.k) ? __ldg(row + e0 + 1) : -1;
                v[qd].z = (e0 + 2 < a.k) ? __ldg(row + e0 + 2) : -1;
                v[qd].w = (e0 + 3 < a.k) ? __ldg(row + e0 + 3) : -1;
              }
            }
#pragma unroll
            for (int qd = 0; qd < 4; ++qd) {
              const int vals[4] = {v[qd].x, v[qd].y, v[qd].z, v[qd].w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int x = vals[e];
                const bool ok = (x >= 0) && (x < a.N);
                bad += (x < -1 || x >= a.N) ? 1 : 0;
                const uint32_t m = __ballot_sync(0xffffffffu, ok);
                if (ok) dst[cnt + __popc(m & ((1u << lane) - 1u))] = x;
                cnt += __popc(m);
              }
            }
          }
        } else {
          for (int base = 0; base < a.k; base += 32) {
            const int e = base + lane;
            const int x = (e < a.k) ? __ldg(row + e) : -1;
            const bool ok = (x >= 0) && (x < a.N);
            bad += (x < -1 || x >= a.N) ? 1 : 0;
            const uint32_t m = __ballot_sync(0xffffffffu, ok);
            if (ok) dst[cnt + __popc(m & ((1u << lane) - 1u))] = x;
            cnt += __popc(m);
          }
        }
        bad = __reduce_add_sync(0xffffffffu, bad);
        if (lane == 0) {
          if (bad) atomicAdd(err + ERR_BAD_INDEX, (unsigned)bad);
          meta[buf] = cnt;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[B_IDX_FULL + buf]);
      }
    } else if (warp >= 8) {
      // ----------------------------------------------------------------
      // TMA producers: twelve warps in two independent streams.
      //   warps 8-13:  q per token (warp 8), and the D_QK/64 key chunks of
      //                every tile into the K ring; warp 8+s owns K slot s
      //                and issues the whole chunk (lane l: rows 4l..4l+3).
      //   warps 14-19: the four 128-column V units of every tile into the
      //                V ring (unit m in slot m mod 2); all six warps take
      //                part in every unit, lanes 0-10 of each sharing its
      //                64 gather4 (a unit's refill is on the P.V critical
      //                path twice per tile, so its issue time matters).
      // Neither stream waits on the other, so QK of the next tile streams
      // while this tile's softmax runs and V lands ahead of PV.  TMA issue
      // cost is serial per warp, so many issuing warps keep many copies in
      // flight.  The leader of a stage arms its byte count; copies from
      // other issuers may complete first, which only drives the
      // transaction count negative until then.
      // ----------------------------------------------------------------
      const bool kstream = warp < 8 + C::NKR;
      const int kw = warp - 8;                      // K slot owned (K stream)
      const int e = (warp - 14) * 11 + (lane < 11 ? lane : 64);   // V gather index 0..63 of a unit
      const bool v_issuer = !kstream && e < 64;
      const int g = kstream ? lane : (e & 31);       // row group
      const int vcc = e >> 5;                       // V swizzle column
      const bool leader = (lane == 0) && (kstream || warp == 14);
      const uint32_t q_s = sbase + C::OFF_Q;
      int lt = 0, lt_nz = 0;
      uint32_t gt = 0, pos = 0;  // tiles and stages of this stream so far
      int64_t last_armed = -1;   // last stage this warp's leader armed
      bool ok = true;
      for (int t = blockIdx.x; t < T && ok; t += stride_t, ++lt) {
        const int buf = lt & 1;
        if (!mbar_wait_warp(&bars[B_IDX_FULL + buf], (lt >> 1) & 1, abort_flag, err)) { ok = false; break; }
        const int nvalid = meta[buf];
        const int ntiles = (nvalid + BK - 1) / BK;
        const int32_t* kl = kidx + buf * KMAX;
        if (ntiles > 0) {
          if (warp == 8) {
            // q[t]: rows t*H .. t*H+H-1 of q viewed [T*H, D_QK], one box per swizzle column
            if (!mbar_wait_warp(&bars[B_Q_EMPTY], (lt_nz & 1) ^ 1, abort_flag, err)) { ok = false; break; }
            if (lane == 0) {
              mbar_arrive_expect_tx(&bars[B_Q_FULL], C::Q_BYTES);
              for (int c = 0; c < NC; ++c)
                tma_load_2d(q_s + c * (H * 128), &a.tmap_q, c * 64, t * H, &bars[B_Q_FULL]);
            }
          }
          for (int j = 0; j < ntiles && ok; ++j, ++gt) {
            if (warp == 8 && lane == 0) DSA_TRACE(a.tr, gt, 0);
            // this lane's 4 rows; keys past the valid count read as zeros
            const int key = j * BK + 4 * g;
            int4 r = *reinterpret_cast<const int4*>(kl + key);
            if (key + 0 >= nvalid) r.x = -1;
            if (key + 1 >= nvalid) r.y = -1;
            if (key + 2 >= nvalid) r.z = -1;
            if (key + 3 >= nvalid) r.w = -1;
            if (kstream) {
              for (int c = 0; c < NC; ++c, ++pos) {
                if ((int)(pos % C::NKR) != kw) continue;
                if (!mbar_wait_warp(&bars[B_KR_EMPTY + kw], ((pos / C::NKR) & 1) ^ 1, abort_flag, err)) {
                  ok = false;
                  break;
                }
                if (leader) mbar_arrive_expect_tx(&bars[B_KR_FULL + kw], C::CHUNK_BYTES);
                tma_gather4(sbase + C::OFF_KR + kw * C::CHUNK_BYTES + g * 512, &a.tmap_kv, c * 64, r.x, r.y, r.z, r.w,
                            &bars[B_KR_FULL + kw]);
                last_armed = pos;
              }
            } else {
              for (int m = 0; m < 4; ++m, ++pos) {
                const int vgroup = (int)(pos % C::NVR);   // V slot of this unit
                if (!mbar_wait_warp(&bars[B_VR_EMPTY + vgroup], ((pos / C::NVR) & 1) ^ 1, abort_flag, err)) {
                  ok = false;
                  break;
                }
                if (leader) mbar_arrive_expect_tx(&bars[B_VR_FULL + vgroup], C::UNIT_BYTES);
                if (v_issuer)
                  tma_gather4(sbase + C::OFF_VR + vgroup * C::UNIT_BYTES + vcc * C::CHUNK_BYTES + g * 512, &a.tmap_kv,
                              (2 * m + vcc) * 64, r.x, r.y, r.z, r.w, &bars[B_VR_FULL + vgroup]);
                last_armed = pos;
              }
            }
          }
          ++lt_nz;
        }
        if (!ok) break;
        // this warp's copies of the token are issued (row indices were read at issue)
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[B_IDX_EMPTY + buf]);
      }
      // Let copies still in flight land before the CTA can exit: the last
      // phase of the slot this warp fills completes only once every byte
      // of it has landed.
      if (leader) {
        if (warp == 8 && lt_nz > 0) mbar_wait_drain(&bars[B_Q_FULL], (lt_nz - 1) & 1, err);
        if (last_armed >= 0) {
          if (kstream)
            mbar_wait_drain(&bars[B_KR_FULL + kw], (uint32_t)(last_armed / C::NKR) & 1, err);
          else
            for (int64_t p = last_armed; p >= 0 && p > last_armed - C::NVR; --p)
              mbar_wait_drain(&bars[B_VR_FULL + (int)(p % C::NVR)], (uint32_t)(p / C::NVR) & 1, err);
        }
      }
      __syncwarp();
    } else if (warp == 4) {
      // ----------------------------------------------------------------
      // QK issuer (one thread): S^T = K q^T into the S double buffer, one
      // K-ring chunk (64 columns, four MMAs) at a time; each chunk goes
      // back to the producers as soon as its MMAs complete.
      // ----------------------------------------------------------------
      if (lane == 0) {
        constexpr uint32_t IDESC_QK = idesc_bf16_f32(128, H, false, false);
        const uint32_t q_s = sbase + C::OFF_Q;
        int lt = 0, lt_nz = 0;
        uint32_t gt = 0, kpos = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < T && ok; t += stride_t, ++lt) {
          const int buf = lt & 1;
          if (!mbar_wait(&bars[B_IDX_FULL + buf], (lt >> 1) & 1, abort_flag, err)) { ok = false; break; }
          const int nvalid = meta[buf];
          mbar_arrive(&bars[B_IDX_EMPTY + buf]);
          const int ntiles = (nvalid + BK - 1) / BK;
          if (ntiles == 0) continue;
          if (!mbar_wait(&bars[B_Q_FULL], lt_nz & 1, abort_flag, err)) { ok = false; break; }
          tc_fence_after();
          for (int j = 0; j < ntiles && ok; ++j, ++gt) {
            const int sb = gt & 1;
            const uint32_t d_s = tmem + C::COL_S + sb * H;
            if (!mbar_wait(&bars[B_S_EMPTY + sb], ((gt >> 1) & 1) ^ 1, abort_flag, err)) { ok = false; break; }
            DSA_TRACE(a.tr, gt, 2);
            tc_fence_after();
            for (int c = 0; c < NC; ++c, ++kpos) {
              const uint32_t slot = kpos % C::NKR;
              if (!mbar_wait(&bars[B_KR_FULL + slot], (kpos / C::NKR) & 1, abort_flag, err)) { ok = false; break; }
              tc_fence_after();
              const uint32_t abase = sbase + C::OFF_KR + slot * C::CHUNK_BYTES;
              const uint32_t bbase = q_s + c * (H * 128);
              mma_bf16_ss_x4(d_s, sdesc_sw128(abase, 16, 1024), sdesc_sw128(bbase, 16, 1024), 2u, 2u, IDESC_QK,
                             c > 0 ? 1u : 0u);
              mma_commit(&bars[B_KR_EMPTY + slot]);
            }
            if (!ok) break;
            DSA_TRACE(a.tr, gt, 1);
            mma_commit(&bars[B_S_FULL + sb]);
            if (j == ntiles - 1) mma_commit(&bars[B_Q_EMPTY]);
          }
          ++lt_nz;
        }
        // wait until every MMA issued above has completed
        mma_commit(&bars[B_DRAIN + 0]);
        mbar_wait(&bars[B_DRAIN + 0], 0, abort_flag, err);
      }
      __syncwarp();
    } else if (warp == 5 || warp == 7) {
      // ----------------------------------------------------------------
      // PV issuers (one thread in each of warps 5 and 7): O^T += V^T P^T,
      // warp 5 for units 0 and 2, warp 7 for units 1 and 3 of every tile,
      // each V-ring unit released as soon as its MMAs complete.
      // ----------------------------------------------------------------
      const int pvi = (warp == 5) ? 0 : 1;
      if (lane == 0) {
        constexpr uint32_t IDESC_PV = idesc_bf16_f32(128, H, true, false);
        const uint32_t p_s = sbase + C::OFF_P;
        int lt = 0, lt_nz = 0;
        uint32_t gt = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < T && ok; t += stride_t, ++lt) {
          const int buf = lt & 1;
          if (!mbar_wait(&bars[B_IDX_FULL + buf], (lt >> 1) & 1, abort_flag, err)) { ok = false; break; }
          const int nvalid = meta[buf];
          mbar_arrive(&bars[B_IDX_EMPTY + buf]);
          const int ntiles = (nvalid + BK - 1) / BK;
          if (ntiles == 0) continue;
          const int ob = lt_nz & 1;
          for (int j = 0; j < ntiles && ok; ++j, ++gt) {
            if (!mbar_wait(&bars[B_P_FULL], gt & 1, abort_flag, err)) { ok = false; break; }
            if (pvi == 0) DSA_TRACE(a.tr, gt, 7);
            tc_fence_after();
            if (j == 0) {
              if (!mbar_wait(&bars[B_O_EMPTY + ob], ((lt_nz >> 1) & 1) ^ 1, abort_flag, err)) { ok = false; break; }
              tc_fence_after();
            }
            for (int m = pvi; m < 4 && ok; m += 2) {
              const uint32_t vp = gt * 4 + m;
              const uint32_t slot = vp % C::NVR;
              if (!mbar_wait(&bars[B_VR_FULL + slot], (vp / C::NVR) & 1, abort_flag, err)) { ok = false; break; }
              tc_fence_after();
              const uint32_t ubase = sbase + C::OFF_VR + slot * C::UNIT_BYTES;
              const uint32_t d_o = tmem + C::COL_O + ob * (4 * H) + m * H;
#pragma unroll
              for (int hf = 0; hf < 2; ++hf) {
                // 16 keys (2048 B of V^T, MN-major; the unit's two swizzle
                // columns CHUNK_BYTES apart) per MMA; P^T one 64-key swizzle
                // column per half
                const uint64_t adesc = sdesc_sw128(ubase + hf * 4 * 2048, C::CHUNK_BYTES, 1024);
                const uint64_t bdesc = sdesc_sw128(p_s + hf * (H * 128), 16, 1024);
                mma_bf16_ss_x4(d_o, adesc, bdesc, 128u, 2u, IDESC_PV, (j > 0 || hf > 0) ? 1u : 0u);
              }
              mma_commit(&bars[B_VR_EMPTY + slot]);
            }
            if (!ok) break;
            mma_commit(&bars[B_P_EMPTY]);
            if (j == ntiles - 1) mma_commit(&bars[B_O_FULL + ob]);
          }
          ++lt_nz;
        }
        mma_commit(&bars[B_DRAIN + 1 + pvi]);
        mbar_wait(&bars[B_DRAIN + 1 + pvi], 0, abort_flag, err);
      }
      __syncwarp();
    }
  } else {
    regs_inc<REGS_SOFTMAX>();
    // ------------------------------------------------------------------
    // softmax + epilogue (warps 0-3, thread i <-> TMEM lane i)
    // ------------------------------------------------------------------
    const int tid = threadIdx.x;  // 0..127
    const float scale_log2 = a.scale * 1.4426950408889634f;
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    uint8_t* p_tile = smem + C::OFF_P;
    int lt = 0, lt_nz = 0;
    uint32_t gt = 0;
    uint32_t sync_phase = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < T && ok; t += stride_t, ++lt) {
      const int buf = lt & 1;
      if (!mbar_wait_warp(&bars[B_IDX_FULL + buf], (lt >> 1) & 1, abort_flag, err)) { ok = false; break; }
      const int nvalid = meta[buf];
      if (!group_sync(&bars[B_SMX_SYNC], sync_phase, abort_flag, err)) { ok = false; break; }
      if (tid == 0) mbar_arrive(&bars[B_IDX_EMPTY + buf]);
      const int ntiles = (nvalid + BK - 1) / BK;
      uint16_t* out_t = a.out + (size_t)t * H * 512;
      if (ntiles == 0) {
        for (int i = tid; i < H * 512; i += 128) out_t[i] = 0;
        if (tid < H) a.lse[(size_t)t * H + tid] = -INFINITY;
        continue;
      }
      const int ob = lt_nz & 1;
      float m_run[H], l_part[H];
#pragma unroll
      for (int h = 0; h < H; ++h) { m_run[h] = -INFINITY; l_part[h] = 0.f; }
      for (int j = 0; j < ntiles; ++j, ++gt) {
        const int sb = gt & 1;
        if (!mbar_wait_warp(&bars[B_S_FULL + sb], (gt >> 1) & 1, abort_flag, err)) { ok = false; break; }
        if (tid == 0) DSA_TRACE(a.tr, gt, 3);
        tc_fence_after();
        float s[H];
        tmem_ld_cols<H>(tmem + lane_off + C::COL_S + sb * H, s);
        tmem_ld_wait();
        tc_fence_before();
        mbar_arrive(&bars[B_S_EMPTY + sb]);
        const bool valid = (j * BK + tid) < nvalid;
        bool mine = false;
#pragma unroll
        for (int h = 0; h < H; ++h) {
          s[h] = valid ? s[h] * scale_log2 : -INFINITY;
          mine |= (s[h] > m_run[h] + kTau);
        }
        // Lazy rescale: the tile max matters only when some score exceeds
        // the running max by more than kTau.  Each warp votes; a warp that
        // votes yes publishes its per-head max.  The new reference is the
        // max over those warps, which bounds every score of the tile (the
        // others lie within kTau of the old reference) as the full tile max
        // would.
        const bool wneed = __any_sync(0xffffffffu, mine);
        float* redb = red + (gt & 1) * (4 * H);
        volatile uint32_t* vote = misc + 4 + (gt & 1) * 4;
        if (wneed) {
          float r[H];
#pragma unroll
          for (int h = 0; h < H; ++h) r[h] = s[h];
          const float wmax = warp_transpose_reduce<H, true>(r);
          if (lane < H) redb[warp * H + lane] = wmax;
        }
        if (lane == 0) vote[warp] = wneed ? 1u : 0u;
        if (!group_sync(&bars[B_SMX_SYNC], sync_phase, abort_flag, err)) { ok = false; break; }
        uint32_t vw[4];
#pragma unroll
        for (int w = 0; w < 4; ++w) vw[w] = vote[w];
        const bool need = (vw[0] | vw[1] | vw[2] | vw[3]) != 0;
        float tmax[H];
        if (need) {
#pragma unroll
          for (int h = 0; h < H; ++h) tmax[h] = -INFINITY;
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            if (vw[w]) {
#pragma unroll
              for (int h = 0; h < H; h += 4) {
                const float4 x = *reinterpret_cast<const float4*>(redb + w * H + h);
                tmax[h + 0] = fmaxf(tmax[h + 0], x.x);
                tmax[h + 1] = fmaxf(tmax[h + 1], x.y);
                tmax[h + 2] = fmaxf(tmax[h + 2], x.z);
                tmax[h + 3] = fmaxf(tmax[h + 3], x.w);
              }
            }
          }
        }
        if (tid == 0) DSA_TRACE(a.tr, gt, 4);
        // Everything that does not touch P^T or O first: the new running
        // max, the rescale factors, P (bf16, packed in registers) and the
        // row sums; only the O rescale and the P^T stores wait for the
        // previous P.V, so the exponentials overlap it.
        float alpha[H];
        if (need) {
#pragma unroll
          for (int h = 0; h < H; ++h) {
            const float mn = fmaxf(m_run[h], tmax[h]);
            alpha[h] = (m_run[h] == -INFINITY) ? 0.f : exp2f(m_run[h] - mn);
            m_run[h] = mn;
            l_part[h] *= alpha[h];
          }
        }
        uint32_t pk[H / 2];
#pragma unroll
        for (int h = 0; h < H; h += 2) {
          const float mr0 = (m_run[h] == -INFINITY) ? 0.f : m_run[h];
          const float mr1 = (m_run[h + 1] == -INFINITY) ? 0.f : m_run[h + 1];
          const uint16_t b0 = f32_to_bf16_rn(exp2f(s[h] - mr0));
          const uint16_t b1 = f32_to_bf16_rn(exp2f(s[h + 1] - mr1));
          l_part[h] += bf16_to_f32(b0);
          l_part[h + 1] += bf16_to_f32(b1);
          pk[h / 2] = (uint32_t)b0 | ((uint32_t)b1 << 16);
        }
        // the previous PV must be done before P is overwritten or O rescaled
        if (!mbar_wait_warp(&bars[B_P_EMPTY], (gt & 1) ^ 1, abort_flag, err)) { ok = false; break; }
        if (tid == 0) DSA_TRACE(a.tr, gt, 5);
        tc_fence_after();
        if (need && j > 0) {
#pragma unroll 1
          for (int m = 0; m < 4; ++m) {
            float o[H];
            const uint32_t ta = tmem + lane_off + C::COL_O + ob * (4 * H) + m * H;
            tmem_ld_cols<H>(ta, o);
            tmem_ld_wait();
#pragma unroll
            for (int h = 0; h < H; ++h) o[h] *= alpha[h];
            tmem_st_cols<H>(ta, o);
          }
          tmem_st_wait();
        }
        // P^T[h][key] (K-major swizzled, 2 columns of 64 keys)
        {
          const uint32_t kcol = tid & 63;
          uint8_t* pcol = p_tile + (tid >> 6) * (H * 128);
#pragma unroll
          for (int h = 0; h < H; ++h)
            *reinterpret_cast<uint16_t*>(pcol + sw128_offset(h, kcol)) =
                (uint16_t)((h & 1) ? (pk[h / 2] >> 16) : (pk[h / 2] & 0xffffu));
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(&bars[B_P_FULL]);
        if (tid == 0) DSA_TRACE(a.tr, gt, 6);
      }
      if (!ok) break;
      // -------- epilogue --------
      float lsum[H];
#pragma unroll
      for (int h = 0; h < H; ++h) lsum[h] = l_part[h];
      const float wsum = warp_transpose_reduce<H, false>(lsum);
      float* redb = red + (gt & 1) * (4 * H);  // not in use by the tile path now
      if (!group_sync(&bars[B_SMX_SYNC], sync_phase, abort_flag, err)) { ok = false; break; }
      if (lane < H) redb[warp * H + lane] = wsum;
      if (!group_sync(&bars[B_SMX_SYNC], sync_phase, abort_flag, err)) { ok = false; break; }
      float inv_l[H];
#pragma unroll
      for (int h = 0; h < H; ++h) {
        const float l = redb[0 * H + h] + redb[1 * H + h] + redb[2 * H + h] + redb[3 * H + h];
        inv_l[h] = (l > 0.f) ? 1.0f / l : 0.f;
        if (tid == h) a.lse[(size_t)t * H + h] = (l > 0.f) ? (m_run[h] + log2f(l)) * 0.6931471805599453f : -INFINITY;
      }
      if (!group_sync(&bars[B_SMX_SYNC], sync_phase, abort_flag, err)) { ok = false; break; }
      if (!mbar_wait_warp(&bars[B_O_FULL + ob], (lt_nz >> 1) & 1, abort_flag, err)) { ok = false; break; }
      tc_fence_after();
#pragma unroll 1
      for (int m = 0; m < 4; ++m) {
        float o[H];
        tmem_ld_cols<H>(tmem + lane_off + C::COL_O + ob * (4 * H) + m * H, o);
        tmem_ld_wait();
#pragma unroll
        for (int h = 0; h < H; ++h) out_t[h * 512 + m * 128 + tid] = f32_to_bf16_rn(o[h] * inv_l[h]);
      }
      tc_fence_before();
      mbar_arrive(&bars[B_O_EMPTY + ob]);
      ++lt_nz;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 4) tmem_dealloc(tmem, C::TMEM_COLS);
}

template <int H, int NC>
static int launch_t(const SparseArgs& a, int num_sms, cudaStream_t stream) {
  using C = Cfg<H, NC>;
  static int attr_set[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set[dev]) {
    if (cudaFuncSetAttribute(sparse_prefill_kernel<H, NC>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::SMEM_BYTES) != cudaSuccess)
      return -1;
    attr_set[dev] = 1;
  }
  const int grid = a.T < num_sms ? a.T : num_sms;
  sparse_prefill_kernel<H, NC><<<grid, NTHREADS, C::SMEM_BYTES, stream>>>(a);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace sparse

int launch_sparse_prefill(const SparseArgs& a, int num_sms, cudaStream_t stream) {
  const int nc = a.d_qk / 64;
  if (a.H == 16 && nc == 9) return sparse::launch_t<16, 9>(a, num_sms, stream);
  if (a.H == 32 && nc == 9) return sparse::launch_t<32, 9>(a, num_sms, stream);
  if (a.H == 16 && nc == 8) return sparse::launch_t<16, 8>(a, num_sms, stream);
  if (a.H == 32 && nc == 8) return sparse::launch_t<32, 8>(a, num_sms, stream);
  return -2;
}

}  // namespace dsa
