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
//               In the streamed instance (STREAM: q and the indices arrive
//               from host memory while the kernel runs) it also waits for
//               each token's chunk to land and counts the CTA's finished
//               tokens for the copy stream that reads them back.
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
//
// FP8 rows (the same kernel with F8 = true; row = 512 e4m3 codes | 4 fp32
// block scales | bf16 RoPE): the key rows are gathered as codes, half the
// bytes, and turned into bf16 on chip with the dequantize arithmetic
// (e4m3x4_dequant_bf16x4), so the result is bit-for-bit that of the bf16
// kernel on the dequantized table.  Sixteen producer warps (8-23), thread =
// key row:
//   warps 8-15  K stream: every 128-code block (and the RoPE columns) is
//               gathered into a code ring (tile::gather4, 4 rows x 128 bytes),
//               then each thread converts its row's half block and writes it
//               with tcgen05.st into a TMEM chunk ring, which the QK MMAs
//               read as their A operand (no bf16 K tile in shared memory).
//   warps 16-23 V stream: the same blocks again into a second code ring,
//               converted into the 128B-swizzled V units the P.V MMAs read.
//   Warps 0-3 run at 176 registers, warps 4-23 at 56 (768 threads at 80).
#include "dsa_device.cuh"
#include "dsa_kernels.h"

namespace dsa {
namespace sparse {

template <bool B>
struct BoolConst {
  static constexpr bool value = B;
};

constexpr int BK = 128;         // keys per tile (the MMA's M)
constexpr int KMAX = 2048;      // longest index row the kernel compacts
constexpr int REGS_SOFTMAX = 192; // warpgroup 0 after rebalancing
constexpr float kTau = 8.0f;    // lazy-rescale threshold (log2 units)

template <int H, int NC, bool F8>
struct Cfg {
  // bf16 rows: 20 warps launched at 96 registers; the softmax warpgroup
  // raised to 192, warpgroups 1-4 lowered to 72 (4*32*192 + 16*32*72 =
  // 640*96).  FP8 rows: 24 warps at 80; softmax 176, the other five
  // warpgroups 56 (128*176 + 640*56 <= 768*80).  One setmaxnreg for all the
  // warps after the softmax warpgroup: a per-warpgroup choice behind a branch
  // cost the bf16 kernel 12 % (ptxas then allocates those regions more
  // conservatively), and giving the MMA warpgroup 64 did not pay here.
  static constexpr int NTHREADS = F8 ? 768 : 640;
  static constexpr int REGS_SMX = F8 ? 176 : REGS_SOFTMAX;
  static constexpr int REGS_WG1 = F8 ? 56 : 72;
  static constexpr int REGS_PROD = F8 ? 56 : 72;
  static_assert(128 * REGS_SMX + 128 * REGS_WG1 + (NTHREADS - 256) * REGS_PROD <= NTHREADS * (F8 ? 80 : 96),
                "registers");
  static constexpr uint32_t CHUNK_BYTES = BK * 128u;            // 128 keys x 64 columns: one swizzle column
  static constexpr uint32_t UNIT_BYTES = 2u * CHUNK_BYTES;      // 128 keys x 128 columns: one PV M-block
  static constexpr uint32_t Q_BYTES = NC * H * 128u;
  static constexpr uint32_t P_BYTES = 2u * H * 128u;            // 128 keys = 2 swizzle columns
  static constexpr uint32_t KIDX_BYTES = 2u * KMAX * 4u;
  static constexpr uint32_t RED_BYTES = 2u * 4u * H * 4u;
  static constexpr int NBAR = F8 ? 92 : 44;
  static constexpr uint32_t TAIL = NBAR * 8u + 64u + 1024u;     // barriers, misc words, alignment slack
  static constexpr uint32_t SMEM_LIMIT = 227u * 1024u;
  // FP8 rows: one fp32 block scale per row of each code slot (at most 6 slots)
  static constexpr uint32_t SCL_BYTES = F8 ? 6u * BK * 4u : 0u;
  static constexpr uint32_t FIXED = Q_BYTES + P_BYTES + KIDX_BYTES + RED_BYTES + SCL_BYTES + TAIL;
  // V ring: 128-column units for PV; K ring: 64-column chunks for QK.
  // Every thread that waits on a ring barrier must pass through each of
  // its phases in order (a phase two ahead has the parity of one that
  // already completed).  With two V slots, unit m of every tile sits in
  // slot m mod 2, filled by V producer group m mod 2 and consumed by PV
  // issuer m mod 2; K slot s is filled by K producer warp s and consumed
  // by the QK issuer, which takes every chunk.
  static constexpr int NVR = 2;
  static constexpr int NFIT = (int)((SMEM_LIMIT - FIXED - NVR * UNIT_BYTES) / CHUNK_BYTES);
  // bf16 rows: K ring of NKR chunk slots in shared memory, one per K-stream warp.
  static constexpr int NKR = F8 ? 0 : 6;
  // FP8 rows: code rings of 16 KB slots (128 rows x 128 bytes), NKC for the
  // K stream and NVC for the V stream; the K chunks live in TMEM (NKT slots).
  static constexpr int NVC = F8 ? 2 : 0;
  static constexpr int NKC = F8 ? (NFIT - NVC < 4 ? NFIT - NVC : 4) : 0;
  static constexpr int NKT = F8 ? 6 : 0;
  static_assert(NFIT >= NKR + NKC + NVC, "shared memory budget");
  static_assert(!F8 || NKC >= 2, "shared memory budget");
  static_assert(NKC + NVC <= 6, "scale words");
  static_assert(NVR == 2, "V slot = unit mod 2 = PV issuer");
  static constexpr uint32_t OFF_KR = 0;
  static constexpr uint32_t OFF_KC = 0;
  static constexpr uint32_t OFF_VC = OFF_KC + NKC * CHUNK_BYTES;
  static constexpr uint32_t OFF_VR = NKR * CHUNK_BYTES + (NKC + NVC) * CHUNK_BYTES;
  static constexpr uint32_t OFF_Q = OFF_VR + NVR * UNIT_BYTES;
  static constexpr uint32_t OFF_P = OFF_Q + Q_BYTES;
  static constexpr uint32_t OFF_KIDX = OFF_P + P_BYTES;
  static constexpr uint32_t OFF_RED = OFF_KIDX + KIDX_BYTES;
  static constexpr uint32_t OFF_SCL = OFF_RED + RED_BYTES;
  static constexpr uint32_t OFF_BAR = OFF_SCL + SCL_BYTES;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8u;
  static constexpr uint32_t SMEM_BYTES = OFF_MISC + 64u + 1024u;
  static_assert(SMEM_BYTES <= SMEM_LIMIT, "shared memory budget");
  // TMEM columns: O^T double buffer (2 x 4H) + S^T double buffer (2 x H)
  // [+ FP8 rows: NKT K chunks of 128 keys x 64 bf16 = 32 columns each]
  static constexpr uint32_t COL_O = 0;
  static constexpr uint32_t COL_S = 8u * H;
  static constexpr uint32_t COL_KT = 10u * H;
  static constexpr uint32_t TMEM_USED = COL_KT + 32u * NKT;
  static constexpr uint32_t TMEM_COLS = (TMEM_USED <= 256) ? 256u : 512u;
  static_assert(TMEM_USED <= 512, "tensor memory budget");
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
  B_KR_FULL = 20,    // [NKR <= 6]
  B_OUT_DONE = 26,   // [2] streamed: a token without keys stored (softmax warpgroup, 128)
  B_KR_EMPTY = 28,   // [NKR <= 8]
  B_VR_FULL = 36,    // [NVR <= 4]
  B_VR_EMPTY = 40,   // [NVR <= 4]
  // FP8 rows only (the K ring slots above are then TMEM chunk slots)
  B_KC_FULL = 44,    // [NKC <= 4][4 row quarters]
  B_KC_EMPTY = 60,   // [NKC <= 4][4]
  B_VC_FULL = 76,    // [NVC <= 2][4]
  B_VC_EMPTY = 84,   // [NVC <= 2][4]
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

// Index loads: the read-only path, or (streamed calls) L2-only loads, since a
// streamed row was written by a copy engine while the kernel runs.
template <bool STREAM>
__device__ __forceinline__ int4 load_idx4(const int4* p) {
  if constexpr (STREAM) return ld_cg_i4(p);
  else return __ldg(p);
}
template <bool STREAM>
__device__ __forceinline__ int load_idx(const int* p) {
  if constexpr (STREAM) return ld_cg_i32(p);
  else return __ldg(p);
}

template <int H, int NC, bool F8, bool STREAM>
__global__ void __launch_bounds__(Cfg<H, NC, F8>::NTHREADS, 1)
sparse_prefill_kernel(const __grid_constant__ SparseArgs a) {
  using C = Cfg<H, NC, F8>;
  static_assert(!(F8 && STREAM), "the FP8 rows are never streamed");
  static_assert(C::NKR <= 6 && C::NKT <= 6, "B_OUT_DONE sits in K ring slots 6 and 7");
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
    // 3 MMA, softmax, 12 (bf16) or 16 (FP8) producer warps
    mbar_init(&bars[B_IDX_EMPTY + 0], F8 ? 20 : 16);
    mbar_init(&bars[B_IDX_EMPTY + 1], F8 ? 20 : 16);
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
    if constexpr (STREAM) {
      mbar_init(&bars[B_OUT_DONE + 0], 128);
      mbar_init(&bars[B_OUT_DONE + 1], 128);
    }
    // bf16: the chunk / unit leader's byte count; FP8: one arrival per
    // converting warp (4 row quarters per TMEM chunk, 8 warps per V unit)
    for (int i = 0; i < (F8 ? C::NKT : C::NKR); ++i) {
      mbar_init(&bars[B_KR_FULL + i], F8 ? 4 : 1);
      mbar_init(&bars[B_KR_EMPTY + i], 1);
    }
    for (int i = 0; i < C::NVR; ++i) {
      mbar_init(&bars[B_VR_FULL + i], F8 ? 8 : 1);
      mbar_init(&bars[B_VR_EMPTY + i], 1);
    }
    if constexpr (F8) {
      // code slots: per row quarter, the two warps that gather and read it
      for (int i = 0; i < 4 * C::NKC; ++i) {
        mbar_init(&bars[B_KC_FULL + i], 2);
        mbar_init(&bars[B_KC_EMPTY + i], 2);
      }
      for (int i = 0; i < 4 * C::NVC; ++i) {
        mbar_init(&bars[B_VC_FULL + i], 2);
        mbar_init(&bars[B_VC_EMPTY + i], 2);
      }
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
    // the warpgroups after the first give registers back
    if constexpr (C::REGS_WG1 == C::REGS_PROD) {
      regs_dec<C::REGS_PROD>();
    } else {
      if (warp < 8)
        regs_dec<C::REGS_WG1>();
      else
        regs_dec<C::REGS_PROD>();
    }
    if (warp == 6) {
      // ------------------------------------------------------------------
      // index compaction
      // ------------------------------------------------------------------
      // Streamed calls: this warp also counts the CTA's tokens done, in order.
      // Once the softmax warps have stored a token (they arrive on B_O_EMPTY
      // after the stores, or on B_OUT_DONE for a token without keys), a fence
      // makes those stores visible device-wide and a release add counts the
      // token; the copy stream that reads the token back waits for that
      // count.  Token lt - 2 is counted before token lt is compacted (the
      // softmax needs token lt's indices before it can arrive twice on one
      // barrier).
      int lc = 0;              // tokens counted
      int tc = blockIdx.x;     // the next token to count
      uint32_t nz = 0;         // of them with keys (O buffer uses)
      uint32_t ez = 0;         // without keys, two bits: uses of B_OUT_DONE 0 and 1 so far
      auto count_next = [&](bool wait) -> bool {
        bool w = true;
        if (wait) {
          // the counted token's valid-key count (its index buffer is reused
          // only for token lc + 2, compacted after this)
          if (meta[lc & 1] > 0) {
            w = mbar_wait_warp(&bars[B_O_EMPTY + (nz & 1)], (nz >> 1) & 1, abort_flag, err);
            ++nz;
          } else {
            const uint32_t b = lc & 1;
            w = mbar_wait_warp(&bars[B_OUT_DONE + b], (ez >> b) & 1, abort_flag, err);
            ez ^= 1u << b;
          }
        }
        // (counted even when the wait gave up: a count that never completes
        // would hold the copy stream; the timeout counter reports the failure)
        if (lane == 0) {
          __threadfence();
          red_release_gpu_add(a.done + tc / a.done_blk, 1u);
        }
        __syncwarp();
        ++lc;
        tc += stride_t;
        return w;
      };
      bool ok = true;
      int lt = 0;
      for (int t = blockIdx.x; t < T; t += stride_t, ++lt) {
        const int buf = lt & 1;
        if constexpr (STREAM) {
          if (lt >= 2 && !count_next(true)) { ok = false; break; }
        }
        if (!mbar_wait_warp(&bars[B_IDX_EMPTY + buf], ((lt >> 1) & 1) ^ 1, abort_flag, err)) { ok = false; break; }
        if constexpr (STREAM) {
          // the token's chunk must have landed
          if (!wait_ready_warp(a.ready, (uint32_t)t, abort_flag, err)) { ok = false; break; }
        }
        const int32_t* row = a.idx + (size_t)t * a.ld;
        int32_t* dst = kidx + buf * KMAX;
        int cnt = 0, bad = 0;
        const bool vec = ((a.ld & 3) == 0) && ((reinterpret_cast<uintptr_t>(a.idx) & 15) == 0);
        if (vec) {
          constexpr int QD = 4;   // four 16-byte loads in flight per lane
          for (int base = 0; base < a.k; base += 128 * QD) {
            int4 v[QD];
#pragma unroll
            for (int qd = 0; qd < QD; ++qd) {
              const int e0 = base + qd * 128 + lane * 4;
              if (e0 + 3 < a.k) {
                v[qd] = load_idx4<STREAM>(reinterpret_cast<const int4*>(row + e0));
              } else {
                v[qd].x = (e0 + 0 < a.k) ? load_idx<STREAM>(row + e0 + 0) : -1;
                v[qd].y = (e0 + 1 < a.k) ? load_idx<STREAM>(row + e0 + 1) : -1;
                v[qd].z = (e0 + 2 < a.k) ? load_idx<STREAM>(row + e0 + 2) : -1;
                v[qd].w = (e0 + 3 < a.k) ? load_idx<STREAM>(row + e0 + 3) : -1;
              }
            }
#pragma unroll
            for (int qd = 0; qd < QD; ++qd) {
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
            const int x = (e < a.k) ? load_idx<STREAM>(row + e) : -1;
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
      if constexpr (STREAM) {
        // the tokens not counted yet (after a failure, without waiting)
        while (tc < T) ok = count_next(ok) && ok;
      }
    } else if (warp >= 8) {
      if constexpr (F8) {
        // ----------------------------------------------------------------
        // FP8 producers, thread = key row.  Warps 8-15 feed QK, warps 16-23
        // P.V.  In each stream warp w converts rows 32*(w & 3) + lane of
        // every tile (its TMEM lane quarter) and half hf of every 128-code
        // block (codes 64*hf .. 64*hf+63: bf16 chunk 2b+hf).  An item is
        // one 128-byte column block of the tile's 128 rows: code block b at
        // byte 128b, and for the K stream with RoPE columns a fifth item at
        // byte 528 (the RoPE columns, bf16, copied into TMEM unchanged).
        // Items flow through a ring of 16 KB code slots; the two warps of a
        // row quarter each gather 16 of its rows (lanes 0-3, 4 rows each)
        // and both read it.  A warp issues items NS-1 ahead of the one it
        // converts, within each token.  The row's block scale of an item
        // comes with it: the hf = 0 warp copies it (cp.async, 4 bytes) into
        // the slot's scale words, tracked by the slot's own barrier.
        // ----------------------------------------------------------------
        auto stream = [&](auto kstream_tag) {
          constexpr bool KS = decltype(kstream_tag)::value;
          constexpr bool ROPE = (NC == 9);
          constexpr int IPT = (KS && ROPE) ? 5 : 4;         // items per tile
          constexpr int NS = KS ? C::NKC : C::NVC;
          constexpr int LAG = NS - 1;
          const int q4 = warp & 3;
          const int hf = ((warp - 8) >> 2) & 1;
          const int row = 32 * q4 + lane;                          // row this thread converts
          const int grow = 32 * q4 + 16 * hf + 4 * (lane & 3);     // rows this lane gathers (lanes 0-3)
          const uint32_t cring = sbase + (KS ? C::OFF_KC : C::OFF_VC);
          const int bfull = (KS ? B_KC_FULL : B_VC_FULL) + q4;     // + 4 * slot
          const int bempty = (KS ? B_KC_EMPTY : B_VC_EMPTY) + q4;
          const uint32_t scl = sbase + C::OFF_SCL + (KS ? 0u : (uint32_t)C::NKC * BK * 4u) + row * 4u;   // + 512 * slot
          const uint32_t rsw = (uint32_t)(row & 7);               // 128B swizzle phase of this row
          uint32_t cpos = 0;   // items of this stream so far
          uint32_t opos = 0;   // TMEM chunks (K) or V units (V) so far
          int lt = 0;
          bool ok = true;
          int drain_lo = 0, drain_hi = 0;   // after an abort: items of the token that may still be in flight
          int lt_nz = 0;                            // tokens with at least one tile
          for (int t = blockIdx.x; t < T && ok; t += stride_t, ++lt) {
            const int buf = lt & 1;
            if (!mbar_wait_warp(&bars[B_IDX_FULL + buf], (lt >> 1) & 1, abort_flag, err)) { ok = false; break; }
            const int nvalid = meta[buf];
            const int ntiles = (nvalid + BK - 1) / BK;
            const int32_t* kl = kidx + buf * KMAX;
            const int nitems = ntiles * IPT;
            if (KS && warp == 8 && ntiles > 0) {
              // q[t]: rows t*H .. t*H+H-1 of q viewed [T*H, D_QK], one box per swizzle column
              if (!mbar_wait_warp(&bars[B_Q_EMPTY], (lt_nz & 1) ^ 1, abort_flag, err)) { ok = false; break; }
              if (lane == 0) {
                mbar_arrive_expect_tx(&bars[B_Q_FULL], C::Q_BYTES);
                for (int c = 0; c < NC; ++c)
                  tma_load_2d(sbase + C::OFF_Q + c * (H * 128), &a.tmap_q, c * 64, t * H, &bars[B_Q_FULL]);
              }
            }
            if (ntiles > 0) ++lt_nz;
            for (int i = 0; i < nitems + LAG; ++i) {
              if (i < nitems) {
                // ---- issue item i
                const int j = i / IPT, b = i - j * IPT;
                const uint32_t cp = cpos + i, s = cp % NS;
                if (!mbar_wait_warp(&bars[bempty + 4 * s], ((cp / NS) & 1) ^ 1, abort_flag, err)) {
                  ok = false;
                  drain_lo = i > LAG ? i - LAG : 0;
                  drain_hi = i;
                  break;
                }
                if (hf == 0 && b < 4) {
                  // this row's scale of block b (zero for a key past the valid count); the
                  // slot's phase cannot complete before this warp's arrival below
                  const int key = j * BK + row;
                  const bool v = key < nvalid;
                  cp_async4(scl + s * (BK * 4), v ? a.kv8 + (size_t)kl[key] * a.row_bytes + 512 + 4 * b : a.kv8,
                            v ? 4u : 0u);
                  cp_async_mbar_arrive(&bars[bfull + 4 * s]);
                }
                __syncwarp();
                if (lane < 4) {
                  const int gk = j * BK + grow;
                  int4 r = *reinterpret_cast<const int4*>(kl + gk);
                  if (gk + 0 >= nvalid) r.x = -1;
                  if (gk + 1 >= nvalid) r.y = -1;
                  if (gk + 2 >= nvalid) r.z = -1;
                  if (gk + 3 >= nvalid) r.w = -1;
                  if (lane == 0) mbar_arrive_expect_tx(&bars[bfull + 4 * s], 16u * 128u);
                  tma_gather4(cring + s * C::CHUNK_BYTES + grow * 128, &a.tmap_kv, b < 4 ? 128 * b : 528, r.x, r.y,
                              r.z, r.w, &bars[bfull + 4 * s]);
                }
              }
              if (i >= LAG) {
                // ---- convert item i - LAG
                const int ic = i - LAG;
                const int j = ic / IPT, b = ic - j * IPT;
                const uint32_t cp = cpos + ic, s = cp % NS;
                // (on an abort from here on, items ic .. min(i, nitems - 1) may still be in flight)
                drain_lo = ic;
                drain_hi = i < nitems ? i + 1 : nitems;
                if (!mbar_wait_warp(&bars[bfull + 4 * s], (cp / NS) & 1, abort_flag, err)) { ok = false; break; }
                if (KS && warp == 8 && lane == 0 && b == 0) DSA_TRACE(a.tr, opos / NC + j, 0);
                const uint32_t src = cring + s * C::CHUNK_BYTES + row * 128;
                const float sc = lds_f32(scl + s * (BK * 4));   // (unused for the RoPE item)
                if constexpr (KS) {
                  const bool rope = ROPE && b == 4;
                  if (!rope || hf == 0) {
                    const uint32_t kt = opos + j * NC + (rope ? 8 : 2 * b + hf);
                    const uint32_t ts = kt % C::NKT;
                    if (!mbar_wait_warp(&bars[B_KR_EMPTY + ts], ((kt / C::NKT) & 1) ^ 1, abort_flag, err)) {
                      ok = false;
                      break;
                    }
                    tc_fence_after();
                    const uint32_t taddr = tmem + ((uint32_t)(q4 * 32) << 16) + C::COL_KT + ts * 32;
                    if (rope) {
                      // bf16 RoPE columns: 8 pieces of 8 values, copied as they are
#pragma unroll 1
                      for (int pp = 0; pp < 8; pp += 2) {
                        const uint4 w0 = lds128(src + ((((uint32_t)pp) ^ rsw) << 4));
                        const uint4 w1 = lds128(src + ((((uint32_t)(pp + 1)) ^ rsw) << 4));
                        const uint32_t v[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
                        tmem_st8_u32(taddr + 4 * pp, v);
                      }
                    } else {
                      // codes 64hf .. 64hf+63: pieces 4hf .. 4hf+3, 16 codes = 8 columns each
#pragma unroll 1
                      for (int pp = 0; pp < 4; ++pp) {
                        const uint4 w = lds128(src + ((((uint32_t)(4 * hf + pp)) ^ rsw) << 4));
                        uint32_t v[8];
                        e4m3x4_dequant_bf16x4(w.x, sc, v[0], v[1]);
                        e4m3x4_dequant_bf16x4(w.y, sc, v[2], v[3]);
                        e4m3x4_dequant_bf16x4(w.z, sc, v[4], v[5]);
                        e4m3x4_dequant_bf16x4(w.w, sc, v[6], v[7]);
                        tmem_st8_u32(taddr + 8 * pp, v);
                      }
                    }
                    tmem_st_wait();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bars[B_KR_FULL + ts]);
                  }
                } else {
                  const uint32_t vp = opos + j * 4 + b;
                  const uint32_t vs = vp % C::NVR;
                  if (!mbar_wait_warp(&bars[B_VR_EMPTY + vs], ((vp / C::NVR) & 1) ^ 1, abort_flag, err)) {
                    ok = false;
                    break;
                  }
                  // this row of the unit's bf16 chunk hf (K-major, 128B-swizzled as the gathers lay it out)
                  const uint32_t dst = sbase + C::OFF_VR + vs * C::UNIT_BYTES + hf * C::CHUNK_BYTES + row * 128;
#pragma unroll 1
                  for (int pp = 0; pp < 4; ++pp) {
                    const uint4 w = lds128(src + ((((uint32_t)(4 * hf + pp)) ^ rsw) << 4));
                    uint32_t v[8];
                    e4m3x4_dequant_bf16x4(w.x, sc, v[0], v[1]);
                    e4m3x4_dequant_bf16x4(w.y, sc, v[2], v[3]);
                    e4m3x4_dequant_bf16x4(w.z, sc, v[4], v[5]);
                    e4m3x4_dequant_bf16x4(w.w, sc, v[6], v[7]);
                    sts128(dst + ((((uint32_t)(2 * pp)) ^ rsw) << 4), v[0], v[1], v[2], v[3]);
                    sts128(dst + ((((uint32_t)(2 * pp + 1)) ^ rsw) << 4), v[4], v[5], v[6], v[7]);
                  }
                  fence_proxy_async_smem();
                  __syncwarp();
                  if (lane == 0) mbar_arrive(&bars[B_VR_FULL + vs]);
                }
                // every code of the slot this warp reads has been consumed
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars[bempty + 4 * s]);
              }
            }
            if (!ok) break;
            cpos += nitems;
            opos += KS ? ntiles * NC : ntiles * 4;
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[B_IDX_EMPTY + buf]);
          }
          // After an abort, let the copies still in flight land before the
          // CTA can exit (each slot's phase completes once its bytes land).
          if (!ok && lane == 0) {
            for (int c = drain_lo; c < drain_hi; ++c) {
              const uint32_t cp = cpos + c, s = cp % NS;
              mbar_wait_drain(&bars[bfull + 4 * s], (cp / NS) & 1, err);
            }
            if (KS && warp == 8 && lt_nz > 0) mbar_wait_drain(&bars[B_Q_FULL], (lt_nz - 1) & 1, err);
          }
          __syncwarp();
        };
        if (warp < 16)
          stream(BoolConst<true>{});
        else
          stream(BoolConst<false>{});
      } else {
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
          if constexpr (STREAM) fence_proxy_async_global();   // q and kv were written by a copy engine
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
      }
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
              constexpr uint32_t NK = F8 ? C::NKT : C::NKR;
              const uint32_t slot = kpos % NK;
              if (!mbar_wait(&bars[B_KR_FULL + slot], (kpos / NK) & 1, abort_flag, err)) { ok = false; break; }
              tc_fence_after();
              const uint32_t bbase = q_s + c * (H * 128);
              if constexpr (F8) {
                // A = the chunk in TMEM (lane = key, 8 columns per 16 keys' K step)
                mma_bf16_ts_x4(d_s, tmem + C::COL_KT + slot * 32, sdesc_sw128(bbase, 16, 1024), 8u, 2u, IDESC_QK,
                               c > 0 ? 1u : 0u);
              } else {
                const uint32_t abase = sbase + C::OFF_KR + slot * C::CHUNK_BYTES;
                mma_bf16_ss_x4(d_s, sdesc_sw128(abase, 16, 1024), sdesc_sw128(bbase, 16, 1024), 2u, 2u, IDESC_QK,
                               c > 0 ? 1u : 0u);
              }
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
    regs_inc<C::REGS_SMX>();
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
    // Streamed calls: the index warp counts each token done once its out and
    // lse stores are in, seeing them through B_O_EMPTY (arrived on after the
    // stores) or, for a token without keys, B_OUT_DONE.
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
        if constexpr (STREAM) mbar_arrive(&bars[B_OUT_DONE + (lt & 1)]);
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

template <int H, int NC, bool F8, bool STREAM>
static int launch_t(const SparseArgs& a, int num_sms, cudaStream_t stream) {
  using C = Cfg<H, NC, F8>;
  static int attr_set[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set[dev]) {
    if (cudaFuncSetAttribute(sparse_prefill_kernel<H, NC, F8, STREAM>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::SMEM_BYTES) != cudaSuccess)
      return -1;
    attr_set[dev] = 1;
  }
  const int grid = a.T < num_sms ? a.T : num_sms;
  sparse_prefill_kernel<H, NC, F8, STREAM><<<grid, C::NTHREADS, C::SMEM_BYTES, stream>>>(a);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

template <bool F8, bool STREAM>
static int launch_f(const SparseArgs& a, int num_sms, cudaStream_t stream) {
  const int nc = a.d_qk / 64;
  if (a.H == 16 && nc == 9) return launch_t<16, 9, F8, STREAM>(a, num_sms, stream);
  if (a.H == 32 && nc == 9) return launch_t<32, 9, F8, STREAM>(a, num_sms, stream);
  if (a.H == 16 && nc == 8) return launch_t<16, 8, F8, STREAM>(a, num_sms, stream);
  if (a.H == 32 && nc == 8) return launch_t<32, 8, F8, STREAM>(a, num_sms, stream);
  return -2;
}

}  // namespace sparse

int launch_sparse_prefill(const SparseArgs& a, int num_sms, cudaStream_t stream) {
  // the streamed instance only for streamed calls: its extra waits and
  // counting stay out of the ordinary kernel's code
  if (a.ready != nullptr && a.done != nullptr) return sparse::launch_f<false, true>(a, num_sms, stream);
  return sparse::launch_f<false, false>(a, num_sms, stream);
}

int launch_sparse_prefill_fp8(const SparseArgs& a, int num_sms, cudaStream_t stream) {
  return sparse::launch_f<true, false>(a, num_sms, stream);
}

}  // namespace dsa
