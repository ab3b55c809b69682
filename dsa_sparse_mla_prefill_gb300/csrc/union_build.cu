// Union list + head-group membership mask builder for the grouped form.
//
// "[Perf][DSA] Grouped sparse prefill with the FlashMLA head-group-mask
// kernel", How: for every group of G consecutive tokens of a request, a
// bitmap over the KV positions is filled from the tokens' top-k rows, a
// prefix sum over the bitmap's popcounts compacts the set bits into a sorted
// union list, and every token gets one membership bit per union slot.  The
// review snippet on that page sizes the buffers: union_pad = ceil(G*k / UB) * UB
// slots per group and ceil(N / 32) bitmap words.
//
// One CTA per group, everything in shared memory.  Two variants of the
// same steps:
//   byte map (when N bytes plus two words per 32 positions fit in a small
//   share of shared memory): one membership byte per KV position, bit j set
//   when token j of the group selects that row.  The union word of 32
//   positions is the non-zero test of their bytes, its popcounts are scanned
//   into prefix[W], and the compaction writes each union slot's row and its
//   membership byte (read straight off the map), with no second pass over the
//   indices and no atomics on the mask;
//   one bitmap (any N up to the shared-memory limit): bitmap[W] -> prefix[W]
//   -> union[g, pos] = set-bit positions in ascending order, then a second
//   pass over the indices sets mask[g, pos] |= 1 << j (bytes packed 4 per
//   word, atomics).
// Slots past the union length hold -1 in the list and 0 in the mask.
#include "dsa_device.cuh"
#include "dsa_kernels.h"

namespace dsa {
namespace unionb {

constexpr int NT = 512;
constexpr int GMAX = 8;   // tokens per group (one mask bit each)

__device__ __forceinline__ void group_of(const ReqTable& rq, int G, int g, int& t0, int& n) {
  int r = 0;
  while (r + 1 < rq.num_req && rq.cu_g[r + 1] <= g) ++r;
  t0 = rq.cu_q[r] + (g - rq.cu_g[r]) * G;
  const int end = rq.cu_q[r + 1];
  n = min(G, end - t0);
}

// Block-wide exclusive scan of one value per thread; returns the exclusive
// prefix and writes the block total.
__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t v, uint32_t* warp_tot, uint32_t& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_tot[warp] = x;
  __syncthreads();
  if (warp == 0) {
    uint32_t w = (lane < NT / 32) ? warp_tot[lane] : 0u;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < NT / 32) warp_tot[lane] = w;  // inclusive warp totals
  }
  __syncthreads();
  const uint32_t before = (warp > 0) ? warp_tot[warp - 1] : 0u;
  total = warp_tot[NT / 32 - 1];
  return before + x - v;
}

// Fills row[lo, hi) with v: single stores up to a 16-byte boundary, then
// 16-byte stores (row is 16-byte aligned and hi a multiple of 4).
__device__ __forceinline__ void fill_i32(int32_t* row, uint32_t lo, uint32_t hi, int32_t v) {
  const uint32_t a4 = min((lo + 3u) & ~3u, hi);
  for (uint32_t u = lo + threadIdx.x; u < a4; u += NT) row[u] = v;
  int4* r4 = reinterpret_cast<int4*>(row);
  const int4 v4 = make_int4(v, v, v, v);
  for (uint32_t u = a4 / 4 + threadIdx.x; u < hi / 4; u += NT) r4[u] = v4;
}

// Zeroes bytes [lo, hi) of row: single bytes up to a 16-byte boundary, then
// 16-byte stores (row is 16-byte aligned and hi a multiple of 16).
__device__ __forceinline__ void fill_u8_zero(uint8_t* row, uint32_t lo, uint32_t hi) {
  const uint32_t a16 = min((lo + 15u) & ~15u, hi);
  for (uint32_t u = lo + threadIdx.x; u < a16; u += NT) row[u] = 0;
  uint4* r16 = reinterpret_cast<uint4*>(row);
  for (uint32_t u = a16 / 16 + threadIdx.x; u < hi / 16; u += NT) r16[u] = make_uint4(0u, 0u, 0u, 0u);
}

// Zeroes n 32-bit words of shared memory at p (16-byte aligned): 16-byte
// stores, then the tail.
__device__ __forceinline__ void zero_smem(uint32_t* p, int n) {
  uint4* p4 = reinterpret_cast<uint4*>(p);
  for (int i = threadIdx.x; i < n / 4; i += NT) p4[i] = make_uint4(0u, 0u, 0u, 0u);
  for (int i = (n & ~3) + threadIdx.x; i < n; i += NT) p[i] = 0u;
}

__global__ void __launch_bounds__(NT) union_build_kernel(UnionArgs a) {
  extern __shared__ __align__(16) uint32_t sm[];
  const int W = (a.N + 31) >> 5;
  const int Wp = (W + 3) & ~3;
  uint32_t* bitmap = sm;                 // [W]
  uint32_t* prefix = sm + Wp;            // [W]
  uint32_t* maskw = sm + 2 * Wp;         // [union_pad / 4], 16-byte aligned
  __shared__ uint32_t warp_tot[NT / 32];
  __shared__ uint32_t s_total;

  const int g = blockIdx.x;
  int t0, n;
  group_of(a.req, a.G, g, t0, n);

  zero_smem(bitmap, W);
  zero_smem(maskw, a.union_pad / 4);
  __syncthreads();

  // 1) bitmap of every valid row of the group's tokens.  Register path: each
  // thread loads entries 4t .. 4t+3 of all the group's token rows up front
  // (independent 16-byte loads, one memory latency) and keeps them for step
  // 4; otherwise a strided loop over each row.
  const bool vec = a.k <= 4 * NT && (a.k & 3) == 0 && (a.ld & 3) == 0 &&
                   (reinterpret_cast<uintptr_t>(a.idx) & 15u) == 0;
  int4 xs[GMAX];
  int bad = 0;
  if (vec) {
#pragma unroll
    for (int j = 0; j < GMAX; ++j) {
      xs[j] = make_int4(-1, -1, -1, -1);
      if (j < n && 4 * (int)threadIdx.x < a.k)
        xs[j] = __ldg(reinterpret_cast<const int4*>(a.idx + (size_t)(t0 + j) * a.ld) + threadIdx.x);
    }
#pragma unroll
    for (int j = 0; j < GMAX; ++j) {
      const int v[4] = {xs[j].x, xs[j].y, xs[j].z, xs[j].w};
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int x = v[c];
        if (x >= 0 && x < a.N) {
          atomicOr(&bitmap[x >> 5], 1u << (x & 31));
        } else if (x != -1) {
          ++bad;
        }
      }
    }
  } else {
    for (int j = 0; j < n; ++j) {
      const int32_t* row = a.idx + (size_t)(t0 + j) * a.ld;
      for (int e = threadIdx.x; e < a.k; e += NT) {
        const int x = __ldg(row + e);
        if (x >= 0 && x < a.N) {
          atomicOr(&bitmap[x >> 5], 1u << (x & 31));
        } else if (x != -1) {
          ++bad;
        }
      }
    }
  }
  bad = __reduce_add_sync(0xffffffffu, bad);
  if ((threadIdx.x & 31) == 0 && bad) atomicAdd(a.err + ERR_BAD_INDEX, (unsigned)bad);
  __syncthreads();

  // 2) exclusive prefix of the popcounts; thread i scans a contiguous run of words
  const int per = (W + NT - 1) / NT;
  const int w0 = threadIdx.x * per;
  uint32_t local = 0;
  for (int w = w0; w < min(W, w0 + per); ++w) local += __popc(bitmap[w]);
  uint32_t total;
  uint32_t run = block_exclusive_scan(local, warp_tot, total);
  for (int w = w0; w < min(W, w0 + per); ++w) {
    prefix[w] = run;
    run += __popc(bitmap[w]);
  }
  if (threadIdx.x == 0) s_total = total;
  __syncthreads();
  const uint32_t U = s_total;
  const uint32_t Ucap = min(U, (uint32_t)a.union_pad);
  if (threadIdx.x == 0 && U > (uint32_t)a.union_pad) atomicAdd(a.err + ERR_UNION_OVERFLOW, 1u);

  // 3) compaction: ascending set-bit positions
  int32_t* urow = a.union_idx + (size_t)g * a.union_pad;
  for (int w = threadIdx.x; w < W; w += NT) {
    uint32_t bits = bitmap[w];
    uint32_t pos = prefix[w];
    while (bits) {
      const int b = __ffs(bits) - 1;
      bits &= bits - 1;
      if (pos < Ucap) urow[pos] = (w << 5) + b;
      ++pos;
    }
  }
  fill_i32(urow, Ucap, (uint32_t)a.union_pad, -1);

  // 4) membership bits: slot of row x = prefix[x>>5] + popc(bits below x)
  auto member = [&](int x, int j) {
    if (x >= 0 && x < a.N) {
      const uint32_t w = (uint32_t)x >> 5;
      const uint32_t pos = prefix[w] + __popc(bitmap[w] & ((1u << (x & 31)) - 1u));
      if (pos < Ucap) atomicOr(&maskw[pos >> 2], (1u << j) << ((pos & 3) * 8));
    }
  };
  if (vec) {
#pragma unroll
    for (int j = 0; j < GMAX; ++j) {
      member(xs[j].x, j);
      member(xs[j].y, j);
      member(xs[j].z, j);
      member(xs[j].w, j);
    }
  } else {
    for (int j = 0; j < n; ++j) {
      const int32_t* row = a.idx + (size_t)(t0 + j) * a.ld;
      for (int e = threadIdx.x; e < a.k; e += NT) member(__ldg(row + e), j);
    }
  }
  __syncthreads();

  // 5) mask row out (16-byte stores; union_pad is a multiple of 16)
  uint4* mrow = reinterpret_cast<uint4*>(a.mask + (size_t)g * a.union_pad);
  const uint4* ms = reinterpret_cast<const uint4*>(maskw);
  for (int i = threadIdx.x; i < a.union_pad / 16; i += NT) mrow[i] = ms[i];
  if (threadIdx.x == 0) a.union_len[g] = (int32_t)Ucap;
}

// Non-zero test of the eight bytes of lo (positions 0-3) and hi (4-7): bit i
// of the result is set when byte i is not zero.  Per byte, (b & 0x7f) + 0x7f
// has bit 7 set when b & 0x7f is not zero and never carries into the next
// byte; or-ing b itself covers b = 0x80.  The eight flags, placed at bits
// 0, 8, 16, 24 (lo) and 4, 12, 20, 28 (hi), are moved to bits 24..31 by one
// multiply: every other partial product lands at a distinct bit below 24 or
// above 31, so nothing carries into the result.
__device__ __forceinline__ uint32_t nonzero_bytes8(uint32_t lo, uint32_t hi) {
  const uint32_t fl = (((lo & 0x7f7f7f7fu) + 0x7f7f7f7fu) | lo) & 0x80808080u;
  const uint32_t fh = (((hi & 0x7f7f7f7fu) + 0x7f7f7f7fu) | hi) & 0x80808080u;
  return (((fl >> 7) | (fh >> 3)) * 0x01020408u) >> 24;
}

// Byte-map variant (see the top of the file).  Shared memory: one membership
// byte per KV position (32 Wp bytes), the union words ub[Wp] and prefix[Wp].
__global__ void __launch_bounds__(NT, 4) union_build_bytemap_kernel(UnionArgs a) {
  extern __shared__ __align__(16) uint32_t sm[];
  const int W = (a.N + 31) >> 5;
  const int Wp = (W + 3) & ~3;
  uint32_t* memw = sm;            // [8 Wp]: byte x = membership byte of position x
  uint32_t* ub = sm + 8 * Wp;     // [Wp]: bit i of word w = position 32w + i is in the union
  uint32_t* prefix = ub + Wp;     // [Wp]: union slots before word w
  const uint8_t* memb = reinterpret_cast<const uint8_t*>(memw);
  __shared__ uint32_t warp_tot[NT / 32];

  const bool vec = a.k <= 4 * NT && (a.k & 3) == 0 && (a.ld & 3) == 0 &&
                   (reinterpret_cast<uintptr_t>(a.idx) & 15u) == 0;
  const int g = blockIdx.x;
  int t0, n;
  group_of(a.req, a.G, g, t0, n);

  zero_smem(memw, 8 * Wp);
  __syncthreads();

  // 1) membership bits of every valid row of the group's tokens.  16-byte
  // loads of entries 4t .. 4t+3 of four token rows at a time, all four issued
  // before any is used, when the row layout allows; else a strided loop.
  int bad = 0;
  auto put = [&](int x, int j) {
    if ((unsigned)x < (unsigned)a.N) {
      atomicOr(&memw[x >> 2], (1u << j) << ((x & 3) << 3));
    } else if (x != -1) {
      ++bad;
    }
  };
  if (vec) {
    const bool in = 4 * (int)threadIdx.x < a.k;
#pragma unroll
    for (int j0 = 0; j0 < GMAX; j0 += 4) {
      if (j0 >= n) break;   // (G = 4, or the group at a request's end)
      int4 xs[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        xs[j] = make_int4(-1, -1, -1, -1);
        if (j0 + j < n && in)
          xs[j] = __ldg(reinterpret_cast<const int4*>(a.idx + (size_t)(t0 + j0 + j) * a.ld) + threadIdx.x);
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        put(xs[j].x, j0 + j);
        put(xs[j].y, j0 + j);
        put(xs[j].z, j0 + j);
        put(xs[j].w, j0 + j);
      }
    }
  } else {
    for (int j = 0; j < n; ++j) {
      const int32_t* row = a.idx + (size_t)(t0 + j) * a.ld;
      for (int e = threadIdx.x; e < a.k; e += NT) put(__ldg(row + e), j);
    }
  }
  bad = __reduce_add_sync(0xffffffffu, bad);
  if ((threadIdx.x & 31) == 0 && bad) atomicAdd(a.err + ERR_BAD_INDEX, (unsigned)bad);
  __syncthreads();

  // 2) union words from the byte map and the exclusive prefix of their
  // popcounts.  Thread t takes words t and NT + t of each pair of NT-word
  // rows; one block scan covers both rows, their counts packed into the two
  // 16-bit halves of one word (a row holds at most 32 NT = 16384 bits, so the
  // low half never carries into the high one).
  uint32_t carry = 0;
  for (int r0 = 0; r0 * NT < W; r0 += 2) {
    const int wa = r0 * NT + threadIdx.x, wb = wa + NT;
    uint32_t cnt[2] = {0u, 0u};
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int w = h ? wb : wa;
      if (w < W) {
        const uint4 b0 = reinterpret_cast<const uint4*>(memw)[2 * w];
        const uint4 b1 = reinterpret_cast<const uint4*>(memw)[2 * w + 1];
        const uint32_t u = nonzero_bytes8(b0.x, b0.y) | (nonzero_bytes8(b0.z, b0.w) << 8) |
                           (nonzero_bytes8(b1.x, b1.y) << 16) | (nonzero_bytes8(b1.z, b1.w) << 24);
        ub[w] = u;
        cnt[h] = __popc(u);
      }
    }
    uint32_t tot;
    const uint32_t ex = block_exclusive_scan(cnt[0] | (cnt[1] << 16), warp_tot, tot);
    if (wa < W) prefix[wa] = carry + (ex & 0xffffu);
    if (wb < W) prefix[wb] = carry + (tot & 0xffffu) + (ex >> 16);
    carry += (tot & 0xffffu) + (tot >> 16);
    __syncthreads();   // warp_tot is reused by the next rows; ub and prefix are read below
  }
  const uint32_t U = carry;
  const uint32_t Ucap = min(U, (uint32_t)a.union_pad);
  if (threadIdx.x == 0 && U > (uint32_t)a.union_pad) atomicAdd(a.err + ERR_UNION_OVERFLOW, 1u);

  // 3) compaction, balanced by union slot: thread t writes slots
  // [c t, c t + c), c = ceil(Ucap / NT), each slot's row (ascending set-bit
  // positions) and membership byte (read off the byte map).  The word holding
  // its first slot is the last word whose prefix is at most that slot (a
  // binary search over prefix[]); from there it walks the set bits forward.
  // (A word per thread would leave the warp holding the densest words looping
  // once per bit while the rest of the CTA waits.)
  int32_t* urow = a.union_idx + (size_t)g * a.union_pad;
  uint8_t* mrow = a.mask + (size_t)g * a.union_pad;
  {
    const uint32_t c = (Ucap + NT - 1) / NT;
    uint32_t s = c * threadIdx.x;
    const uint32_t s_end = min(s + c, Ucap);
    if (s < s_end) {
      int lo = 0, hi = W - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (prefix[mid] <= s) lo = mid; else hi = mid - 1;
      }
      int w = lo;
      uint32_t bits = ub[w];
      for (uint32_t r = s - prefix[w]; r > 0; --r) bits &= bits - 1;   // the word's bits before slot s
      for (; s < s_end; ++s) {
        while (bits == 0u) bits = ub[++w];   // (slot s < U: a later word holds it)
        const int x = (w << 5) + (__ffs(bits) - 1);
        bits &= bits - 1;
        urow[s] = x;
        mrow[s] = memb[x];
      }
    }
  }
  // 4) slots past the union: -1 in the list, 0 in the mask
  fill_i32(urow, Ucap, (uint32_t)a.union_pad, -1);
  fill_u8_zero(mrow, Ucap, (uint32_t)a.union_pad);
  if (threadIdx.x == 0) a.union_len[g] = (int32_t)Ucap;
}

}  // namespace unionb

int launch_union_build(const UnionArgs& a, cudaStream_t stream) {
  if (a.num_groups == 0) return 0;
  const int64_t bsm = union_build_bytemap_smem_bytes(a.N);
  if (bsm <= kUnionBytemapMaxSmem) {
    if (bsm > 48 * 1024 &&
        cudaFuncSetAttribute(unionb::union_build_bytemap_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bsm) !=
            cudaSuccess)
      return -1;
    // one CTA per group: the hardware scheduler hands a finished CTA's SM the
    // next group (a persistent grid with each CTA walking groups, with or
    // without an L2 prefetch of its next group's index rows, measured slower)
    unionb::union_build_bytemap_kernel<<<a.num_groups, unionb::NT, (size_t)bsm, stream>>>(a);
    return cudaGetLastError() == cudaSuccess ? 0 : -1;
  }
  const int smem = union_build_smem_bytes(a.N, a.union_pad);
  if (smem > 48 * 1024) {
    if (cudaFuncSetAttribute(unionb::union_build_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
        cudaSuccess)
      return -1;
  }
  unionb::union_build_kernel<<<a.num_groups, unionb::NT, smem, stream>>>(a);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace dsa
