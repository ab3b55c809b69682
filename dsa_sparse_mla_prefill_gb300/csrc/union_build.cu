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
//   token bitmaps (when G bitmaps of W = ceil(N/32) words fit in a small
//   share of shared memory): one bitmap per token; the union word is the OR
//   of the tokens' words, its popcounts are scanned into prefix[W], and the
//   compaction writes each union slot's row and, read straight off the
//   tokens' words, its membership byte (bit j = token j), with no second
//   pass over the indices and no atomics on the mask;
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

// Token-bitmap variant (see the top of the file).  Shared memory: G token
// bitmaps of WS = Wp | 1 words each (an odd stride puts the G words of one
// position in different banks), prefix[Wp], and the mask bytes of the row.
__global__ void __launch_bounds__(NT, 4) union_build_tokbits_kernel(UnionArgs a) {
  extern __shared__ __align__(16) uint32_t sm[];
  const int W = (a.N + 31) >> 5;
  const int Wp = (W + 3) & ~3;
  const int WS = Wp | 1;
  uint32_t* maskw = sm;                                  // [union_pad / 4], 16-byte aligned
  uint32_t* prefix = sm + a.union_pad / 4;               // [Wp]
  uint32_t* tb = prefix + Wp;                            // [G][WS]
  uint8_t* maskb = reinterpret_cast<uint8_t*>(maskw);
  __shared__ uint32_t warp_tot[NT / 32];
  __shared__ uint32_t s_total;

  const int g = blockIdx.x;
  int t0, n;
  group_of(a.req, a.G, g, t0, n);

  zero_smem(tb, a.G * WS);
  zero_smem(maskw, a.union_pad / 4);
  __syncthreads();

  // 1) token j's bitmap from its valid rows (16-byte loads of entries 4t..4t+3
  // when the row layout allows, else a strided loop)
  const bool vec = a.k <= 4 * NT && (a.k & 3) == 0 && (a.ld & 3) == 0 &&
                   (reinterpret_cast<uintptr_t>(a.idx) & 15u) == 0;
  int bad = 0;
  auto set_bit = [&](int x, int j) {
    if (x >= 0 && x < a.N) {
      atomicOr(&tb[j * WS + (x >> 5)], 1u << (x & 31));
    } else if (x != -1) {
      ++bad;
    }
  };
  if (vec) {
#pragma unroll
    for (int j = 0; j < GMAX; ++j) {
      if (j < n && 4 * (int)threadIdx.x < a.k) {
        const int4 x = __ldg(reinterpret_cast<const int4*>(a.idx + (size_t)(t0 + j) * a.ld) + threadIdx.x);
        set_bit(x.x, j);
        set_bit(x.y, j);
        set_bit(x.z, j);
        set_bit(x.w, j);
      }
    }
  } else {
    for (int j = 0; j < n; ++j) {
      const int32_t* row = a.idx + (size_t)(t0 + j) * a.ld;
      for (int e = threadIdx.x; e < a.k; e += NT) set_bit(__ldg(row + e), j);
    }
  }
  bad = __reduce_add_sync(0xffffffffu, bad);
  if ((threadIdx.x & 31) == 0 && bad) atomicAdd(a.err + ERR_BAD_INDEX, (unsigned)bad);
  __syncthreads();

  auto union_word = [&](int w) {
    uint32_t u = 0u;
    for (int j = 0; j < n; ++j) u |= tb[j * WS + w];
    return u;
  };
  // 2) exclusive prefix of the union words' popcounts (contiguous run per thread)
  const int per = (W + NT - 1) / NT;
  const int w0 = threadIdx.x * per;
  uint32_t local = 0;
  for (int w = w0; w < min(W, w0 + per); ++w) local += __popc(union_word(w));
  uint32_t total;
  uint32_t run = block_exclusive_scan(local, warp_tot, total);
  for (int w = w0; w < min(W, w0 + per); ++w) {
    prefix[w] = run;
    run += __popc(union_word(w));
  }
  if (threadIdx.x == 0) s_total = total;
  __syncthreads();
  const uint32_t U = s_total;
  const uint32_t Ucap = min(U, (uint32_t)a.union_pad);
  if (threadIdx.x == 0 && U > (uint32_t)a.union_pad) atomicAdd(a.err + ERR_UNION_OVERFLOW, 1u);

  // 3) compaction: ascending set-bit positions, each slot's membership byte
  // from the tokens' words
  int32_t* urow = a.union_idx + (size_t)g * a.union_pad;
  for (int w = threadIdx.x; w < W; w += NT) {
    uint32_t tw[GMAX];
    uint32_t bits = 0u;
#pragma unroll
    for (int j = 0; j < GMAX; ++j) {
      tw[j] = (j < n) ? tb[j * WS + w] : 0u;
      bits |= tw[j];
    }
    uint32_t pos = prefix[w];
    while (bits) {
      const int b = __ffs(bits) - 1;
      bits &= bits - 1;
      if (pos < Ucap) {
        urow[pos] = (w << 5) + b;
        uint32_t m = 0u;
#pragma unroll
        for (int j = 0; j < GMAX; ++j) m |= ((tw[j] >> b) & 1u) << j;
        maskb[pos] = (uint8_t)m;
      }
      ++pos;
    }
  }
  fill_i32(urow, Ucap, (uint32_t)a.union_pad, -1);
  __syncthreads();

  // 4) mask row out (16-byte stores; union_pad is a multiple of 16)
  uint4* mrow = reinterpret_cast<uint4*>(a.mask + (size_t)g * a.union_pad);
  const uint4* ms = reinterpret_cast<const uint4*>(maskw);
  for (int i = threadIdx.x; i < a.union_pad / 16; i += NT) mrow[i] = ms[i];
  if (threadIdx.x == 0) a.union_len[g] = (int32_t)Ucap;
}

}  // namespace unionb

int launch_union_build(const UnionArgs& a, cudaStream_t stream) {
  if (a.num_groups == 0) return 0;
  const int64_t tsm = union_build_tokbits_smem_bytes(a.N, a.G, a.union_pad);
  if (tsm <= kUnionTokbitsMaxSmem) {
    if (tsm > 48 * 1024 &&
        cudaFuncSetAttribute(unionb::union_build_tokbits_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)tsm) !=
            cudaSuccess)
      return -1;
    unionb::union_build_tokbits_kernel<<<a.num_groups, unionb::NT, (size_t)tsm, stream>>>(a);
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
