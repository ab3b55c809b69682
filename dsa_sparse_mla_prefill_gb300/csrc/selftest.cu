// Self-test of the tcgen05 building blocks used by the kernels: one
// D[128, N] = A[128, K] . B[N, K]^T product through shared memory in the
// 128B-swizzled K-major or MN-major layouts, accumulated in TMEM and read
// back with 32x32b loads.  Built into a separate test library.
#include "dsa_device.cuh"

namespace {

using namespace dsa;

__global__ void __launch_bounds__(128, 1)
selftest_mma_kernel(const uint16_t* A, const uint16_t* B, float* D, int N, int K, int a_mn, int b_mn,
                    unsigned int* status) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  uint8_t* As = smem;                          // 128 x K bf16
  uint8_t* Bs = smem + 128 * K * 2;            // N x K bf16
  __shared__ uint64_t bar;
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  const int tid = threadIdx.x, warp = tid >> 5;

  // stage A and B in the requested layout (a_mn == 2: A goes to TMEM below)
  for (int i = tid; i < 128 * K && a_mn != 2; i += 128) {
    const int m = i / K, k = i % K;
    uint32_t off = a_mn ? (m / 64) * (K * 128) + sw128_offset(k, m % 64)
                        : (k / 64) * (128 * 128) + sw128_offset(m, k % 64);
    *reinterpret_cast<uint16_t*>(As + off) = A[i];
  }
  for (int i = tid; i < N * K; i += 128) {
    const int n = i / K, k = i % K;
    uint32_t off = b_mn ? (n / 64) * (K * 128) + sw128_offset(k, n % 64)
                        : (k / 64) * (N * 128) + sw128_offset(n, k % 64);
    *reinterpret_cast<uint16_t*>(Bs + off) = B[i];
  }
  fence_proxy_async_smem();
  if (tid == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(&tmem_slot, 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  if (a_mn == 2) {
    // row tid of A into TMEM columns 128.., two bf16 per column (lower K in the low half)
    for (int c = 0; c < K / 2; c += 16) {
      uint32_t r[16];
      for (int i = 0; i < 16; ++i) {
        const uint32_t lo = A[(size_t)tid * K + 2 * (c + i)];
        const uint32_t hi = A[(size_t)tid * K + 2 * (c + i) + 1];
        r[i] = lo | (hi << 16);
      }
      tmem_st16_u32(tmem + ((uint32_t)(warp * 32) << 16) + 128 + c, r);
    }
    tmem_st_wait();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
  }
  if (tid == 0) {
    const uint32_t idesc = idesc_bf16_f32(128, N, a_mn == 1, b_mn != 0);
    const uint32_t a0 = smem_u32(As), b0 = smem_u32(Bs);
    // four MMAs per issue statement (K = 64 per group), as the kernels do
    for (int ks = 0; ks < K / 16; ks += 4) {
      const uint64_t ad = a_mn ? sdesc_sw128(a0 + ks * 2048, K * 128, 1024)
                               : sdesc_sw128(a0 + (ks / 4) * (128 * 128), 16, 1024);
      const uint64_t bd = b_mn ? sdesc_sw128(b0 + ks * 2048, K * 128, 1024)
                               : sdesc_sw128(b0 + (ks / 4) * (N * 128), 16, 1024);
      const uint32_t da = a_mn ? 128u : 2u, db = b_mn ? 128u : 2u;
      if (a_mn == 2)
        mma_bf16_ts_x4(tmem, tmem + 128 + ks * 8, bd, 8u, db, idesc_bf16_f32(128, N, false, b_mn != 0),
                       ks > 0 ? 1u : 0u);
      else
        mma_bf16_ss_x4(tmem, ad, bd, da, db, idesc, ks > 0 ? 1u : 0u);
    }
    mma_commit(&bar);
  }
  __syncwarp();
  const bool ok = mbar_wait(&bar, 0, &abort_flag, status);
  tc_fence_after();
  if (ok) {
    for (int c = 0; c < N; c += 16) {
      float v[16];
      tmem_ld16(tmem + ((uint32_t)(warp * 32) << 16) + c, v);
      tmem_ld_wait();
      for (int i = 0; i < 16; ++i) D[(size_t)tid * N + c + i] = v[i];
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, 256);
}

}  // namespace

extern "C" int dsa_selftest_mma(const uint16_t* A, const uint16_t* B, float* D, int N, int K, int a_mn, int b_mn,
                                unsigned int* status, cudaStream_t stream) {
  if (N < 16 || N > 256 || (N % 16) || K < 16 || (K % 64) || (a_mn == 1 && K > 128) || (b_mn && K > 128)) return 1;
  if (a_mn == 2 && (N > 128 || K > 256)) return 1;  // D in columns 0..127, A in 128..255
  if (b_mn && (N % 64)) return 1;
  const int smem = 128 * K * 2 + N * K * 2 + 1024;
  if (cudaFuncSetAttribute(selftest_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return 3;
  selftest_mma_kernel<<<1, 128, smem, stream>>>(A, B, D, N, K, a_mn, b_mn, status);
  return cudaGetLastError() == cudaSuccess ? 0 : 3;
}

// ---------------------------------------------------------------------------
// MMA timing: one CTA issues `reps` accumulating M=128 x N x K=16 bf16 MMAs
// (A and B K-major, 128B swizzle, shared memory) and records clock64 before
// the first issue, after the last issue and after the commit completed.
// ---------------------------------------------------------------------------
namespace {
__global__ void __launch_bounds__(128, 1) selftest_mma_timing_kernel(int N, int reps, int precomputed,
                                                                    long long* out, unsigned int* status) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  constexpr int K = 256;  // 4 swizzle columns, cycled through
  uint8_t* As = smem;
  uint8_t* Bs = smem + 128 * K * 2;
  __shared__ uint64_t bar;
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  const int tid = threadIdx.x, warp = tid >> 5;
  for (int i = tid; i < (128 + N) * K / 8; i += 128) reinterpret_cast<uint4*>(As)[i] = make_uint4(0, 0, 0, 0);
  fence_proxy_async_smem();
  if (tid == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(&tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  if (precomputed == 2 && (tid == 0 || tid == 32)) {
    // two warps issue half of the MMAs each, into different accumulators
    const uint32_t idesc = idesc_bf16_f32(128, N, false, false);
    const uint64_t ad0 = sdesc_sw128(smem_u32(As), 16, 1024), bd0 = sdesc_sw128(smem_u32(Bs), 16, 1024);
    const uint32_t d = tmem + (tid == 0 ? 0u : 128u);
    const long long t0 = clock64();
    for (int r = 0; r < reps / 2; ++r) {
      const int ks = r & 15;
      const uint64_t ad = ad0 + (uint64_t)(((ks >> 2) * (128 * 128) + (ks & 3) * 32) >> 4);
      const uint64_t bd = bd0 + (uint64_t)(((ks >> 2) * (N * 128) + (ks & 3) * 32) >> 4);
      mma_bf16_ss(d, ad, bd, idesc, r > 0 ? 1u : 0u);
    }
    const long long t1 = clock64();
    if (tid == 0) {
      mma_commit(&bar);
      mbar_wait(&bar, 0, &abort_flag, status);
      out[0] = t1 - t0;
      out[1] = clock64() - t0;
    }
  } else if (precomputed == 5 && warp > 0) {
    // TMEM load traffic from warps 1-3 (columns 384..447 of their lane
    // quarters) while warp 0 issues the MMAs below; a fixed count
    float v[16];
    float acc = 0.f;
    for (int it = 0; it < reps; ++it) {
      tmem_ld16(tmem + ((uint32_t)(warp * 32) << 16) + 384 + (it & 3) * 16, v);
      tmem_ld_wait();
      acc += v[it & 15];
    }
    if (acc == 12345.f) out[1] = 0;  // keep the loads
  } else if (precomputed == 6 && warp > 0) {
    // warps 1-3 poll a barrier phase that does not complete (fixed count)
    uint32_t hits = 0;
    for (int it = 0; it < reps * 4; ++it) hits += mbar_try_wait(smem_u32(&bar), 0u) ? 0u : 1u;
    if (hits == 0xffffffffu) out[1] = 0;
  } else if (precomputed == 7 && warp > 0) {
    // warps 1-3 store 16-byte pieces into the upper half of the A region
    uint4* dst = reinterpret_cast<uint4*>(As) + 2048;
    for (int it = 0; it < reps * 4; ++it) dst[(it * 96 + tid) & 1023] = make_uint4(it, it, it, it);
  } else if ((precomputed >= 4 && precomputed <= 7) && tid == 0) {
    // A from tensor memory (columns 256..383), four MMAs per asm statement
    const uint32_t idesc = idesc_bf16_f32(128, N, false, false);
    const uint64_t bd0 = sdesc_sw128(smem_u32(Bs), 16, 1024);
    const long long t0 = clock64();
    for (int r = 0; r < reps; r += 4) {
      const int ch = (r >> 2) & 3;
      const uint64_t bd = bd0 + (uint64_t)((ch * (N * 128)) >> 4);
      mma_bf16_ts_x4(tmem, tmem + 256 + ch * 32, bd, 8u, 2u, idesc, r > 0 ? 1u : 0u);
    }
    const long long t1 = clock64();
    mma_commit(&bar);
    mbar_wait(&bar, 0, &abort_flag, status);
    out[0] = t1 - t0;
    out[1] = clock64() - t0;
  } else if (precomputed == 3 && tid == 0) {
    // four MMAs per asm statement, one predicate setup
    const uint32_t idesc = idesc_bf16_f32(128, N, false, false);
    const uint64_t ad0 = sdesc_sw128(smem_u32(As), 16, 1024), bd0 = sdesc_sw128(smem_u32(Bs), 16, 1024);
    const long long t0 = clock64();
    for (int r = 0; r < reps; r += 4) {
      const int ks = r & 15;
      const uint64_t ad = ad0 + (uint64_t)(((ks >> 2) * (128 * 128)) >> 4);
      const uint64_t bd = bd0 + (uint64_t)(((ks >> 2) * (N * 128)) >> 4);
      asm volatile(
          "{\n\t.reg .pred p;\n\t"
          "setp.ne.b32 p, %4, 0;\n\t"
          "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t"
          "tcgen05.mma.cta_group::1.kind::f16 [%0], %5, %6, %3, 1;\n\t"
          "tcgen05.mma.cta_group::1.kind::f16 [%0], %7, %8, %3, 1;\n\t"
          "tcgen05.mma.cta_group::1.kind::f16 [%0], %9, %10, %3, 1;\n\t}"
          ::"r"(tmem), "l"(ad), "l"(bd), "r"(idesc), "r"(r > 0 ? 1u : 0u), "l"(ad + 2), "l"(bd + 2), "l"(ad + 4),
          "l"(bd + 4), "l"(ad + 6), "l"(bd + 6)
          : "memory");
    }
    const long long t1 = clock64();
    mma_commit(&bar);
    mbar_wait(&bar, 0, &abort_flag, status);
    out[0] = t1 - t0;
    out[1] = clock64() - t0;
  } else if (precomputed < 2 && tid == 0) {
    const uint32_t idesc = idesc_bf16_f32(128, N, false, false);
    const uint32_t a0 = smem_u32(As), b0 = smem_u32(Bs);
    const uint64_t ad0 = sdesc_sw128(a0, 16, 1024), bd0 = sdesc_sw128(b0, 16, 1024);
    const long long t0 = clock64();
    for (int r = 0; r < reps; ++r) {
      const int ks = r & 15;
      if (precomputed) {
        // start-address field += byte offset >> 4
        const uint64_t ad = ad0 + (uint64_t)(((ks >> 2) * (128 * 128) + (ks & 3) * 32) >> 4);
        const uint64_t bd = bd0 + (uint64_t)(((ks >> 2) * (N * 128) + (ks & 3) * 32) >> 4);
        mma_bf16_ss(tmem, ad, bd, idesc, r > 0 ? 1u : 0u);
      } else {
        mma_bf16_ss(tmem, sdesc_sw128(a0 + (ks >> 2) * (128 * 128) + (ks & 3) * 32, 16, 1024),
                    sdesc_sw128(b0 + (ks >> 2) * (N * 128) + (ks & 3) * 32, 16, 1024), idesc, r > 0 ? 1u : 0u);
      }
    }
    const long long t1 = clock64();
    mma_commit(&bar);
    mbar_wait(&bar, 0, &abort_flag, status);
    const long long t2 = clock64();
    out[0] = t1 - t0;
    out[1] = t2 - t0;
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, 512);
}
}  // namespace

extern "C" int dsa_selftest_mma_timing(int N, int reps, int precomputed, long long* out, unsigned int* status,
                                       cudaStream_t stream) {
  if (N < 16 || N > 256 || (N % 16) || reps < 1) return 1;
  const int smem = (128 + N) * 256 * 2 + 1024;
  if (cudaFuncSetAttribute(selftest_mma_timing_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
      cudaSuccess)
    return 3;
  selftest_mma_timing_kernel<<<1, 128, smem, stream>>>(N, reps, precomputed, out, status);
  return cudaGetLastError() == cudaSuccess ? 0 : 3;
}

// ---------------------------------------------------------------------------
// TMA gather4 layout check: 128 listed rows (columns 64c .. 64c+63) gathered
// into one 16 KB tile, 4 rows per instruction; the raw shared-memory image is
// copied out so the host can compare it with the 128B-swizzled layout the
// MMAs read (row r at r*128, 16-byte piece p at (p ^ (r & 7)) * 16).
// ---------------------------------------------------------------------------
#include "dsa_tmap.h"

namespace {
__global__ void __launch_bounds__(128, 1) selftest_gather4_kernel(const __grid_constant__ CUtensorMap map,
                                                                 const int* rows, int col, uint16_t* out,
                                                                 unsigned int* status) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* tile = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  const int tid = threadIdx.x;
  if (tid == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (tid == 0) {
    mbar_arrive_expect_tx(&bar, 128 * 128);
    for (int g = 0; g < 32; ++g)
      tma_gather4(smem_u32(tile) + g * 512, &map, col, rows[4 * g], rows[4 * g + 1], rows[4 * g + 2],
                  rows[4 * g + 3], &bar);
  }
  const bool ok = mbar_wait(&bar, 0, &abort_flag, status);
  if (ok)
    for (int i = tid; i < 128 * 64; i += 128) out[i] = reinterpret_cast<const uint16_t*>(tile)[i];
}
}  // namespace

extern "C" int dsa_selftest_gather4(const uint16_t* kv, int N, int ld, const int* rows_dev, int col, uint16_t* out,
                                    unsigned int* status, cudaStream_t stream) {
  if (N < 1 || ld < 64 || (ld & 7) || col < 0 || (col & 7) || col + 64 > ld) return 1;
  CUtensorMap map;
  if (!dsa::make_row_gather_map(&map, kv, N, ld, ld)) return 2;
  const int smem = 128 * 128 + 1024;
  selftest_gather4_kernel<<<1, 128, smem, stream>>>(map, rows_dev, col, out, status);
  return cudaGetLastError() == cudaSuccess ? 0 : 3;
}

// ---------------------------------------------------------------------------
// Multicast gather4 into a 2-CTA cluster: CTA r gathers the 64 listed rows
// 64r .. 64r+63 (columns col .. col+63) for both CTAs, so each CTA ends up
// with all 128 rows; each copies its shared-memory image to out[rank].
// ---------------------------------------------------------------------------
namespace {
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(128, 1)
    selftest_gather4_mc_kernel(const __grid_constant__ CUtensorMap map, const int* rows, int col, uint16_t* out,
                               unsigned int* status) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* tile = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  const int tid = threadIdx.x;
  const int rank = (int)cluster_ctarank();
  if (tid == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  cluster_sync();
  if (tid == 0) {
    mbar_arrive_expect_tx(&bar, 128 * 128);
    for (int g = 16 * rank; g < 16 * rank + 16; ++g)
      tma_gather4_mc(smem_u32(tile) + g * 512, &map, col, rows[4 * g], rows[4 * g + 1], rows[4 * g + 2],
                     rows[4 * g + 3], &bar, (uint16_t)3);
  }
  const bool ok = mbar_wait(&bar, 0, &abort_flag, status);
  if (ok)
    for (int i = tid; i < 128 * 64; i += 128) out[rank * 128 * 64 + i] = reinterpret_cast<const uint16_t*>(tile)[i];
  __syncthreads();
  cluster_sync();
}
}  // namespace

extern "C" int dsa_selftest_gather4_mc(const uint16_t* kv, int N, int ld, const int* rows_dev, int col,
                                       uint16_t* out, unsigned int* status, cudaStream_t stream) {
  if (N < 1 || ld < 64 || (ld & 7) || col < 0 || (col & 7) || col + 64 > ld) return 1;
  CUtensorMap map;
  if (!dsa::make_row_gather_map(&map, kv, N, ld, ld)) return 2;
  const int smem = 128 * 128 + 1024;
  selftest_gather4_mc_kernel<<<2, 128, smem, stream>>>(map, rows_dev, col, out, status);
  return cudaGetLastError() == cudaSuccess ? 0 : 3;
}

// ---------------------------------------------------------------------------
// TMA gather4 issue timing: `total` gathers of 4 rows x 128 B (rows spread
// over the table) into a 64 KB ring, issued by `lanes` lanes of each of
// `warps` warps; records cycles from first issue to all bytes landed.
// ---------------------------------------------------------------------------
namespace {
__global__ void __launch_bounds__(512, 1) selftest_gather4_timing_kernel(const __grid_constant__ CUtensorMap map,
                                                                        int N, int total, int warps, int lanes,
                                                                        long long* out, unsigned int* status) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* ring = smem_raw + (((raw + 1023u) & ~1023u) - raw);  // 64 KB
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  __shared__ long long t_start;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (tid == 0) {
    mbar_arrive_expect_tx(&bar, (uint32_t)total * 512u);
    t_start = clock64();
  }
  __syncthreads();
  const int issuers = warps * lanes;
  if (warp < warps && lane < lanes) {
    const int me = warp * lanes + lane;
    for (int g = me; g < total; g += issuers) {
      const int r = (g * 37) % (N - 4);
      tma_gather4(smem_u32(ring) + (g & 127) * 512, &map, 0, r, r + 1, r + 2, r + 3, &bar);
    }
  }
  if (tid == 0) {
    mbar_wait(&bar, 0, &abort_flag, status);
    out[0] = clock64() - t_start;
  }
}
}  // namespace

extern "C" int dsa_selftest_gather4_timing(const uint16_t* kv, int N, int ld, int total, int warps, int lanes,
                                           long long* out, unsigned int* status, cudaStream_t stream) {
  if (N < 8 || ld < 64 || (ld & 7) || warps < 1 || warps > 16 || lanes < 1 || lanes > 32 || total < 1) return 1;
  CUtensorMap map;
  if (!dsa::make_row_gather_map(&map, kv, N, ld, ld)) return 2;
  const int smem = 65536 + 1024;
  if (cudaFuncSetAttribute(selftest_gather4_timing_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
      cudaSuccess)
    return 3;
  selftest_gather4_timing_kernel<<<1, 512, smem, stream>>>(map, N, total, warps, lanes, out, status);
  return cudaGetLastError() == cudaSuccess ? 0 : 3;
}
