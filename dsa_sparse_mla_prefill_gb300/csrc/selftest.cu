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
// Pair (cta_group::2) check: D[256, N] = A[256, K] . B[N, K]^T as pair MMAs of
// a 2-CTA cluster.  CTA r stages A rows 128r .. 128r+127 and B rows (N/2) r ..
// (N/2)(r+1)-1 in its own shared memory (same offsets in both CTAs), in the
// K-major or MN-major 128B-swizzled layout, either by plain stores or (gather
// = 1, K-major A) by tile::gather4 loads of its own A rows whose bytes
// complete on the even CTA's barrier; one thread of the even CTA issues the
// pair MMAs and commits to both CTAs' barriers; each CTA reads its 128 rows
// of D back from its own tensor memory.
// ---------------------------------------------------------------------------
namespace {
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(128, 1)
    selftest_mma_pair_kernel(const __grid_constant__ CUtensorMap amap, const uint16_t* A, const uint16_t* B,
                             float* D, int N, int K, int a_mn, int b_mn, int gather, unsigned int* status) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  const int Nh = N / 2;
  uint8_t* As = smem;                          // 128 x K bf16 (this CTA's rows of A)
  uint8_t* Bs = smem + 128 * K * 2;            // N/2 x K bf16 (this CTA's rows of B)
  __shared__ uint64_t bar_full, bar_done;
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  const int tid = threadIdx.x, warp = tid >> 5;
  const int rank = (int)cluster_ctarank();
  const bool tma_a = gather && !a_mn;

  for (int i = tid; i < 128 * K && !tma_a; i += 128) {
    const int m = i / K, k = i % K;
    uint32_t off = a_mn ? (m / 64) * (K * 128) + sw128_offset(k, m % 64)
                        : (k / 64) * (128 * 128) + sw128_offset(m, k % 64);
    *reinterpret_cast<uint16_t*>(As + off) = A[(size_t)(128 * rank) * K + i];
  }
  for (int i = tid; i < Nh * K; i += 128) {
    const int n = i / K, k = i % K;
    uint32_t off = b_mn ? (n / 64) * (K * 128) + sw128_offset(k, n % 64)
                        : (k / 64) * (Nh * 128) + sw128_offset(n, k % 64);
    *reinterpret_cast<uint16_t*>(Bs + off) = B[(size_t)(Nh * rank) * K + i];
  }
  fence_proxy_async_smem();
  if (tid == 0) {
    mbar_init(&bar_full, 1);
    mbar_init(&bar_done, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc_pair(&tmem_slot, 256);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();   // both CTAs' operands and barriers exist before any load or MMA
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  if (tma_a) {
    const uint32_t full0 = map_peer(smem_u32(&bar_full), 0);
    if (rank == 0 && tid == 0) mbar_arrive_expect_tx(&bar_full, 2u * 128u * (uint32_t)K * 2u);
    if (tid < 32)
      for (int c = 0; c < K / 64; ++c) {
        const int r0 = 128 * rank + 4 * tid;
        tma_gather4_pair(smem_u32(As) + c * (128 * 128) + tid * 512, &amap, c * 64, r0, r0 + 1, r0 + 2, r0 + 3,
                         full0);
      }
  } else if (rank == 0 && tid == 0) {
    mbar_arrive(&bar_full);
  }
  if (rank == 0 && tid == 0) {
    if (mbar_wait_cluster(&bar_full, 0, &abort_flag, status)) {
      tc_fence_after();
      const uint32_t idesc = idesc_bf16_f32(256, N, a_mn == 1, b_mn != 0);
      const uint32_t a0 = smem_u32(As), b0 = smem_u32(Bs);
      for (int ks = 0; ks < K / 16; ks += 4) {
        const uint64_t ad = a_mn ? sdesc_sw128(a0 + ks * 2048, K * 128, 1024)
                                 : sdesc_sw128(a0 + (ks / 4) * (128 * 128), 16, 1024);
        const uint64_t bd = b_mn ? sdesc_sw128(b0 + ks * 2048, K * 128, 1024)
                                 : sdesc_sw128(b0 + (ks / 4) * (Nh * 128), 16, 1024);
        mma_pair_bf16_ss_x4(tmem, ad, bd, a_mn ? 128u : 2u, b_mn ? 128u : 2u, idesc, ks > 0 ? 1u : 0u);
      }
      mma_pair_commit(&bar_done, (uint16_t)3);
    }
  }
  __syncwarp();
  const bool ok = mbar_wait_cluster(&bar_done, 0, &abort_flag, status);
  tc_fence_after();
  if (ok) {
    for (int c = 0; c < N; c += 16) {
      float v[16];
      tmem_ld16(tmem + ((uint32_t)(warp * 32) << 16) + c, v);
      tmem_ld_wait();
      for (int i = 0; i < 16; ++i) D[(size_t)(128 * rank + tid) * N + c + i] = v[i];
    }
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();   // neither CTA frees tensor memory while the pair may still use it
  tc_fence_after();
  if (warp == 0) tmem_dealloc_pair(tmem, 256);
}
}  // namespace

extern "C" int dsa_selftest_mma_pair(const uint16_t* A, const uint16_t* B, float* D, int N, int K, int a_mn, int b_mn,
                                     int gather, unsigned int* status, cudaStream_t stream) {
  if (N < 32 || N > 256 || (N % 32) || K < 64 || (K % 64) || (a_mn && K > 128) || (b_mn && K > 128)) return 1;
  if (b_mn && ((N / 2) % 64)) return 1;
  const int smem = 128 * K * 2 + (N / 2) * K * 2 + 1024;
  if (smem > 227 * 1024) return 1;
  CUtensorMap map;
  if (!dsa::make_row_gather_map(&map, A, 256, K, K)) return 2;
  if (cudaFuncSetAttribute(selftest_mma_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
      cudaSuccess)
    return 3;
  selftest_mma_pair_kernel<<<2, 128, smem, stream>>>(map, A, B, D, N, K, a_mn, b_mn, gather, status);
  return cudaGetLastError() == cudaSuccess ? 0 : 3;
}
