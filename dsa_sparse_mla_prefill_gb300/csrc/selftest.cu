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
    for (int ks = 0; ks < K / 16; ++ks) {
      const uint64_t ad = a_mn ? sdesc_sw128(a0 + ks * 2048, K * 128, 1024)
                               : sdesc_sw128(a0 + (ks / 4) * (128 * 128) + (ks % 4) * 32, 16, 1024);
      const uint64_t bd = b_mn ? sdesc_sw128(b0 + ks * 2048, K * 128, 1024)
                               : sdesc_sw128(b0 + (ks / 4) * (N * 128) + (ks % 4) * 32, 16, 1024);
      if (a_mn == 2)
        mma_bf16_ts(tmem, tmem + 128 + ks * 8, bd, idesc_bf16_f32(128, N, false, b_mn != 0), ks > 0 ? 1u : 0u);
      else
        mma_bf16_ss(tmem, ad, bd, idesc, ks > 0 ? 1u : 0u);
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
