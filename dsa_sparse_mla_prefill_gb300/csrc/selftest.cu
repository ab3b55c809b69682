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
  __shared__ uint64_t bar, bar2, bar3;  // bar3 is never armed: its parity-1 phase counts as complete
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  const int tid = threadIdx.x, warp = tid >> 5;
  for (int i = tid; i < (128 + N) * K / 8; i += 128) reinterpret_cast<uint4*>(As)[i] = make_uint4(0, 0, 0, 0);
  fence_proxy_async_smem();
  if (tid == 0) {
    mbar_init(&bar, 1);
    mbar_init(&bar2, 1);
    mbar_init(&bar3, 1);
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
  } else if (precomputed >= 8 && precomputed <= 13 && tid == 0) {
    // batches of four MMAs and a commit, the pattern of one K chunk: out[0]
    // = cycles the issuing thread spent in the batches; with 9 the thread
    // also waits for each batch to complete before the next one; 10: no
    // commits; 11: a commit every second batch; 12: a commit to a barrier
    // nobody waits on in between (a second one); 13: no clock reads
    const uint32_t idesc = idesc_bf16_f32(128, N, false, false);
    const uint64_t ad0 = sdesc_sw128(smem_u32(As), 16, 1024), bd0 = sdesc_sw128(smem_u32(Bs), 16, 1024);
    const int nb = reps / 4;
    long long issue = 0;
    const long long t0 = clock64();
    for (int bI = 0; bI < nb; ++bI) {
      const int ks = (bI * 4) & 15;
      const uint64_t ad = ad0 + (uint64_t)(((ks >> 2) * (128 * 128)) >> 4);
      const uint64_t bd = bd0 + (uint64_t)(((ks >> 2) * (N * 128)) >> 4);
      const long long ta = precomputed == 13 ? 0 : clock64();
      mma_bf16_ss_x4(tmem, ad, bd, 2u, 2u, idesc, bI > 0 ? 1u : 0u);
      if (precomputed == 8 || precomputed == 9 || precomputed == 13 || (precomputed == 11 && (bI & 1)))
        mma_commit(&bar);
      if (precomputed == 12) mma_commit(&bar2);
      if (precomputed != 13) issue += clock64() - ta;
      if (precomputed == 9 && !mbar_wait(&bar, (uint32_t)bI & 1u, &abort_flag, status)) break;
    }
    if (precomputed == 8 || precomputed == 13) mbar_wait(&bar, (uint32_t)(nb - 1) & 1u, &abort_flag, status);
    if (precomputed == 11) mbar_wait(&bar, (uint32_t)(nb / 2 - 1) & 1u, &abort_flag, status);
    if (precomputed == 10 || precomputed == 12) {
      mma_commit(&bar);
      mbar_wait(&bar, 0u, &abort_flag, status);
    }
    out[0] = issue;
    out[1] = clock64() - t0;
  } else if (precomputed >= 14 && precomputed <= 19 && tid == 0) {
    // what between MMA blocks drains the pipeline: 14 -- blocks of 8 MMAs and
    // a commit; 15 -- a tcgen05 fence after each 4-MMA block; 16 -- a test of
    // a completed barrier phase after each block; 17 -- nine blocks, then nine
    // commits to nine barriers; 18 -- a commit after each block, its barrier
    // tested (complete or not) before the next block; 19 -- blocks of 16 MMAs
    // and a commit
    const uint32_t idesc = idesc_bf16_f32(128, N, false, false);
    const uint64_t ad0 = sdesc_sw128(smem_u32(As), 16, 1024), bd0 = sdesc_sw128(smem_u32(Bs), 16, 1024);
    const int nb = reps / 4;
    const long long t0 = clock64();
    uint32_t phases = 0;
    for (int bI = 0; bI < nb; ++bI) {
      const int ks = (bI * 4) & 15;
      const uint64_t ad = ad0 + (uint64_t)(((ks >> 2) * (128 * 128)) >> 4);
      const uint64_t bd = bd0 + (uint64_t)(((ks >> 2) * (N * 128)) >> 4);
      mma_bf16_ss_x4(tmem, ad, bd, 2u, 2u, idesc, bI > 0 ? 1u : 0u);
      if (precomputed == 14 && (bI & 1)) { mma_commit(&bar); ++phases; }
      if (precomputed == 19 && (bI & 3) == 3) { mma_commit(&bar); ++phases; }
      if (precomputed == 15) tc_fence_after();
      if (precomputed == 16) (void)mbar_try_wait(smem_u32(&bar2), 1u);
      if (precomputed == 17 && (bI % 9) == 8)
        for (int c = 0; c < 9; ++c) { mma_commit(&bar); ++phases; }
      if (precomputed == 18) {
        mma_commit(&bar);
        ++phases;
        (void)mbar_try_wait(smem_u32(&bar), (phases - 1) & 1u);
      }
    }
    mma_commit(&bar2);
    mbar_wait(&bar2, 0u, &abort_flag, status);
    out[0] = phases;
    out[1] = clock64() - t0;
  } else if ((precomputed == 20 || precomputed == 21 || precomputed == 22) && tid == 0) {
    // the loop of mode 3 issued through the x4 helper (20), with a commit to a
    // second barrier after every block (21), or with the blocks' descriptors
    // built as in the kernels, sdesc_sw128 of a byte address per block (22)
    const uint32_t idesc = idesc_bf16_f32(128, N, false, false);
    const uint64_t ad0 = sdesc_sw128(smem_u32(As), 16, 1024), bd0 = sdesc_sw128(smem_u32(Bs), 16, 1024);
    const long long t0 = clock64();
    for (int r = 0; r < reps; r += 4) {
      const int ks = r & 15;
      const uint64_t ad = precomputed == 22 ? sdesc_sw128(smem_u32(As) + (ks >> 2) * (128 * 128), 16, 1024)
                                            : ad0 + (uint64_t)(((ks >> 2) * (128 * 128)) >> 4);
      const uint64_t bd = precomputed == 22 ? sdesc_sw128(smem_u32(Bs) + (ks >> 2) * (N * 128), 16, 1024)
                                            : bd0 + (uint64_t)(((ks >> 2) * (N * 128)) >> 4);
      mma_bf16_ss_x4(tmem, ad, bd, 2u, 2u, idesc, r > 0 ? 1u : 0u);
      if (precomputed == 21) mma_commit(&bar2);
    }
    const long long t1 = clock64();
    mma_commit(&bar);
    mbar_wait(&bar, 0, &abort_flag, status);
    out[0] = t1 - t0;
    out[1] = clock64() - t0;
  } else if ((precomputed == 23 || precomputed == 24) && (tid & 31) == 0 && warp < (precomputed == 23 ? 2 : 4)) {
    // 2 (23) or 4 (24) warps each issue reps / nw MMAs in x4 blocks into
    // their own 64-column accumulator; warp 0 records the time until all
    // of its MMAs completed (the others finish at about the same time)
    const int nw = precomputed == 23 ? 2 : 4;
    const uint32_t idesc = idesc_bf16_f32(128, N, false, false);
    const uint64_t ad0 = sdesc_sw128(smem_u32(As), 16, 1024), bd0 = sdesc_sw128(smem_u32(Bs), 16, 1024);
    const uint32_t d = tmem + (uint32_t)warp * 64u;
    const long long t0 = clock64();
    for (int r = 0; r < reps / nw; r += 4) {
      const int ks = r & 15;
      const uint64_t ad = ad0 + (uint64_t)(((ks >> 2) * (128 * 128)) >> 4);
      const uint64_t bd = bd0 + (uint64_t)(((ks >> 2) * (N * 128)) >> 4);
      mma_bf16_ss_x4(d, ad, bd, 2u, 2u, idesc, r > 0 ? 1u : 0u);
    }
    const long long t1 = clock64();
    if (warp == 0) {
      mma_commit(&bar);
      mbar_wait(&bar, 0, &abort_flag, status);
      out[0] = t1 - t0;
      out[1] = clock64() - t0;
    }
  } else if (precomputed >= 25 && precomputed <= 28 && (tid & 31) == 0 && warp < (precomputed == 27 ? 2 : 1)) {
    // the QK issue loop of the sparse kernels with its data always ready:
    // per 4-MMA block a barrier wait (a completed phase), a tcgen05 fence,
    // the MMAs and a commit (25); without the fence (26); split over two
    // warps with their own accumulators (27); two blocks per wait-fence
    // group (28, still one commit per block)
    const int nw = precomputed == 27 ? 2 : 1;
    const uint32_t idesc = idesc_bf16_f32(128, N, false, false);
    const uint64_t ad0 = sdesc_sw128(smem_u32(As), 16, 1024), bd0 = sdesc_sw128(smem_u32(Bs), 16, 1024);
    const uint32_t d = tmem + (uint32_t)warp * 64u;
    const long long t0 = clock64();
    const int step = precomputed == 28 ? 8 : 4;
    for (int r = 0; r < reps / nw; r += step) {
      const int ks = r & 15;
      const uint64_t ad = ad0 + (uint64_t)(((ks >> 2) * (128 * 128)) >> 4);
      const uint64_t bd = bd0 + (uint64_t)(((ks >> 2) * (N * 128)) >> 4);
      if (!mbar_wait(&bar3, 1u, &abort_flag, status)) break;
      if (precomputed == 28 && !mbar_wait(&bar3, 1u, &abort_flag, status)) break;
      if (precomputed != 26) tc_fence_after();
      mma_bf16_ss_x4(d, ad, bd, 2u, 2u, idesc, r > 0 ? 1u : 0u);
      mma_commit(&bar2);
      if (precomputed == 28) {
        mma_bf16_ss_x4(d, ad + 8, bd + 8, 2u, 2u, idesc, 1u);
        mma_commit(&bar2);
      }
    }
    const long long t1 = clock64();
    if (warp == 0) {
      mma_commit(&bar);
      mbar_wait(&bar, 0, &abort_flag, status);
      out[0] = t1 - t0;
      out[1] = clock64() - t0;
    }
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

// ---------------------------------------------------------------------------
// Whole-GPU TMA gather4 rate: every CTA of a grid of two-CTA clusters issues
// `per_cta` gathers (rows taken from `rows`, four per gather, 128 B each)
// into a 64 KB ring, from `warps` warps x `lanes` lanes; with `mc` each
// gather is multicast to both CTAs of the cluster.  out[cta] = cycles from
// the start (after a cluster barrier) until every byte bound for this CTA
// landed.  Used to size the gather streams of the kernels.
// ---------------------------------------------------------------------------
namespace {
constexpr int kRateMaxBars = 64;

__global__ void __launch_bounds__(512, 1) selftest_gather4_rate_kernel(const __grid_constant__ CUtensorMap map,
                                                                      const int* rows, int per_cta, int warps,
                                                                      int lanes, int mc, int flags, long long* out,
                                                                      unsigned int* status) {
  // flags: bit 0 -- 128 KB ring (gathers land in distinct places for up to
  // 256 gathers); bit 1 -- one completion barrier per 32 gathers (else 256);
  // bit 2 -- each batch of 32 gathers reads another 64-column slice (9 in a
  // row of 576); bit 3 -- every gather is preceded by a completed-phase
  // barrier test of the warp (the check a ring producer makes)
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* ring = smem_raw + (((raw + 1023u) & ~1023u) - raw);  // 64 or 128 KB
  const int kRateBatch = (flags & 2) ? 32 : 256;
  const int ring_mask = (flags & 1) ? 255 : 127;
  __shared__ uint64_t bars[kRateMaxBars + 1];  // the last one is never armed
  __shared__ int abort_flag;
  __shared__ long long t_start;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nb = (per_cta + kRateBatch - 1) / kRateBatch;
  if (tid == 0) {
    for (int b = 0; b <= kRateMaxBars; ++b) mbar_init(&bars[b], 1);
    abort_flag = 0;
    fence_mbar_init();
    for (int b = 0; b < nb; ++b) {
      const int cnt = min(kRateBatch, per_cta - b * kRateBatch);
      mbar_arrive_expect_tx(&bars[b], (uint32_t)cnt * 512u * (mc ? 2u : 1u));
    }
  }
  __syncthreads();
  cluster_sync();
  if (tid == 0) t_start = clock64();
  __syncthreads();
  const int issuers = warps * lanes;
  if (warp < warps && lane < lanes) {
    const int me = warp * lanes + lane;
    const int* my_rows = rows + (size_t)blockIdx.x * per_cta * 4;
    for (int g = me; g < per_cta; g += issuers) {
      const int4 r = *reinterpret_cast<const int4*>(my_rows + 4 * g);
      const uint32_t dst = smem_u32(ring) + (g & ring_mask) * 512;
      const int x = (flags & 4) ? ((g / 32) % 9) * 64 : 0;
      if (flags & 8) {
        // parity 1 of a barrier still in phase 0: complete by definition
        if (!mbar_wait(&bars[kRateMaxBars], 1u, &abort_flag, status)) break;
        __syncwarp(__activemask());
      }
      if (mc)
        tma_gather4_mc(dst, &map, x, r.x, r.y, r.z, r.w, &bars[g / kRateBatch], (uint16_t)3);
      else
        tma_gather4(dst, &map, x, r.x, r.y, r.z, r.w, &bars[g / kRateBatch]);
    }
  }
  if (tid == 0) {
    for (int b = 0; b < nb; ++b) mbar_wait(&bars[b], 0, &abort_flag, status);
    out[blockIdx.x] = clock64() - t_start;
  }
  __syncthreads();
  cluster_sync();  // the peer's copies into this CTA have landed (counted above)
}
}  // namespace

extern "C" int dsa_selftest_gather4_rate(const uint16_t* kv, int N, int ld, const int* rows_dev, int grid,
                                         int per_cta, int warps, int lanes, int mc, int flags, long long* out,
                                         unsigned int* status, cudaStream_t stream) {
  if (N < 8 || ld < 64 || (ld & 7) || warps < 1 || warps > 16 || lanes < 1 || lanes > 32 || per_cta < 1 ||
      per_cta > ((flags & 2) ? 32 : 256) * kRateMaxBars || grid < 2 || (grid & 1) || ((flags & 4) && ld < 576))
    return 1;
  CUtensorMap map;
  if (!dsa::make_row_gather_map(&map, kv, N, ld, ld)) return 2;
  const int smem = 131072 + 1024;
  if (cudaFuncSetAttribute(selftest_gather4_rate_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
      cudaSuccess)
    return 3;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(512, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = 2;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, selftest_gather4_rate_kernel, map, rows_dev, per_cta, warps, lanes, mc, flags, out,
                         status) !=
      cudaSuccess)
    return 3;
  return cudaGetLastError() == cudaSuccess ? 0 : 3;
}

// ---------------------------------------------------------------------------
// Gather ring turnaround: the K-stream pattern of the prefill kernels with no
// MMAs.  Each CTA of a two-CTA cluster streams `chunks` stages of 128 rows x
// 64 columns (16 KB) through a ring of `stages` slots.  The 32 gathers of a
// stage come from `warps` x `lanes` issuers; with `mc` each CTA issues half
// of them with multicast and a stage is refilled only after both CTAs
// released it.  One consumer thread waits for each stage, holds it for `hold`
// cycles and releases it.  out[cta] = cycles for the whole stream.  flags:
// bit 0 -- producers poll the empty barrier from lane 0 only; bit 1 -- with
// a short sleep between polls; bit 2 -- every gather reads columns 0..63;
// bit 4 -- the consumer arms a stage's next phase as soon as it has seen the
// current one complete (so no bytes land before the phase is armed); bit 5 --
// stage ownership: warp w fills only stage w (warps == stages), its `lanes`
// lanes sharing the stage's gathers; bit 6 -- no empty-barrier wait on the
// first pass over the ring (those phases are free anyway); bit 7 -- every
// stage gathers the rows of another tile (no row is fetched by consecutive
// stages).
// ---------------------------------------------------------------------------
namespace {
constexpr int kRingMaxStages = 8;

__global__ void __launch_bounds__(512, 1) selftest_ring_rate_kernel(const __grid_constant__ CUtensorMap map,
                                                                   const int* rows, int ntiles, int chunks,
                                                                   int stages, int warps, int lanes, int mc,
                                                                   int hold, int flags, long long* out,
                                                                   unsigned int* status) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* ring = smem_raw + (((raw + 1023u) & ~1023u) - raw);  // stages x 16 KB
  __shared__ uint64_t full[kRingMaxStages], empty[kRingMaxStages];
  __shared__ int abort_flag;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int rank = (int)cluster_ctarank();
  const int cl = blockIdx.x >> 1;
  if (tid == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], mc ? 2 : 1);
    }
    abort_flag = 0;
    if (flags & 16)
      for (int s = 0; s < stages; ++s) mbar_arrive_expect_tx(&full[s], 16384u);
    fence_mbar_init();
  }
  __syncthreads();
  cluster_sync();
  const int per_chunk = mc ? 16 : 32;  // gathers this CTA issues per stage
  if (warp < warps) {
    const bool owned = (flags & 32) != 0;
    const int me = owned ? lane : warp * lanes + lane;
    const int pstride = owned ? lanes : per_chunk;  // gathers per issuing lane: per_chunk / pstride
    const bool issuer = lane < lanes && me < per_chunk;
    for (int pos = owned ? warp : 0; pos < chunks; pos += owned ? stages : 1) {
      const int s = pos % stages;
      const uint32_t par = ((pos / stages) & 1) ^ 1;
      if ((flags & 64) && pos < stages) {
      } else if (flags & 1) {
        int ok = 1;
        if (lane == 0) {
          const uint32_t a = smem_u32(&empty[s]);
          const uint64_t t0 = globaltimer();
          while (!mbar_try_wait(a, par)) {
            if (flags & 2) __nanosleep(32);
            volatile int* af = &abort_flag;
            if (*af || globaltimer() - t0 > kWaitTimeoutNs) {
              *af = 1;
              ok = 0;
              break;
            }
          }
        }
        if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      } else if (!mbar_wait_warp(&empty[s], par, &abort_flag, status)) {
        break;
      }
      if ((owned || warp == 0) && lane == 0 && !(flags & 16)) mbar_arrive_expect_tx(&full[s], 16384u);
      const int x = (flags & 4) ? 0 : (pos % 9) * 64;
      const int tile = (flags & 128) ? pos % ntiles : (pos / 9) % ntiles;
      for (int q = me; issuer && q < per_chunk; q += pstride) {
        const int rg = mc ? 16 * rank + q : q;
        const int4 r = __ldg(reinterpret_cast<const int4*>(rows + ((size_t)(cl * ntiles + tile) * 32 + rg) * 4));
        const uint32_t dst = smem_u32(ring) + s * 16384 + rg * 512;
        if (mc)
          tma_gather4_mc(dst, &map, x, r.x, r.y, r.z, r.w, &full[s], (uint16_t)3);
        else
          tma_gather4(dst, &map, x, r.x, r.y, r.z, r.w, &full[s]);
      }
    }
  } else if (warp == 15 && lane == 0) {
    const long long t0 = clock64();
    for (int pos = 0; pos < chunks; ++pos) {
      const int s = pos % stages;
      if (!mbar_wait(&full[s], (pos / stages) & 1, &abort_flag, status)) break;
      if ((flags & 16) && pos + stages < chunks) mbar_arrive_expect_tx(&full[s], 16384u);
      const long long th = clock64();
      while (clock64() - th < hold) {
      }
      mbar_arrive(&empty[s]);
      if (mc) mbar_arrive_remote(map_peer(smem_u32(&empty[s]), (uint32_t)(rank ^ 1)));
    }
    out[blockIdx.x] = clock64() - t0;
    // the last stages' bytes have landed here (waited above); the peer's
    // copies into this CTA are part of them
  }
  __syncthreads();
  cluster_sync();
}
}  // namespace

extern "C" int dsa_selftest_ring_rate(const uint16_t* kv, int N, int ld, const int* rows_dev, int ntiles, int grid,
                                      int chunks, int stages, int warps, int lanes, int mc, int hold, int flags,
                                      long long* out, unsigned int* status, cudaStream_t stream) {
  if (N < 8 || ld < 576 || (ld & 7) || warps < 1 || warps > 15 || lanes < 1 || lanes > 32 || chunks < 1 ||
      stages < 1 || stages > kRingMaxStages || ntiles < 1 || grid < 2 || (grid & 1) || hold < 0 || hold > 100000 ||
      ((flags & 32) ? warps != stages : warps * lanes < (mc ? 16 : 32)))
    return 1;
  CUtensorMap map;
  if (!dsa::make_row_gather_map(&map, kv, N, ld, ld)) return 2;
  const int smem = kRingMaxStages * 16384 + 1024;
  if (cudaFuncSetAttribute(selftest_ring_rate_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
      cudaSuccess)
    return 3;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(512, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = 2;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, selftest_ring_rate_kernel, map, rows_dev, ntiles, chunks, stages, warps, lanes, mc,
                         hold, flags, out, status) != cudaSuccess)
    return 3;
  return cudaGetLastError() == cudaSuccess ? 0 : 3;
}
