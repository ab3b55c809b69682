// Top-k -> packed per-token key mask for the masked dense-MHA form.
//
// "[2/N][Attention] Enable masked MHA for sparse MLA prefills", commit log:
// the masked path scatters each token's top-k indices into a key mask that
// is zeroed inside the kernel.  Bit n of row t (word n >> 5, bit n & 31,
// LSB first) stands for key cu_seqlens_kv[r] + n of the token's request r.
//
// One CTA per token: zero the row in shared memory, set the bits with
// shared-memory atomics, write the row out with coalesced stores.
#include "dsa_device.cuh"
#include "dsa_kernels.h"

namespace dsa {
namespace keymask {

constexpr int NT = 256;

__global__ void __launch_bounds__(NT) topk_to_key_mask_kernel(KeyMaskArgs a) {
  extern __shared__ uint32_t row_s[];
  const int t = blockIdx.x;
  int r = 0;
  while (r + 1 < a.req.num_req && a.req.cu_q[r + 1] <= t) ++r;
  const int kv0 = a.req.cu_kv[r];
  const int nk = a.req.cu_kv[r + 1] - kv0;
  const int nbits = min(nk, a.words * 32);

  for (int i = threadIdx.x; i < a.words; i += NT) row_s[i] = 0u;
  __syncthreads();
  const int32_t* idx = a.idx + (size_t)t * a.ld;
  int bad = 0;
  for (int e = threadIdx.x; e < a.k; e += NT) {
    const int x = __ldg(idx + e);
    if (x == -1) continue;
    const int n = x - kv0;
    if (x >= 0 && n >= 0 && n < nbits) {
      atomicOr(&row_s[n >> 5], 1u << (n & 31));
    } else {
      ++bad;
    }
  }
  bad = __reduce_add_sync(0xffffffffu, bad);
  if ((threadIdx.x & 31) == 0 && bad) atomicAdd(a.err + ERR_BAD_INDEX, (unsigned)bad);
  __syncthreads();
  uint32_t* out = a.key_mask + (size_t)t * a.words;
  for (int i = threadIdx.x; i < a.words; i += NT) out[i] = row_s[i];
}

}  // namespace keymask

int launch_topk_to_key_mask(const KeyMaskArgs& a, cudaStream_t stream) {
  const int smem = a.words * 4;
  if (smem > 48 * 1024) {
    if (cudaFuncSetAttribute(keymask::topk_to_key_mask_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem) != cudaSuccess)
      return -1;
  }
  if (a.T == 0) return 0;
  keymask::topk_to_key_mask_kernel<<<a.T, keymask::NT, smem, stream>>>(a);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace dsa
