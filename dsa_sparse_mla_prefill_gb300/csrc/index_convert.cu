// Request-local -> physical KV row conversion for the sparse forms.
//
// "[Perf][DSA] Grouped sparse prefill with the FlashMLA head-group-mask
// kernel", How: the selected positions are request-local (position x of the
// request's KV sequence) and are mapped to physical rows of the paged KV
// cache before the attention reads them.  With the request's block table
// (one physical block id per logical block of block_size positions):
//     row(x) = block_table[r][x / block_size] * block_size + x % block_size
// for 0 <= x < kv_len[r] with a mapped block (id >= 0) and a row inside the
// table; -1 stays -1, columns at or past k become -1, and every other entry
// becomes -1 and is counted as an ignored index entry.
//
// One CTA per token, coalesced over the row (16-byte accesses when the row
// stride allows); in place is allowed (each entry is read and written by the
// same thread).
#include "dsa_device.cuh"
#include "dsa_kernels.h"

namespace dsa {
namespace convert {

constexpr int NT = 256;

__device__ __forceinline__ int request_of(const ReqTable& rq, int t) {
  int lo = 0, hi = rq.num_req - 1;   // largest r with cu_q[r] <= t
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (rq.cu_q[mid] <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__device__ __forceinline__ int32_t to_row(int32_t x, int e, const ConvertArgs& a, const int32_t* bt, int kv_len,
                                          int& bad) {
  if (e >= a.k || x == -1) return -1;
  if (x < 0 || x >= kv_len) {
    ++bad;
    return -1;
  }
  const int32_t blk = __ldg(bt + x / a.block_size);
  const int64_t row = (int64_t)blk * a.block_size + x % a.block_size;
  if (blk < 0 || row >= a.N) {
    ++bad;
    return -1;
  }
  return (int32_t)row;
}

__global__ void __launch_bounds__(NT) local_to_global_kernel(ConvertArgs a) {
  const int t = blockIdx.x;
  const int r = request_of(a.req, t);
  const int kv_len = a.req.cu_kv[r + 1] - a.req.cu_kv[r];
  const int32_t* bt = a.block_table + (size_t)r * a.max_blocks;
  const int32_t* src = a.idx_local + (size_t)t * a.ld;
  int32_t* dst = a.idx_global + (size_t)t * a.ld;
  int bad = 0;
  if (a.vec) {
    for (int e4 = threadIdx.x; e4 < a.ld / 4; e4 += NT) {
      const int4 x = reinterpret_cast<const int4*>(src)[e4];
      int4 y;
      y.x = to_row(x.x, 4 * e4 + 0, a, bt, kv_len, bad);
      y.y = to_row(x.y, 4 * e4 + 1, a, bt, kv_len, bad);
      y.z = to_row(x.z, 4 * e4 + 2, a, bt, kv_len, bad);
      y.w = to_row(x.w, 4 * e4 + 3, a, bt, kv_len, bad);
      reinterpret_cast<int4*>(dst)[e4] = y;
    }
  } else {
    for (int e = threadIdx.x; e < a.ld; e += NT) dst[e] = to_row(src[e], e, a, bt, kv_len, bad);
  }
  bad = __reduce_add_sync(0xffffffffu, bad);
  if ((threadIdx.x & 31) == 0 && bad) atomicAdd(a.err + ERR_BAD_INDEX, (unsigned)bad);
}

}  // namespace convert

int launch_local_to_global(const ConvertArgs& a, cudaStream_t stream) {
  if (a.T == 0) return 0;
  convert::local_to_global_kernel<<<a.T, convert::NT, 0, stream>>>(a);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace dsa
