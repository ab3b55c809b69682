// dsa_sparse_prefill_host without a caller workspace (host code plus one
// file-scope device array).
//
// Some callers cannot hand the library device memory: a plug-in that runs
// inside a host program whose allocator owns the whole GPU (every byte
// already reserved by a caching allocator, so a cudaMalloc of its own would
// fail), or a runtime that forbids device allocation once it is serving.
// For them this entry point runs the same chunked, copy-overlapped pipeline
// as dsa_sparse_prefill_host, with its buffer sets in a fixed scratch array
// that is part of the library's own device image: the array exists on every
// device where this file's device code is loaded, for as long as the process
// runs, and no call allocates or frees anything.
//
// Host code may not use the array's name as a device address (on the host it
// names a stand-in object), so the first call on each device asks the runtime
// for the array's device address with that device current and keeps it.
#include <cstdint>

#include <cuda_runtime.h>

#include "../../include/dsa.h"

namespace {

// The scratch: DSA_HOST_NOALLOC_SCRATCH_BYTES, 256-byte aligned as the
// pipeline's buffer sets require.  Shared by every call on a device.
static __device__ __align__(256) uint8_t g_host_scratch[DSA_HOST_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDev = 64;
void* g_scratch_addr[kMaxDev] = {};

}  // namespace

extern "C" {

int dsa_sparse_prefill_host_noalloc(const uint16_t* q, const uint16_t* kv, int kv_on_host, int N, int ld_kv,
                                    const int32_t* idx, int T, int H, int d_qk, int d_v, int k, int ld, float scale,
                                    uint16_t* out, float* lse, int chunk_tokens, dsa_stream_t stream) {
  if (T < 0 || N < 0 || k < 0 || ld < k || ld_kv < d_qk || chunk_tokens < 1) return DSA_ERR_INVALID_ARG;
  const int64_t need =
      dsa_sparse_prefill_host_workspace(T, N, ld_kv, H, d_qk, d_v, ld, chunk_tokens, kv_on_host);
  if (need < 0) return DSA_ERR_INVALID_ARG;
  // the shape's buffers do not fit the fixed scratch: a smaller chunk_tokens
  // (or kv already on the device) needs less
  if (need > (int64_t)DSA_HOST_NOALLOC_SCRATCH_BYTES) return DSA_ERR_UNSUPPORTED;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) {
    cudaGetLastError();
    return DSA_ERR_CUDA;
  }
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_host_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return DSA_ERR_CUDA;
    }
    g_scratch_addr[dev] = p;
  }
  return dsa_sparse_prefill_host(q, kv, kv_on_host, N, ld_kv, idx, T, H, d_qk, d_v, k, ld, scale, out, lse,
                                 g_scratch_addr[dev], (int64_t)DSA_HOST_NOALLOC_SCRATCH_BYTES, chunk_tokens, stream);
}

}  // extern "C"
