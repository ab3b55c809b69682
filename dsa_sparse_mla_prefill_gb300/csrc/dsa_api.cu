// C-ABI shim: argument validation, host-side request tables and kernel
// launches for the entry points declared in include/dsa.h.
#include <cstdint>
#include <cstring>
#include <vector>

#include <cuda_runtime.h>

#include "../../include/dsa.h"
#include "dsa_kernels.h"
#include "dsa_tmap.h"

namespace {

// Device error counters (see dsa_last_device_error).  One copy per device
// that loads the library.
__device__ unsigned int g_dsa_err[4];

constexpr int kMaxDev = 64;

struct DevInfo {
  bool init = false;
  int num_sms = 0;
  unsigned int* err = nullptr;
};
DevInfo g_dev[kMaxDev];

// diagnostic timeline buffer (dsa_debug_trace)
dsa::TraceArgs g_trace = {nullptr, 0};

// Per-device set-up: SM count and the device address of the error counters.
bool dev_info(DevInfo** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return false;
  DevInfo& d = g_dev[dev];
  if (!d.init) {
    if (cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return false;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_dsa_err) != cudaSuccess) return false;
    d.err = static_cast<unsigned int*>(p);
    d.init = true;
  }
  *out = &d;
  return true;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

// Fills a request table from host offsets (NULL = one request of T tokens).
// With G > 0, cu_g holds group offsets (G tokens of one request per group).
int fill_req(dsa::ReqTable& rq, const int32_t* cu_q, const int32_t* cu_kv, int num_req, int T, int Nkv,
             int G) {
  if (cu_q == nullptr) {
    if (cu_kv != nullptr) return DSA_ERR_INVALID_ARG;
    num_req = 1;
  }
  if (num_req < 1) return DSA_ERR_INVALID_ARG;
  if (num_req > dsa::kMaxReq) return DSA_ERR_UNSUPPORTED;
  rq.num_req = num_req;
  rq.cu_q[0] = 0;
  rq.cu_kv[0] = 0;
  rq.cu_g[0] = 0;
  for (int r = 0; r < num_req; ++r) {
    const int q0 = cu_q ? cu_q[r] : 0, q1 = cu_q ? cu_q[r + 1] : T;
    // without KV offsets the (single) request spans Nkv rows; Nkv < 0 = not used
    const int k0 = cu_kv ? cu_kv[r] : 0, k1 = cu_kv ? cu_kv[r + 1] : (Nkv > 0 ? Nkv : 0);
    if (q1 < q0 || k1 < k0) return DSA_ERR_INVALID_ARG;
    if (r == 0 && (q0 != 0 || k0 != 0)) return DSA_ERR_INVALID_ARG;
    rq.cu_q[r + 1] = q1;
    rq.cu_kv[r + 1] = k1;
    const int ng = (G > 0) ? (q1 - q0 + G - 1) / G : 0;
    rq.cu_g[r + 1] = rq.cu_g[r] + ng;
  }
  if (rq.cu_q[num_req] != T) return DSA_ERR_INVALID_ARG;
  if (Nkv >= 0 && cu_kv && rq.cu_kv[num_req] != Nkv) return DSA_ERR_INVALID_ARG;
  return DSA_OK;
}

constexpr int kMaxSmem = 232448;

}  // namespace

extern "C" {

const char* dsa_status_string(int status) {
  switch (status) {
    case DSA_OK: return "DSA_OK";
    case DSA_ERR_INVALID_ARG: return "DSA_ERR_INVALID_ARG";
    case DSA_ERR_UNSUPPORTED: return "DSA_ERR_UNSUPPORTED";
    case DSA_ERR_CUDA: return "DSA_ERR_CUDA";
    case DSA_ERR_DEVICE: return "DSA_ERR_DEVICE";
    default: return "DSA_ERR_UNKNOWN";
  }
}

int dsa_version(void) { return 100; }

int64_t dsa_union_pad(int G, int k, int union_block) {
  if (G <= 0 || k <= 0 || union_block <= 0) return -1;
  const int64_t n = (int64_t)G * k;
  return (n + union_block - 1) / union_block * union_block;
}

int dsa_num_groups(const int32_t* cu_seqlens_q_host, int num_req, int T, int G, int* num_groups) {
  if (num_groups == nullptr || G <= 0 || T < 0) return DSA_ERR_INVALID_ARG;
  if (cu_seqlens_q_host == nullptr) {
    *num_groups = (T + G - 1) / G;
    return DSA_OK;
  }
  if (num_req < 1 || cu_seqlens_q_host[0] != 0 || cu_seqlens_q_host[num_req] != T) return DSA_ERR_INVALID_ARG;
  int64_t n = 0;
  for (int r = 0; r < num_req; ++r) {
    const int len = cu_seqlens_q_host[r + 1] - cu_seqlens_q_host[r];
    if (len < 0) return DSA_ERR_INVALID_ARG;
    n += (len + G - 1) / G;
  }
  *num_groups = (int)n;
  return DSA_OK;
}

int dsa_union_build(const int32_t* idx, int T, int k, int ld, int G, const int32_t* cu_seqlens_q_host,
                    int num_req, int N, int32_t* union_idx, int32_t* union_len, uint8_t* mask, int union_pad,
                    dsa_stream_t stream) {
  if (T < 0 || k < 0 || ld < k || G < 1 || N < 0 || union_pad < 0) return DSA_ERR_INVALID_ARG;
  if (G > 8) return DSA_ERR_UNSUPPORTED;
  if ((union_pad & 15) != 0) return DSA_ERR_INVALID_ARG;
  const int64_t need = (int64_t)G * k < N ? (int64_t)G * k : N;
  if (union_pad < need) return DSA_ERR_INVALID_ARG;
  if (dsa::union_build_smem_bytes(N, union_pad) > kMaxSmem) return DSA_ERR_UNSUPPORTED;
  if (T == 0) return DSA_OK;
  if (!idx || !union_idx || !union_len || !mask) return DSA_ERR_INVALID_ARG;
  if (!aligned4(idx) || !aligned16(union_idx) || !aligned16(mask) || !aligned4(union_len))
    return DSA_ERR_INVALID_ARG;
  dsa::UnionArgs a;
  int st = fill_req(a.req, cu_seqlens_q_host, nullptr, num_req, T, -1, G);
  if (st != DSA_OK) return st;
  DevInfo* d;
  if (!dev_info(&d)) return DSA_ERR_CUDA;
  a.idx = idx;
  a.union_idx = union_idx;
  a.union_len = union_len;
  a.mask = mask;
  a.err = d->err;
  a.T = T;
  a.k = k;
  a.ld = ld;
  a.G = G;
  a.N = N;
  a.union_pad = union_pad;
  a.num_groups = a.req.cu_g[a.req.num_req];
  return dsa::launch_union_build(a, (cudaStream_t)stream) == 0 ? DSA_OK : DSA_ERR_CUDA;
}

int dsa_sparse_prefill(const uint16_t* q, const uint16_t* kv, int N, int ld_kv, const int32_t* idx, int T,
                       int H, int d_qk, int d_v, int k, int ld, float scale, uint16_t* out, float* lse,
                       dsa_stream_t stream) {
  return dsa::sparse_prefill_streamed(q, kv, N, ld_kv, idx, T, H, d_qk, d_v, k, ld, scale, out, lse, nullptr,
                                      nullptr, 0, (cudaStream_t)stream);
}

}  // extern "C"

namespace dsa {

int sparse_prefill_streamed(const uint16_t* q, const uint16_t* kv, int N, int ld_kv, const int32_t* idx, int T,
                            int H, int d_qk, int d_v, int k, int ld, float scale, uint16_t* out, float* lse,
                            const uint32_t* ready, uint32_t* done, int done_blk, cudaStream_t stream) {
  if (T < 0 || N < 0 || k < 0 || ld < k || ld_kv < d_qk) return DSA_ERR_INVALID_ARG;
  if (!(H == 16 || H == 32) || !(d_qk == 576 || d_qk == 512) || d_v != 512 || k > 2048)
    return DSA_ERR_UNSUPPORTED;
  if ((ld_kv & 7) != 0) return DSA_ERR_INVALID_ARG;
  if (T == 0) return DSA_OK;
  // (kv may be null only for an empty table, N = 0)
  if (!q || (!kv && N > 0) || !idx || !out || !lse) return DSA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(kv) || !aligned4(idx) || !aligned4(out) || !aligned4(lse))
    return DSA_ERR_INVALID_ARG;
  DevInfo* d;
  if (!dev_info(&d)) return DSA_ERR_CUDA;
  dsa::SparseArgs a;
  a.q = q;
  a.kv = kv;
  a.kv8 = nullptr;
  a.row_bytes = 0;
  a.idx = idx;
  a.out = out;
  a.lse = lse;
  a.err = d->err;
  a.T = T;
  a.H = H;
  a.d_qk = d_qk;
  a.N = N;
  a.ld_kv = ld_kv;
  a.k = k;
  a.ld = ld;
  a.scale = scale;
  a.tr = g_trace;
  a.ready = ready;
  a.done = done;
  a.done_blk = done_blk;
  if ((ready == nullptr) != (done == nullptr) || (done != nullptr && done_blk < 1)) return DSA_ERR_INVALID_ARG;
  // With N = 0 every index is out of range, no tile is formed and the map is
  // never used: it is encoded over q so that it is well formed.
  if (!dsa::make_row_gather_map(&a.tmap_kv, N > 0 ? (const void*)kv : (const void*)q, N > 0 ? N : 1,
                                N > 0 ? ld_kv : d_qk, N > 0 ? ld_kv : d_qk))
    return DSA_ERR_CUDA;
  if (!dsa::make_tile_map(&a.tmap_q, q, (int64_t)T * H, d_qk, d_qk, H)) return DSA_ERR_CUDA;
  const int r = dsa::launch_sparse_prefill(a, d->num_sms, stream);
  return r == 0 ? DSA_OK : (r == -2 ? DSA_ERR_UNSUPPORTED : DSA_ERR_CUDA);
}

}  // namespace dsa

extern "C" {

int dsa_grouped_prefill(const uint16_t* q, const uint16_t* kv, int N, int ld_kv, const int32_t* union_idx,
                        const int32_t* union_len, const uint8_t* mask, int union_pad, int G,
                        const int32_t* cu_seqlens_q_host, int num_req, int T, int H, int d_qk, int d_v,
                        float scale, uint16_t* out, float* lse, dsa_stream_t stream) {
  if (T < 0 || N < 0 || G < 1 || H < 1 || union_pad < 0 || ld_kv < d_qk) return DSA_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !(scale < INFINITY)) return DSA_ERR_INVALID_ARG;
  if (G > 8 || G * H != 128 || !(d_qk == 576 || d_qk == 512) || d_v != 512) return DSA_ERR_UNSUPPORTED;
  if ((ld_kv & 7) != 0 || (union_pad & 15) != 0) return DSA_ERR_INVALID_ARG;
  if (T == 0) return DSA_OK;
  // (kv may be null only for an empty table, N = 0)
  if (!q || (!kv && N > 0) || !union_idx || !union_len || !mask || !out || !lse) return DSA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(kv) || !aligned16(union_idx) || !aligned16(mask) || !aligned16(out) ||
      !aligned4(lse))
    return DSA_ERR_INVALID_ARG;
  dsa::GroupedArgs a;
  int st = fill_req(a.req, cu_seqlens_q_host, nullptr, num_req, T, -1, G);
  if (st != DSA_OK) return st;
  DevInfo* d;
  if (!dev_info(&d)) return DSA_ERR_CUDA;
  a.q = q;
  a.kv = kv;
  a.union_idx = union_idx;
  a.union_len = union_len;
  a.mask = mask;
  a.out = out;
  a.lse = lse;
  a.err = d->err;
  a.T = T;
  a.H = H;
  a.G = G;
  a.d_qk = d_qk;
  a.N = N;
  a.ld_kv = ld_kv;
  a.union_pad = union_pad;
  a.num_groups = a.req.cu_g[a.req.num_req];
  a.scale = scale;
  a.tr = g_trace;
  // With N = 0 every union is empty and the map is never used (encoded over q).
  if (!dsa::make_row_gather_map(&a.tmap_kv, N > 0 ? (const void*)kv : (const void*)q, N > 0 ? N : 1,
                                N > 0 ? ld_kv : d_qk, N > 0 ? ld_kv : d_qk))
    return DSA_ERR_CUDA;
  if (!dsa::make_tile_map(&a.tmap_q, q, (int64_t)T * H, d_qk, d_qk, 64)) return DSA_ERR_CUDA;
  if (!dsa::make_tile_map(&a.tmap_kv_blk, N > 0 ? (const void*)kv : (const void*)q, N > 0 ? N : 1,
                          N > 0 ? ld_kv : d_qk, N > 0 ? ld_kv : d_qk, 64))
    return DSA_ERR_CUDA;
  const int r = dsa::launch_grouped_prefill(a, d->num_sms, (cudaStream_t)stream);
  return r == 0 ? DSA_OK : (r == -2 ? DSA_ERR_UNSUPPORTED : DSA_ERR_CUDA);
}

int dsa_topk_to_key_mask(const int32_t* idx, int T, int k, int ld, const int32_t* cu_seqlens_q_host,
                         const int32_t* cu_seqlens_kv_host, int num_req, uint32_t* key_mask, int words,
                         dsa_stream_t stream) {
  if (T < 0 || k < 0 || ld < k || words < 1) return DSA_ERR_INVALID_ARG;
  if ((cu_seqlens_q_host == nullptr) != (cu_seqlens_kv_host == nullptr)) return DSA_ERR_INVALID_ARG;
  if (words * 4 > kMaxSmem) return DSA_ERR_UNSUPPORTED;
  if (T == 0) return DSA_OK;
  if (!idx || !key_mask || !aligned4(idx) || !aligned4(key_mask)) return DSA_ERR_INVALID_ARG;
  dsa::KeyMaskArgs a;
  // one request without offsets: every key of [0, 32*words) is request-local
  int st = fill_req(a.req, cu_seqlens_q_host, cu_seqlens_kv_host, num_req, T,
                    cu_seqlens_kv_host ? -1 : 32 * words, 0);
  if (st != DSA_OK) return st;
  for (int r = 0; r < a.req.num_req; ++r)
    if (a.req.cu_kv[r + 1] - a.req.cu_kv[r] > 32 * words) return DSA_ERR_INVALID_ARG;
  DevInfo* d;
  if (!dev_info(&d)) return DSA_ERR_CUDA;
  a.idx = idx;
  a.key_mask = key_mask;
  a.err = d->err;
  a.T = T;
  a.k = k;
  a.ld = ld;
  a.words = words;
  return dsa::launch_topk_to_key_mask(a, (cudaStream_t)stream) == 0 ? DSA_OK : DSA_ERR_CUDA;
}

int dsa_local_to_global(const int32_t* idx_local, int T, int k, int ld, const int32_t* cu_seqlens_q_host,
                        const int32_t* kv_lens_host, int num_req, const int32_t* block_table, int max_blocks,
                        int block_size, int N, int32_t* idx_global, dsa_stream_t stream) {
  if (T < 0 || k < 0 || ld < k || block_size < 1 || max_blocks < 1 || N < 0) return DSA_ERR_INVALID_ARG;
  if (kv_lens_host == nullptr) return DSA_ERR_INVALID_ARG;
  if (cu_seqlens_q_host == nullptr) num_req = 1;
  if (num_req < 1) return DSA_ERR_INVALID_ARG;
  if (num_req > dsa::kMaxReq) return DSA_ERR_UNSUPPORTED;
  // cumulative KV lengths stand in for the KV offsets of the request table
  std::vector<int32_t> cu_kv(num_req + 1, 0);
  for (int r = 0; r < num_req; ++r) {
    if (kv_lens_host[r] < 0 || (int64_t)kv_lens_host[r] > (int64_t)max_blocks * block_size)
      return DSA_ERR_INVALID_ARG;
    if ((int64_t)cu_kv[r] + kv_lens_host[r] > INT32_MAX) return DSA_ERR_UNSUPPORTED;
    cu_kv[r + 1] = cu_kv[r] + kv_lens_host[r];
  }
  dsa::ConvertArgs a;
  const int32_t one_req[2] = {0, T};   // NULL cu_seqlens_q: one request of T tokens
  int st = fill_req(a.req, cu_seqlens_q_host ? cu_seqlens_q_host : one_req, cu_kv.data(), num_req, T, -1, 0);
  if (st != DSA_OK) return st;
  if (T == 0) return DSA_OK;
  if (!idx_local || !idx_global || !block_table || !aligned4(idx_local) || !aligned4(idx_global) ||
      !aligned4(block_table))
    return DSA_ERR_INVALID_ARG;
  DevInfo* d;
  if (!dev_info(&d)) return DSA_ERR_CUDA;
  a.idx_local = idx_local;
  a.idx_global = idx_global;
  a.block_table = block_table;
  a.err = d->err;
  a.T = T;
  a.k = k;
  a.ld = ld;
  a.max_blocks = max_blocks;
  a.block_size = block_size;
  a.N = N;
  a.vec = (ld % 4 == 0) && aligned16(idx_local) && aligned16(idx_global) ? 1 : 0;
  return dsa::launch_local_to_global(a, (cudaStream_t)stream) == 0 ? DSA_OK : DSA_ERR_CUDA;
}

int dsa_masked_mha_prefill_strided(const uint16_t* q, int64_t q_stride_t, int64_t q_stride_h, const uint16_t* k,
                                   int64_t k_stride_t, int64_t k_stride_h, const uint16_t* k_pe,
                                   int64_t k_pe_stride_t, const uint16_t* v, int64_t v_stride_t, int64_t v_stride_h,
                                   const uint32_t* key_mask, int words, const int32_t* cu_seqlens_q_host,
                                   const int32_t* cu_seqlens_kv_host, int num_req, int T, int H, int d_qk,
                                   int d_rope, int d_v, float scale, uint16_t* out, float* lse, dsa_stream_t stream) {
  if (T < 0 || H < 1 || words < 1) return DSA_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !(scale < INFINITY)) return DSA_ERR_INVALID_ARG;
  if ((cu_seqlens_q_host == nullptr) != (cu_seqlens_kv_host == nullptr)) return DSA_ERR_INVALID_ARG;
  if (!((d_qk == 192 && d_v == 128) || (d_qk == 256 && d_v == 256))) return DSA_ERR_UNSUPPORTED;
  if (d_rope != 0 && d_rope != 64) return DSA_ERR_UNSUPPORTED;
  if (T == 0) return DSA_OK;
  const int d_k = d_qk - d_rope;   // columns of each key row read from k
  if (!q || !k || !v || !key_mask || !out || !lse || (d_rope > 0 && !k_pe)) return DSA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(key_mask) || !aligned16(out) ||
      !aligned4(lse) || (d_rope > 0 && !aligned16(k_pe)))
    return DSA_ERR_INVALID_ARG;
  // strides in elements: multiples of 8 (16 bytes, the TMA rule), heads and
  // rows not overlapping
  auto strides_ok = [&](int64_t st, int64_t sh, int cols) {
    return (st % 8) == 0 && (sh % 8) == 0 && sh >= cols && st >= (int64_t)H * sh;
  };
  if (!strides_ok(q_stride_t, q_stride_h, d_qk) || !strides_ok(k_stride_t, k_stride_h, d_k) ||
      !strides_ok(v_stride_t, v_stride_h, d_v))
    return DSA_ERR_INVALID_ARG;
  if (d_rope > 0 && ((k_pe_stride_t % 8) != 0 || k_pe_stride_t < d_rope)) return DSA_ERR_INVALID_ARG;
  if ((words & 3) != 0) return DSA_ERR_INVALID_ARG;  // 128-key tiles read 4 words per row
  dsa::MaskedArgs a;
  memset(&a, 0, sizeof(a));
  // query tiles of 128 per request
  int st = fill_req(a.req, cu_seqlens_q_host, cu_seqlens_kv_host, num_req, T, cu_seqlens_kv_host ? -1 : T, 128);
  if (st != DSA_OK) return st;
  for (int r = 0; r < a.req.num_req; ++r)
    if (a.req.cu_kv[r + 1] - a.req.cu_kv[r] > 32 * words) return DSA_ERR_INVALID_ARG;
  DevInfo* d;
  if (!dev_info(&d)) return DSA_ERR_CUDA;
  a.k_chunks = d_k / 64;
  a.key_mask = key_mask;
  a.out = out;
  a.lse = lse;
  a.err = d->err;
  a.T = T;
  a.H = H;
  a.d_qk = d_qk;
  a.d_v = d_v;
  a.words = words;
  a.num_qtiles = a.req.cu_g[a.req.num_req];
  a.scale = scale;
  a.tr = g_trace;
  // (with no keys no key tile is loaded; the maps still need one row)
  const int64_t nk = a.req.cu_kv[a.req.num_req] > 0 ? a.req.cu_kv[a.req.num_req] : 1;
  const int v_box = d_v > 128 ? 64 : 128;   // keys per V stage of the kernel
  if (!dsa::make_head_tile_map_strided(&a.tmap_q, q, T, H, d_qk, q_stride_h, q_stride_t, 128) ||
      !dsa::make_head_tile_map_strided(&a.tmap_k, k, nk, H, d_k, k_stride_h, k_stride_t, 128) ||
      !dsa::make_head_tile_map_strided(&a.tmap_v, v, nk, H, d_v, v_stride_h, v_stride_t, v_box) ||
      (d_rope > 0 && !dsa::make_tile_map(&a.tmap_kpe, k_pe, nk, d_rope, k_pe_stride_t, 128)))
    return DSA_ERR_CUDA;
  const int r = dsa::launch_masked_mha(a, d->num_sms, (cudaStream_t)stream);
  return r == 0 ? DSA_OK : (r == -2 ? DSA_ERR_UNSUPPORTED : DSA_ERR_CUDA);
}

int dsa_masked_mha_prefill(const uint16_t* q, const uint16_t* k, const uint16_t* v, const uint32_t* key_mask,
                           int words, const int32_t* cu_seqlens_q_host, const int32_t* cu_seqlens_kv_host,
                           int num_req, int T, int H, int d_qk, int d_v, float scale, uint16_t* out, float* lse,
                           dsa_stream_t stream) {
  return dsa_masked_mha_prefill_strided(q, (int64_t)H * d_qk, d_qk, k, (int64_t)H * d_qk, d_qk, nullptr, 0, v,
                                        (int64_t)H * d_v, d_v, key_mask, words, cu_seqlens_q_host,
                                        cu_seqlens_kv_host, num_req, T, H, d_qk, 0, d_v, scale, out, lse, stream);
}

int dsa_debug_trace(void* device_buffer, int capacity) {
  if (capacity < 0) return DSA_ERR_INVALID_ARG;
  if (device_buffer == nullptr || capacity == 0) {
    g_trace.trace = nullptr;
    g_trace.trace_cap = 0;
    return DSA_OK;
  }
  if ((reinterpret_cast<uintptr_t>(device_buffer) & 7u) != 0) return DSA_ERR_INVALID_ARG;
  g_trace.trace = static_cast<unsigned long long*>(device_buffer);
  g_trace.trace_cap = capacity;
  return DSA_OK;
}

int64_t dsa_kv_fp8_row_bytes(int d_rope) { return (d_rope == 0 || d_rope == 64) ? 528 + 2 * d_rope : -1; }

static int kv_fp8_call(const uint16_t* kv, uint16_t* kv_out, uint8_t* fp8, const void* fp8_in, int N, int ld_kv,
                       int d_rope, bool quantize, dsa_stream_t stream) {
  if (N < 0 || ld_kv < 512 + d_rope || (ld_kv & 7) != 0) return DSA_ERR_INVALID_ARG;
  if (d_rope != 0 && d_rope != 64) return DSA_ERR_UNSUPPORTED;
  if (N == 0) return DSA_OK;
  const void* bf = quantize ? (const void*)kv : (const void*)kv_out;
  const void* f8 = quantize ? (const void*)fp8 : fp8_in;
  if (!bf || !f8 || !aligned16(bf) || !aligned16(f8)) return DSA_ERR_INVALID_ARG;
  DevInfo* d;
  if (!dev_info(&d)) return DSA_ERR_CUDA;
  dsa::Fp8KvArgs a;
  a.kv = kv;
  a.kv_out = kv_out;
  a.fp8 = quantize ? fp8 : const_cast<uint8_t*>(static_cast<const uint8_t*>(fp8_in));
  a.N = N;
  a.ld_kv = ld_kv;
  a.d_rope = d_rope;
  return dsa::launch_kv_fp8(a, quantize, d->num_sms, (cudaStream_t)stream) == 0 ? DSA_OK : DSA_ERR_CUDA;
}

int dsa_kv_fp8_quantize(const uint16_t* kv, int N, int ld_kv, int d_rope, uint8_t* kv_fp8, dsa_stream_t stream) {
  return kv_fp8_call(kv, nullptr, kv_fp8, nullptr, N, ld_kv, d_rope, true, stream);
}

int dsa_kv_fp8_dequantize(const uint8_t* kv_fp8, int N, int d_rope, uint16_t* kv, int ld_kv, dsa_stream_t stream) {
  return kv_fp8_call(nullptr, kv, nullptr, kv_fp8, N, ld_kv, d_rope, false, stream);
}

int dsa_sparse_prefill_fp8(const uint16_t* q, const uint8_t* kv_fp8, int N, int d_rope, const int32_t* idx, int T,
                           int H, int d_qk, int d_v, int k, int ld, float scale, uint16_t* out, float* lse,
                           dsa_stream_t stream) {
  if (T < 0 || N < 0 || k < 0 || ld < k) return DSA_ERR_INVALID_ARG;
  if (!(H == 16 || H == 32) || !(d_rope == 0 || d_rope == 64) || d_qk != 512 + d_rope || d_v != 512 || k > 2048)
    return DSA_ERR_UNSUPPORTED;
  if (T == 0) return DSA_OK;
  if (!q || (!kv_fp8 && N > 0) || !idx || !out || !lse) return DSA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(kv_fp8) || !aligned4(idx) || !aligned4(out) || !aligned4(lse))
    return DSA_ERR_INVALID_ARG;
  DevInfo* d;
  if (!dev_info(&d)) return DSA_ERR_CUDA;
  const int rb = (int)dsa_kv_fp8_row_bytes(d_rope);
  dsa::SparseArgs a;
  a.q = q;
  a.kv = nullptr;
  a.kv8 = kv_fp8;
  a.row_bytes = rb;
  a.ready = nullptr;
  a.done = nullptr;
  a.done_blk = 0;
  a.idx = idx;
  a.out = out;
  a.lse = lse;
  a.err = d->err;
  a.T = T;
  a.H = H;
  a.d_qk = d_qk;
  a.N = N;
  a.ld_kv = 0;
  a.k = k;
  a.ld = ld;
  a.scale = scale;
  a.tr = g_trace;
  // With N = 0 no tile is formed and the map is never used: it is encoded
  // over q (T*H rows of 2*d_qk >= rb bytes) so that it is well formed.
  if (!dsa::make_row_gather_map_u8(&a.tmap_kv, N > 0 ? (const void*)kv_fp8 : (const void*)q,
                                   N > 0 ? N : (int64_t)T * H, N > 0 ? rb : 2 * d_qk))
    return DSA_ERR_CUDA;
  if (!dsa::make_tile_map(&a.tmap_q, q, (int64_t)T * H, d_qk, d_qk, H)) return DSA_ERR_CUDA;
  const int r = dsa::launch_sparse_prefill_fp8(a, d->num_sms, (cudaStream_t)stream);
  return r == 0 ? DSA_OK : (r == -2 ? DSA_ERR_UNSUPPORTED : DSA_ERR_CUDA);
}

int dsa_debug_wait_timeout(dsa_stream_t stream) {
  DevInfo* d;
  if (!dev_info(&d)) return DSA_ERR_CUDA;
  return dsa::launch_wait_timeout(d->err, (cudaStream_t)stream) == 0 ? DSA_OK : DSA_ERR_CUDA;
}

int dsa_last_device_error(dsa_stream_t stream, uint32_t* counts) {
  if (!counts) return DSA_ERR_INVALID_ARG;
  DevInfo* d;
  if (!dev_info(&d)) return DSA_ERR_CUDA;
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return DSA_ERR_CUDA;
  unsigned int h[4] = {0, 0, 0, 0};
  if (cudaMemcpy(h, d->err, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) return DSA_ERR_CUDA;
  const unsigned int z[4] = {0, 0, 0, 0};
  if (cudaMemcpy(d->err, z, sizeof(z), cudaMemcpyHostToDevice) != cudaSuccess) return DSA_ERR_CUDA;
  for (int i = 0; i < 4; ++i) counts[i] = h[i];
  return (h[1] || h[2]) ? DSA_ERR_DEVICE : DSA_OK;
}

}  // extern "C"
