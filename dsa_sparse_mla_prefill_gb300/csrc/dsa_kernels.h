// Internal interface between the C-ABI shim (dsa_api.cu) and the kernels.
// Not installed; callers use include/dsa.h.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace dsa {

// Requests whose host-side sequence offsets travel inside the launch
// parameters (no device copy, no allocation).
constexpr int kMaxReq = 512;

struct ReqTable {
  int num_req;
  int32_t cu_q[kMaxReq + 1];    // query token offsets
  int32_t cu_kv[kMaxReq + 1];   // KV row offsets (masked mode / key mask)
  int32_t cu_g[kMaxReq + 1];    // group (or query tile) offsets
};

// Diagnostic timeline (dsa_debug_trace): when `trace` is set, CTAs 0 and 1
// record clock64() at up to 8 events of each of their first `trace_cap`
// tiles into trace[(cta * trace_cap + tile) * 8 + event].
struct TraceArgs {
  unsigned long long* trace;
  int trace_cap;
};

struct SparseArgs {
  CUtensorMap tmap_kv;  // kv rows, 64-column x 1-row box (row gathers)
  CUtensorMap tmap_q;   // q viewed [T*H, d_qk], 64-column x H-row box
  const uint16_t* q;    // [T, H, d_qk] bf16
  const uint16_t* kv;   // [N, ld_kv] bf16
  const uint8_t* kv8;   // FP8 rows [N, row_bytes] (the FP8 kernel; tmap_kv is then a byte map over them)
  int row_bytes;
  const int32_t* idx;   // [T, ld]
  uint16_t* out;        // [T, H, 512] bf16
  float* lse;           // [T, H]
  unsigned int* err;    // device error counters
  int T, H, d_qk, N, ld_kv, k, ld;
  float scale;
  TraceArgs tr;
  // Streamed from host memory (null otherwise): token t's q and index row may
  // be read once *ready > t (a copy stream raises it after each chunk lands);
  // once token t's out and lse are stored, done[t / done_blk] is incremented
  // (a copy stream waits on those counters before reading a chunk back).  A
  // CTA that gives up still counts its remaining tokens, so every counter
  // reaches its total.
  const uint32_t* ready;
  uint32_t* done;
  int done_blk;
};

struct UnionArgs {
  const int32_t* idx;   // [T, ld]
  int32_t* union_idx;   // [groups, union_pad]
  int32_t* union_len;   // [groups]
  uint8_t* mask;        // [groups, union_pad]
  unsigned int* err;
  int T, k, ld, G, N, union_pad, num_groups;
  ReqTable req;
};

struct Fp8KvArgs {
  const uint16_t* kv;   // quantize: bf16 rows [N, ld_kv]
  uint16_t* kv_out;     // dequantize: bf16 rows [N, ld_kv]
  uint8_t* fp8;         // FP8 rows [N, 528 + 2 d_rope] (quantize writes, dequantize reads)
  int N, ld_kv, d_rope;
};

struct KeyMaskArgs {
  const int32_t* idx;   // [T, ld] global rows
  uint32_t* key_mask;   // [T, words]
  unsigned int* err;
  int T, k, ld, words;
  ReqTable req;
};

struct ConvertArgs {
  const int32_t* idx_local;    // [T, ld] request-local positions
  int32_t* idx_global;         // [T, ld] physical rows (may alias idx_local)
  const int32_t* block_table;  // [num_req, max_blocks] physical block ids
  unsigned int* err;
  int T, k, ld, max_blocks, block_size, N;
  int vec;                     // 16-byte row accesses (ld % 4 == 0, aligned pointers)
  ReqTable req;                // cu_q: token offsets; cu_kv: cumulative KV lengths
};

struct GroupedArgs {
  CUtensorMap tmap_kv;      // kv rows for tile::gather4 (box 64 columns x 1 row, 128B swizzle)
  CUtensorMap tmap_q;       // q viewed [T*H, d_qk], box 64 columns x 64 rows
  CUtensorMap tmap_kv_blk;  // kv rows, box 64 columns x 64 rows (contiguous runs of the union)
  const uint16_t* q;
  const uint16_t* kv;
  const int32_t* union_idx;
  const int32_t* union_len;
  const uint8_t* mask;
  uint16_t* out;
  float* lse;
  unsigned int* err;
  int T, H, G, d_qk, N, ld_kv, union_pad, num_groups;
  float scale;
  ReqTable req;
  TraceArgs tr;
};

struct MaskedArgs {
  CUtensorMap tmap_q;   // q [T, H, d_qk] (strided): box 64 columns x 1 head x 128 rows
  CUtensorMap tmap_k;   // k [Nk, H, 64 * k_chunks] (strided): same box
  CUtensorMap tmap_v;   // v [Nk, H, d_v] (strided): box 64 columns x 1 head x (128 or 64) rows
  CUtensorMap tmap_kpe; // shared RoPE columns [Nk, d_qk - 64 * k_chunks]: box 64 columns x 128 rows
  int k_chunks;         // 64-column chunks of each key row read from tmap_k (the rest from tmap_kpe)
  const uint32_t* key_mask;  // [T, words]
  uint16_t* out;        // [T, H, d_v]
  float* lse;           // [T, H]
  unsigned int* err;
  int T, H, d_qk, d_v, words, num_qtiles;
  float scale;
  ReqTable req;         // cu_g = query-tile offsets per request
  TraceArgs tr;
};

// Shared memory of the union builder: bitmap and prefix (W words each, W
// rounded up to a multiple of 4 so the mask staging stays 16-byte aligned)
// plus one mask byte per union slot.
inline int union_build_smem_bytes(int N, int union_pad) {
  const int W = (N + 31) / 32;
  const int Wp = (W + 3) & ~3;
  return 8 * Wp + union_pad;
}

// The byte-map variant: one membership byte per KV position (32 Wp bytes),
// the union words and their prefix (Wp words each); used when it needs at
// most kUnionBytemapMaxSmem bytes (two or more CTAs per SM).
constexpr int kUnionBytemapMaxSmem = 96 * 1024;
inline int64_t union_build_bytemap_smem_bytes(int N) {
  const int64_t W = (N + 31) / 32;
  const int64_t Wp = (W + 3) & ~3;
  return 40 * Wp;
}

// Each returns 0 on success, -1 on a CUDA launch error, -2 if the shape has
// no kernel instance.
int launch_sparse_prefill(const SparseArgs& a, int num_sms, cudaStream_t stream);
int launch_sparse_prefill_fp8(const SparseArgs& a, int num_sms, cudaStream_t stream);
int launch_union_build(const UnionArgs& a, cudaStream_t stream);

int launch_topk_to_key_mask(const KeyMaskArgs& a, cudaStream_t stream);
int launch_local_to_global(const ConvertArgs& a, cudaStream_t stream);
int launch_grouped_prefill(const GroupedArgs& a, int num_sms, cudaStream_t stream);
int launch_masked_mha(const MaskedArgs& a, int num_sms, cudaStream_t stream);
int launch_wait_timeout(unsigned int* err, cudaStream_t stream);
int launch_kv_fp8(const Fp8KvArgs& a, bool quantize, int num_sms, cudaStream_t stream);

// dsa_sparse_prefill with the streamed-call fields of SparseArgs (ready, done,
// done_blk; all null / 0 for an ordinary call).  Same checks and DSA_* status
// as dsa_sparse_prefill.
int sparse_prefill_streamed(const uint16_t* q, const uint16_t* kv, int N, int ld_kv, const int32_t* idx, int T,
                            int H, int d_qk, int d_v, int k, int ld, float scale, uint16_t* out, float* lse,
                            const uint32_t* ready, uint32_t* done, int done_blk, cudaStream_t stream);

}  // namespace dsa
