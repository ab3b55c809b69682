/*
 * dsa.h - C ABI of the GB300 (sm_103a) DeepSeek-Sparse-Attention prefill
 * library (libdsa.so).
 *
 * The operation: DSA prefill over an MLA latent KV cache.  Every query token
 * t with H heads attends only to its own top-k selected latent rows:
 *
 *     out[t,h,:] = softmax_j( scale * q[t,h,0:D_QK] . kv[idx_j, 0:D_QK] ) . kv[idx_j, 0:D_V]
 *     lse[t,h]   = log sum_j exp( scale * q[t,h,:] . kv[idx_j, 0:D_QK] )      (natural log)
 *
 * with D_QK = 576 (512 NoPE + 64 RoPE) or 512 (NoPE layout) and D_V = 512,
 * V being the first 512 columns of the same latent row ("[Perf][DSA] Grouped
 * sparse prefill with the FlashMLA head-group-mask kernel", commit message
 * and Why; "[Perf][GLM-5.3-Flash] Dense/masked-MHA sparse prefill for the
 * NoPE (256, 0, 256) layout + skip the NoPE K concat", Purpose).  The
 * library offers the three forms the pages describe: per-token sparse,
 * grouped sparse (union list + head-group mask), and masked dense MHA.
 *
 * Conventions for every call
 *  - Tensor pointers are DEVICE pointers to caller-owned, contiguous memory
 *    laid out as stated; bf16 tensors are passed as uint16_t bit patterns.
 *    Arrays documented as HOST are read during the call (their values are
 *    copied into the launch) and may be freed when it returns.
 *  - No memory is allocated on any call (dsa_sparse_prefill_host creates
 *    three streams and a few events per device on its first use).  Every
 *    compute call is asynchronous on `stream` (NULL = the legacy default
 *    stream) and returns once the work is queued.
 *  - Return value: DSA_OK, or an error code; on an error nothing was
 *    launched.  DSA_ERR_INVALID_ARG: a null pointer, a negative or
 *    inconsistent size, a misaligned pointer or stride.  DSA_ERR_UNSUPPORTED:
 *    a shape the kernels do not implement.  DSA_ERR_CUDA: the launch failed.
 *  - Index entries equal to -1 mean "no selection" and may appear anywhere
 *    in the first k columns of a row; columns k..ld-1 are ignored.  Any
 *    other entry outside [0, N) is treated as absent and counted (see
 *    dsa_last_device_error).  A token without any valid entry gets out = 0
 *    and lse = -inf.  Duplicate valid entries in one row are not supported
 *    (results unspecified).
 *  - Causality is carried entirely by the indices (sparse forms) or by the
 *    key mask (masked form); no positional mask is applied.
 */
#ifndef DSA_H_
#define DSA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st* dsa_stream_t;

enum dsa_status {
  DSA_OK = 0,
  DSA_ERR_INVALID_ARG = 1,
  DSA_ERR_UNSUPPORTED = 2,
  DSA_ERR_CUDA = 3,
  DSA_ERR_DEVICE = 4
};

/* Largest number of requests one call accepts (host offset arrays). */
#define DSA_MAX_REQUESTS 512

/* Human-readable name of a status code (static string, never NULL). */
const char* dsa_status_string(int status);

/* Library version as major*10000 + minor*100 + patch. */
int dsa_version(void);

/* ------------------------------------------------------------------------
 * Host-side sizing helpers (no GPU work).
 * ---------------------------------------------------------------------- */

/* Per-group capacity of the union list: ceil(G*k / union_block) * union_block
 * ("[Perf][DSA] Grouped sparse prefill ...", review snippet of the union
 * builder's sizes).  Returns the value, or -1 for non-positive arguments. */
int64_t dsa_union_pad(int G, int k, int union_block);

/* Number of groups of G consecutive tokens of one request (a request's last
 * group may be short).  cu_seqlens_q_host: HOST int32 [num_req + 1],
 * ascending offsets starting at 0; NULL means one request of T tokens.
 * Writes *num_groups.  Returns DSA_OK or DSA_ERR_INVALID_ARG. */
int dsa_num_groups(const int32_t* cu_seqlens_q_host, int num_req, int T, int G, int* num_groups);

/* ------------------------------------------------------------------------
 * Union list + head-group membership mask ("[Perf][DSA] Grouped sparse
 * prefill with the FlashMLA head-group-mask kernel", How: bitmap over KV
 * positions -> prefix-sum compaction -> sorted union, plus per-token
 * membership bits).
 *
 * idx          [T, ld] int32 global KV rows (first k columns used).
 * G            tokens per group, 1..8 (one mask bit per token).
 * cu_seqlens_q HOST int32 [num_req + 1] or NULL (one request of T tokens);
 *              groups never straddle requests.
 * N            KV rows: valid indices lie in [0, N).  The bitmap and the
 *              mask staging live in shared memory, so 8*ceil(N/32) +
 *              union_pad must not exceed 232448 bytes (N up to ~440k rows
 *              at union_pad = 16384); larger shapes are DSA_ERR_UNSUPPORTED.
 * union_idx    out [num_groups, union_pad] int32: slots 0..len-1 hold the
 *              group's distinct valid rows in ascending order; the rest -1.
 * union_len    out [num_groups] int32.
 * mask         out [num_groups, union_pad] uint8: bit j of slot u is set iff
 *              union_idx[g,u] is among token j's valid rows (token j = j-th
 *              token of the group); 0 in the padding.
 * union_pad    >= min(G*k, N) and a multiple of 16 (dsa_union_pad with a
 *              block of 16 or more qualifies).  A union longer than
 *              union_pad is truncated and counted as a device error.
 * ---------------------------------------------------------------------- */
int dsa_union_build(const int32_t* idx, int T, int k, int ld, int G, const int32_t* cu_seqlens_q_host,
                    int num_req, int N, int32_t* union_idx, int32_t* union_len, uint8_t* mask, int union_pad,
                    dsa_stream_t stream);

/* ------------------------------------------------------------------------
 * Per-token sparse MLA prefill ("[Perf][DSA] Grouped sparse prefill ...",
 * commit message: each token gathers its own 2048 selected rows).
 *
 * q     [T, H, d_qk] bf16.        kv  [N, ld_kv] bf16, row n = latent row n
 *       (kv may be null when N = 0: every index is then out of range).
 * idx   [T, ld] int32 global rows, first k columns used; k <= 2048.
 * out   [T, H, d_v] bf16 (out).   lse [T, H] fp32 (out, natural log).
 * H in {16, 32}; d_qk in {576, 512}; d_v = 512; ld_kv >= d_qk and a
 * multiple of 8; q, kv 16-byte aligned.
 * ---------------------------------------------------------------------- */
int dsa_sparse_prefill(const uint16_t* q, const uint16_t* kv, int N, int ld_kv, const int32_t* idx, int T,
                       int H, int d_qk, int d_v, int k, int ld, float scale, uint16_t* out, float* lse,
                       dsa_stream_t stream);

/* ------------------------------------------------------------------------
 * Grouped sparse prefill ("[Perf][DSA] Grouped sparse prefill ...", commit
 * message and How): the G = 128 / H consecutive tokens of a group act as 128
 * pseudo-heads p = j*H + h over the group's union list; the mask restricts
 * pseudo-head p to the slots whose bit j is set, so the result equals the
 * per-token form.  Pseudo-heads past a short group's tokens are dropped.
 *
 * q, kv, out, lse, d_qk, d_v, ld_kv as for dsa_sparse_prefill.
 * union_idx, union_len, mask, union_pad, G, cu_seqlens_q, num_req exactly as
 * produced by / passed to dsa_union_build.  H * G must equal 128 and
 * G <= 8 (the gate on the same page, review snippet).  scale must be
 * positive and finite (the kernel takes the row max on unscaled scores);
 * otherwise DSA_ERR_INVALID_ARG.
 * ---------------------------------------------------------------------- */
int dsa_grouped_prefill(const uint16_t* q, const uint16_t* kv, int N, int ld_kv, const int32_t* union_idx,
                        const int32_t* union_len, const uint8_t* mask, int union_pad, int G,
                        const int32_t* cu_seqlens_q_host, int num_req, int T, int H, int d_qk, int d_v,
                        float scale, uint16_t* out, float* lse, dsa_stream_t stream);

/* ------------------------------------------------------------------------
 * Top-k -> packed key mask ("[2/N][Attention] Enable masked MHA for sparse
 * MLA prefills", commit log: scatter of the top-k into a per-token mask that
 * the kernel zeroes itself).
 *
 * idx           [T, ld] int32 global KV rows (first k columns used).
 * cu_seqlens_q  HOST int32 [num_req + 1]; cu_seqlens_kv HOST int32
 *               [num_req + 1] (KV row offsets).  NULL/NULL = one request.
 * key_mask      out [T, words] uint32: bit (n & 31) of word (n >> 5) of row
 *               t is set iff row cu_seqlens_kv[r] + n is among token t's
 *               valid top-k (r = the token's request).  Every word is written.
 * words         >= ceil(longest request's KV length / 32).
 * Indices outside the token's own request are treated as absent and counted.
 * ---------------------------------------------------------------------- */
int dsa_topk_to_key_mask(const int32_t* idx, int T, int k, int ld, const int32_t* cu_seqlens_q_host,
                         const int32_t* cu_seqlens_kv_host, int num_req, uint32_t* key_mask, int words,
                         dsa_stream_t stream);

/* ------------------------------------------------------------------------
 * Request-local -> physical KV rows ("[Perf][DSA] Grouped sparse prefill
 * ...", How: the selected positions are mapped to physical rows of the paged
 * KV cache through the request -> global index conversion).  Run it on the
 * per-token index rows before dsa_sparse_prefill / dsa_union_build, so that
 * the union is sorted by physical row as dsa_grouped_prefill requires.
 *
 * idx_local    [T, ld] int32: position x in the KV sequence of the token's
 *              request (0 <= x < kv_len), -1 = absent; first k columns used.
 * cu_seqlens_q HOST int32 [num_req + 1] or NULL (one request of T tokens).
 * kv_lens      HOST int32 [num_req]: KV length of each request.
 * block_table  DEVICE int32 [num_req, max_blocks]: physical block of each
 *              logical block of block_size positions; negative = unmapped.
 * N            physical KV rows (rows outside [0, N) are not produced).
 * idx_global   out [T, ld] int32: block_table[r][x / block_size] * block_size
 *              + x % block_size for every valid x; -1 for -1 entries, for
 *              columns >= k and for every other entry (positions outside
 *              [0, kv_len), unmapped blocks, rows outside [0, N)), which are
 *              also counted in counts[0] of dsa_last_device_error.
 *              idx_global may equal idx_local (in place).
 * Requires block_size >= 1, max_blocks >= 1, kv_len <= max_blocks *
 * block_size for every request; idx pointers 4-byte aligned.
 * ---------------------------------------------------------------------- */
int dsa_local_to_global(const int32_t* idx_local, int T, int k, int ld, const int32_t* cu_seqlens_q_host,
                        const int32_t* kv_lens_host, int num_req, const int32_t* block_table, int max_blocks,
                        int block_size, int N, int32_t* idx_global, dsa_stream_t stream);

/* ------------------------------------------------------------------------
 * Masked dense MHA simulating DSA ("[2/N][Attention] Enable masked MHA for
 * sparse MLA prefills", Purpose; "[Perf][GLM-5.3-Flash] ...", Purpose): per
 * head, token t of request r attends to the keys n of its request whose mask
 * bit is set, with per-head (decompressed) q/k/v.
 *
 * q   [T, H, d_qk] bf16; k [Nk, H, d_qk] bf16; v [Nk, H, d_v] bf16, where
 *     Nk = cu_seqlens_kv[num_req].
 * key_mask [T, words] uint32 as written by dsa_topk_to_key_mask.
 * out [T, H, d_v] bf16 (out); lse [T, H] fp32 (out, natural log).
 * (d_qk, d_v) = (192, 128) (DeepSeek-V3.2) or (256, 256) (GLM-5 and the
 * GLM-5.3-Flash NoPE layout), the geometries of the masked-MHA allow-list
 * ("[Perf][GLM-5.3-Flash] ...", review snippets); others return
 * DSA_ERR_UNSUPPORTED.  Any H >= 1.
 * scale must be positive and finite (the kernel takes the row max on
 * unscaled scores); otherwise DSA_ERR_INVALID_ARG.
 * Chunked context: a request's queries may be the last q_len of its kv_len
 * keys (cu_seqlens_q and cu_seqlens_kv differ); the mask rows of the chunk's
 * tokens are rows of the whole prompt's mask.
 * ---------------------------------------------------------------------- */
int dsa_masked_mha_prefill(const uint16_t* q, const uint16_t* k, const uint16_t* v, const uint32_t* key_mask,
                           int words, const int32_t* cu_seqlens_q_host, const int32_t* cu_seqlens_kv_host,
                           int num_req, int T, int H, int d_qk, int d_v, float scale, uint16_t* out, float* lse,
                           dsa_stream_t stream);

/* ------------------------------------------------------------------------
 * The same with strided per-head operands and the key's RoPE columns in a
 * buffer of their own ("[Perf][GLM-5.3-Flash] ...", commit messages: with no
 * RoPE part the concatenated K is k_nope itself, so no copy; here neither
 * layout forms the concatenated K).  Key row n of head h is
 *     [ k[n * k_stride_t + h * k_stride_h + 0 .. d_qk - d_rope - 1],
 *       k_pe[n * k_pe_stride_t + 0 .. d_rope - 1] ]
 * and q[t, h, :] = q[t * q_stride_t + h * q_stride_h + ...], v likewise, so
 * k and v may be views into the per-head kv projection output (e.g. k =
 * kv[..., :256], v = kv[..., 256:] of a [Nk, H, 512] tensor).
 *
 * Strides are in elements, multiples of 8 (16 bytes), with stride_h >= the
 * columns read and stride_t >= H * stride_h; k_pe_stride_t >= d_rope and a
 * multiple of 8.  d_rope = 0 (k_pe unused, may be NULL) or 64 (k_pe [Nk, 64]
 * shared by all heads, required).  d_qk - d_rope must be a multiple of 64.
 * out is contiguous [T, H, d_v].  Everything else as dsa_masked_mha_prefill.
 * ---------------------------------------------------------------------- */
int dsa_masked_mha_prefill_strided(const uint16_t* q, int64_t q_stride_t, int64_t q_stride_h, const uint16_t* k,
                                   int64_t k_stride_t, int64_t k_stride_h, const uint16_t* k_pe,
                                   int64_t k_pe_stride_t, const uint16_t* v, int64_t v_stride_t, int64_t v_stride_h,
                                   const uint32_t* key_mask, int words, const int32_t* cu_seqlens_q_host,
                                   const int32_t* cu_seqlens_kv_host, int num_req, int T, int H, int d_qk,
                                   int d_rope, int d_v, float scale, uint16_t* out, float* lse, dsa_stream_t stream);

/* ------------------------------------------------------------------------
 * Device error counters of the current device.  Synchronizes `stream`, then
 * copies and clears the counters: counts[0] = ignored out-of-range index
 * entries, counts[1] = bounded waits that ran out (a kernel stopped early;
 * its outputs are incomplete), counts[2] = truncated union lists, counts[3]
 * reserved.  `counts` is a HOST array of 4.  Returns DSA_ERR_DEVICE if
 * counts[1] or counts[2] is nonzero, DSA_ERR_CUDA if the stream reported an
 * error, else DSA_OK.
 * ---------------------------------------------------------------------- */
int dsa_last_device_error(dsa_stream_t stream, uint32_t* counts);

/* ------------------------------------------------------------------------
 * dsa_sparse_prefill from and to HOST memory, with the copies overlapped
 * with the attention (the end-to-end call: inputs that live on the host,
 * results wanted there).  Three internal streams of the library carry the
 * host -> device copies of q and the indices, the per-token kernel, and the
 * device -> host copies of out and lse.  Two forms, chosen by the workspace:
 *
 * streamed (a workspace of dsa_sparse_prefill_host_workspace(..., chunk_tokens
 *   >= T, ...) bytes, which holds every token): ONE kernel launch over all
 *   tokens.  The inputs are copied in chunks (of at most chunk_tokens and at
 *   most 2 tokens per SM); after each chunk a stream write raises a counter,
 *   and the kernel takes up a token only once the counter is past it.  The
 *   kernel counts finished tokens per block of one token per CTA, and each
 *   chunk's outputs are copied back once the blocks it covers are counted
 *   (stream waits on those counters).  Needs the driver's stream memory
 *   operations (DSA_ERR_UNSUPPORTED without them).  A kernel that gives up
 *   (a bounded wait ran out, counted in dsa_last_device_error) still
 *   completes every counter, so no copy waits forever; its outputs are then
 *   incomplete.
 * ring (a smaller workspace, of dsa_sparse_prefill_host_workspace(...,
 *   chunk_tokens < T, ...) bytes): the tokens go through in chunks of
 *   chunk_tokens, one kernel launch per chunk, so that chunk i+1 arrives and
 *   chunk i-1 leaves while chunk i is computed (3 chunks in flight).
 *
 * q, idx, out, lse: HOST pointers, laid out as for dsa_sparse_prefill;
 *   page-locked (pinned) memory is needed for the copies to overlap.
 * kv: HOST (kv_on_host = 1, copied once per call) or DEVICE (0) [N, ld_kv].
 * workspace: DEVICE scratch, 256-byte aligned, of at least
 *   dsa_sparse_prefill_host_workspace(...) bytes (same arguments); the
 *   library allocates nothing.  Calls that share a workspace must be
 *   ordered on one stream.
 * stream: the copies start after the work queued on it before the call, and
 *   work queued on it after the call waits for the last outputs to be back
 *   in host memory and the kernel to end (synchronize the stream before
 *   reading out and lse).
 * Shapes and errors as dsa_sparse_prefill; DSA_ERR_INVALID_ARG also for
 * chunk_tokens < 1 or a workspace that is too small or misaligned.  A CUDA
 * error part way returns DSA_ERR_CUDA with the work queued so far left to
 * finish (the caller's stream waits for it).  The results are bit for bit
 * those of dsa_sparse_prefill on device copies of the same inputs, in either
 * form.  The library's streams and events are per device and shared by all
 * calls: calls on one device must not run from several host threads at once.
 * ---------------------------------------------------------------------- */
int64_t dsa_sparse_prefill_host_workspace(int T, int N, int ld_kv, int H, int d_qk, int d_v, int ld,
                                          int chunk_tokens, int kv_on_host);

/* The chunk sizes dsa_sparse_prefill_host uses for T tokens on a GPU with
 * num_sms SMs (host only): middle chunks of the largest multiple of num_sms
 * not above min(chunk_tokens, T) (the persistent kernel deals tokens to one
 * CTA per SM, so no CTA is left a token behind), and first and last chunks
 * that ramp num_sms, 2 num_sms, 4 num_sms ... while the ramps still leave
 * room for a full chunk.  Writes up to max_chunks sizes (HOST int32) and
 * *num_chunks; DSA_ERR_INVALID_ARG if they do not fit or for bad sizes. */
int dsa_sparse_prefill_host_plan(int T, int chunk_tokens, int num_sms, int32_t* sizes, int max_chunks,
                                 int* num_chunks);

int dsa_sparse_prefill_host(const uint16_t* q, const uint16_t* kv, int kv_on_host, int N, int ld_kv,
                            const int32_t* idx, int T, int H, int d_qk, int d_v, int k, int ld, float scale,
                            uint16_t* out, float* lse, void* workspace, int64_t workspace_bytes, int chunk_tokens,
                            dsa_stream_t stream);

/* ------------------------------------------------------------------------
 * dsa_sparse_prefill_host for callers that cannot give the library device
 * memory (no counterpart on the pages; it exists for the deployment, not
 * for the method).  Some host programs cannot call cudaMalloc for a
 * workspace: their allocator has reserved the whole GPU up front, so a
 * private allocation would fail, or their runtime forbids device
 * allocation once it is serving.  This call takes no workspace: its buffer
 * sets live in a fixed scratch array of DSA_HOST_NOALLOC_SCRATCH_BYTES
 * (64 MiB) that belongs to the library's device image, held on every GPU
 * where the library's device code is loaded until the process exits.  The
 * call allocates and frees nothing.
 *
 * Arguments, results and errors as dsa_sparse_prefill_host (out and lse are
 * bit for bit the same), with one more error: DSA_ERR_UNSUPPORTED when
 * dsa_sparse_prefill_host_workspace(...) for these arguments exceeds
 * DSA_HOST_NOALLOC_SCRATCH_BYTES; a smaller chunk_tokens, or kv already in
 * device memory, needs less (the 16384-token, H = 32, top-2048 chunk fits
 * with chunk_tokens = 152 and kv on the host).
 *
 * - Set-up: the first call on a device looks up the scratch array's device
 *   address with that device current (and creates the library's copy
 *   streams, as dsa_sparse_prefill_host does); make that first call before
 *   any stream capture.
 * - Every call on a device shares the one array, which keeps whatever the
 *   last call left there; nothing in it needs to start at zero, since each
 *   call writes every byte it reads.  Calls whose work overlaps on the GPU
 *   (different streams, or several host threads) race on the array: order
 *   them on one stream.
 * ---------------------------------------------------------------------- */
#define DSA_HOST_NOALLOC_SCRATCH_BYTES (64ull << 20)

int dsa_sparse_prefill_host_noalloc(const uint16_t* q, const uint16_t* kv, int kv_on_host, int N, int ld_kv,
                                    const int32_t* idx, int T, int H, int d_qk, int d_v, int k, int ld, float scale,
                                    uint16_t* out, float* lse, int chunk_tokens, dsa_stream_t stream);

/* ------------------------------------------------------------------------
 * FP8 latent rows for the KV cache.  The pages keep the cache in bf16 (the
 * grouped gate in "[Perf][DSA] Grouped sparse prefill ...", review
 * snippets, refuses a quantized cache); an FP8 row here holds the 512 NoPE
 * columns as float8 e4m3 with one fp32 scale per 128 of them, then the RoPE
 * columns in bf16:
 *     bytes [0, 512) codes | [512, 528) 4 scales | [528, 528 + 2 d_rope) RoPE
 * (656 bytes per row at d_rope = 64, 528 for the NoPE layout; rows packed).
 * Quantize: scale = block amax / 448 (1 for an all-zero block), code =
 * e4m3(x / scale) with the division in IEEE float32 and round-to-nearest-even
 * conversion saturating at 448.  Dequantize: e4m3 value times the block's
 * scale in float32, rounded to bf16; the attention forms then run on the
 * bf16 rows.
 * kv: DEVICE bf16 [N, ld_kv], ld_kv >= 512 + d_rope and a multiple of 8;
 * kv_fp8: DEVICE [N, dsa_kv_fp8_row_bytes(d_rope)]; both 16-byte aligned.
 * d_rope in {0, 64}, else DSA_ERR_UNSUPPORTED.
 * ---------------------------------------------------------------------- */
int64_t dsa_kv_fp8_row_bytes(int d_rope);
int dsa_kv_fp8_quantize(const uint16_t* kv, int N, int ld_kv, int d_rope, uint8_t* kv_fp8, dsa_stream_t stream);
int dsa_kv_fp8_dequantize(const uint8_t* kv_fp8, int N, int d_rope, uint16_t* kv, int ld_kv, dsa_stream_t stream);

/* Per-token sparse MLA prefill reading FP8 latent rows directly (the pages'
 * per-token form, as dsa_sparse_prefill, over the row layout above).  Each
 * selected row is gathered as codes + scales + RoPE (656 bytes at d_rope =
 * 64 against 1152 in bf16) and dequantized on chip with exactly the
 * dsa_kv_fp8_dequantize arithmetic, so out and lse are bit-for-bit those of
 * dsa_kv_fp8_dequantize followed by dsa_sparse_prefill, without the bf16
 * table.
 * q      DEVICE [T, H, d_qk] bf16, 16-byte aligned; d_qk = 512 + d_rope.
 * kv_fp8 DEVICE [N, dsa_kv_fp8_row_bytes(d_rope)], 16-byte aligned (may be
 *        null when N = 0).
 * idx, k, ld, out, lse, scale: as dsa_sparse_prefill.  H in {16, 32};
 * d_rope in {0, 64}; d_v = 512; k <= 2048, else DSA_ERR_UNSUPPORTED. */
int dsa_sparse_prefill_fp8(const uint16_t* q, const uint8_t* kv_fp8, int N, int d_rope, const int32_t* idx, int T,
                           int H, int d_qk, int d_v, int k, int ld, float scale, uint16_t* out, float* lse,
                           dsa_stream_t stream);

/* ------------------------------------------------------------------------
 * Form choice (host only, no GPU call).  "[Perf][GLM-5.3-Flash] ...", commit
 * messages: prompts within the top-k budget run dense MHA, longer ones masked
 * MHA up to a length threshold (36k tokens at TP4, 64k at TP8) and the
 * per-token kernel beyond; "[Perf][DSA] Grouped sparse prefill ...", How:
 * the grouped form may take everything longer than the top-k budget.  Here
 * the three exact forms are compared by predicted time, each form's work (its
 * dominant kernel's roofline quantity) over the fraction of the measured peak
 * that form reaches, plus fixed costs:
 *   per-token  sum_t n_t * 2 d_qk bytes gathered (n_t = min(k, position + 1))
 *              + q, out, indices, lse bytes, at per_token_frac of HBM;
 *   grouped    2 * 128 * U * (d_qk + 512) FLOPs (U = sum of union rows) at
 *              grouped_frac of bf16, + the union build (T * k * 4 bytes at
 *              union_frac of HBM); only where 128 % H == 0 and 128 / H <= 8;
 *   masked     2 * H * sum_r (q_r (q_r + 1) / 2 + q_r * ctx_r) * (d_qk + d_v)
 *              FLOPs at masked_frac of bf16, + the key mask; only for the
 *              masked geometries (192, 128) and (256, 256), i.e. where the
 *              caller has per-head k and v.
 * U comes from the caller (sum of union_len after dsa_union_build) or is
 * estimated per group as min(last position + 1, n_last (1 + union_growth)).
 * ---------------------------------------------------------------------- */
enum dsa_form { DSA_FORM_PER_TOKEN = 0, DSA_FORM_GROUPED = 1, DSA_FORM_MASKED = 2 };

typedef struct dsa_form_calibration {
  double hbm_gbs, bf16_tflops;               /* measured peaks */
  double per_token_frac, per_token_ms0;      /* of HBM; fixed ms */
  double union_frac, union_ms0;              /* union build: of HBM on index bytes; fixed ms */
  double grouped_frac_576, grouped_frac_512; /* of bf16, by latent key width */
  double grouped_ms0;
  double masked_frac_192, masked_frac_256;   /* of bf16, by per-head d_qk */
  double masked_ms0;
  double key_mask_frac, key_mask_ms0;        /* key mask: of HBM on index + mask bytes */
  double union_growth;                       /* union of a group / one token's rows - 1 */
} dsa_form_calibration;

typedef struct dsa_form_query {
  int num_req;
  const int32_t* q_lens;     /* HOST [num_req] query tokens (the last q_len positions) */
  const int32_t* kv_lens;    /* HOST [num_req] KV positions, >= q_len */
  int H;                     /* query heads on this GPU */
  int k;                     /* top-k per token */
  int d_qk;                  /* latent key width of the sparse forms: 576 or 512 */
  int masked_d_qk;           /* per-head geometry when the masked form can run, else 0 */
  int masked_d_v;
  double union_rows;         /* sum of union rows if known, else < 0 (estimated) */
} dsa_form_query;

typedef struct dsa_form_estimate {
  double ms[3];              /* predicted ms by dsa_form; < 0 = not applicable */
  int form;                  /* the fastest applicable form */
  double union_rows;         /* union rows used for the grouped estimate */
} dsa_form_estimate;

/* The calibration measured on GB300 (defaults of dsa_choose_form). */
int dsa_form_calibration_default(dsa_form_calibration* calib);

/* Fills *out; calib NULL = the GB300 default.  DSA_ERR_INVALID_ARG on null
 * pointers, num_req < 1, H < 1, k < 1, kv_len < q_len or a non-positive
 * fraction; DSA_ERR_UNSUPPORTED for d_qk other than 512 / 576. */
int dsa_choose_form(const dsa_form_query* query, const dsa_form_calibration* calib, dsa_form_estimate* out);

/* ------------------------------------------------------------------------
 * Failure-path check (no counterpart on the pages).  Launches one CTA whose
 * bounded wait on an mbarrier that nothing completes runs out after the
 * library's wait limit (2 s): the kernel records the timeout, releases the
 * tensor memory it holds and returns, as every pipeline kernel does when a
 * wait runs out.  Afterwards dsa_last_device_error reports counts[1] >= 1
 * and DSA_ERR_DEVICE, and the context stays usable.  Asynchronous on stream.
 * ---------------------------------------------------------------------- */
int dsa_debug_wait_timeout(dsa_stream_t stream);

/* ------------------------------------------------------------------------
 * Diagnostic timeline (no counterpart on the pages; a profiling aid).  While
 * a buffer is set, the first two CTAs of every per-token, grouped and masked
 * launch write clock64() stamps of up to 8 pipeline events for each of their
 * first `capacity` tiles into it: u64 slot [(cta * capacity + tile) * 8 +
 * event]; untouched slots keep their contents.  `device_buffer` is caller-owned
 * device memory of at least 2 * capacity * 8 * 8 bytes; NULL (or capacity 0)
 * switches recording off.  Host-only call; returns DSA_OK or
 * DSA_ERR_INVALID_ARG.
 * ---------------------------------------------------------------------- */
int dsa_debug_trace(void* device_buffer, int capacity);

#ifdef __cplusplus
}
#endif

#endif /* DSA_H_ */
