// Per-token sparse prefill from and to host memory, with the copies
// overlapped with the attention (host code only).
//
// The tokens go through in chunks; three internal streams per device carry
// the host -> device copies of a chunk's q and indices, the per-token kernel
// of the chunk, and the device -> host copies of its out and lse, so that
// chunk i+1 arrives and chunk i-1 leaves while chunk i is computed.  A ring
// of NB device buffer sets in the caller's workspace holds the chunks in
// flight; events order each buffer's reuse (the copy into set b waits for the
// kernel that last read it, the kernel for the copy that last drained it).
// The caller's stream is joined at both ends: the copies start after the work
// queued on it so far, and work queued on it after the call starts once the
// last chunk is back in host memory.
//
// Chunk sizes: the per-token kernel runs one persistent CTA per SM with the
// tokens dealt round-robin, so a chunk that is a multiple of the SM count
// leaves no CTA a token behind the others; the middle chunks are the largest
// such multiple the workspace allows, and the first and last chunks ramp
// (one, two, four ... tokens per SM) so that the copy before the first
// kernel and the copy after the last are short.
//
// Streamed form (a workspace that holds every token's buffers): one kernel
// launch covers all tokens and the copies flow around it.  After each chunk's
// inputs land, the host-to-device stream raises a `ready` word to the chunk's
// end (a stream write, ordered after the copies); the kernel reads a token's
// inputs only once `ready` is past it.  The kernel counts finished tokens in
// blocks of one token per CTA, and the device-to-host stream waits (stream
// waits on those counters) before it reads a chunk back.  This removes the
// per-chunk launch (each launch fills and drains every CTA's pipeline once).
// Every upload is queued before the kernel and no read-back wait is queued
// unless the kernel launched; a CTA that gives up still completes its
// counters, so no stream waits for a value that never comes.
#include <cstdint>
#include <cstring>
#include <initializer_list>
#include <vector>

#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/dsa.h"
#include "dsa_kernels.h"

namespace {

constexpr int NB = 3;          // buffer sets in flight
constexpr int kMaxDev = 64;
constexpr int64_t kAlign = 256;

struct Pipe {
  bool init = false;
  int num_sms = 0;
  cudaStream_t h2d = nullptr, cmp = nullptr, d2h = nullptr;
  cudaEvent_t entry = nullptr, kv_in = nullptr, exit = nullptr;
  cudaEvent_t in[NB] = {}, done[NB] = {}, out[NB] = {};
};
Pipe g_pipe[kMaxDev];

// Releases whatever a failed set-up created, so that a later call starts clean.
void pipe_release(Pipe& s) {
  for (cudaStream_t* st : {&s.h2d, &s.cmp, &s.d2h})
    if (*st) {
      cudaStreamDestroy(*st);
      *st = nullptr;
    }
  for (cudaEvent_t* ev : {&s.entry, &s.kv_in, &s.exit})
    if (*ev) {
      cudaEventDestroy(*ev);
      *ev = nullptr;
    }
  for (int b = 0; b < NB; ++b)
    for (cudaEvent_t* ev : {&s.in[b], &s.done[b], &s.out[b]})
      if (*ev) {
        cudaEventDestroy(*ev);
        *ev = nullptr;
      }
}

bool pipe_of(Pipe** p) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return false;
  Pipe& s = g_pipe[dev];
  if (!s.init) {
    const unsigned ef = cudaEventDisableTiming;
    bool ok = cudaStreamCreateWithFlags(&s.h2d, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&s.cmp, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&s.d2h, cudaStreamNonBlocking) == cudaSuccess &&
              cudaEventCreateWithFlags(&s.entry, ef) == cudaSuccess &&
              cudaEventCreateWithFlags(&s.kv_in, ef) == cudaSuccess &&
              cudaEventCreateWithFlags(&s.exit, ef) == cudaSuccess &&
              cudaDeviceGetAttribute(&s.num_sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess &&
              s.num_sms >= 1;
    for (int b = 0; b < NB && ok; ++b)
      ok = cudaEventCreateWithFlags(&s.in[b], ef) == cudaSuccess &&
           cudaEventCreateWithFlags(&s.done[b], ef) == cudaSuccess &&
           cudaEventCreateWithFlags(&s.out[b], ef) == cudaSuccess;
    if (!ok) {
      pipe_release(s);
      cudaGetLastError();
      return false;
    }
    s.init = true;
  }
  *p = &s;
  return true;
}

int64_t up(int64_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

// Stream memory operations of the driver API, found through the runtime.
typedef CUresult (*PfnStreamValue32)(CUstream, CUdeviceptr, cuuint32_t, unsigned int);
struct MemOps {
  bool tried = false;
  PfnStreamValue32 write = nullptr, wait = nullptr;
};
MemOps g_memops;

const MemOps* mem_ops() {
  if (!g_memops.tried) {
    g_memops.tried = true;
    void* pw = nullptr;
    void* pa = nullptr;
    cudaDriverEntryPointQueryResult qw, qa;
    if (cudaGetDriverEntryPointByVersion("cuStreamWriteValue32", &pw, 12000, cudaEnableDefault, &qw) ==
            cudaSuccess &&
        qw == cudaDriverEntryPointSuccess &&
        cudaGetDriverEntryPointByVersion("cuStreamWaitValue32", &pa, 12000, cudaEnableDefault, &qa) ==
            cudaSuccess &&
        qa == cudaDriverEntryPointSuccess && pw && pa) {
      g_memops.write = reinterpret_cast<PfnStreamValue32>(pw);
      g_memops.wait = reinterpret_cast<PfnStreamValue32>(pa);
    } else {
      cudaGetLastError();
    }
  }
  return g_memops.write ? &g_memops : nullptr;
}

// Chunk sizes for T tokens, none above `cap`, as described at the top.
std::vector<int> plan_chunks(int T, int cap, int unit) {
  std::vector<int> out;
  const int full = cap >= unit ? cap / unit * unit : cap;
  std::vector<int> ramp;   // unit, 2 unit, 4 unit, ... below the full size
  int64_t ramp_sum = 0;
  for (int64_t r = unit; r < full && 2 * (ramp_sum + r) + full <= T; r *= 2) {
    ramp.push_back((int)r);
    ramp_sum += r;
  }
  for (int r : ramp) out.push_back(r);
  int64_t mid = T - 2 * ramp_sum;
  while (mid > 0) {
    const int n = (int)(mid < full ? mid : full);
    out.push_back(n);
    mid -= n;
  }
  for (int i = (int)ramp.size() - 1; i >= 0; --i) out.push_back(ramp[i]);
  return out;
}

// Byte sizes of one buffer set and of the whole workspace.
struct Layout {
  int64_t q, idx, out, lse, set, kv, total;
};

Layout layout(int chunk, int N, int ld_kv, int H, int d_qk, int d_v, int ld, bool kv_host) {
  Layout l;
  l.q = up((int64_t)chunk * H * d_qk * 2);
  l.idx = up((int64_t)chunk * ld * 4);
  l.out = up((int64_t)chunk * H * d_v * 2);
  l.lse = up((int64_t)chunk * H * 4);
  l.set = l.q + l.idx + l.out + l.lse;
  l.kv = kv_host ? up((int64_t)N * ld_kv * 2) : 0;
  l.total = l.kv + NB * l.set;
  return l;
}

// Streamed form: the table, one buffer set for all T tokens, then the
// `ready` word and the done counters (one word per token at most).
int64_t streamed_bytes(int T, int N, int ld_kv, int H, int d_qk, int d_v, int ld, bool kv_host) {
  const Layout l = layout(T, N, ld_kv, H, d_qk, d_v, ld, kv_host);
  return l.kv + l.set + up(4 * ((int64_t)T + 1));
}

// Chunks of the streamed form: at most this many tokens per SM.  Small
// chunks keep the uploads just ahead of the kernel (a CTA's next token is at
// most two chunks away) and the last read-back short; their cost is a few
// queued operations each.
constexpr int kStreamTokensPerSm = 2;

}  // namespace

extern "C" {

int dsa_sparse_prefill_host_plan(int T, int chunk_tokens, int num_sms, int32_t* sizes, int max_chunks,
                                 int* num_chunks) {
  if (T < 0 || chunk_tokens < 1 || num_sms < 1 || max_chunks < 0 || !num_chunks || (max_chunks > 0 && !sizes))
    return DSA_ERR_INVALID_ARG;
  if (T == 0) {
    *num_chunks = 0;
    return DSA_OK;
  }
  const std::vector<int> plan = plan_chunks(T, chunk_tokens < T ? chunk_tokens : T, num_sms);
  *num_chunks = (int)plan.size();
  for (int i = 0; i < (int)plan.size() && i < max_chunks; ++i) sizes[i] = plan[i];
  return (int)plan.size() <= max_chunks ? DSA_OK : DSA_ERR_INVALID_ARG;
}

int64_t dsa_sparse_prefill_host_workspace(int T, int N, int ld_kv, int H, int d_qk, int d_v, int ld,
                                          int chunk_tokens, int kv_on_host) {
  if (T < 0 || N < 0 || ld_kv < 1 || H < 1 || d_qk < 1 || d_v < 1 || ld < 1 || chunk_tokens < 1) return -1;
  if (chunk_tokens >= T) return streamed_bytes(T, N, ld_kv, H, d_qk, d_v, ld, kv_on_host != 0 && N > 0);
  return layout(chunk_tokens, N, ld_kv, H, d_qk, d_v, ld, kv_on_host != 0).total;
}

int dsa_sparse_prefill_host(const uint16_t* q, const uint16_t* kv, int kv_on_host, int N, int ld_kv,
                            const int32_t* idx, int T, int H, int d_qk, int d_v, int k, int ld, float scale,
                            uint16_t* out, float* lse, void* workspace, int64_t workspace_bytes, int chunk_tokens,
                            dsa_stream_t stream) {
  if (T < 0 || N < 0 || k < 0 || ld < k || ld_kv < d_qk || chunk_tokens < 1) return DSA_ERR_INVALID_ARG;
  if (!(H == 16 || H == 32) || !(d_qk == 576 || d_qk == 512) || d_v != 512 || k > 2048) return DSA_ERR_UNSUPPORTED;
  if ((ld_kv & 7) != 0) return DSA_ERR_INVALID_ARG;
  if (T == 0) return DSA_OK;
  if (!q || (!kv && N > 0) || !idx || !out || !lse || !workspace) return DSA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) != 0) return DSA_ERR_INVALID_ARG;
  const int chunk = chunk_tokens < T ? chunk_tokens : T;
  const bool kv_host = kv_on_host != 0 && N > 0;
  const Layout L = layout(chunk, N, ld_kv, H, d_qk, d_v, ld, kv_host);
  // the streamed form when the workspace holds every token (and the driver
  // has stream memory operations), else the ring of chunk launches
  const bool fits_all = workspace_bytes >= streamed_bytes(T, N, ld_kv, H, d_qk, d_v, ld, kv_host);
  const bool streamed = fits_all && mem_ops() != nullptr;
  if (!streamed && workspace_bytes < L.total) return fits_all ? DSA_ERR_UNSUPPORTED : DSA_ERR_INVALID_ARG;
  Pipe* p;
  if (!pipe_of(&p)) return DSA_ERR_CUDA;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  auto ok = [](cudaError_t e) { return e == cudaSuccess; };
  // On an error after work was queued on the library's streams, the caller's
  // stream still waits for all of it, so no copy into the caller's buffers is
  // left in flight behind the caller's next work (the first error is the one
  // returned; errors of these joins are not).
  auto fail = [&](int st) {
    const cudaStream_t ss[3] = {p->h2d, p->cmp, p->d2h};
    for (cudaStream_t s : ss)
      if (cudaEventRecord(p->exit, s) == cudaSuccess) cudaStreamWaitEvent((cudaStream_t)stream, p->exit, 0);
    return st;
  };
  // start after the work already queued on the caller's stream
  if (!ok(cudaEventRecord(p->entry, (cudaStream_t)stream)) || !ok(cudaStreamWaitEvent(p->h2d, p->entry, 0)) ||
      !ok(cudaStreamWaitEvent(p->cmp, p->entry, 0)) || !ok(cudaStreamWaitEvent(p->d2h, p->entry, 0)))
    return fail(DSA_ERR_CUDA);
  if (streamed) {
    const MemOps* mo = mem_ops();
    const Layout F = layout(T, N, ld_kv, H, d_qk, d_v, ld, kv_host);
    uint8_t* set = ws + F.kv;
    uint16_t* dq = reinterpret_cast<uint16_t*>(set);
    int32_t* didx = reinterpret_cast<int32_t*>(set + F.q);
    uint16_t* dout = reinterpret_cast<uint16_t*>(set + F.q + F.idx);
    float* dlse = reinterpret_cast<float*>(set + F.q + F.idx + F.out);
    uint32_t* ready = reinterpret_cast<uint32_t*>(set + F.set);
    uint32_t* done = ready + 1;
    const int blk = T < p->num_sms ? T : p->num_sms;   // one token per CTA (the kernel's grid)
    const int nblk = (T + blk - 1) / blk;
    const CUstream h2d = (CUstream)p->h2d, d2h = (CUstream)p->d2h;
    // counters cleared before the kernel and the read-backs start
    if (!ok(cudaMemsetAsync(ready, 0, 4 * ((size_t)nblk + 1), p->h2d)) || !ok(cudaEventRecord(p->kv_in, p->h2d)) ||
        !ok(cudaStreamWaitEvent(p->cmp, p->kv_in, 0)) || !ok(cudaStreamWaitEvent(p->d2h, p->kv_in, 0)))
      return fail(DSA_ERR_CUDA);
    const uint16_t* kv_dev = kv;
    if (kv_host) {
      if (!ok(cudaMemcpyAsync(ws, kv, (size_t)N * ld_kv * 2, cudaMemcpyHostToDevice, p->h2d))) return fail(DSA_ERR_CUDA);
      kv_dev = reinterpret_cast<const uint16_t*>(ws);
    }
    const int cap = chunk < kStreamTokensPerSm * p->num_sms ? chunk : kStreamTokensPerSm * p->num_sms;
    const std::vector<int> plan = plan_chunks(T, cap, p->num_sms);
    auto upload = [&](int64_t t0, int n) {
      return ok(cudaMemcpyAsync(dq + t0 * H * d_qk, q + t0 * H * d_qk, (size_t)n * H * d_qk * 2,
                                cudaMemcpyHostToDevice, p->h2d)) &&
             ok(cudaMemcpyAsync(didx + t0 * ld, idx + t0 * ld, (size_t)n * ld * 4, cudaMemcpyHostToDevice, p->h2d)) &&
             mo->write(h2d, (CUdeviceptr)ready, (cuuint32_t)(t0 + n), CU_STREAM_WRITE_VALUE_DEFAULT) == CUDA_SUCCESS;
    };
    // the table and the first chunk, then the kernel (so that it starts while
    // the host queues the rest), then the other chunks' uploads
    if (!upload(0, plan[0])) return fail(DSA_ERR_CUDA);
    const int st = dsa::sparse_prefill_streamed(dq, kv_dev, N, ld_kv, didx, T, H, d_qk, d_v, k, ld, scale, dout,
                                                dlse, ready, done, blk, p->cmp);
    if (st != DSA_OK) return fail(st);
    if (!ok(cudaEventRecord(p->done[0], p->cmp))) return fail(DSA_ERR_CUDA);
    int64_t t0 = plan[0];
    for (size_t i = 1; i < plan.size(); t0 += plan[i], ++i)
      if (!upload(t0, plan[i])) {
        // release the kernel rather than leave it waiting out its bound (the
        // call reports the error; no read-back was queued)
        mo->write(h2d, (CUdeviceptr)ready, (cuuint32_t)T, CU_STREAM_WRITE_VALUE_DEFAULT);
        return fail(DSA_ERR_CUDA);
      }
    // each chunk back once every block of tokens it touches is counted done
    t0 = 0;
    int waited = -1;   // blocks already waited for
    for (int n : plan) {
      const int b_last = (int)((t0 + n - 1) / blk);
      for (int b = waited + 1; b <= b_last; ++b) {
        const int64_t cnt = (int64_t)T - (int64_t)b * blk < blk ? (int64_t)T - (int64_t)b * blk : blk;
        if (mo->wait(d2h, (CUdeviceptr)(done + b), (cuuint32_t)cnt, CU_STREAM_WAIT_VALUE_GEQ) != CUDA_SUCCESS)
          return fail(DSA_ERR_CUDA);
      }
      waited = b_last;
      if (!ok(cudaMemcpyAsync(out + t0 * H * d_v, dout + t0 * H * d_v, (size_t)n * H * d_v * 2, cudaMemcpyDeviceToHost,
                              p->d2h)) ||
          !ok(cudaMemcpyAsync(lse + t0 * H, dlse + t0 * H, (size_t)n * H * 4, cudaMemcpyDeviceToHost, p->d2h)))
        return fail(DSA_ERR_CUDA);
      t0 += n;
    }
    // the caller's stream continues once the outputs are in host memory and
    // the kernel has ended
    if (!ok(cudaEventRecord(p->exit, p->d2h)) || !ok(cudaStreamWaitEvent((cudaStream_t)stream, p->exit, 0)) ||
        !ok(cudaStreamWaitEvent((cudaStream_t)stream, p->done[0], 0)))
      return DSA_ERR_CUDA;
    return DSA_OK;
  }
  const uint16_t* kv_dev = kv;
  if (kv_host) {
    if (!ok(cudaMemcpyAsync(ws, kv, (size_t)N * ld_kv * 2, cudaMemcpyHostToDevice, p->h2d)) ||
        !ok(cudaEventRecord(p->kv_in, p->h2d)) || !ok(cudaStreamWaitEvent(p->cmp, p->kv_in, 0)))
      return fail(DSA_ERR_CUDA);
    kv_dev = reinterpret_cast<const uint16_t*>(ws);
  }
  const std::vector<int> plan = plan_chunks(T, chunk, p->num_sms);
  const int nchunks = (int)plan.size();
  int64_t t0 = 0;
  for (int i = 0; i < nchunks; t0 += plan[i], ++i) {
    const int b = i % NB;
    const int n = plan[i];
    uint8_t* set = ws + L.kv + b * L.set;
    uint16_t* dq = reinterpret_cast<uint16_t*>(set);
    int32_t* didx = reinterpret_cast<int32_t*>(set + L.q);
    uint16_t* dout = reinterpret_cast<uint16_t*>(set + L.q + L.idx);
    float* dlse = reinterpret_cast<float*>(set + L.q + L.idx + L.out);
    // inputs of chunk i, once the kernel of chunk i - NB has read set b
    if (i >= NB && !ok(cudaStreamWaitEvent(p->h2d, p->done[b], 0))) return fail(DSA_ERR_CUDA);
    if (!ok(cudaMemcpyAsync(dq, q + t0 * H * d_qk, (size_t)n * H * d_qk * 2, cudaMemcpyHostToDevice, p->h2d)) ||
        !ok(cudaMemcpyAsync(didx, idx + t0 * ld, (size_t)n * ld * 4, cudaMemcpyHostToDevice, p->h2d)) ||
        !ok(cudaEventRecord(p->in[b], p->h2d)))
      return fail(DSA_ERR_CUDA);
    // the kernel, once its inputs are in and set b's previous outputs left
    if (!ok(cudaStreamWaitEvent(p->cmp, p->in[b], 0)) || (i >= NB && !ok(cudaStreamWaitEvent(p->cmp, p->out[b], 0))))
      return fail(DSA_ERR_CUDA);
    const int st = dsa_sparse_prefill(dq, kv_dev, N, ld_kv, didx, n, H, d_qk, d_v, k, ld, scale, dout, dlse,
                                      (dsa_stream_t)p->cmp);
    if (st != DSA_OK) return fail(st);
    if (!ok(cudaEventRecord(p->done[b], p->cmp))) return fail(DSA_ERR_CUDA);
    // outputs of chunk i back to the host
    if (!ok(cudaStreamWaitEvent(p->d2h, p->done[b], 0)) ||
        !ok(cudaMemcpyAsync(out + t0 * H * d_v, dout, (size_t)n * H * d_v * 2, cudaMemcpyDeviceToHost, p->d2h)) ||
        !ok(cudaMemcpyAsync(lse + t0 * H, dlse, (size_t)n * H * 4, cudaMemcpyDeviceToHost, p->d2h)) ||
        !ok(cudaEventRecord(p->out[b], p->d2h)))
      return fail(DSA_ERR_CUDA);
  }
  // the caller's stream continues once the last outputs are in host memory
  if (!ok(cudaEventRecord(p->exit, p->d2h)) || !ok(cudaStreamWaitEvent((cudaStream_t)stream, p->exit, 0)))
    return DSA_ERR_CUDA;
  return DSA_OK;
}

}  // extern "C"
