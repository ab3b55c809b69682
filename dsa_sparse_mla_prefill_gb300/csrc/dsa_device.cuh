// Device-side building blocks for the sm_103a kernels: mbarriers with bounded
// waits, cp.async gathers, the tcgen05 tensor-core instructions (TMEM
// allocation, MMA issue, commit, TMEM loads/stores) and the shared-memory /
// instruction descriptors they take.  Inline PTX only; no library code.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace dsa {

// ---------------------------------------------------------------------------
// error counters (in device global memory, owned by the library)
//   [0] index entries outside [-1, N) that were ignored
//   [1] bounded waits that ran out (the kernel stopped early)
//   [2] union lists that did not fit in union_pad (truncated)
//   [3] reserved
// ---------------------------------------------------------------------------
enum { ERR_BAD_INDEX = 0, ERR_TIMEOUT = 1, ERR_UNION_OVERFLOW = 2 };

// A bounded wait gives up after this long (ns of %globaltimer).
constexpr uint64_t kWaitTimeoutNs = 2000000000ull;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t lane_id() { return threadIdx.x & 31; }

__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ---------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// The same with a suspend-time hint: a thread whose phase is not complete
// sleeps until it completes (or the hint, in ns, runs out) instead of
// returning at once, so waiting warps do not take issue slots from the warps
// doing the work.
constexpr uint32_t kSuspendHintNs = 50000;
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "n"(kSuspendHintNs)
      : "memory");
  return ok != 0;
}

// Waits until the phase with the given parity has completed.  Returns false
// (and raises the CTA's abort flag and the timeout counter) when the wait ran
// out or another thread of the CTA already gave up.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          unsigned int* err) {
  const uint32_t a = smem_u32(bar);
  if (mbar_try_wait(a, parity)) return true;
  const uint64_t t0 = globaltimer();
  while (true) {
    if (mbar_try_wait_sleep(a, parity)) return true;
    if (*abort_flag) return false;
    if (globaltimer() - t0 > kWaitTimeoutNs) {
      *abort_flag = 1;
      atomicAdd(err + ERR_TIMEOUT, 1u);
      return false;
    }
  }
}

// Warp-uniform bounded wait: every lane waits, and the warp proceeds only if
// all lanes saw the phase complete (so .sync.aligned instructions that follow
// never run with a partial warp).
__device__ __forceinline__ bool mbar_wait_warp(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                               unsigned int* err) {
  const bool ok = mbar_wait(bar, parity, abort_flag, err);
  return __all_sync(0xffffffffu, ok);
}

// Bounded barrier among the `count` threads that share one mbarrier
// (initialised with that count): arrive, then wait for the phase.  Unlike
// bar.sync it cannot hang if a thread of the group has given up.
__device__ __forceinline__ bool group_sync(uint64_t* bar, uint32_t& phase, volatile int* abort_flag,
                                           unsigned int* err) {
  mbar_arrive(bar);
  const bool ok = mbar_wait(bar, phase, abort_flag, err);
  phase ^= 1u;
  return ok;
}

// Same as mbar_wait, with cluster-scope acquire: for barriers that receive
// arrivals (and data) from the peer CTA of a cluster.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool mbar_try_wait_cluster_sleep(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "n"(kSuspendHintNs)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                                  unsigned int* err) {
  const uint32_t a = smem_u32(bar);
  if (mbar_try_wait_cluster(a, parity)) return true;
  const uint64_t t0 = globaltimer();
  while (true) {
    if (mbar_try_wait_cluster_sleep(a, parity)) return true;
    if (*abort_flag) return false;
    if (globaltimer() - t0 > kWaitTimeoutNs) {
      *abort_flag = 1;
      atomicAdd(err + ERR_TIMEOUT, 1u);
      return false;
    }
  }
}
__device__ __forceinline__ bool mbar_wait_cluster_warp(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                                       unsigned int* err) {
  const bool ok = mbar_wait_cluster(bar, parity, abort_flag, err);
  return __all_sync(0xffffffffu, ok);
}

// ---------------------------------------------------------------------------
// clusters / distributed shared memory
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_id_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t nclusters_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}
// Address of the same shared-memory offset in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_peer(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
__device__ __forceinline__ void st_cluster_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared::cluster.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
               : "memory");
}
__device__ __forceinline__ float4 ld_cluster_v4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}
__device__ __forceinline__ void st_cluster_f32(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}
// Arrive on an mbarrier of another CTA of the cluster (release at cluster scope).
// Asynchronous 16-byte store into a peer CTA's shared memory that counts
// its bytes on the peer's mbarrier (transaction count), so the receiver
// learns of the data by waiting on its own barrier; no release fence on the
// sender.  Both addresses come from map_peer.
__device__ __forceinline__ void st_async_v4(uint32_t remote_addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d,
                                            uint32_t remote_bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
                   remote_addr),
               "r"(a), "r"(b), "r"(c), "r"(d), "r"(remote_bar)
               : "memory");
}

// The same for one 32-bit value.
__device__ __forceinline__ void st_async_f32(uint32_t remote_addr, float v, uint32_t remote_bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(remote_addr),
               "r"(__float_as_uint(v)), "r"(remote_bar)
               : "memory");
}

// Arrival on a peer CTA's barrier without release semantics: for signalling
// that values loaded earlier are no longer needed, when every one of those
// loads has already been consumed by an instruction before the arrival (so
// it has completed and the peer may overwrite the buffer).
__device__ __forceinline__ void mbar_arrive_remote_relaxed(uint32_t remote_bar) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(remote_bar) : "memory");
}

// Two floats to a bf16 pair with round-to-nearest-even: lo in bits 0-15.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// ---------------------------------------------------------------------------
// FP8 latent rows: float8 e4m3 codes times a per-block fp32 scale, rounded to
// bf16.  Every e4m3 value is exact in f16 and f32; the product is one IEEE
// float32 multiply that keeps subnormals (no .ftz, while the library is
// otherwise built to flush them), then round-to-nearest-even to bf16.  The
// dequantize kernel and the attention kernels that read FP8 rows share this
// one routine, so the two paths give the same bits.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t f16x2_scaled_bf16x2(uint32_t h, float s) {
  const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h));   // .x: the low half
  float lo, hi;
  asm("{.reg .b64 x, y, d;\n\t"
      "mov.b64 x, {%2, %3};\n\t"
      "mov.b64 y, {%4, %4};\n\t"
      "mul.rn.f32x2 d, x, y;\n\t"
      "mov.b64 {%0, %1}, d;}"
      : "=f"(lo), "=f"(hi) : "f"(f.x), "f"(f.y), "f"(s));
  return pack_bf16x2(lo, hi);
}
// four codes (byte i of w = code i) -> bf16 pairs: lo = codes 0, 1; hi = codes 2, 3
__device__ __forceinline__ void e4m3x4_dequant_bf16x4(uint32_t w, float s, uint32_t& lo, uint32_t& hi) {
  uint32_t h0, h1;
  asm("{.reg .b16 l, h;\n\t"
      "mov.b32 {l, h}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, l;\n\t"
      "cvt.rn.f16x2.e4m3x2 %1, h;}"
      : "=r"(h0), "=r"(h1) : "r"(w));
  lo = f16x2_scaled_bf16x2(h0, s);
  hi = f16x2_scaled_bf16x2(h1, s);
}

// cp.async of 4 bytes (src_bytes = 0: zero fill), and an arrival on an
// mbarrier once this thread's earlier cp.async copies have landed (the
// barrier's pending count is raised now and lowered then).
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_mbar_arrive(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ float lds_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr));
  return v;
}

// 16-byte shared-memory accesses by 32-bit shared address
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}
__device__ __forceinline__ void sts128(uint32_t addr, uint32_t x, uint32_t y, uint32_t z, uint32_t w) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(x), "r"(y), "r"(z), "r"(w) : "memory");
}

__device__ __forceinline__ void mbar_arrive_remote(uint32_t remote_bar) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(remote_bar) : "memory");
}
__device__ __forceinline__ void fence_proxy_async_cluster() {
  asm volatile("fence.proxy.async.shared::cluster;" ::: "memory");
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Diagnostic timeline stamp (see TraceArgs): CTAs 0 and 1 only.
#define DSA_TRACE(tr, slot, ev)                                                              \
  do {                                                                                       \
    if ((tr).trace != nullptr && blockIdx.x < 2 && (int)(slot) < (tr).trace_cap)             \
      (tr).trace[((size_t)blockIdx.x * (tr).trace_cap + (slot)) * 8 + (ev)] = clock64();     \
  } while (0)

// Arrive and add `bytes` to the transaction count the phase waits for.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

// TMA row gather: rows r0..r3 (columns x .. x+63 of a 64x1-box, 128B-swizzled
// map) into 4 consecutive 128-byte rows at `dst`; the bytes complete on `bar`.
// x must be a multiple of 8 elements (16 bytes); rows outside the map read as
// zeros.
__device__ __forceinline__ void tma_gather4(uint32_t dst, const CUtensorMap* map, int x, int r0, int r1, int r2,
                                            int r3, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(r0), "r"(r1), "r"(r2), "r"(r3), "r"(smem_u32(bar))
      : "memory");
}

// TMA tiled 3-D load of one box (columns x .. x+63, head y, rows z .. z+box-1).
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y, int z,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}

// TMA tiled 2-D load of one box (columns x .. x+63, rows y .. y+box-1).
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// ---------------------------------------------------------------------------
// CTA pairs (cta_group::2).  Two CTAs of a cluster (ranks 2i, 2i+1) act as
// one: a pair MMA issued by one thread of the even CTA computes an M = 256
// tile whose A rows 0-127 and B columns 0..N/2-1 come from the even CTA's
// shared memory and A rows 128-255 and B columns N/2..N-1 from the odd
// CTA's (same offsets), and writes D rows 0-127 to the even CTA's tensor
// memory and rows 128-255 to the odd CTA's (same address).  Every tcgen05
// instruction of such a kernel uses cta_group::2; allocation, relinquish and
// deallocation are executed by one warp of each CTA of the pair.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// Four accumulating pair MMAs (see mma_bf16_ss_x4): A and B descriptors
// address the same offsets in both CTAs' shared memory.
__device__ __forceinline__ void mma_pair_bf16_ss_x4(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t da,
                                                    uint32_t db, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %5, %6, %3, 1;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %7, %8, %3, 1;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %9, %10, %3, 1;\n\t}"
      ::"r"(d_tmem), "l"(a), "l"(b), "r"(idesc), "r"(accumulate), "l"(a + da), "l"(b + db), "l"(a + 2ull * da),
      "l"(b + 2ull * db), "l"(a + 3ull * da), "l"(b + 3ull * db)
      : "memory");
}

// One arrival on the barrier at the offset of `bar` in every CTA of
// cta_mask once every pair tcgen05 op issued so far by this thread has
// completed (the completion signal; no data moves).
__device__ __forceinline__ void mma_pair_commit(uint64_t* bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_u32(bar)),
      "h"(cta_mask)
      : "memory");
}

// TMA loads into this CTA's own shared memory whose bytes complete on a
// barrier of either CTA of the pair (`bar_cluster`: a shared::cluster
// address, e.g. map_peer(smem_u32(bar), 0) for the even CTA's barrier), so
// that the pair's MMA issuer learns of both CTAs' operands on one barrier.
__device__ __forceinline__ void tma_gather4_pair(uint32_t dst, const CUtensorMap* map, int x, int r0, int r1, int r2,
                                                 int r3, uint32_t bar_cluster) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes.cta_group::2 "
      "[%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(r0), "r"(r1), "r"(r2), "r"(r3), "r"(bar_cluster)
      : "memory");
}
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, int x, int y,
                                                 uint32_t bar_cluster) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2 "
      "[%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar_cluster)
      : "memory");
}

// Bulk copy of `bytes` (a multiple of 16, both addresses 16-byte aligned)
// from this CTA's shared memory into a peer CTA's, by the copy engine (the
// async proxy); the bytes complete on `bar_cluster`, a barrier of the
// destination CTA.  The source may be rewritten once the destination has
// observed the barrier phase (every byte was read by then).
__device__ __forceinline__ void bulk_copy_to_peer(uint32_t dst_cluster, uint32_t src, uint32_t bytes,
                                                  uint32_t bar_cluster) {
  asm volatile("cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   dst_cluster),
               "r"(src), "r"(bytes), "r"(bar_cluster)
               : "memory");
}

// Arrive-and-expect on a barrier given by its shared::cluster address (a
// barrier of this CTA or of the peer).
__device__ __forceinline__ void mbar_arrive_expect_tx_cluster(uint32_t bar_cluster, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cluster.shared::cluster.b64 _, [%0], %1;" ::"r"(bar_cluster),
               "r"(bytes)
               : "memory");
}

// Bounded wait that ignores the CTA abort flag: used on the way out to let
// copies already in flight land before the CTA exits.
__device__ __forceinline__ bool mbar_wait_drain(uint64_t* bar, uint32_t parity, unsigned int* err) {
  const uint32_t a = smem_u32(bar);
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(a, parity)) {
    if (globaltimer() - t0 > kWaitTimeoutNs) {
      atomicAdd(err + ERR_TIMEOUT, 1u);
      return false;
    }
  }
  return true;
}

// Non-blocking probe of a phase with cluster-scope acquire (barriers that
// receive arrivals and data from the peer CTA).
__device__ __forceinline__ bool mbar_ready_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Non-blocking probe of a phase.
__device__ __forceinline__ bool mbar_ready(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// ---------------------------------------------------------------------------
// cp.async (16-byte, L2-only) with zero fill, and proxy fences
// ---------------------------------------------------------------------------
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Makes this thread's generic-proxy shared-memory writes visible to the async
// proxy (the tensor core reads shared memory through it).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// The same for global memory: orders what this thread has observed through
// the generic proxy (a flag it acquired) before the TMA reads it issues next.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// ---------------------------------------------------------------------------
// flags shared with the copy engines (streamed host calls)
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void red_release_gpu_add(uint32_t* p, uint32_t v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Loads cached in L2 only: for data another agent (a copy engine) may have
// written while the kernel runs, which the non-coherent path must not serve.
__device__ __forceinline__ int4 ld_cg_i4(const int4* p) {
  int4 v;
  asm volatile("ld.global.cg.v4.s32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ int ld_cg_i32(const int* p) {
  int v;
  asm volatile("ld.global.cg.s32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}

// Bounded wait (lane 0 polls, the warp follows) until *ready > t.  Returns
// false, raising the CTA's abort flag and the timeout counter, when it ran
// out or another thread of the CTA already gave up.
__device__ __forceinline__ bool wait_ready_warp(const uint32_t* ready, uint32_t t, volatile int* abort_flag,
                                                unsigned int* err) {
  bool ok = true;
  if (lane_id() == 0 && ld_acquire_gpu(ready) <= t) {
    const uint64_t t0 = globaltimer();
    while (true) {
      __nanosleep(256);
      if (ld_acquire_gpu(ready) > t) break;
      if (*abort_flag) {
        ok = false;
        break;
      }
      if (globaltimer() - t0 > kWaitTimeoutNs) {
        *abort_flag = 1;
        atomicAdd(err + ERR_TIMEOUT, 1u);
        ok = false;
        break;
      }
    }
  }
  ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
  __syncwarp();
  return ok;
}

// ---------------------------------------------------------------------------
// tcgen05: TMEM allocation
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
// Warpgroup register rebalancing: every warp of a 4-warp-aligned group
// executes the same call; the sum over the CTA must stay within the
// registers the CTA was launched with.
template <int N>
__device__ __forceinline__ void regs_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;\n" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void regs_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;\n" ::"n"(N));
}

__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// ---------------------------------------------------------------------------
// tcgen05: descriptors
// ---------------------------------------------------------------------------
// Instruction descriptor for kind::f16 with bf16 A/B and an fp32 accumulator.
//   bits 4-5 D format (1 = f32), 7-9 A format (1 = bf16), 10-12 B format,
//   15 A major (0 = K-major, 1 = MN-major), 16 B major, 17-22 N>>3, 24-28 M>>4.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, bool a_mn_major, bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn_major ? 1u : 0u) << 15) |
         ((b_mn_major ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Shared-memory matrix descriptor, 128-byte swizzle.
//   bits 0-13 start>>4, 16-29 leading byte offset>>4, 32-45 stride byte
//   offset>>4, 46-47 version (1), 49-51 base offset (0: atoms 1024-aligned),
//   61-63 layout (2 = 128-byte swizzle).
// K-major: the swizzle atom is 8 rows x 128 B (64 bf16 of K); SBO = stride
//   between 8-row groups along M/N; LBO unused.
// MN-major: the atom is 8 K-rows x 128 B (64 bf16 of M/N); LBO = stride
//   between 64-element groups along M/N, SBO = stride between 8-row groups
//   along K.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// Byte offset of element (row, col) inside a K-major 128B-swizzled tile whose
// rows are 64 bf16 wide (one swizzle column): row r at r*128, 16-byte chunk
// c at (c ^ (r & 7)) * 16.
__host__ __device__ __forceinline__ uint32_t sw128_offset(uint32_t row, uint32_t col) {
  return row * 128u + ((((col >> 3) ^ row) & 7u) << 4) + (col & 7u) * 2u;
}

// ---------------------------------------------------------------------------
// tcgen05: MMA issue and commit (single thread)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mma_bf16_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
      ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// A operand from tensor memory (M = 128 rows in lanes, 16-bit elements packed
// two per 32-bit column, consecutive K in consecutive columns), B from
// shared memory.
__device__ __forceinline__ void mma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
      ::"r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void tmem_st8_u32(uint32_t taddr, const uint32_t* r) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(r[0]),
               "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
               : "memory");
}
__device__ __forceinline__ void tmem_st16_u32(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

// Four accumulating MMAs in one statement (one predicate setup, no per-MMA
// descriptor rebuild): MMA e uses a + e*da and b + e*db, where da/db advance
// the descriptors' start-address field (units of 16 bytes).  The first MMA
// accumulates iff accumulate != 0, the other three always accumulate.
// Issuing them together roughly halves the per-MMA issue cost.
__device__ __forceinline__ void mma_bf16_ss_x4(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t da, uint32_t db,
                                               uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %5, %6, %3, 1;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %7, %8, %3, 1;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %9, %10, %3, 1;\n\t}"
      ::"r"(d_tmem), "l"(a), "l"(b), "r"(idesc), "r"(accumulate), "l"(a + da), "l"(b + db), "l"(a + 2ull * da),
      "l"(b + 2ull * db), "l"(a + 3ull * da), "l"(b + 3ull * db)
      : "memory");
}
// Same with the A operand in tensor memory (A column advance ta per MMA).
__device__ __forceinline__ void mma_bf16_ts_x4(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t ta, uint32_t db,
                                               uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%5], %6, %3, 1;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%7], %8, %3, 1;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%9], %10, %3, 1;\n\t}"
      ::"r"(d_tmem), "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate), "r"(a_tmem + ta), "l"(b + db),
      "r"(a_tmem + 2 * ta), "l"(b + 2ull * db), "r"(a_tmem + 3 * ta), "l"(b + 3ull * db)
      : "memory");
}

// One arrival on the barrier at the offset of `bar` in every CTA of
// cta_mask once every tcgen05 op issued so far by this thread has completed.
__device__ __forceinline__ void mma_commit_mc(uint64_t* bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_u32(bar)),
      "h"(cta_mask)
      : "memory");
}

// The barrier gets one arrival once every tcgen05 op issued so far by this
// thread has completed.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

// ---------------------------------------------------------------------------
// tcgen05: TMEM <-> registers.  32x32b shape: warp w (w % 4) reads lanes
// 32*(w%4) .. +31, thread i gets lane 32*(w%4)+i, consecutive columns.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float* v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float* v) {
  uint32_t r[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) r[i] = __float_as_uint(v[i]);
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

// N consecutive columns (N a multiple of 16) of this thread's lane.
template <int N>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, float* v) {
#pragma unroll
  for (int i = 0; i < N / 16; ++i) tmem_ld16(taddr + 16 * i, v + 16 * i);
}
template <int N>
__device__ __forceinline__ void tmem_st_cols(uint32_t taddr, const float* v) {
#pragma unroll
  for (int i = 0; i < N / 16; ++i) tmem_st16(taddr + 16 * i, v + 16 * i);
}

// ---------------------------------------------------------------------------
// small numeric helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint16_t f32_to_bf16_rn(float x) {
  // round-to-nearest-even via the hardware conversion
  uint16_t r;
  asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(r) : "f"(x));
  return r;
}
__device__ __forceinline__ float bf16_to_f32(uint16_t b) { return __uint_as_float(((uint32_t)b) << 16); }

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

}  // namespace dsa
