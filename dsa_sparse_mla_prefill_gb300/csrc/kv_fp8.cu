// FP8 latent rows for the KV cache: quantize bf16 rows, dequantize them back.
//
// The pages keep the KV cache in bf16 ("[Perf][DSA] Grouped sparse prefill
// ...", review snippets: the grouped path refuses a quantized KV cache); an
// FP8 row here is the plainest layout for the latent row: the 512 NoPE
// columns as float8 e4m3, one fp32 scale per 128 of them (block amax / 448,
// 1 for an all-zero block), then the RoPE columns in bf16:
//     bytes [0, 512) codes | [512, 528) 4 scales | [528, 528 + 2 d_rope) RoPE
// Quantize: code = e4m3(x / scale), the division in IEEE float32 and the
// conversion round-to-nearest-even, saturating at 448.  Dequantize: the e4m3
// value times its block's scale in float32, rounded to bf16.
//
// The float32 steps are IEEE operations that keep subnormal values (written
// as PTX without .ftz, since the library is otherwise built to flush them),
// so tiny values and tiny scales follow the definition exactly.  The
// dequantize arithmetic is the shared e4m3x4_dequant_bf16x4, which the
// attention kernels that read FP8 rows directly also use.
//
// One warp per 128-column block (lane l: columns 4l .. 4l+3 of the block),
// four warps per row; a CTA takes eight rows at a time and issues all their
// loads before it converts any of them.
#include <cuda_fp16.h>

#include "dsa_device.cuh"
#include "dsa_kernels.h"

namespace dsa {
namespace fp8kv {

constexpr int NT = 128;
constexpr int RPI = 8;   // rows per CTA per iteration

__device__ __forceinline__ uint16_t f32x2_to_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;   // low byte: lo's code
}

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t b) { return __uint_as_float(b << 16); }

// IEEE float32 operations that keep subnormals
__device__ __forceinline__ float div_ieee(float a, float b) {
  float r;
  asm("div.rn.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ float max_ieee(float a, float b) {
  float r;
  asm("max.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ float abs_ieee(float a) {
  float r;
  asm("abs.f32 %0, %1;" : "=f"(r) : "f"(a));
  return r;
}

__global__ void __launch_bounds__(NT) quantize_kernel(Fp8KvArgs a) {
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rb = 528 + 2 * a.d_rope;
  for (int n0 = blockIdx.x * RPI; n0 < a.N; n0 += gridDim.x * RPI) {
    // every row's load first, so RPI loads per thread are in flight
    uint2 raw[RPI];
    uint32_t rope[RPI];
#pragma unroll
    for (int r = 0; r < RPI; ++r) {
      raw[r] = make_uint2(0, 0);
      rope[r] = 0;
      if (n0 + r < a.N) {
        const uint16_t* src = a.kv + (size_t)(n0 + r) * a.ld_kv;
        raw[r] = *reinterpret_cast<const uint2*>(src + 128 * w + 4 * lane);
        if (w == 0 && 2 * lane < a.d_rope) rope[r] = *reinterpret_cast<const uint32_t*>(src + 512 + 2 * lane);
      }
    }
#pragma unroll
    for (int r = 0; r < RPI; ++r) {
      const float v[4] = {bf16_bits_to_f32(raw[r].x & 0xffffu), bf16_bits_to_f32(raw[r].x >> 16),
                          bf16_bits_to_f32(raw[r].y & 0xffffu), bf16_bits_to_f32(raw[r].y >> 16)};
      float amax = max_ieee(max_ieee(abs_ieee(v[0]), abs_ieee(v[1])), max_ieee(abs_ieee(v[2]), abs_ieee(v[3])));
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) amax = max_ieee(amax, __shfl_xor_sync(0xffffffffu, amax, o));
      if (n0 + r >= a.N) continue;
      uint8_t* dst = a.fp8 + (size_t)(n0 + r) * rb;
      // (amax is +0 or positive: a zero bit pattern is an all-zero block)
      const float scale = __float_as_uint(amax) != 0u ? div_ieee(amax, 448.f) : 1.f;
      const uint32_t lo = f32x2_to_e4m3x2(div_ieee(v[0], scale), div_ieee(v[1], scale));
      const uint32_t hi = f32x2_to_e4m3x2(div_ieee(v[2], scale), div_ieee(v[3], scale));
      *reinterpret_cast<uint32_t*>(dst + 128 * w + 4 * lane) = lo | (hi << 16);
      if (lane == 0) *reinterpret_cast<float*>(dst + 512 + 4 * w) = scale;
      if (w == 0 && 2 * lane < a.d_rope)   // RoPE columns: 2 per lane
        *reinterpret_cast<uint32_t*>(dst + 528 + 4 * lane) = rope[r];
    }
  }
}

__global__ void __launch_bounds__(NT) dequantize_kernel(Fp8KvArgs a) {
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rb = 528 + 2 * a.d_rope;
  for (int n0 = blockIdx.x * RPI; n0 < a.N; n0 += gridDim.x * RPI) {
    uint32_t codes[RPI], rope[RPI];
    float scale[RPI];
#pragma unroll
    for (int r = 0; r < RPI; ++r) {
      codes[r] = 0;
      rope[r] = 0;
      scale[r] = 0.f;
      if (n0 + r < a.N) {
        const uint8_t* src = a.fp8 + (size_t)(n0 + r) * rb;
        codes[r] = *reinterpret_cast<const uint32_t*>(src + 128 * w + 4 * lane);
        scale[r] = *reinterpret_cast<const float*>(src + 512 + 4 * w);
        if (w == 0 && 2 * lane < a.d_rope) rope[r] = *reinterpret_cast<const uint32_t*>(src + 528 + 4 * lane);
      }
    }
#pragma unroll
    for (int r = 0; r < RPI; ++r) {
      if (n0 + r >= a.N) break;
      uint16_t* dst = a.kv_out + (size_t)(n0 + r) * a.ld_kv;
      uint2 out;
      e4m3x4_dequant_bf16x4(codes[r], scale[r], out.x, out.y);
      *reinterpret_cast<uint2*>(dst + 128 * w + 4 * lane) = out;
      if (w == 0 && 2 * lane < a.d_rope) *reinterpret_cast<uint32_t*>(dst + 512 + 2 * lane) = rope[r];
    }
  }
}

}  // namespace fp8kv

int launch_kv_fp8(const Fp8KvArgs& a, bool quantize, int num_sms, cudaStream_t stream) {
  if (a.N == 0) return 0;
  // RPI rows per CTA, each thread's RPI loads issued before any of them is
  // used, 16 CTAs (2048 threads) per SM: the copy is latency-bound, so the
  // bytes in flight per SM set its rate; larger tables loop over rows
  const int cap = 16 * num_sms;
  const int need = (a.N + fp8kv::RPI - 1) / fp8kv::RPI;
  const int grid = need < cap ? need : cap;
  if (quantize)
    fp8kv::quantize_kernel<<<grid, fp8kv::NT, 0, stream>>>(a);
  else
    fp8kv::dequantize_kernel<<<grid, fp8kv::NT, 0, stream>>>(a);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace dsa
