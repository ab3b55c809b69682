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
// four warps per row, rows strided over the grid.
#include <cuda_fp16.h>

#include "dsa_device.cuh"
#include "dsa_kernels.h"

namespace dsa {
namespace fp8kv {

constexpr int NT = 128;

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
  for (int n = blockIdx.x; n < a.N; n += gridDim.x) {
    const uint16_t* src = a.kv + (size_t)n * a.ld_kv;
    uint8_t* dst = a.fp8 + (size_t)n * rb;
    const uint2 raw = *reinterpret_cast<const uint2*>(src + 128 * w + 4 * lane);
    float v[4] = {bf16_bits_to_f32(raw.x & 0xffffu), bf16_bits_to_f32(raw.x >> 16),
                  bf16_bits_to_f32(raw.y & 0xffffu), bf16_bits_to_f32(raw.y >> 16)};
    float amax = max_ieee(max_ieee(abs_ieee(v[0]), abs_ieee(v[1])), max_ieee(abs_ieee(v[2]), abs_ieee(v[3])));
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) amax = max_ieee(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    // (amax is +0 or positive: a zero bit pattern is an all-zero block)
    const float scale = __float_as_uint(amax) != 0u ? div_ieee(amax, 448.f) : 1.f;
    const uint32_t lo = f32x2_to_e4m3x2(div_ieee(v[0], scale), div_ieee(v[1], scale));
    const uint32_t hi = f32x2_to_e4m3x2(div_ieee(v[2], scale), div_ieee(v[3], scale));
    *reinterpret_cast<uint32_t*>(dst + 128 * w + 4 * lane) = lo | (hi << 16);
    if (lane == 0) *reinterpret_cast<float*>(dst + 512 + 4 * w) = scale;
    if (w == 0 && 2 * lane < a.d_rope)   // RoPE columns: 2 per lane
      *reinterpret_cast<uint32_t*>(dst + 528 + 4 * lane) = *reinterpret_cast<const uint32_t*>(src + 512 + 2 * lane);
  }
}

__global__ void __launch_bounds__(NT) dequantize_kernel(Fp8KvArgs a) {
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rb = 528 + 2 * a.d_rope;
  for (int n = blockIdx.x; n < a.N; n += gridDim.x) {
    const uint8_t* src = a.fp8 + (size_t)n * rb;
    uint16_t* dst = a.kv_out + (size_t)n * a.ld_kv;
    const uint32_t codes = *reinterpret_cast<const uint32_t*>(src + 128 * w + 4 * lane);
    const float scale = *reinterpret_cast<const float*>(src + 512 + 4 * w);
    uint2 out;
    e4m3x4_dequant_bf16x4(codes, scale, out.x, out.y);
    *reinterpret_cast<uint2*>(dst + 128 * w + 4 * lane) = out;
    if (w == 0 && 2 * lane < a.d_rope)
      *reinterpret_cast<uint32_t*>(dst + 512 + 2 * lane) = *reinterpret_cast<const uint32_t*>(src + 528 + 4 * lane);
  }
}

}  // namespace fp8kv

int launch_kv_fp8(const Fp8KvArgs& a, bool quantize, int num_sms, cudaStream_t stream) {
  if (a.N == 0) return 0;
  const int grid = a.N < 8 * num_sms ? a.N : 8 * num_sms;
  if (quantize)
    fp8kv::quantize_kernel<<<grid, fp8kv::NT, 0, stream>>>(a);
  else
    fp8kv::dequantize_kernel<<<grid, fp8kv::NT, 0, stream>>>(a);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace dsa
