// Host-side tensor-map encoding for TMA row gathers.  The driver entry point
// is looked up through the runtime (no link-time dependency on libcuda), so
// the library still loads on machines without a GPU driver.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace dsa {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_tiled_fn() {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
    else
      cudaGetLastError();
  }
  return fn;
}

// 2-D bf16 map over `rows` rows of `cols` elements (row pitch `ld` elements):
// box = 64 columns x 1 row with 128-byte swizzle, the shape a tile::gather4
// load takes (4 rows of 128 bytes per instruction).  Rows outside [0, rows)
// read as zeros.  Returns false if the map cannot be encoded.
inline bool make_row_gather_map(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, int64_t ld) {
  EncodeTiledFn fn = encode_tiled_fn();
  if (fn == nullptr || rows < 1 || cols < 64) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)ld * 2u};
  cuuint32_t box[2] = {64u, 1u};
  cuuint32_t es[2] = {1u, 1u};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D byte map over `rows` rows of `row_bytes` bytes (also the row pitch, a
// multiple of 16): box = 128 bytes x 1 row with 128-byte swizzle, so one
// tile::gather4 load brings 4 rows of 128 bytes, as over bf16 rows.  Rows
// outside [0, rows) read as zero bytes.  For the FP8 latent rows.
inline bool make_row_gather_map_u8(CUtensorMap* m, const void* base, int64_t rows, int64_t row_bytes) {
  EncodeTiledFn fn = encode_tiled_fn();
  if (fn == nullptr || rows < 1 || row_bytes < 128 || (row_bytes % 16) != 0) return false;
  cuuint64_t dims[2] = {(cuuint64_t)row_bytes, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
  cuuint32_t box[2] = {128u, 1u};
  cuuint32_t es[2] = {1u, 1u};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D bf16 map with box = 64 columns x `box_rows` rows, 128-byte swizzle: a
// tile of box_rows rows lands as box_rows consecutive 128-byte rows, the
// K-major layout of one swizzle column of an MMA operand.
inline bool make_tile_map(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, int64_t ld, int box_rows) {
  EncodeTiledFn fn = encode_tiled_fn();
  if (fn == nullptr || rows < 1 || cols < 64 || box_rows < 1 || box_rows > 256) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)ld * 2u};
  cuuint32_t box[2] = {64u, (cuuint32_t)box_rows};
  cuuint32_t es[2] = {1u, 1u};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D bf16 map over a strided [rows, heads, cols] view (element strides
// stride_h between heads and stride_t between rows, both multiples of 8):
// box = 64 columns x 1 head x box_rows rows, 128-byte swizzle, so a box of
// one head lands as box_rows consecutive 128-byte rows, the K-major layout of
// one swizzle column of an MMA operand.  Rows outside [0, rows) read as zeros.
inline bool make_head_tile_map_strided(CUtensorMap* m, const void* base, int64_t rows, int64_t heads, int64_t cols,
                                       int64_t stride_h, int64_t stride_t, int box_rows) {
  EncodeTiledFn fn = encode_tiled_fn();
  if (fn == nullptr || rows < 1 || heads < 1 || cols < 64 || box_rows < 1 || box_rows > 256) return false;
  cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)heads, (cuuint64_t)rows};
  cuuint64_t strides[2] = {(cuuint64_t)stride_h * 2u, (cuuint64_t)stride_t * 2u};
  cuuint32_t box[3] = {64u, 1u, (cuuint32_t)box_rows};
  cuuint32_t es[3] = {1u, 1u, 1u};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The same over a contiguous [rows, heads, cols] tensor.
inline bool make_head_tile_map(CUtensorMap* m, const void* base, int64_t rows, int64_t heads, int64_t cols,
                               int box_rows) {
  return make_head_tile_map_strided(m, base, rows, heads, cols, cols, heads * cols, box_rows);
}

}  // namespace dsa
