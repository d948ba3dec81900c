// attn_common.cuh -- tile geometry, tensor-map encoding and shared-memory
// layout helpers shared by the sparse-tree attention kernels.
//
// Tiles are 128 query rows x 128 key rows.  Every bf16 operand tile lives in
// shared memory in the canonical 128-byte-swizzled layout that TMA writes
// (box = 64 elements x rows, SWIZZLE_128B): a [rows x D] tile is D/64 "column
// blocks" of rows x 128 bytes, 16-byte chunk c of row r stored at chunk
// c ^ (r % 8).  The same bytes serve as a K-major operand (rows = M or N,
// D = K) and as an MN-major operand (rows = K, D = N or M).
#pragma once

#include <cudaTypedefs.h>

#include "internal.h"
#include "ptx.cuh"

namespace stt {

constexpr int kTile = 128;       // query rows and key rows per tile
constexpr int kColBlock = 64;    // bf16 elements per 128-byte swizzle row
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Number of 128-key tiles of the causal block 0 that query tile [q0, q0+128)
// sees: keys 0..min(q0+127, T-1).  Zero when T == 0.
__host__ __device__ __forceinline__ int causal_kv_tiles(int q0, int T) {
  if (T <= 0) return 0;
  const int lim = min(q0 + kTile - 1, T - 1);
  return lim / kTile + 1;
}

// Last key row query q sees in block 0 (keys 0..lim); -1 if none.
__host__ __device__ __forceinline__ int causal_row_limit(int q, int T) { return min(q, T - 1); }

// Byte offset of 16-byte chunk `c` (0..D/8-1) of row `r` in a swizzled
// [rows x D] bf16 tile with `rows` rows.
__device__ __forceinline__ uint32_t swz_chunk_offset(int r, int c, int rows) {
  const int cb = c >> 3, cc = c & 7;
  return (uint32_t)(cb * rows * 128 + r * 128 + ((cc ^ (r & 7)) << 4));
}

// Encodes a 3-D bf16 tensor map over [outer][rows][D] with a 64 x box_rows box
// and 128-byte swizzle; out-of-range rows read as zero.
inline cudaError_t encode_tile_map(CUtensorMap* map, const void* base, int D, int rows, int outer,
                                   int box_rows) {
  auto enc = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(tensor_map_encoder());
  if (!enc) return cudaErrorNotSupported;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)rows, (cuuint64_t)outer};
  cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)D * 2 * (cuuint64_t)rows};
  cuuint32_t box[3] = {(cuuint32_t)kColBlock, (cuuint32_t)box_rows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                   box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// fp32 [outer][rows][D] tensor map with a 32 x box_rows box (128-byte rows) and
// 128-byte swizzle: the staging layout used for reduce-add of gradients.
inline cudaError_t encode_f32_map(CUtensorMap* map, const void* base, int D, int rows, int outer,
                                  int box_rows) {
  auto enc = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(tensor_map_encoder());
  if (!enc) return cudaErrorNotSupported;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)rows, (cuuint64_t)outer};
  cuuint64_t strides[2] = {(cuuint64_t)D * 4, (cuuint64_t)D * 4 * (cuuint64_t)rows};
  cuuint32_t box[3] = {32, (cuuint32_t)box_rows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(base), dims, strides,
                   box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// max(a, b, c) in one instruction.
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}
// Packed fp32 pairs (lo in the low word) and the paired FMA / add.
__device__ __forceinline__ uint64_t f32x2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void unpack_f32x2(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t fma_f32x2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint64_t mul_f32x2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t add_f32x2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}

__device__ __forceinline__ float bf16lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

// Dot product of two bf16 rows of length D in global memory (fp32 accumulate).
template <int D>
__device__ __forceinline__ float dot_bf16_rows(const __nv_bfloat16* a, const __nv_bfloat16* b) {
  const uint4* a4 = reinterpret_cast<const uint4*>(a);
  const uint4* b4 = reinterpret_cast<const uint4*>(b);
  float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
  for (int c = 0; c < D / 8; ++c) {
    const uint4 x = __ldg(a4 + c), y = __ldg(b4 + c);
    acc0 = fmaf(bf16lo(x.x), bf16lo(y.x), acc0);
    acc1 = fmaf(bf16hi(x.x), bf16hi(y.x), acc1);
    acc0 = fmaf(bf16lo(x.y), bf16lo(y.y), acc0);
    acc1 = fmaf(bf16hi(x.y), bf16hi(y.y), acc1);
    acc0 = fmaf(bf16lo(x.z), bf16lo(y.z), acc0);
    acc1 = fmaf(bf16hi(x.z), bf16hi(y.z), acc1);
    acc0 = fmaf(bf16lo(x.w), bf16lo(y.w), acc0);
    acc1 = fmaf(bf16hi(x.w), bf16hi(y.w), acc1);
  }
  return acc0 + acc1;
}

}  // namespace stt
