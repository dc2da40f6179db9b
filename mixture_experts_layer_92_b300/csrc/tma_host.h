// Host-side TMA tensor maps (cuTensorMapEncodeTiled) shared by the tensor-core GEMMs.
#pragma once
#include <mutex>

#include "common.cuh"

namespace moe {

inline PFN_cuTensorMapEncodeTiled_v12000& encoder_slot() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  return fn;
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no libcuda link).
inline bool get_encoder() {
  static std::once_flag once;
  PFN_cuTensorMapEncodeTiled_v12000& g_encode = encoder_slot();
  std::call_once(once, [&g_encode]() {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPoint("cuTensorMapEncodeTiled", &fn, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode != nullptr;
}

inline CUtensorMapSwizzle swizzle_of(int kb) {
  return kb == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
}

// 2-D bf16 map over a row-major [rows, inner] matrix; box = [box_rows, kb], kb*2-byte swizzle.
inline bool encode_2d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint32_t box_rows,
               int kb) {
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {inner * 2};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(kb), box_rows};
  cuuint32_t es[2] = {1, 1};
  return encoder_slot()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                  box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle_of(kb),
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

// 3-D bf16 map over [groups, rows, inner]; box = [1, box_rows, kb], kb*2-byte swizzle.
inline bool encode_3d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint64_t groups,
               uint32_t box_rows, int kb) {
  cuuint64_t dims[3] = {inner, rows, groups};
  cuuint64_t strides[2] = {inner * 2, inner * rows * 2};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(kb), box_rows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return encoder_slot()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                  box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle_of(kb),
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

// 3-D uint8 map over [groups, rows, inner] bytes (8-bit weights); box = [1, box_rows, kb],
// no swizzle (the converters read it row by row).
inline bool encode_3d_u8(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint64_t groups,
                  uint32_t box_rows, int kb) {
  cuuint64_t dims[3] = {inner, rows, groups};
  cuuint64_t strides[2] = {inner, inner * rows};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(kb), box_rows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return encoder_slot()(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box,
                  es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

// 2-D bf16 map over a row-major [rows, inner] matrix whose tiles are read MN-major: box =
// [64 rows, 64 inner elements] with a 128-byte swizzle, i.e. a 64-wide slice of the
// contiguous dimension for 64 consecutive rows (the K rows of the MMA operand).
inline bool encode_2d_mn(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows,
                         uint64_t row_stride_elems) {
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {row_stride_elems * 2};
  cuuint32_t box[2] = {64, 64};
  cuuint32_t es[2] = {1, 1};
  return encoder_slot()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                        strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D bf16 map over [groups, rows, inner] read MN-major: box = [1, 64 rows, 64 inner].
inline bool encode_3d_mn(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows,
                         uint64_t groups) {
  cuuint64_t dims[3] = {inner, rows, groups};
  cuuint64_t strides[2] = {inner * 2, inner * rows * 2};
  cuuint32_t box[3] = {64, 64, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return encoder_slot()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                        strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D fp32 map over [groups, rows, inner] for tensor stores of 32-row blocks: box =
// [1, 32 rows, cols] with cols = 32 (128-byte rows, 128-byte swizzle) or 16 (64-byte rows,
// 64-byte swizzle).
inline bool encode_3d_f32_store(CUtensorMap* m, void* base, uint64_t inner, uint64_t rows,
                                uint64_t groups, int cols) {
  cuuint64_t dims[3] = {inner, rows, groups};
  cuuint64_t strides[2] = {inner * 4, inner * rows * 4};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(cols), 32, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return encoder_slot()(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE,
                        cols == 32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                        CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

// 2-D map for tensor stores of 16-bit outputs (bf16 or fp16 bits) [rows, cols] with row
// stride ld elements: box = [32 rows, box_cols] with box_cols = 32 (64-byte rows, 64-byte
// swizzle) or 16 (32-byte rows, 32-byte swizzle). False when the base or the row stride is
// not 16-byte aligned (the caller then stores element-wise).
inline bool encode_2d_out16(CUtensorMap* m, void* base, uint64_t cols, uint64_t rows, uint64_t ld,
                            int box_cols) {
  if (base == nullptr || (reinterpret_cast<uintptr_t>(base) & 15) != 0 || (ld * 2) % 16 != 0 ||
      cols == 0 || rows == 0 || cols > ld)
    return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {ld * 2};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), 32};
  cuuint32_t es[2] = {1, 1};
  return encoder_slot()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE,
                        box_cols == 32 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B,
                        CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

// 2-D map for tensor stores of 8-bit codes [rows, cols] (row stride ld bytes): box = [32 rows,
// 32 bytes], 32-byte swizzle. False when the base or the row stride is not 16-byte aligned.
inline bool encode_2d_out8(CUtensorMap* m, void* base, uint64_t cols, uint64_t rows, uint64_t ld) {
  if (base == nullptr || (reinterpret_cast<uintptr_t>(base) & 15) != 0 || ld % 16 != 0 ||
      cols == 0 || rows == 0 || cols > ld)
    return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {ld};
  cuuint32_t box[2] = {32, 32};
  cuuint32_t es[2] = {1, 1};
  return encoder_slot()(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, base, dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_32B,
                        CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

// 2-D map over bytes [rows, inner] (8-bit codes): box = [box_rows, 128 bytes], 128-byte swizzle.
inline bool encode_2d_u8_sw128(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows,
                               uint32_t box_rows) {
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {inner};
  cuuint32_t box[2] = {128, box_rows};
  cuuint32_t es[2] = {1, 1};
  return encoder_slot()(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims,
                        strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D map over bytes [groups, rows, inner]: box = [1, box_rows, 128 bytes], 128-byte swizzle.
inline bool encode_3d_u8_sw128(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows,
                               uint64_t groups, uint32_t box_rows) {
  cuuint64_t dims[3] = {inner, rows, groups};
  cuuint64_t strides[2] = {inner, inner * rows};
  cuuint32_t box[3] = {128, box_rows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return encoder_slot()(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims,
                        strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D map over 4-bit values packed two per byte, [groups, rows, inner values]: each group of
// 16 values (8 bytes) lands in 16 bytes of shared memory (8 empty), i.e. one byte per value
// as the block-scaled MMA reads 4-bit operands; box = [1, box_rows, 128 values] (the
// required inner box), 128-byte swizzle. inner % 128 == 0; base 32-byte aligned.
inline bool encode_3d_e2m1_sw128(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows,
                                 uint64_t groups, uint32_t box_rows) {
  cuuint64_t dims[3] = {inner, rows, groups};
  cuuint64_t strides[2] = {inner / 2, inner / 2 * rows};
  cuuint32_t box[3] = {128, box_rows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return encoder_slot()(m, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 3, const_cast<void*>(base), dims,
                        strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace moe
