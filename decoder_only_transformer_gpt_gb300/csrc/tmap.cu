// TMA descriptor construction (host). cuTensorMapEncodeTiled is a driver API
// function; it is looked up through the runtime's driver-entry-point query so
// the library does not link against libcuda directly.
#include "kernels.h"

#include <mutex>

namespace gptgb {

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

}  // namespace

bool make_tmap_2d_bf16(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows,
                       uint64_t ld) {
  EncodeTiledFn fn = encode_fn();
  if (ld == 0) ld = cols;
  if (!fn || !base || (reinterpret_cast<uintptr_t>(base) & 15u) || ((ld * 2) & 15u) || ld < cols) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {ld * 2};
  const cuuint32_t box[2] = {64, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_tmap_2d(CUtensorMap* map, const void* base, int elem_bytes, uint64_t rows, uint64_t cols,
                  uint32_t box_cols, uint32_t box_rows, uint64_t ld) {
  EncodeTiledFn fn = encode_fn();
  if (ld == 0) ld = cols;
  if (!fn || !base || (reinterpret_cast<uintptr_t>(base) & 15u) || ((ld * elem_bytes) & 15u) || ld < cols) return false;
  if (elem_bytes != 2 && elem_bytes != 4) return false;
  if (box_cols * static_cast<uint32_t>(elem_bytes) != 128) return false;      // one 128-byte swizzle row
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {ld * static_cast<uint64_t>(elem_bytes)};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUtensorMapDataType dt = elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  return fn(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_tmap_qkv(CUtensorMap* map, const void* base, int B, int T, int C3, int D) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || !base || (reinterpret_cast<uintptr_t>(base) & 15u) || ((C3 * 2) & 15) || (D != 32 && D != 64))
    return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(C3), static_cast<cuuint64_t>(T), static_cast<cuuint64_t>(B)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(C3) * 2, static_cast<cuuint64_t>(C3) * 2 * T};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(D), static_cast<cuuint32_t>(kAttnBQ), 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUtensorMapSwizzle swz = (D == 64) ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// An fp32 [B][T][C] tensor with a box of 32 rows x 32 columns (128 bytes, 128-byte swizzle; one batch):
// the attention derivative adds its dQ tiles into it with TMA reduce-adds. Rows past T are clipped.
bool make_tmap_bt_f32(CUtensorMap* map, const void* base, int B, int T, int C) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || !base || (reinterpret_cast<uintptr_t>(base) & 15u) || ((C * 4) & 15)) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(C), static_cast<cuuint64_t>(T), static_cast<cuuint64_t>(B)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(C) * 4, static_cast<cuuint64_t>(C) * 4 * T};
  const cuuint32_t box[3] = {32, 32, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The attention output y viewed as [B][T][C] bf16 with a box of 32 rows x D columns (one batch),
// for the TMA store of each warp's 32 query rows of one head: rows past T are clipped by the copy.
bool make_tmap_attn_out(CUtensorMap* map, const void* base, int B, int T, int C, int D) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || !base || (reinterpret_cast<uintptr_t>(base) & 15u) || ((C * 2) & 15) || (D != 32 && D != 64))
    return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(C), static_cast<cuuint64_t>(T), static_cast<cuuint64_t>(B)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(C) * 2, static_cast<cuuint64_t>(C) * 2 * T};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(D), 32, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUtensorMapSwizzle swz = (D == 64) ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_NONE,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace gptgb
