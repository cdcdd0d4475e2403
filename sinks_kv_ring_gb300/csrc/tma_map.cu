// tma_map.cu -- 2-D TMA tensor maps over the K/V tensors, encoded through the
// driver entry point (looked up once through the runtime, so the library does
// not link the driver library directly).
#include <cuda.h>

#include "launch.h"

namespace kvr {
namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

}  // namespace

bool make_tma_map_2d(CUtensorMap *m, const void *ptr, long long rows, int width, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)width, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)width * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_tma_map_rows3d(CUtensorMap *m, const void *ptr, long long rows, int width, int box_rows, bool one_part) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || width % 64) return false;
  const int parts = width / 64;
  cuuint64_t dims[3] = {64, (cuuint64_t)parts, (cuuint64_t)rows};
  cuuint64_t strides[2] = {128, (cuuint64_t)width * 2};
  cuuint32_t box[3] = {64, one_part ? 1u : (cuuint32_t)parts, (cuuint32_t)box_rows};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_tma_map_tokens4d(CUtensorMap *m, const void *ptr, long long T, int hkv, int width, int box_rows,
                           bool one_part, int heads_per_box) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || width % 64 || heads_per_box < 1 || heads_per_box > hkv) return false;
  const int parts = width / 64;
  cuuint64_t dims[4] = {64, (cuuint64_t)parts, (cuuint64_t)hkv, (cuuint64_t)T};
  cuuint64_t strides[3] = {128, (cuuint64_t)width * 2, (cuuint64_t)hkv * width * 2};
  cuuint32_t box[4] = {64, one_part ? 1u : (cuuint32_t)parts, (cuuint32_t)heads_per_box, (cuuint32_t)box_rows};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(ptr), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_tma_map_heads3d(CUtensorMap *m, const void *ptr, long long rows, int hq, int width, int G) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || G < 1 || 128 % G || hq % G || width % 64) return false;
  cuuint64_t dims[3] = {(cuuint64_t)width, (cuuint64_t)hq, (cuuint64_t)rows};
  cuuint64_t strides[2] = {(cuuint64_t)width * 2, (cuuint64_t)hq * width * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)G, (cuuint32_t)(128 / G)};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace kvr
