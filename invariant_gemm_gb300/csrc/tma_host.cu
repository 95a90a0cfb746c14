// Host side of the tensor-memory-accelerator (TMA) copies: encoding of 2-D
// and 3-D tensor maps through the driver entry point (the library does not
// link libcuda; the runtime hands out the driver function).
#include <cudaTypedefs.h>
#include <mutex>

#include "ig_common.cuh"

namespace ig {

namespace {
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_once;

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  std::call_once(g_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode;
}
}  // namespace

int encode_map_2d(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                  uint64_t row_stride_bytes, uint32_t box_cols, uint32_t box_rows, int swizzle) {
  if (!encoder()) return IG_ERR_CUDA;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {row_stride_bytes};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        static_cast<CUtensorMapSwizzle>(swizzle),
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? IG_OK : IG_ERR_CUDA;
}

int encode_map_a3(CUtensorMap* map, const void* base, uint64_t rows, uint64_t K,
                  uint32_t box_rows) {
  if (!encoder() || K % 64 != 0) return IG_ERR_CUDA;
  const cuuint64_t dims[3] = {64, rows, K / 64};
  const cuuint64_t strides[2] = {K * 2, 128};
  const cuuint32_t box[3] = {64, box_rows, 4};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? IG_OK : IG_ERR_CUDA;
}

}  // namespace ig
