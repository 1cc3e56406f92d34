// TMA tensor maps of the [rows, heads, D] tensors (host side), encoded with
// the driver's cuTensorMapEncodeTiled found through the runtime's entry-point
// query (no link-time dependency on libcuda).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>
#include <string>

#include "kernels.hpp"

namespace cpattn {

static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// [rows, heads, D] bf16 viewed as a 3-D tensor (D, heads, rows); box = 64
// columns x 1 head x box_rows rows (128 for Q, 64 for a K/V piece), 128-byte
// swizzle.
static bool make_map_bf16(CUtensorMap* m, const void* base, int64_t rows, int heads, int D, int box_rows,
                     std::string* err) {
  auto enc = tensor_map_encoder();
  if (!enc) {
    *err = "cuTensorMapEncodeTiled is not available from the driver";
    return false;
  }
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)heads, (cuuint64_t)rows};
  cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)heads * D * 2};
  cuuint32_t box[3] = {64, 1, (cuuint32_t)box_rows};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    *err = "cuTensorMapEncodeTiled failed (" + std::to_string((int)r) + ")";
    return false;
  }
  return true;
}

bool make_tensor_map_bf16(CUtensorMap* m, const void* base, int64_t rows, int heads, int D, int box_rows,
                          std::string* err) {
  return make_map_bf16(m, base, rows, heads, D, box_rows, err);
}

// [rows, heads, D] fp32 as (D, heads, rows); box = D columns x 1 head x
// box_rows rows, no swizzle (the tile of a reduce-add from shared memory).
bool make_tensor_map_f32(CUtensorMap* m, const void* base, int64_t rows, int heads, int D, int box_rows,
                         std::string* err) {
  auto enc = tensor_map_encoder();
  if (!enc) {
    *err = "cuTensorMapEncodeTiled is not available from the driver";
    return false;
  }
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)heads, (cuuint64_t)rows};
  cuuint64_t strides[2] = {(cuuint64_t)D * 4, (cuuint64_t)heads * D * 4};
  cuuint32_t box[3] = {(cuuint32_t)D, 1, (cuuint32_t)box_rows};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    *err = "cuTensorMapEncodeTiled (fp32) failed (" + std::to_string((int)r) + ")";
    return false;
  }
  return true;
}

}  // namespace cpattn
