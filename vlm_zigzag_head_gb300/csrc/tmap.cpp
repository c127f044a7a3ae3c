// TMA tensor maps over THD tensors (driver entry point resolved at run time,
// so the library does not link libcuda directly).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>

#include "tc.h"

namespace cpattn {

namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

}  // namespace

// dims (innermost first): {d, H, rows}; box {64, 1, rows_per_box}; a box row is
// 64 bf16 = 128 bytes, laid out by the hardware in the 128-byte swizzle that
// the tensor-core shared-memory descriptors expect.
bool make_tmap_thd(CUtensorMap* map, const void* base, int64_t rows, int H, int d,
                   int rows_per_box, const char** err, bool f16) {
  auto fn = encode_fn();
  if (!fn) {
    *err = "cuTensorMapEncodeTiled unavailable";
    return false;
  }
  if (rows < 1) rows = 1;  // an empty tensor is never read; keep the map valid
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)rows};
  cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)H * d * 2};
  cuuint32_t box[3] = {64, 1, (cuuint32_t)rows_per_box};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                  const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    *err = "cuTensorMapEncodeTiled failed";
    return false;
  }
  return true;
}

bool make_tmap_f32_sw128(CUtensorMap* map, void* base, int64_t rows, int H, int d, int box_rows,
                         const char** err) {
  auto fn = encode_fn();
  if (!fn) {
    *err = "cuTensorMapEncodeTiled unavailable";
    return false;
  }
  if (rows < 1) rows = 1;
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)rows};
  cuuint64_t strides[2] = {(cuuint64_t)d * 4, (cuuint64_t)H * d * 4};
  cuuint32_t box[3] = {32, 1, (cuuint32_t)box_rows};   // 32 fp32 = one 128-byte swizzle row
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    *err = "cuTensorMapEncodeTiled failed (swizzled fp32 rows)";
    return false;
  }
  return true;
}

bool make_tmap_ld(CUtensorMap* map, const void* base, int64_t pitch, int H, int box_rows,
                  const char** err) {
  auto fn = encode_fn();
  if (!fn) {
    *err = "cuTensorMapEncodeTiled unavailable";
    return false;
  }
  cuuint64_t dims[3] = {(cuuint64_t)pitch, (cuuint64_t)H, 2};
  cuuint64_t strides[2] = {(cuuint64_t)pitch * 4, (cuuint64_t)pitch * H * 4};
  cuuint32_t box[3] = {(cuuint32_t)box_rows, 1, 2};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    *err = "cuTensorMapEncodeTiled failed (lse2/D planes)";
    return false;
  }
  return true;
}

}  // namespace cpattn
