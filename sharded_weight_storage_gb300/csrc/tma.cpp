// Tensor maps for TMA tile loads of byte matrices (e4m3 weights and codes).
#include <cudaTypedefs.h>

#include <mutex>

#include "sws_internal.h"

namespace sws {
namespace {

// cuTensorMapEncodeTiled through the runtime's driver entry point, so the
// library needs no direct link against the driver library.
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

}  // namespace

int encode_u8_tile_map(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, int box_rows, int box_cols) {
  auto fn = encode_fn();
  if (!fn) return fail(SWS_E_CUDA, "cuTensorMapEncodeTiled is unavailable");
  if (rows <= 0 || cols <= 0 || cols % 16 != 0 || box_rows <= 0 || box_rows > 256 ||
      (box_cols != 128 && box_cols != 64))
    return fail(SWS_E_INVALID, "tensor map: shape [%lld, %lld], box %d x %d", (long long)rows, (long long)cols,
                box_rows, box_cols);
  cuuint64_t gdim[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t gstride[1] = {(cuuint64_t)cols};
  cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
  cuuint32_t estride[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), gdim, gstride, box, estride,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, box_cols == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(SWS_E_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return SWS_OK;
}

}  // namespace sws
