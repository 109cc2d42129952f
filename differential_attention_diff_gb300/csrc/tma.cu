// tma.cu — host-side TMA descriptor encoding.  cuTensorMapEncodeTiled is a
// driver API; it is fetched through the runtime's entry-point query so that
// the library does not link against libcuda (and loads on hosts without a
// GPU driver).
#include <cudaTypedefs.h>

#include <mutex>

#include "kernels.h"
#include "tma.cuh"

namespace da {
namespace {

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

void fetch_encode() {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                       &q) == cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
}

}  // namespace

bool tma_available() {
  std::call_once(g_encode_once, fetch_encode);
  return g_encode != nullptr;
}

bool encode_tmap_bf16_4d(CUtensorMap* map, const da_t4& t, int B, int N, int H, int D,
                         int rows) {
  if (!tma_available()) return false;
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H),
                        static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(B)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(t.sh) * 2, static_cast<cuuint64_t>(t.sn) * 2,
                           static_cast<cuuint64_t>(t.sb) * 2};
  // a dimension of extent 1 may carry any stride; keep it a valid multiple of 16
  for (int i = 0; i < 3; ++i)
    if (strides[i] == 0) strides[i] = 16;
  cuuint32_t box[4] = {64, 1, static_cast<cuuint32_t>(rows), 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, t.ptr, dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool encode_tmap_f32_4d(CUtensorMap* map, void* ptr, int B, int N, int H, int D, int rows, int box_d) {
  if (!tma_available()) return false;
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H),
                        static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(B)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(D) * 4, static_cast<cuuint64_t>(H) * D * 4,
                           static_cast<cuuint64_t>(N) * H * D * 4};
  cuuint32_t box[4] = {static_cast<cuuint32_t>(box_d > 0 ? box_d : D), 1, static_cast<cuuint32_t>(rows), 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, ptr, dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool encode_tmap_f32_slots(CUtensorMap* map, void* ptr, int units, int slots, int rows, int D, int box_d) {
  if (!tma_available()) return false;
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(rows),
                        static_cast<cuuint64_t>(slots), static_cast<cuuint64_t>(units)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(D) * 4, static_cast<cuuint64_t>(rows) * D * 4,
                           static_cast<cuuint64_t>(slots) * rows * D * 4};
  cuuint32_t box[4] = {static_cast<cuuint32_t>(box_d > 0 ? box_d : D), static_cast<cuuint32_t>(rows), 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, ptr, dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace da
