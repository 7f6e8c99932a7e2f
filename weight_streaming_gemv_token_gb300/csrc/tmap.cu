// Tiled TMA descriptors (tensor maps) for the persistent decode kernel's
// weight boxes and the tensor-core GEMM's operand tiles, encoded on the host
// through the runtime's driver entry point (no link against the driver
// library).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "common.h"

namespace wsg {

namespace {

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

}  // namespace

dec_status encode_map_2d(void* out, const void* base, long long rows, long long cols, int elem, int box_cols,
                         int box_rows, bool swizzle128, std::string* err) {
  static_assert(sizeof(CUtensorMap) == 128, "tensor map size");
  auto enc = tensor_map_encoder();
  if (!enc) return fail(err, DEC_ECUDA, "cuTensorMapEncodeTiled is not available");
  if (elem != 2 && elem != 4) return fail(err, DEC_EINVAL, "tensor map: element size %d", elem);
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * elem};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  const CUresult r =
      enc(static_cast<CUtensorMap*>(out), elem == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
          2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
          swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(err, DEC_EINVAL, "cuTensorMapEncodeTiled failed (%d) for a %lld x %lld matrix, box %d x %d",
                static_cast<int>(r), rows, cols, box_rows, box_cols);
  return DEC_OK;
}

}  // namespace wsg
