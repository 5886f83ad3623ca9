// tma_host.cu -- host-side encoding of TMA tensor maps through the driver entry point
// (obtained from the runtime, so the library does not link libcuda directly).
#include <cudaTypedefs.h>

#include <mutex>

#include "tma.cuh"

namespace ssm {

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

bool encode_tmap_3d(CUtensorMap* map, const void* base, int esize, uint64_t d0, uint64_t d1,
                    uint64_t d2, uint64_t stride1, uint64_t stride2, uint32_t b0, uint32_t b1,
                    uint32_t b2, int swizzle) {
  auto fn = encode_fn();
  if (!fn) return false;
  const CUtensorMapDataType dt =
      esize == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {stride1 * (uint64_t)esize, stride2 * (uint64_t)esize};  // bytes
  cuuint32_t box[3] = {b0, b1, b2};
  cuuint32_t estr[3] = {1, 1, 1};
  const CUtensorMapSwizzle sw = swizzle == 32    ? CU_TENSOR_MAP_SWIZZLE_32B
                               : swizzle == 64  ? CU_TENSOR_MAP_SWIZZLE_64B
                               : swizzle == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                                : CU_TENSOR_MAP_SWIZZLE_NONE;
  if (swizzle && (sw == CU_TENSOR_MAP_SWIZZLE_NONE || b0 * (uint32_t)esize > (uint32_t)swizzle))
    return false;
  const CUresult r = fn(map, dt, 3, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace ssm
