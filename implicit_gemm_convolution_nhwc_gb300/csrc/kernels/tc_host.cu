// Host helpers for the tensor-core kernels: tensor-map encoding through the
// driver entry point, and the device error word.
#include <cudaTypedefs.h>

#include <mutex>

#include "tc_common.cuh"

namespace cig {

// Bits set by kernels when a bounded wait gave up (see tc_common.cuh).
__device__ unsigned g_conv_device_errors = 0u;

namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    else
      cudaGetLastError();
  });
  return fn;
}

}  // namespace

bool encode_tmap(CUtensorMap* map, CUtensorMapDataType dtype, int rank, const void* base, const uint64_t* dims,
                 const uint64_t* strides_bytes, const uint32_t* box, CUtensorMapSwizzle swizzle,
                 const uint32_t* element_strides) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t d[5], st[4];
  cuuint32_t b[5], es[5];
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    b[i] = box[i];
    es[i] = element_strides ? element_strides[i] : 1;
    if (i + 1 < rank) st[i] = strides_bytes[i];
  }
  CUresult r = fn(map, dtype, (cuuint32_t)rank, const_cast<void*>(base), d, st, b, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

unsigned* device_error_word() {
  static unsigned* cached[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return nullptr;
  if (dev < 64 && cached[dev]) return cached[dev];
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_conv_device_errors) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  if (dev < 64) cached[dev] = static_cast<unsigned*>(p);
  return static_cast<unsigned*>(p);
}

}  // namespace cig

extern "C" conv_status conv_device_errors(uint32_t* flags, int32_t clear) {
  if (!flags) return CONV_ERR_INVALID_ARG;
  unsigned v = 0;
  if (cudaMemcpyFromSymbol(&v, cig::g_conv_device_errors, sizeof(v)) != cudaSuccess) {
    cudaGetLastError();
    return CONV_ERR_CUDA;
  }
  *flags = v;
  if (clear) {
    const unsigned zero = 0;
    if (cudaMemcpyToSymbol(cig::g_conv_device_errors, &zero, sizeof(zero)) != cudaSuccess) {
      cudaGetLastError();
      return CONV_ERR_CUDA;
    }
  }
  return CONV_OK;
}
