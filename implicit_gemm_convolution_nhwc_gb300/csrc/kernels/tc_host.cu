// Host helpers for the tensor-core kernels: tensor-map encoding through the
// driver entry point, and the device error word.
#include <cudaTypedefs.h>

#include <mutex>

#include "tc_common.cuh"
#include "../kernel_entry.h"

namespace cig {

// Bits set by kernels when a bounded wait gave up (see tc_common.cuh).
__device__ unsigned g_conv_device_errors = 0u;
// Result words of conv_selftest_wait_timeout.
__device__ unsigned g_selftest_out[2];

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

// Looked up on every call, not cached: after a device reset the module reloads
// in a new context and the word may live at another address.
unsigned* device_error_word() {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_conv_device_errors) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return static_cast<unsigned*>(p);
}

namespace {

// One CTA waits on an mbarrier that nothing ever arrives on, with the given
// limit: the wait gives up, records the timeout in the device error word and
// the kernel returns. out[0] = 1 when the wait gave up as it should.
__global__ void selftest_wait_timeout_kernel(unsigned long long limit_ns, unsigned* err, unsigned* out) {
  __shared__ uint64_t bar;
  __shared__ uint32_t abort_word;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_word = 0u;
    mbar_fence_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const bool ok = mbar_wait(&bar, 0u, &abort_word, err, limit_ns);
    out[0] = ok ? 0u : 1u;
    out[1] = abort_word;
  }
}

}  // namespace

}  // namespace cig

extern "C" conv_status conv_selftest_wait_timeout(uint64_t limit_ns, uint32_t* gave_up, void* stream) {
  if (!gave_up || limit_ns == 0 || limit_ns > 1000000000ull) return CONV_ERR_INVALID_ARG;  // at most 1 s
  unsigned* err = cig::device_error_word();
  if (!err) return CONV_ERR_CUDA;
  unsigned* out = nullptr;
  if (cudaGetSymbolAddress(reinterpret_cast<void**>(&out), cig::g_selftest_out) != cudaSuccess) {
    cudaGetLastError();
    return CONV_ERR_CUDA;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cig::selftest_wait_timeout_kernel<<<1, 32, 0, s>>>(limit_ns, err, out);
  if (cudaGetLastError() != cudaSuccess) return CONV_ERR_CUDA;
  unsigned host[2] = {0u, 0u};
  if (cudaMemcpyFromSymbolAsync(host, cig::g_selftest_out, sizeof(host), 0, cudaMemcpyDeviceToHost, s) !=
          cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return CONV_ERR_CUDA;
  *gave_up = host[0] == 1u && host[1] == 1u ? 1u : 0u;
  return CONV_OK;
}

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
