// wq_tensor_map.h -- host-side lookup of the driver's tiled tensor-map
// encoder (cuTensorMapEncodeTiled), shared by the kernels that stage data
// with TMA.  The runtime hands out the driver entry point, so the library
// does not link libcuda directly.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

namespace wq {

typedef CUresult (*TensorMapEncodeFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                      const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                      const cuuint32_t*, CUtensorMapInterleave,
                                      CUtensorMapSwizzle, CUtensorMapL2promotion,
                                      CUtensorMapFloatOOBfill);

// The encoder, or nullptr when the driver does not provide it.
inline TensorMapEncodeFn tensor_map_encoder() {
  static TensorMapEncodeFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<TensorMapEncodeFn>(f);
  });
  return fn;
}

}  // namespace wq
