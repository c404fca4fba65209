// Host helpers shared by the kernel launchers: per-device one-time opt-in to
// large dynamic shared memory, and the SM count of the current device.
#pragma once
#include <cuda_runtime.h>

#include <cmath>
#include <mutex>
#include <set>
#include <utility>

namespace m2 {

// 1 / s when that is exact (s > 0 a power of two with a normal inverse), else
// 0: kernels then multiply instead of divide and get the identical quotient.
inline float exact_inverse(float s) {
  int e = 0;
  if (!(s > 0.f) || std::frexp(s, &e) != 0.5f) return 0.f;
  const float inv = 1.0f / s;
  return (std::isnormal(inv) && inv * s == 1.0f) ? inv : 0.f;
}

// cudaFuncSetAttribute(MaxDynamicSharedMemorySize) once per (device, kernel).
inline cudaError_t ensure_smem_optin(const void* func, int bytes) {
  static std::mutex mu;
  static std::set<std::pair<int, const void*>> done;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  if (done.count({dev, func})) return cudaSuccess;
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done.insert({dev, func});
  return e;
}

inline int device_sm_count() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 148;
}

}  // namespace m2

namespace m2 {

// Launch with programmatic dependent launch allowed: the kernel may start
// while the previous kernel on the stream is finishing.  Every kernel of this
// library calls pdl_wait() before its first global-memory access, so it only
// touches data after the previous kernel has completed and flushed.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace m2
