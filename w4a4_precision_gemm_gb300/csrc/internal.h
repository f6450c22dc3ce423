// internal.h - host-side helpers shared by the library's translation units.
#pragma once
#include <cuda_runtime.h>
#include <cstdint>
#include <cstddef>
#include <utility>

#include "../../include/lpq.h"

namespace lpq {

// Record a CUDA error for lpq_last_cuda_error() and map it to a status.
lpq_status record_cuda(cudaError_t e);
// Count one kernel launch (per host thread).
void count_launch(uint64_t n = 1);
// Device address of the library's error word (set up once per device).
uint32_t* error_word_ptr();
// Number of SMs of the current device (cached per device).
int sm_count();
// Check the result of a kernel launch (cudaGetLastError) and count it.
inline lpq_status after_launch() {
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return record_cuda(e);
  count_launch();
  return LPQ_OK;
}

// Launch a kernel with programmatic stream serialization (the kernel calls
// pdl_wait() before touching global memory), then check and count it.
template <typename... KArgs, typename... Args>
inline lpq_status launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                             int cluster_x, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  int n = 1;
  if (cluster_x > 1) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = static_cast<unsigned>(cluster_x);
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    n = 2;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
  if (e != cudaSuccess) return record_cuda(e);
  count_launch();
  return LPQ_OK;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace lpq

#define LPQ_CHECK_NULL(p) \
  do {                    \
    if ((p) == nullptr) return LPQ_ERR_NULL; \
  } while (0)
#define LPQ_CHECK_ALIGN(p) \
  do {                     \
    if (!lpq::aligned16(p)) return LPQ_ERR_ALIGN; \
  } while (0)
