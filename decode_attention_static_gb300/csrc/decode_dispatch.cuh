// Instantiation and launch of the decode kernel for one storage type over
// head_dim in {64, 128} and group size in {1, 2, 4, 8}.
#pragma once

#include "decode_kernel.cuh"
#include "launch.h"

namespace da {

template <typename T, int D, int G>
cudaError_t launch_decode_t(const DecodeParams& p, cudaStream_t stream, const cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.splits, p.n_kv_head, p.B);
  cfg.blockDim = dim3(kDecodeThreads);
  cfg.dynamicSmemBytes = DecodeShape<D, G>::kSmemBytes;
  cfg.stream = stream;
  cfg.attrs = const_cast<cudaLaunchAttribute*>(attr);
  cfg.numAttrs = attr ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, decode_split_kernel<T, D, G>, p);
}

// Applies the shared-memory opt-in for the current device and reports the
// occupancy of one instance.
template <typename T, int D, int G>
cudaError_t decode_info_t(DecodeKernelInfo* info) {
  const int smem = DecodeShape<D, G>::kSmemBytes;
  cudaError_t e = cudaFuncSetAttribute(decode_split_kernel<T, D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  int n = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_split_kernel<T, D, G>, kDecodeThreads, smem);
  if (e != cudaSuccess) return e;
  info->smem_bytes = smem;
  info->ctas_per_sm = n;
  return cudaSuccess;
}

#define DA_DISPATCH_GROUP(T, D, FN, ...)                 \
  switch (group) {                                       \
    case 1: return FN<T, D, 1>(__VA_ARGS__);             \
    case 2: return FN<T, D, 2>(__VA_ARGS__);             \
    case 4: return FN<T, D, 4>(__VA_ARGS__);             \
    case 8: return FN<T, D, 8>(__VA_ARGS__);             \
    default: return cudaErrorInvalidValue;               \
  }

#define DA_DISPATCH(T, FN, ...)                                         \
  if (head_dim == 128) { DA_DISPATCH_GROUP(T, 128, FN, __VA_ARGS__) }   \
  if (head_dim == 64) { DA_DISPATCH_GROUP(T, 64, FN, __VA_ARGS__) }     \
  return cudaErrorInvalidValue;

}  // namespace da
