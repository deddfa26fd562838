// Instantiation and launch of the decode kernel for one storage type over
// head_dim in {64, 128} and group size in {1, 2, 4, 8}; RP selects the
// instances of the fused step with rotary embedding, `flavor` one of the
// InstanceConfig flavours (distinct kernels for four or more heads per KV
// head only).
#pragma once

#include "decode_kernel.cuh"
#include "launch.h"

namespace da {

template <int D, int G, int F>
using ConfiguredShape = DecodeShape<D, G, DecodeConfig<D, G>::kWarps, DecodeConfig<D, G>::kPerLane,
                                    InstanceConfig<D, G, F>::kStages, InstanceConfig<D, G, F>::kTensorScores>;

template <typename T, int D, int G, bool RP, int F>
constexpr auto configured_kernel() {
  using C = InstanceConfig<D, G, F>;
  return decode_split_kernel<T, D, G, DecodeConfig<D, G>::kWarps, DecodeConfig<D, G>::kPerLane, C::kStages, RP,
                             C::kTensorScores, C::kMinBlocks>;
}

template <typename T, int D, int G, bool RP, int F>
cudaError_t launch_decode_t(const DecodeParams& p, cudaStream_t stream, const cudaLaunchAttribute* pdl) {
  using Shape = ConfiguredShape<D, G, F>;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.splits, p.n_kv_head, p.B);
  cfg.blockDim = dim3(Shape::kThreads);
  cfg.dynamicSmemBytes = Shape::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attrs[2];
  int n = 0;
  if (pdl) attrs[n++] = *pdl;
  if (p.cluster > 1) {
    attrs[n].id = cudaLaunchAttributeClusterDimension;
    attrs[n].val.clusterDim.x = p.cluster;
    attrs[n].val.clusterDim.y = 1;
    attrs[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attrs;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, configured_kernel<T, D, G, RP, F>(), p);
}

// Applies the shared-memory and cluster-size opt-ins for the current device
// and reports the occupancy of one instance: resident CTAs per SM and the
// largest cluster (16, else 8) of which at least one fits.
template <typename T, int D, int G, bool RP, int F>
cudaError_t decode_info_t(DecodeKernelInfo* info) {
  using Shape = ConfiguredShape<D, G, F>;
  const int smem = Shape::kSmemBytes;
  auto* fn = configured_kernel<T, D, G, RP, F>();
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e != cudaSuccess) return e;
  int n = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, Shape::kThreads, smem);
  if (e != cudaSuccess) return e;
  info->smem_bytes = smem;
  info->ctas_per_sm = n;
  info->tensor_scores = InstanceConfig<D, G, F>::kTensorScores ? 1 : 0;
  info->flavor = InstanceConfig<D, G, F>::kFlavor;
  info->cluster_max = 1;
  for (int cs = 16; cs >= 1; --cs) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(cs, 1, 1);
    cfg.blockDim = dim3(Shape::kThreads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = cs;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, fn, &cfg) != cudaSuccess) {
      clusters = 0;
      (void)cudaGetLastError();  // a refused size is not an error of the call
    }
    info->active_clusters[cs] = clusters;
    if (clusters > 0 && info->cluster_max == 1) info->cluster_max = cs;
  }
  return cudaSuccess;
}

#define DA_DISPATCH_FLAVOR(T, RP, D, G, FN, ...)                   \
  switch (flavor) {                                                \
    case kFlavorPair: return FN<T, D, G, RP, kFlavorPair>(__VA_ARGS__);        \
    case kFlavorCudaCores: return FN<T, D, G, RP, kFlavorCudaCores>(__VA_ARGS__); \
    default: return FN<T, D, G, RP, kFlavorWide>(__VA_ARGS__);                 \
  }

#define DA_DISPATCH_GROUP(T, RP, D, FN, ...)                          \
  switch (group) {                                                    \
    case 1: return FN<T, D, 1, RP, kFlavorWide>(__VA_ARGS__);         \
    case 2: return FN<T, D, 2, RP, kFlavorWide>(__VA_ARGS__);         \
    case 4: DA_DISPATCH_FLAVOR(T, RP, D, 4, FN, __VA_ARGS__)          \
    case 8: DA_DISPATCH_FLAVOR(T, RP, D, 8, FN, __VA_ARGS__)          \
    default: return cudaErrorInvalidValue;                            \
  }

#define DA_DISPATCH(T, RP, FN, ...)                                         \
  if (head_dim == 128) { DA_DISPATCH_GROUP(T, RP, 128, FN, __VA_ARGS__) }   \
  if (head_dim == 64) { DA_DISPATCH_GROUP(T, RP, 64, FN, __VA_ARGS__) }     \
  return cudaErrorInvalidValue;

}  // namespace da
