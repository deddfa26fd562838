// Host-side launch interface between the C ABI layer and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace da {

// Dynamic shared memory and resident CTAs per SM of one decode-kernel
// instance on `device` (the shared-memory opt-in is applied on first use).
struct DecodeKernelInfo {
  int smem_bytes;
  int ctas_per_sm;
};

bool decode_supported(int head_dim, int group);
cudaError_t decode_kernel_info(int dtype, int head_dim, int group, int device, DecodeKernelInfo* info);
cudaError_t launch_decode(const DecodeParams& p, int dtype, int head_dim, int group, cudaStream_t stream);
cudaError_t launch_combine(const DecodeParams& p, int dtype, int head_dim, cudaStream_t stream);
cudaError_t launch_append(void* k_cache, void* v_cache, const void* k_new, const void* v_new,
                          const int32_t* pos, int B, int n_kv_head, int head_dim, int capacity,
                          int32_t* err_flag, cudaStream_t stream);

// Per-dtype halves of launch_decode / decode_kernel_info (one translation
// unit each, compiled in parallel).
cudaError_t launch_decode_f16(const DecodeParams& p, int head_dim, int group, cudaStream_t stream,
                              const cudaLaunchAttribute* attr);
cudaError_t launch_decode_bf16(const DecodeParams& p, int head_dim, int group, cudaStream_t stream,
                               const cudaLaunchAttribute* attr);
cudaError_t decode_info_f16(int head_dim, int group, DecodeKernelInfo* info);
cudaError_t decode_info_bf16(int head_dim, int group, DecodeKernelInfo* info);

}  // namespace da
