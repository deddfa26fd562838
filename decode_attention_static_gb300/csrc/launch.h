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
  int cluster_max;              // largest cluster size that can be resident
  int active_clusters[17];      // clusters of each size (1..16) resident at once
  int tensor_scores;            // 1: the scores run on the tensor cores (K tiles by TMA tensor copies)
  int flavor;                   // the flavour this kernel is (kFlavor* of decode_kernel.cuh)
};

bool decode_supported(int head_dim, int group);
cudaError_t decode_kernel_info(int dtype, int head_dim, int group, int device, DecodeKernelInfo* info,
                               bool rope = false, int flavor = 0);
cudaError_t launch_decode(const DecodeParams& p, int dtype, int head_dim, int group, int flavor, cudaStream_t stream);
// Scratch bytes of one decode call with `splits` splits in clusters of
// `cluster`: none when one cluster serves a group; otherwise a fixed region
// of 32-bit arrival counters, then fp32 per-cluster partials
// acc [B, n_head, splits / cluster, D] and (m, l) [B, n_head, splits / cluster, 2].
size_t workspace_bytes_for(int B, int n_head, int splits, int cluster, int head_dim);
cudaError_t launch_append(void* k_cache, void* v_cache, const void* k_new, const void* v_new,
                          const int32_t* pos, int B, int n_kv_head, int head_dim, int capacity,
                          int32_t* err_flag, cudaStream_t stream);

// Per-dtype halves of launch_decode / decode_kernel_info (one translation
// unit each, compiled in parallel); `flavor` selects the flavour where an
// instance has several.
cudaError_t launch_decode_f16(const DecodeParams& p, int head_dim, int group, int flavor, cudaStream_t stream,
                              const cudaLaunchAttribute* attr);
cudaError_t launch_decode_bf16(const DecodeParams& p, int head_dim, int group, int flavor, cudaStream_t stream,
                               const cudaLaunchAttribute* attr);
cudaError_t decode_info_f16(int head_dim, int group, int flavor, DecodeKernelInfo* info);
cudaError_t decode_info_bf16(int head_dim, int group, int flavor, DecodeKernelInfo* info);
// The same for the instances of the fused step with rotary embedding.
cudaError_t launch_decode_f16_rope(const DecodeParams& p, int head_dim, int group, int flavor, cudaStream_t stream,
                                   const cudaLaunchAttribute* attr);
cudaError_t launch_decode_bf16_rope(const DecodeParams& p, int head_dim, int group, int flavor, cudaStream_t stream,
                                    const cudaLaunchAttribute* attr);
cudaError_t decode_info_f16_rope(int head_dim, int group, int flavor, DecodeKernelInfo* info);
cudaError_t decode_info_bf16_rope(int head_dim, int group, int flavor, DecodeKernelInfo* info);

}  // namespace da
