// In-place KV-cache append kernel.
#include "common.cuh"
#include "launch.h"

namespace da {

// k_cache[b, g, pos[b], :] = k_new[b, g, :] (and V), 16 bytes per thread.
__global__ void __launch_bounds__(256) append_kernel(uint8_t* k_cache, uint8_t* v_cache, const uint8_t* k_new,
                                                     const uint8_t* v_new, const int32_t* pos, int B,
                                                     int n_kv_head, int row_vecs, int capacity,
                                                     int32_t* err_flag) {
  pdl_wait();
  pdl_trigger();  // the next grid may start its prologue while the rows are copied
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t total = (int64_t)B * n_kv_head * row_vecs;
  if (i >= total) return;
  const int c = (int)(i % row_vecs);
  const int64_t bg = i / row_vecs;
  const int b = (int)(bg / n_kv_head);
  const int p = pos[b];
  if (p < 0 || p >= capacity) {
    if (c == 0 && bg % n_kv_head == 0 && err_flag) atomicOr(err_flag, kErrPosition);
    return;
  }
  const int64_t src = (bg * row_vecs + c) * 16;
  const int64_t dst = ((bg * capacity + p) * row_vecs + c) * 16;
  *reinterpret_cast<uint4*>(k_cache + dst) = ld_global_nc_v4(k_new + src);
  *reinterpret_cast<uint4*>(v_cache + dst) = ld_global_nc_v4(v_new + src);
}

static cudaLaunchAttribute pdl_attribute() {
  cudaLaunchAttribute a;
  a.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  a.val.programmaticStreamSerializationAllowed = 1;
  return a;
}

cudaError_t launch_append(void* k_cache, void* v_cache, const void* k_new, const void* v_new,
                          const int32_t* pos, int B, int n_kv_head, int head_dim, int capacity,
                          int32_t* err_flag, cudaStream_t stream) {
  const int row_vecs = head_dim / 8;
  const int64_t total = (int64_t)B * n_kv_head * row_vecs;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((total + 255) / 256));
  cfg.blockDim = dim3(256);
  cfg.stream = stream;
  cudaLaunchAttribute attr = pdl_attribute();
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, append_kernel, static_cast<uint8_t*>(k_cache), static_cast<uint8_t*>(v_cache),
                            static_cast<const uint8_t*>(k_new), static_cast<const uint8_t*>(v_new), pos, B,
                            n_kv_head, row_vecs, capacity, err_flag);
}

}  // namespace da
