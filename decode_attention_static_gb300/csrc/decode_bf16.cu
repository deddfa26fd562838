// Decode-kernel instances for bf16 caches.
#include "decode_dispatch.cuh"

namespace da {

cudaError_t launch_decode_bf16(const DecodeParams& p, int head_dim, int group, int flavor, cudaStream_t stream,
                              const cudaLaunchAttribute* attr) {
  DA_DISPATCH(__nv_bfloat16, false, launch_decode_t, p, stream, attr)
}

cudaError_t decode_info_bf16(int head_dim, int group, int flavor, DecodeKernelInfo* info) {
  DA_DISPATCH(__nv_bfloat16, false, decode_info_t, info)
}

}  // namespace da
