// Decode-kernel instances of the fused step with rotary embedding for fp16 caches.
#include "decode_dispatch.cuh"

namespace da {

cudaError_t launch_decode_f16_rope(const DecodeParams& p, int head_dim, int group, int flavor, cudaStream_t stream,
                              const cudaLaunchAttribute* attr) {
  DA_DISPATCH(__half, true, launch_decode_t, p, stream, attr)
}

cudaError_t decode_info_f16_rope(int head_dim, int group, int flavor, DecodeKernelInfo* info) {
  DA_DISPATCH(__half, true, decode_info_t, info)
}

}  // namespace da
