// decode_attn_fwd_static_scratch: decode attention for callers that cannot
// allocate device memory. The split partials live in a library-owned
// file-scope device array instead of a caller workspace.
#include <stdint.h>

#include <mutex>

#include "decode_attn.h"
#include "launch.h"

namespace {

constexpr int kMaxDevices = 64;

// Scratch for the split partials of every call on a device. In host code this
// name is only a stand-in for the symbol: its device address comes from
// cudaGetSymbolAddress below, and only that address is passed to kernels.
static __device__ __align__(256) unsigned char g_static_scratch[DA_STATIC_SCRATCH_BYTES];

void* g_scratch_ptr[kMaxDevices] = {};
std::mutex g_scratch_mutex;

// Device address of g_static_scratch on the current device, looked up once
// per device with that device current. The look-up is refused while `stream`
// is being captured (it may load the library's device code, which a capture
// does not allow). Returns DA_OK or DA_ERR_CUDA.
int scratch_address(void** out, cudaStream_t stream) {
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess || device < 0 || device >= kMaxDevices) return DA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (!g_scratch_ptr[device]) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone) return DA_ERR_CUDA;
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_static_scratch) != cudaSuccess || !ptr) return DA_ERR_CUDA;
    g_scratch_ptr[device] = ptr;
  }
  *out = g_scratch_ptr[device];
  return DA_OK;
}

}  // namespace

extern "C" int decode_attn_fwd_static_scratch(const void* q, const void* k_cache, const void* v_cache,
                                              const int32_t* kv_len, int B, int n_head, int n_kv_head,
                                              int head_dim, int capacity, float scale, void* out,
                                              int max_kv_len_hint, int dtype, int32_t* err_flag,
                                              void* stream) {
  // The split count this call will use decides how much scratch it needs
  // (none when it is 1).
  int cluster = 1;
  const int splits =
      decode_attn_splits_for(B, n_head, n_kv_head, head_dim, capacity, max_kv_len_hint, dtype, &cluster);
  if (splits < 0) return splits;
  const size_t need = da::workspace_bytes_for(B, n_head, splits, cluster, head_dim);
  if (need > DA_STATIC_SCRATCH_BYTES) return DA_ERR_SHAPE;
  void* scratch = nullptr;
  if (need > 0) {
    const int rc = scratch_address(&scratch, static_cast<cudaStream_t>(stream));
    if (rc != DA_OK) return rc;
    // This call's arrival counters (one per sequence and KV head, at the start
    // of the array) start at zero whatever an earlier call left there: an
    // overlapping or interrupted call cannot spoil the calls after it.
    if (cudaMemsetAsync(scratch, 0, (size_t)B * n_kv_head * sizeof(unsigned int), static_cast<cudaStream_t>(stream)) !=
        cudaSuccess)
      return DA_ERR_CUDA;
  }
  return decode_attn_fwd(q, k_cache, v_cache, kv_len, B, n_head, n_kv_head, head_dim, capacity, scale, out, scratch,
                         need > 0 ? (size_t)DA_STATIC_SCRATCH_BYTES : 0, max_kv_len_hint, dtype, err_flag, stream);
}
