// Combine kernel (merge of the split-KV partial softmax states) and the
// in-place KV-cache append kernel.
#include "common.cuh"
#include "launch.h"

namespace da {

// out[b, h, :] = sum_s 2^(m_s - M) acc_s / sum_s 2^(m_s - M) l_s, M = max_s m_s,
// over the active splits of sequence b; rounded to the storage type. One warp
// per (b, h); lane i holds elements [i * D/32, (i + 1) * D/32).
template <typename T, int D>
__global__ void __launch_bounds__(128) combine_kernel(const DecodeParams p) {
  using S = Storage<T>;
  constexpr int E = D / 32;
  pdl_wait();
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int bh = blockIdx.x * 4 + warp;
  if (bh >= p.B * p.n_head) return;
  const int b = bh / p.n_head;
  int32_t err_bits = 0;
  const int L = sequence_length(p, b, &err_bits);
  if (L < 0) return;  // the decode kernel wrote NaN rows and the error bit
  const int nsplit = active_splits(L, split_chunk(L, p.splits, tile_rows(D)));
  if (nsplit <= 1) return;  // the decode kernel wrote out directly

  const float* ml = p.ws_ml + (int64_t)bh * p.splits * 2;
  float mm = -INFINITY;
  for (int s = lane; s < nsplit; s += 32) mm = fmaxf(mm, ml[2 * s]);
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) mm = fmaxf(mm, __shfl_xor_sync(0xffffffffu, mm, off));

  float ls = 0.f;
  float acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;
  const float* accs = p.ws_acc + (int64_t)bh * p.splits * D + lane * E;
  for (int s = 0; s < nsplit; ++s) {
    const float ms = ml[2 * s];
    const float f = (ms == -INFINITY) ? 0.f : fast_exp2(ms - mm);
    ls = fmaf(ml[2 * s + 1], f, ls);
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = fmaf(accs[(int64_t)s * D + e], f, acc[e]);
  }
  uint16_t* o = reinterpret_cast<uint16_t*>(p.out) + (int64_t)bh * D + lane * E;
#pragma unroll
  for (int e = 0; e < E; ++e) o[e] = S::round(acc[e] / ls);
}

// k_cache[b, g, pos[b], :] = k_new[b, g, :] (and V), 16 bytes per thread.
__global__ void __launch_bounds__(256) append_kernel(uint8_t* k_cache, uint8_t* v_cache, const uint8_t* k_new,
                                                     const uint8_t* v_new, const int32_t* pos, int B,
                                                     int n_kv_head, int row_vecs, int capacity,
                                                     int32_t* err_flag) {
  pdl_wait();
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

cudaError_t launch_combine(const DecodeParams& p, int dtype, int head_dim, cudaStream_t stream) {
  const int rows = p.B * p.n_head;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((rows + 3) / 4);
  cfg.blockDim = dim3(128);
  cfg.stream = stream;
  cudaLaunchAttribute attr = pdl_attribute();
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  if (dtype == 0) {
    if (head_dim == 128) return cudaLaunchKernelEx(&cfg, combine_kernel<__half, 128>, p);
    return cudaLaunchKernelEx(&cfg, combine_kernel<__half, 64>, p);
  }
  if (head_dim == 128) return cudaLaunchKernelEx(&cfg, combine_kernel<__nv_bfloat16, 128>, p);
  return cudaLaunchKernelEx(&cfg, combine_kernel<__nv_bfloat16, 64>, p);
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
