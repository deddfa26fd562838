// C ABI of the decode-attention library: argument validation, the split
// plan, and the launches on the caller's stream. Nothing here allocates or
// synchronises.
#include <stdint.h>

#include <algorithm>
#include <atomic>
#include <mutex>

#include "decode_attn.h"
#include "launch.h"

namespace da {

namespace {

constexpr int kMaxDevices = 64;
constexpr float kLog2e = 1.4426950408889634f;

struct DeviceState {
  std::atomic<int> sms{0};
  std::atomic<int> ready[4][2][4];  // [dtype + 2 * rotary][head_dim 64/128][log2 group]
  DecodeKernelInfo info[4][2][4];
};

DeviceState g_devices[kMaxDevices];
std::mutex g_mutex;

int group_index(int group) { return group == 1 ? 0 : group == 2 ? 1 : group == 4 ? 2 : 3; }

cudaError_t current_device(int* device) {
  cudaError_t e = cudaGetDevice(device);
  if (e != cudaSuccess) return e;
  if (*device < 0 || *device >= kMaxDevices) return cudaErrorInvalidDevice;
  return cudaSuccess;
}

cudaError_t device_sms(int device, int* sms) {
  int n = g_devices[device].sms.load(std::memory_order_acquire);
  if (n == 0) {
    cudaError_t e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, device);
    if (e != cudaSuccess) return e;
    g_devices[device].sms.store(n, std::memory_order_release);
  }
  *sms = n;
  return cudaSuccess;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_sizes(int B, int n_head, int n_kv_head, int head_dim, int capacity, int dtype) {
  if (dtype != DA_F16 && dtype != DA_BF16) return DA_ERR_DTYPE;
  if (B < 0 || n_head < 1 || n_kv_head < 1 || head_dim < 1 || capacity < 1) return DA_ERR_SHAPE;
  if (n_head % n_kv_head != 0) return DA_ERR_SHAPE;
  if (B > 65535 || n_kv_head > 65535) return DA_ERR_SHAPE;  // grid z / y limits
  if (!decode_supported(head_dim, n_head / n_kv_head)) return DA_ERR_UNSUPPORTED;
  return DA_OK;
}

}  // namespace

size_t workspace_bytes_for(int B, int n_head, int splits, int cluster, int head_dim) {
  const int clusters = splits / (cluster > 0 ? cluster : 1);
  if (clusters <= 1) return 0;
  const size_t rows = (size_t)B * n_head * clusters;
  return kCounterBytes + rows * (head_dim + 2) * sizeof(float);
}

bool decode_supported(int head_dim, int group) {
  return (head_dim == 64 || head_dim == 128) && (group == 1 || group == 2 || group == 4 || group == 8);
}

cudaError_t decode_kernel_info(int dtype, int head_dim, int group, int device, DecodeKernelInfo* info, bool rope) {
  const int ki = dtype + (rope ? 2 : 0);
  const int di = head_dim == 128 ? 1 : 0;
  const int gi = group_index(group);
  DeviceState& st = g_devices[device];
  if (st.ready[ki][di][gi].load(std::memory_order_acquire)) {
    *info = st.info[ki][di][gi];
    return cudaSuccess;
  }
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!st.ready[ki][di][gi].load(std::memory_order_acquire)) {
    DecodeKernelInfo k = {};
    cudaError_t e;
    if (rope) {
      e = dtype == DA_F16 ? decode_info_f16_rope(head_dim, group, &k) : decode_info_bf16_rope(head_dim, group, &k);
    } else {
      e = dtype == DA_F16 ? decode_info_f16(head_dim, group, &k) : decode_info_bf16(head_dim, group, &k);
    }
    if (e != cudaSuccess) return e;
    if (k.ctas_per_sm < 1) return cudaErrorInvalidConfiguration;
    st.info[ki][di][gi] = k;
    st.ready[ki][di][gi].store(1, std::memory_order_release);
  }
  *info = st.info[ki][di][gi];
  return cudaSuccess;
}

cudaError_t launch_decode(const DecodeParams& p, int dtype, int head_dim, int group, cudaStream_t stream) {
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  if (p.rope_cos)
    return dtype == DA_F16 ? launch_decode_f16_rope(p, head_dim, group, stream, &attr)
                           : launch_decode_bf16_rope(p, head_dim, group, stream, &attr);
  return dtype == DA_F16 ? launch_decode_f16(p, head_dim, group, stream, &attr)
                         : launch_decode_bf16(p, head_dim, group, stream, &attr);
}

namespace {

// Profiling hook events of this host thread (see da_set_timing_events).
thread_local cudaEvent_t t_event_before = nullptr;
thread_local cudaEvent_t t_event_after = nullptr;
// Failure-detection test hook (da_test_skip_slot) of this host thread.
thread_local int t_skip_slot = -1;
// Ordering promise (da_set_prefix_ready) of this host thread.
thread_local int t_prefix_ready = 0;

cudaError_t record_event(cudaEvent_t ev, cudaStream_t st) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(st, &cs);
  if (e != cudaSuccess) return e;
  if (cs == cudaStreamCaptureStatusActive) return cudaEventRecordWithFlags(ev, st, cudaEventRecordExternal);
  return cudaEventRecord(ev, st);
}

// Splits and cluster size for the current device: plan + occupancy of the instance.
int plan_for_device(int dtype, int B, int n_kv_head, int head_dim, int group, int bound, int* splits,
                    int* cluster) {
  int device = 0, sms = 0;
  if (current_device(&device) != cudaSuccess) return DA_ERR_CUDA;
  if (device_sms(device, &sms) != cudaSuccess) return DA_ERR_CUDA;
  // One plan serves the plain and the rotary instances (so that a workspace
  // sized for one fits the other): take the smaller occupancy of the two.
  // Querying both also applies both instances' launch attributes.
  DecodeKernelInfo info, info_rope;
  if (decode_kernel_info(dtype, head_dim, group, device, &info) != cudaSuccess) return DA_ERR_CUDA;
  if (decode_kernel_info(dtype, head_dim, group, device, &info_rope, true) != cudaSuccess) return DA_ERR_CUDA;
  info.ctas_per_sm = std::min(info.ctas_per_sm, info_rope.ctas_per_sm);
  info.cluster_max = std::min(info.cluster_max, info_rope.cluster_max);
  for (int c = 0; c <= kMaxClusterSize; ++c)
    info.active_clusters[c] = std::min(info.active_clusters[c], info_rope.active_clusters[c]);
  // the largest cluster size of which one cluster per group is co-resident
  const int64_t units = (int64_t)B * n_kv_head;
  int fit = 1;
  for (int c = std::min(info.cluster_max, kMaxClusterSize); c >= 2; --c) {
    if (info.active_clusters[c] >= units) {
      fit = c;
      break;
    }
  }
  int cs = 1;
  const int s = decode_attn_plan_splits(B, n_kv_head, head_dim, bound, sms, info.ctas_per_sm, fit, &cs);
  if (s < 1) return s;
  *splits = s;
  *cluster = cs;
  return DA_OK;
}

// One decode launch over B sequences. `lens` has lens_period entries (B, or
// a divisor of B when several layers of one batch share their lengths:
// sequence b reads lens[b % lens_period]).
int decode_common(const void* q, const void* k_cache, const void* v_cache, void* k_cache_w, void* v_cache_w,
                  const void* k_new, const void* v_new, const int32_t* lens, int lens_are_positions, int B,
                  int n_head, int n_kv_head, int head_dim, int capacity, float scale, void* out, void* workspace,
                  size_t workspace_bytes, int max_kv_len_hint, int dtype, int32_t* err_flag, void* stream,
                  const float* rope_cos = nullptr, const float* rope_sin = nullptr, int rope_rows = 0,
                  int lens_period = 0) {
  int rc = check_sizes(B, n_head, n_kv_head, head_dim, capacity, dtype);
  if (rc != DA_OK) return rc;
  if (B == 0) return DA_OK;
  if (!q || !k_cache || !v_cache || !lens || !out) return DA_ERR_NULL;
  if (lens_are_positions && (!k_new || !v_new)) return DA_ERR_NULL;
  if ((rope_cos != nullptr) != (rope_sin != nullptr)) return DA_ERR_NULL;
  if (rope_cos) {
    if (!lens_are_positions) return DA_ERR_NULL;  // rotary embedding comes with the fused step only
    if (rope_rows < capacity) return DA_ERR_SHAPE;
    if (!aligned16(rope_cos) || !aligned16(rope_sin)) return DA_ERR_ALIGN;
  }
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) ||
      (k_new && !aligned16(k_new)) || (v_new && !aligned16(v_new)))
    return DA_ERR_ALIGN;
  const int group = n_head / n_kv_head;
  const int bound = max_kv_len_hint > 0 ? std::min(max_kv_len_hint, capacity) : capacity;
  int splits = 1, cluster = 1;
  rc = plan_for_device(dtype, B, n_kv_head, head_dim, group, bound, &splits, &cluster);
  if (rc != DA_OK) return rc;
  const size_t need = workspace_bytes_for(B, n_head, splits, cluster, head_dim);
  if (need > 0) {
    if (!workspace || workspace_bytes < need) return DA_ERR_WORKSPACE;
    if (!aligned16(workspace)) return DA_ERR_ALIGN;
  }

  DecodeParams p = {};
  p.q = static_cast<const uint8_t*>(q);
  p.k_cache = static_cast<const uint8_t*>(k_cache);
  p.v_cache = static_cast<const uint8_t*>(v_cache);
  p.k_cache_w = static_cast<uint8_t*>(k_cache_w);
  p.v_cache_w = static_cast<uint8_t*>(v_cache_w);
  p.k_new = static_cast<const uint8_t*>(k_new);
  p.v_new = static_cast<const uint8_t*>(v_new);
  p.lens = lens;
  p.lens_are_positions = lens_are_positions;
  p.lens_period = lens_period > 0 ? lens_period : B;
  p.B = B;
  p.n_head = n_head;
  p.n_kv_head = n_kv_head;
  p.capacity = capacity;
  p.splits = splits;
  p.cluster = cluster;
  p.rope_cos = rope_cos;
  p.rope_sin = rope_sin;
  p.rope_rows = rope_rows;
  p.len_hint = bound;
  p.skip_slot = t_skip_slot;
  // One length (one sequence, or the layers of one sequence) with an explicit
  // bound: the bound is normally that length, so the kernel issues its first
  // tiles before reading the length.
  p.speculate = (p.lens_period == 1 && max_kv_len_hint > 0) ? 1 : 0;
  p.prefix_ready = (p.speculate && t_prefix_ready) ? 1 : 0;
  p.qscale = scale * kLog2e;
  p.out = static_cast<uint8_t*>(out);
  if (need > 0) {
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    p.counters = reinterpret_cast<unsigned int*>(ws);
    p.ws_acc = reinterpret_cast<float*>(ws + kCounterBytes);
    p.ws_ml = p.ws_acc + (size_t)B * n_head * (splits / cluster) * head_dim;
  }
  p.err_flag = err_flag;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (t_event_before && record_event(t_event_before, st) != cudaSuccess) return DA_ERR_CUDA;
  if (launch_decode(p, dtype, head_dim, group, st) != cudaSuccess) return DA_ERR_CUDA;
  if (t_event_after && record_event(t_event_after, st) != cudaSuccess) return DA_ERR_CUDA;
  return DA_OK;
}

}  // namespace
}  // namespace da

extern "C" {

const char* da_status_string(int status) {
  switch (status) {
    case DA_OK: return "ok";
    case DA_ERR_NULL: return "a required pointer is NULL";
    case DA_ERR_SHAPE: return "a size is out of range or inconsistent";
    case DA_ERR_UNSUPPORTED: return "unsupported head_dim or group size (head_dim in {64,128}, group in {1,2,4,8})";
    case DA_ERR_WORKSPACE: return "workspace is NULL or smaller than decode_attn_workspace_size()";
    case DA_ERR_CUDA: return "a CUDA runtime call or kernel launch failed";
    case DA_ERR_ALIGN: return "a pointer is not 16-byte aligned";
    case DA_ERR_DTYPE: return "unknown dtype code";
    default: return "unknown status";
  }
}

int da_version(void) { return 100; }

int decode_attn_plan_splits(int B, int n_kv_head, int head_dim, int max_kv_len, int num_sms, int ctas_per_sm,
                            int cluster_max, int* cluster_size) {
  if (B < 1 || n_kv_head < 1 || max_kv_len < 1 || num_sms < 1 || ctas_per_sm < 1 || cluster_max < 1)
    return DA_ERR_SHAPE;
  if (head_dim != 64 && head_dim != 128) return DA_ERR_UNSUPPORTED;
  const int64_t units = (int64_t)B * n_kv_head;
  const int64_t slots = (int64_t)num_sms * ctas_per_sm;  // CTAs resident at once
  const int rows = da::tile_rows(head_dim);
  const int64_t tiles = ((int64_t)max_kv_len + rows - 1) / rows;
  // Splits that fit one wave, at most one per tile. In a batch the lengths
  // below the bound are unknown on the host; sizing for two waves keeps the
  // long sequences' CTAs short while the short ones' extra splits exit at once.
  const int64_t waves = B > 1 ? 2 : 1;
  int64_t want = std::min<int64_t>({waves * slots / units, tiles, (int64_t)da::kMaxSplits});
  if (units > da::kMaxCounterGroups) want = 1;
  int64_t cs = 1;
  if (want >= 2) {
    const int64_t fit = std::min<int64_t>(cluster_max, da::kMaxClusterSize);
    if (B == 1 && fit >= 2 && units * fit >= num_sms && tiles >= 2 * fit) {
      // A long prefix of one sequence: one cluster of `fit` CTAs per group
      // already covers every SM, and merges on chip instead of through L2.
      cs = fit;
    } else {
      // A short prefix is latency-bound: one cluster per group, at most one
      // CTA per SM, about ctas_per_sm tiles per CTA. Too short for two
      // CTAs: no split at all.
      const int64_t c = std::min<int64_t>(
          {fit, std::max<int64_t>(1, num_sms / units), (tiles + ctas_per_sm - 1) / ctas_per_sm});
      if (tiles <= da::kClusterTilesPerSplit * std::max<int64_t>(c, 1)) cs = c >= 2 ? c : 0;
    }
    if (cs > 1) {
      want = cs;
    } else if (cs == 0) {
      want = 1;
      cs = 1;
    }
  } else {
    want = 1;
  }
  if (cluster_size) *cluster_size = (int)cs;
  return (int)want;
}

size_t decode_attn_workspace_size(int B, int n_head, int n_kv_head, int head_dim, int capacity) {
  if (da::check_sizes(B, n_head, n_kv_head, head_dim, capacity, DA_F16) != DA_OK) return (size_t)-1;
  if (B == 0) return 0;
  // The plan depends on the length bound: take the largest need over the
  // bounds of up to 4 * 16 tiles (where the short-prefix plans live) and
  // the capacity (beyond those, flat splits only grow with the bound).
  size_t most = 0;
  const int rows = da::tile_rows(head_dim);
  for (int dtype = DA_F16; dtype <= DA_BF16; ++dtype) {
    for (int t = 1; t <= 4 * da::kMaxClusterSize + 1; ++t) {
      const int bound = t * rows < capacity ? t * rows : capacity;
      int splits = 1, cluster = 1;
      if (da::plan_for_device(dtype, B, n_kv_head, head_dim, n_head / n_kv_head, bound, &splits, &cluster) !=
          DA_OK)
        return (size_t)-1;
      most = std::max(most, da::workspace_bytes_for(B, n_head, splits, cluster, head_dim));
      if (bound == capacity) break;
    }
    int splits = 1, cluster = 1;
    if (da::plan_for_device(dtype, B, n_kv_head, head_dim, n_head / n_kv_head, capacity, &splits, &cluster) !=
        DA_OK)
      return (size_t)-1;
    most = std::max(most, da::workspace_bytes_for(B, n_head, splits, cluster, head_dim));
  }
  return most;
}

int decode_attn_workspace_init(void* workspace, size_t workspace_bytes, void* stream) {
  if (!workspace) return workspace_bytes == 0 ? DA_OK : DA_ERR_NULL;
  if (cudaMemsetAsync(workspace, 0, workspace_bytes, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return DA_ERR_CUDA;
  return DA_OK;
}

int decode_attn_splits_for(int B, int n_head, int n_kv_head, int head_dim, int capacity, int max_kv_len_hint,
                           int dtype, int* cluster_size) {
  int rc = da::check_sizes(B, n_head, n_kv_head, head_dim, capacity, dtype);
  if (rc != DA_OK) return rc;
  int splits = 1, cluster = 1;
  if (B > 0) {
    const int bound = max_kv_len_hint > 0 ? std::min(max_kv_len_hint, capacity) : capacity;
    rc = da::plan_for_device(dtype, B, n_kv_head, head_dim, n_head / n_kv_head, bound, &splits, &cluster);
    if (rc != DA_OK) return rc;
  }
  if (cluster_size) *cluster_size = cluster;
  return splits;
}

int decode_attn_shard_heads(int n_head, int n_kv_head, int world, int rank, int* kv_head0, int* n_kv_local,
                            int* head0, int* n_head_local) {
  if (n_head < 1 || n_kv_head < 1 || n_head % n_kv_head != 0 || world < 1 || rank < 0 || rank >= world)
    return DA_ERR_SHAPE;
  if (!kv_head0 || !n_kv_local || !head0 || !n_head_local) return DA_ERR_NULL;
  const int group = n_head / n_kv_head;
  const int base = n_kv_head / world, extra = n_kv_head % world;
  const int first = rank * base + std::min(rank, extra);
  const int count = base + (rank < extra ? 1 : 0);
  *kv_head0 = first;
  *n_kv_local = count;
  *head0 = first * group;
  *n_head_local = count * group;
  return DA_OK;
}

int da_test_skip_slot(int slot) {
  da::t_skip_slot = slot < 0 ? -1 : slot;
  return DA_OK;
}

int da_set_prefix_ready(int on) {
  da::t_prefix_ready = on ? 1 : 0;
  return DA_OK;
}

int da_set_timing_events(void* event_before, void* event_after) {
  const bool on = event_before && event_after;
  da::t_event_before = on ? static_cast<cudaEvent_t>(event_before) : nullptr;
  da::t_event_after = on ? static_cast<cudaEvent_t>(event_after) : nullptr;
  return DA_OK;
}

int kvcache_append(void* k_cache, void* v_cache, const void* k_new, const void* v_new, const int32_t* position_ids,
                   int B, int n_kv_head, int head_dim, int capacity, int dtype, int32_t* err_flag, void* stream) {
  if (dtype != DA_F16 && dtype != DA_BF16) return DA_ERR_DTYPE;
  if (B < 0 || n_kv_head < 1 || capacity < 1 || head_dim < 8 || head_dim % 8 != 0) return DA_ERR_SHAPE;
  if (B == 0) return DA_OK;
  if (!k_cache || !v_cache || !k_new || !v_new || !position_ids) return DA_ERR_NULL;
  if (!da::aligned16(k_cache) || !da::aligned16(v_cache) || !da::aligned16(k_new) || !da::aligned16(v_new))
    return DA_ERR_ALIGN;
  if (da::launch_append(k_cache, v_cache, k_new, v_new, position_ids, B, n_kv_head, head_dim, capacity, err_flag,
                        static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return DA_ERR_CUDA;
  return DA_OK;
}

int decode_attn_fwd(const void* q, const void* k_cache, const void* v_cache, const int32_t* kv_len, int B, int n_head,
                    int n_kv_head, int head_dim, int capacity, float scale, void* out, void* workspace,
                    size_t workspace_bytes, int max_kv_len_hint, int dtype, int32_t* err_flag, void* stream) {
  return da::decode_common(q, k_cache, v_cache, nullptr, nullptr, nullptr, nullptr, kv_len, 0, B, n_head, n_kv_head,
                           head_dim, capacity, scale, out, workspace, workspace_bytes, max_kv_len_hint, dtype,
                           err_flag, stream);
}

int decode_step_fwd(const void* q, void* k_cache, void* v_cache, const void* k_new, const void* v_new,
                    const int32_t* position_ids, int B, int n_head, int n_kv_head, int head_dim, int capacity,
                    float scale, void* out, void* workspace, size_t workspace_bytes, int max_kv_len_hint, int dtype,
                    int32_t* err_flag, void* stream) {
  return da::decode_common(q, k_cache, v_cache, k_cache, v_cache, k_new, v_new, position_ids, 1, B, n_head,
                           n_kv_head, head_dim, capacity, scale, out, workspace, workspace_bytes, max_kv_len_hint,
                           dtype, err_flag, stream);
}

int decode_step_rope_fwd(const void* q, void* k_cache, void* v_cache, const void* k_new, const void* v_new,
                         const float* rope_cos, const float* rope_sin, int rope_rows, const int32_t* position_ids,
                         int B, int n_head, int n_kv_head, int head_dim, int capacity, float scale, void* out,
                         void* workspace, size_t workspace_bytes, int max_kv_len_hint, int dtype, int32_t* err_flag,
                         void* stream) {
  if (B > 0 && (!rope_cos || !rope_sin)) return DA_ERR_NULL;
  return da::decode_common(q, k_cache, v_cache, k_cache, v_cache, k_new, v_new, position_ids, 1, B, n_head,
                           n_kv_head, head_dim, capacity, scale, out, workspace, workspace_bytes, max_kv_len_hint,
                           dtype, err_flag, stream, rope_cos, rope_sin, rope_rows);
}

int decode_step_layers_fwd(const void* q, void* k_cache, void* v_cache, const void* k_new, const void* v_new,
                           const int32_t* position_ids, int layers, int B, int n_head, int n_kv_head, int head_dim,
                           int capacity, float scale, void* out, void* workspace, size_t workspace_bytes,
                           int max_kv_len_hint, int dtype, int32_t* err_flag, void* stream) {
  if (layers < 0) return DA_ERR_SHAPE;
  if (layers == 0 || B == 0) return DA_OK;
  if ((int64_t)layers * B > 65535) return DA_ERR_SHAPE;
  // [layers, B, ...] stacks are [layers * B, ...] batches whose sequence
  // l * B + b has the length of sequence b: every layer in one launch.
  return da::decode_common(q, k_cache, v_cache, k_cache, v_cache, k_new, v_new, position_ids, 1, layers * B, n_head,
                           n_kv_head, head_dim, capacity, scale, out, workspace, workspace_bytes, max_kv_len_hint,
                           dtype, err_flag, stream, nullptr, nullptr, 0, B);
}

}  // extern "C"
