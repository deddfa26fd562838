// C ABI of the decode-attention library: argument validation, the split
// plan, and the launches on the caller's stream. Nothing here allocates or
// synchronises.
#include <cudaTypedefs.h>
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
  std::atomic<int> ready[4][2][4][3];  // [dtype + 2 * rotary][head_dim 64/128][log2 group][flavour]
  DecodeKernelInfo info[4][2][4][3];
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

cudaError_t decode_kernel_info(int dtype, int head_dim, int group, int device, DecodeKernelInfo* info, bool rope,
                               int flavor) {
  const int ki = dtype + (rope ? 2 : 0);
  const int di = head_dim == 128 ? 1 : 0;
  const int gi = group_index(group);
  const int ti = flavor >= 0 && flavor < 3 ? flavor : 0;
  DeviceState& st = g_devices[device];
  if (st.ready[ki][di][gi][ti].load(std::memory_order_acquire)) {
    *info = st.info[ki][di][gi][ti];
    return cudaSuccess;
  }
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!st.ready[ki][di][gi][ti].load(std::memory_order_acquire)) {
    DecodeKernelInfo k = {};
    cudaError_t e;
    if (rope) {
      e = dtype == DA_F16 ? decode_info_f16_rope(head_dim, group, ti, &k)
                          : decode_info_bf16_rope(head_dim, group, ti, &k);
    } else {
      e = dtype == DA_F16 ? decode_info_f16(head_dim, group, ti, &k) : decode_info_bf16(head_dim, group, ti, &k);
    }
    if (e != cudaSuccess) return e;
    if (k.ctas_per_sm < 1) return cudaErrorInvalidConfiguration;
    st.info[ki][di][gi][ti] = k;
    st.ready[ki][di][gi][ti].store(1, std::memory_order_release);
  }
  *info = st.info[ki][di][gi][ti];
  return cudaSuccess;
}

cudaError_t launch_decode(const DecodeParams& p, int dtype, int head_dim, int group, int flavor,
                          cudaStream_t stream) {
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  if (p.rope_cos)
    return dtype == DA_F16 ? launch_decode_f16_rope(p, head_dim, group, flavor, stream, &attr)
                           : launch_decode_bf16_rope(p, head_dim, group, flavor, stream, &attr);
  return dtype == DA_F16 ? launch_decode_f16(p, head_dim, group, flavor, stream, &attr)
                         : launch_decode_bf16(p, head_dim, group, flavor, stream, &attr);
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

// cuTensorMapEncodeTiled of the driver, looked up once (null if unavailable).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = []() -> PFN_cuTensorMapEncodeTiled_v12000 {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult found = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &found) !=
            cudaSuccess ||
        found != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }();
  return fn;
}

static_assert(sizeof(TensorMap) == sizeof(CUtensorMap), "TensorMap holds a CUtensorMap");

// The two K-cache tensor maps of the tensor-core instances: the cache as
// [groups][capacity][head_dim] elements, boxes of 64 columns by one tile's
// rows and by 8 rows, 128-byte swizzle, zero fill past the capacity.
bool encode_k_maps(DecodeParams* p, const void* k_cache, int dtype, int64_t groups, int capacity, int head_dim) {
  const PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)head_dim, (cuuint64_t)capacity, (cuuint64_t)groups};
  const cuuint64_t strides[2] = {(cuuint64_t)head_dim * 2, (cuuint64_t)capacity * head_dim * 2};
  const cuuint32_t box_tile[3] = {64, (cuuint32_t)tile_rows(head_dim), 1};
  const cuuint32_t box_rows8[3] = {64, 8, 1};
  const cuuint32_t unit[3] = {1, 1, 1};
  const CUtensorMapDataType type = dtype == DA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  void* base = const_cast<void*>(k_cache);
  if (enc(reinterpret_cast<CUtensorMap*>(&p->k_tiles), type, 3, base, dims, strides, box_tile, unit,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  return enc(reinterpret_cast<CUtensorMap*>(&p->k_rows8), type, 3, base, dims, strides, box_rows8, unit,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// CTAs that stream at most this many tiles each run the CUDA-core flavour of
// the instances with four or more heads per KV head: its per-tile path is
// shorter (no tensor-memory round trip), which wins until the tensor-core
// flavour's higher streaming rate pays (measured, 32 / 8 heads, one
// sequence, µs per call CUDA-core / tensor-core: kv 1024 and 2048, 2 and 3
// tiles per CTA, 5.30 / 6.14 and 6.30 / 6.43; kv 4096, 12288, 16384 and
// 32768, 6, 11, 14 and 27 tiles, 8.22 / 7.90, 13.97 / 13.54, 16.55 / 15.86
// and 26.45 / 25.25).
constexpr int64_t kCudaCoreChunkTiles = 4;

// Splits and cluster size for the current device: plan + occupancy of the
// instance. *flavor (if given) gets the flavour of the instance the call
// launches (rotary or not): the two-CTAs-per-SM one when the plan is one CTA
// per group and the groups fill more than one wave of the one-per-SM kernel
// (fewer waves), the CUDA-core one when each CTA streams few tiles, else the
// default; *tensor_scores whether that kernel runs its scores on the tensor
// cores (its K tiles then need tensor maps).
int plan_for_device(int dtype, int B, int n_kv_head, int head_dim, int group, int bound, int* splits,
                    int* cluster, bool rope = false, bool* tensor_scores = nullptr, int* flavor = nullptr) {
  int device = 0, sms = 0;
  if (current_device(&device) != cudaSuccess) return DA_ERR_CUDA;
  if (device_sms(device, &sms) != cudaSuccess) return DA_ERR_CUDA;
  // One plan serves the plain and the rotary instances (so that a workspace
  // sized for one fits the other): take the smaller occupancy of the two.
  // Querying both also applies both instances' launch attributes.
  DecodeKernelInfo info, info_rope;
  if (decode_kernel_info(dtype, head_dim, group, device, &info) != cudaSuccess) return DA_ERR_CUDA;
  if (decode_kernel_info(dtype, head_dim, group, device, &info_rope, true) != cudaSuccess) return DA_ERR_CUDA;
  const bool default_tc = (rope ? info_rope.tensor_scores : info.tensor_scores) != 0;
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
  int f = kFlavorWide;
  if (default_tc) {
    if (s == 1 && units > (int64_t)sms * info.ctas_per_sm) {
      // The occupancy query reports one CTA per SM for the pair flavour as
      // well, but two run at once (measured: the 288-group S2-Pro layers call
      // takes 20.5 us instead of 24.6 at kv 634); a plan of one CTA per group
      // never depends on CTAs being co-resident.
      DecodeKernelInfo pair;
      if (decode_kernel_info(dtype, head_dim, group, device, &pair, rope, kFlavorPair) != cudaSuccess)
        return DA_ERR_CUDA;
      if (pair.flavor == kFlavorPair) f = kFlavorPair;
    } else {
      const int64_t rows = tile_rows(head_dim);
      const int64_t tiles = ((int64_t)bound + rows - 1) / rows;
      if ((tiles + s - 1) / s <= kCudaCoreChunkTiles) {
        // Only where the same clusters fit that kernel too.
        DecodeKernelInfo cc;
        if (decode_kernel_info(dtype, head_dim, group, device, &cc, rope, kFlavorCudaCores) != cudaSuccess)
          return DA_ERR_CUDA;
        if (cc.flavor == kFlavorCudaCores && (cs == 1 || cc.active_clusters[cs] >= units)) f = kFlavorCudaCores;
      }
    }
  }
  if (flavor) *flavor = f;
  if (tensor_scores) *tensor_scores = default_tc && f != kFlavorCudaCores;
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
  bool tensor_scores = false;
  int flavor = 0;
  rc = plan_for_device(dtype, B, n_kv_head, head_dim, group, bound, &splits, &cluster, rope_cos != nullptr,
                       &tensor_scores, &flavor);
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
  if (tensor_scores && !encode_k_maps(&p, k_cache, dtype, (int64_t)B * n_kv_head, capacity, head_dim))
    return DA_ERR_CUDA;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (t_event_before && record_event(t_event_before, st) != cudaSuccess) return DA_ERR_CUDA;
  if (launch_decode(p, dtype, head_dim, group, flavor, st) != cudaSuccess) return DA_ERR_CUDA;
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
      // A CTA alone on its SM streams about twice the tiles in the time its
      // cluster merge saves over the workspace merge (measured with four
      // query heads per KV head: clusters of 12 beat 19 flat splits up to
      // 96 tiles), so the bound doubles at one CTA per SM.
      const int64_t per_split = ctas_per_sm == 1 ? 2 * da::kClusterTilesPerSplit : da::kClusterTilesPerSplit;
      if (tiles <= per_split * std::max<int64_t>(c, 1)) cs = c >= 2 ? c : 0;
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

int decode_attn_kernel_for(int B, int n_head, int n_kv_head, int head_dim, int capacity, int max_kv_len_hint,
                           int dtype, int rotary) {
  int rc = da::check_sizes(B, n_head, n_kv_head, head_dim, capacity, dtype);
  if (rc != DA_OK) return rc;
  if (B == 0) return DA_KERNEL_CUDA_CORES;
  const int bound = max_kv_len_hint > 0 ? std::min(max_kv_len_hint, capacity) : capacity;
  int splits = 1, cluster = 1, flavor = 0;
  bool tensor_scores = false;
  rc = da::plan_for_device(dtype, B, n_kv_head, head_dim, n_head / n_kv_head, bound, &splits, &cluster, rotary != 0,
                           &tensor_scores, &flavor);
  if (rc != DA_OK) return rc;
  if (!tensor_scores) return DA_KERNEL_CUDA_CORES;
  return flavor == da::kFlavorPair ? DA_KERNEL_TENSOR_CORES_PAIRED : DA_KERNEL_TENSOR_CORES;
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
