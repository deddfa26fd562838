// Split-KV decode attention over the active prefix of a static KV cache.
//
// One CTA per (split s, KV head g, sequence b). It owns the rows
// [s * chunk, min((s + 1) * chunk, L)) of its sequence's K and V, where L is
// the active length and chunk an even share of L in whole tiles, so every
// byte of the active prefix is read exactly once and nothing beyond it. The
// CTA serves all G query heads of its KV head from that single read
// (grouped-query attention without expansion: fish-speech issue #1310,
// section 2; VoxCPM issue #395, section 4.1, enable_gqa).
//
// Data path: one producer lane streams K and V tiles with bulk TMA copies
// (cp.async.bulk, contiguous rows of the cache) into a kStages-deep ring of
// shared-memory stages guarded by full/empty mbarriers. Four consumer warps
// read the stages with 128-bit shared loads: a row of D elements is spread
// over D/8 lanes holding 8 elements each, and each lane keeps its slice of
// the G query vectors in registers, pre-multiplied by scale * log2(e).
// Scores are reduced across the lanes of a row with xor shuffles; every
// group of lanes keeps an fp32 online-softmax state (running max m, sum l,
// accumulator acc) in the base-2 domain (the max-subtracted fp32 softmax of
// Cuda-Compute-OSS issue #343, "Proposed implementation"). At the end the
// states of all lane groups and warps are merged; a sequence that needs a
// single split writes `out` directly, otherwise the CTA writes its partial
// (m, l, acc) for the combine kernel.
#pragma once

#include "common.cuh"

namespace da {

template <int D, int G>
struct DecodeShape {
  static constexpr int kRowBytes = 2 * D;
  static constexpr int kTileRows = kTileBytes / kRowBytes;          // 32 for D=128, 64 for D=64
  static constexpr int kLanesPerRow = D / 8;                        // 16 or 8
  static constexpr int kRowsPerStep = 32 / kLanesPerRow;            // rows a warp covers per step
  static constexpr int kRowsPerWarp = kTileRows / kConsumerWarps;   // rows of a tile per warp
  static constexpr int kSteps = kRowsPerWarp / kRowsPerStep;        // steps per tile per warp
  static constexpr int kStageBytes = 2 * kTileBytes;                // K tile then V tile
  static constexpr int kRingBytes = kStages * kStageBytes;
  static constexpr int kReduceFloats = kConsumerWarps * G * (D + 2);
  static constexpr int kSmemBytes = kRingBytes + kReduceFloats * 4 + 2 * kStages * 8 + 16;
  static_assert(kRowsPerWarp % kRowsPerStep == 0, "tile rows must split evenly over warps");
};

template <typename T, int D, int G>
__global__ void __launch_bounds__(kDecodeThreads) decode_split_kernel(const DecodeParams p) {
  using Shape = DecodeShape<D, G>;
  using S = Storage<T>;
  constexpr int LPR = Shape::kLanesPerRow;

  extern __shared__ __align__(128) uint8_t smem[];
  float* red = reinterpret_cast<float*>(smem + Shape::kRingBytes);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + Shape::kRingBytes + Shape::kReduceFloats * 4);
  uint64_t* empty = full + kStages;
  int* abort_flag = reinterpret_cast<int*>(empty + kStages);

  const int s = blockIdx.x;
  const int g_kv = blockIdx.y;
  const int b = blockIdx.z;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int H = p.n_head;

  pdl_trigger();
  pdl_wait();

  int32_t err_bits = 0;
  const int L = sequence_length(p, b, &err_bits);
  if (L < 0) {
    // Invalid input: split 0 writes NaN rows for the group's heads.
    if (s == 0) {
      for (int i = threadIdx.x; i < G * D; i += blockDim.x) {
        const int64_t o = ((int64_t)b * H + (int64_t)g_kv * G) * D + i;
        reinterpret_cast<uint16_t*>(p.out)[o] = S::kNaN;
      }
      if (threadIdx.x == 0 && p.err_flag) atomicOr(p.err_flag, err_bits);
    }
    return;
  }
  const int chunk = split_chunk(L, p.splits, Shape::kTileRows);
  const int nsplit = active_splits(L, chunk);
  if (s >= nsplit) return;
  const int r0 = s * chunk;
  const int r1 = min(L, r0 + chunk);
  const int ntiles = (r1 - r0 + Shape::kTileRows - 1) / Shape::kTileRows;
  const bool fused = p.k_new != nullptr;

  const int64_t kv_row0 = ((int64_t)b * p.n_kv_head + g_kv) * p.capacity;  // first row of this (b, g)
  const int64_t new_row = ((int64_t)b * p.n_kv_head + g_kv) * D;           // element offset into k_new

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kConsumerWarps);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kConsumerWarps) {
    // ---------------- producer warp ----------------
    if (fused && s == 0 && lane < D / 8) {
      // The new row goes into the cache; no CTA of this launch reads it back
      // from there (the CTA owning row L-1 takes it from k_new/v_new).
      const int64_t dst = (kv_row0 + (L - 1)) * Shape::kRowBytes + lane * 16;
      const int64_t src = new_row * 2 + lane * 16;
      *reinterpret_cast<uint4*>(p.k_cache_w + dst) = ld_global_nc_v4(p.k_new + src);
      *reinterpret_cast<uint4*>(p.v_cache_w + dst) = ld_global_nc_v4(p.v_new + src);
    }
    if (lane == 0) {
      const uint64_t policy = evict_first_policy();
      int issued = 0;
      for (int t = 0; t < ntiles; ++t) {
        const int stage = t % kStages;
        if (t >= kStages) {
          if (!mbar_wait(&empty[stage], ((t / kStages) & 1) ^ 1)) {
            atomicOr(abort_flag, 1);
            break;
          }
        }
        if (*reinterpret_cast<volatile int*>(abort_flag)) break;
        const int tr0 = r0 + t * Shape::kTileRows;
        const int rows = min(Shape::kTileRows, r1 - tr0);
        const bool new_last = fused && (tr0 + rows == L);
        const int cached = new_last ? rows - 1 : rows;
        uint8_t* kdst = smem + stage * Shape::kStageBytes;
        uint8_t* vdst = kdst + kTileBytes;
        mbar_arrive_expect_tx(&full[stage], 2u * rows * Shape::kRowBytes);
        if (cached > 0) {
          const int64_t off = (kv_row0 + tr0) * Shape::kRowBytes;
          bulk_load(kdst, p.k_cache + off, cached * Shape::kRowBytes, &full[stage], policy);
          bulk_load(vdst, p.v_cache + off, cached * Shape::kRowBytes, &full[stage], policy);
        }
        if (new_last) {
          const int64_t off = new_row * 2;
          bulk_load(kdst + cached * Shape::kRowBytes, p.k_new + off, Shape::kRowBytes, &full[stage], policy);
          bulk_load(vdst + cached * Shape::kRowBytes, p.v_new + off, Shape::kRowBytes, &full[stage], policy);
        }
        ++issued;
      }
      // After an abort, let copies already in flight land before the CTA
      // exits (bounded): the last tile issued to each stage.
      if (*reinterpret_cast<volatile int*>(abort_flag)) {
        for (int t = max(0, issued - kStages); t < issued; ++t) mbar_wait(&full[t % kStages], (t / kStages) & 1);
      }
    }
    __syncwarp();
    return;  // the producer warp takes no part in the epilogue
  }

  // ---------------- consumer warps ----------------
  const int c = lane % LPR;     // which 8-element slice of a row
  const int lrow = lane / LPR;  // which row of a step

  float qf[G][8];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    const int64_t qoff = (((int64_t)b * H + (int64_t)g_kv * G + g) * D + c * 8) * 2;
    float f[8];
    S::unpack(ld_global_nc_v4(p.q + qoff), f);
#pragma unroll
    for (int e = 0; e < 8; ++e) qf[g][e] = f[e] * p.qscale;
  }

  float m[G], l[G], acc[G][8];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    m[g] = -INFINITY;
    l[g] = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[g][e] = 0.f;
  }

  bool aborted = false;
  for (int t = 0; t < ntiles; ++t) {
    const int stage = t % kStages;
    const bool ok_wait = mbar_wait(&full[stage], (t / kStages) & 1);
    if (__any_sync(0xffffffffu, !ok_wait)) {
      aborted = true;
      break;
    }
    const uint8_t* kt = smem + stage * Shape::kStageBytes;
    const uint8_t* vt = kt + kTileBytes;
    const int rows = min(Shape::kTileRows, r1 - (r0 + t * Shape::kTileRows));

    float sc[Shape::kSteps][G];
#pragma unroll
    for (int u = 0; u < Shape::kSteps; ++u) {
      const int r = warp * Shape::kRowsPerWarp + u * Shape::kRowsPerStep + lrow;
      const bool valid = r < rows;
      uint4 kv = make_uint4(0u, 0u, 0u, 0u);
      if (valid) kv = ld_shared_v4(kt + r * Shape::kRowBytes + c * 16);
      float kf[8];
      S::unpack(kv, kf);
      float part[G];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float a0 = qf[g][0] * kf[0];
        float a1 = qf[g][1] * kf[1];
        a0 = fmaf(qf[g][2], kf[2], a0);
        a1 = fmaf(qf[g][3], kf[3], a1);
        a0 = fmaf(qf[g][4], kf[4], a0);
        a1 = fmaf(qf[g][5], kf[5], a1);
        a0 = fmaf(qf[g][6], kf[6], a0);
        a1 = fmaf(qf[g][7], kf[7], a1);
        part[g] = a0 + a1;
      }
#pragma unroll
      for (int off = LPR / 2; off >= 1; off >>= 1) {
#pragma unroll
        for (int g = 0; g < G; ++g) part[g] += __shfl_xor_sync(0xffffffffu, part[g], off);
      }
#pragma unroll
      for (int g = 0; g < G; ++g) sc[u][g] = valid ? part[g] : -INFINITY;
    }

    float pw[Shape::kSteps][G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      float mx = sc[0][g];
#pragma unroll
      for (int u = 1; u < Shape::kSteps; ++u) mx = fmaxf(mx, sc[u][g]);
      const float mnew = fmaxf(m[g], mx);
      const bool none = (mnew == -INFINITY);  // no visible row yet in this lane group
      const float alpha = none ? 1.f : fast_exp2(m[g] - mnew);
      float add = 0.f;
#pragma unroll
      for (int u = 0; u < Shape::kSteps; ++u) {
        pw[u][g] = none ? 0.f : fast_exp2(sc[u][g] - mnew);
        add += pw[u][g];
      }
      l[g] = fmaf(l[g], alpha, add);
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[g][e] *= alpha;
      m[g] = mnew;
    }

#pragma unroll
    for (int u = 0; u < Shape::kSteps; ++u) {
      const int r = warp * Shape::kRowsPerWarp + u * Shape::kRowsPerStep + lrow;
      uint4 vv = make_uint4(0u, 0u, 0u, 0u);
      if (r < rows) vv = ld_shared_v4(vt + r * Shape::kRowBytes + c * 16);
      float vf[8];
      S::unpack(vv, vf);
#pragma unroll
      for (int g = 0; g < G; ++g) {
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[g][e] = fmaf(pw[u][g], vf[e], acc[g][e]);
      }
    }

    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[stage]);
  }
  if (aborted) atomicOr(abort_flag, 1);

  // Merge the lane groups of the warp that hold the same slice c.
#pragma unroll
  for (int off = LPR; off < 32; off <<= 1) {
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float mo = __shfl_xor_sync(0xffffffffu, m[g], off);
      const float lo = __shfl_xor_sync(0xffffffffu, l[g], off);
      const float mm = fmaxf(m[g], mo);
      const float fa = (m[g] == -INFINITY) ? 0.f : fast_exp2(m[g] - mm);
      const float fb = (mo == -INFINITY) ? 0.f : fast_exp2(mo - mm);
      l[g] = l[g] * fa + lo * fb;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float ao = __shfl_xor_sync(0xffffffffu, acc[g][e], off);
        acc[g][e] = acc[g][e] * fa + ao * fb;
      }
      m[g] = mm;
    }
  }

  // Per-warp states to shared memory: red[warp][g][0..D) = acc, [D] = m, [D+1] = l.
  if (lrow == 0) {
#pragma unroll
    for (int g = 0; g < G; ++g) {
      float* dst = red + (warp * G + g) * (D + 2);
#pragma unroll
      for (int e = 0; e < 8; ++e) dst[c * 8 + e] = acc[g][e];
      if (c == 0) {
        dst[D] = m[g];
        dst[D + 1] = l[g];
      }
    }
  }
  asm volatile("bar.sync 1, %0;" ::"n"(kConsumerThreads) : "memory");

  const bool failed = *reinterpret_cast<volatile int*>(abort_flag) != 0;
  if (failed && threadIdx.x == 0 && p.err_flag) atomicOr(p.err_flag, kErrTimeout);

  for (int i = threadIdx.x; i < G * D; i += kConsumerThreads) {
    const int g = i / D;
    const int d = i % D;
    float mm = -INFINITY;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) mm = fmaxf(mm, red[(w * G + g) * (D + 2) + D]);
    float ls = 0.f, as = 0.f;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) {
      const float* src = red + (w * G + g) * (D + 2);
      const float mw = src[D];
      const float f = (mw == -INFINITY) ? 0.f : fast_exp2(mw - mm);
      ls = fmaf(src[D + 1], f, ls);
      as = fmaf(src[d], f, as);
    }
    const int h = g_kv * G + g;
    if (nsplit == 1) {
      const int64_t o = ((int64_t)b * H + h) * D + d;
      reinterpret_cast<uint16_t*>(p.out)[o] = failed ? S::kNaN : S::round(as / ls);
    } else {
      const int64_t base = ((int64_t)b * H + h) * p.splits + s;
      p.ws_acc[base * D + d] = failed ? __int_as_float(0x7fc00000) : as;
      if (d == 0) {
        p.ws_ml[base * 2] = failed ? __int_as_float(0x7fc00000) : mm;
        p.ws_ml[base * 2 + 1] = ls;
      }
    }
  }
}

}  // namespace da
