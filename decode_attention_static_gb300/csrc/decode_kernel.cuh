// Split-KV decode attention over the active prefix of a static KV cache.
//
// One CTA per (split s, KV head g, sequence b). It owns the rows
// [s * chunk, min((s + 1) * chunk, L)) of its sequence's K and V, where L is
// the active length and chunk an even share of L in whole tiles, so every
// byte of the active prefix is read exactly once (the tensor-core variant
// below copies a partial last K tile in 8-row boxes: at most 7 rows past the
// prefix, never weighted). The
// CTA serves all G query heads of its KV head from that single read
// (grouped-query attention without expansion: fish-speech issue #1310,
// section 2; VoxCPM issue #395, section 4.1, enable_gqa).
//
// Data path: one producer lane streams K and V tiles with bulk TMA copies
// (cp.async.bulk, contiguous rows of the cache) into a kStages-deep ring of
// shared-memory stages guarded by full/empty mbarriers. CW consumer warps
// read the stages with 128-bit shared loads: a row of D elements is spread
// over D/8 lanes holding one 16-byte vector each, and each lane keeps its
// slice of the G query vectors in registers (raw 16-bit; scores are scaled
// by scale * log2(e) after the dot product). Scores are reduced across the
// lanes of a row with xor shuffles; every group of lanes keeps an fp32 online-softmax
// state (running max m, sum l, accumulator acc) in the base-2 domain (the
// max-subtracted fp32 softmax of Cuda-Compute-OSS issue #343, "Proposed
// implementation"). The fused step reads the attended row L - 1 from k_new
// and v_new and writes it into the cache; with rotary embedding (RP) q and
// that key row are rotated first (VoxCPM issue #395, section 4.1).
//
// Tensor-core scores (TC, four or more query heads per KV head): the scores
// of a K tile are one tcgen05.mma chain (S^T = K q^T, fp32 in tensor memory)
// issued by an extra warp, K arriving by TMA tensor copies in the swizzled
// operand layout; two groups of four consumer warps take the tiles in turn,
// read the scores from tensor memory and accumulate the weighted V on the
// CUDA cores (see the TC consumer below).
//
// Merge of the splits. The splits of one (b, g) group are launched as
// thread-block clusters of `cluster` CTAs. Each CTA folds its warps' states
// into one (m, l, acc), the thread folding an output storing it straight
// into the rank that merges it (distributed shared memory); after one cluster
// barrier every CTA merges its slice of the G x D outputs over all CTAs of
// its cluster from its own shared memory. A group served by one
// cluster writes `out` there and then; a group served by several clusters
// writes one partial per cluster to the workspace, and the last CTA to
// arrive (a per-group counter) merges those partials into `out`.
#pragma once

#include "common.cuh"

namespace da {

// Largest cluster the merge supports (the hardware limit for non-portable
// cluster sizes).
constexpr int kMaxCluster = 16;

template <int D, int G, int CW, int DPL, int NS, bool TC = false>
struct DecodeShape {
  static constexpr int kStages = NS;                                 // depth of the shared-memory ring
  static constexpr int kConsumerWarps = CW;
  static constexpr int kConsumerThreads = CW * 32;
  // + the producer warp (+ the warp issuing the tensor-core scores)
  static constexpr int kThreads = kConsumerThreads + (TC ? 64 : 32);
  // Warps that release a ring stage once they are done with it: every
  // consumer warp, or with tensor-core scores the four warps of the group
  // that consumed the tile.
  static constexpr int kEmptyArrivals = TC ? 4 : CW;
  static constexpr int kRowBytes = 2 * D;
  static constexpr int kTileRows = kTileBytes / kRowBytes;           // 64 for D=128, 128 for D=64
  static constexpr int kVecs = DPL / 8;                              // 16-byte vectors per lane per row
  static constexpr int kLanesPerRow = D / DPL;
  static constexpr int kRowsPerStep = 32 / kLanesPerRow;             // rows a warp covers per step
  static constexpr int kRowsPerWarp = kTileRows / CW;                // rows of a tile per warp
  static constexpr int kSteps = kRowsPerWarp / kRowsPerStep;         // steps per tile per warp
  // When a quarter-warp (8 lanes, one shared-memory wavefront) spans two rows,
  // odd rows visit their two vectors in the opposite order so that the eight
  // 16-byte loads of a wavefront hit distinct banks.
  static constexpr bool kSwap = kVecs == 2 && kLanesPerRow * 16 < 128;
  static constexpr int kStageBytes = 2 * kTileBytes;                 // K tile then V tile
  static constexpr int kRingBytes = kStages * kStageBytes;
  static constexpr int kMergeFloats = CW * G * (D + 2);              // per-warp states (in the idle ring)
  // Receive area of the cluster merge: (m, l) of up to kMaxCluster ranks and
  // their shares of this CTA's slice of the outputs (at most G*D + 15 floats).
  static constexpr int kRecvFloats = kMaxCluster * 2 * G + G * D + kMaxCluster;
  // Tensor-core scores: the q operand (16 rows of D elements as 64-column
  // halves of 128-byte swizzled rows, 1024-byte aligned), the weights of the
  // two consumer groups' current tiles [2][kTileRows][G], and small
  // per-group arrays: tile maxima [2][4][G], weight sums
  // [2][4][G], running maxima [2][G], the new row's scores [G] and the
  // tensor-memory base address.
  static constexpr int kQOffset = (kRingBytes + kRecvFloats * 4 + 1023) / 1024 * 1024;
  static constexpr int kQBytes = 16 * 2 * D;
  static constexpr int kPOffset = kQOffset + kQBytes;
  static constexpr int kAuxOffset = kPOffset + 2 * kTileRows * G * 4;
  static constexpr int kAuxFloats = 8 * G + 8 * G + 2 * G + G + 1;
  // Layout after the ring: receive area, (tensor-core extras,) then the
  // mbarriers (full, empty, merge, and with tensor-core scores two
  // score-ready and two score-free) and flags.
  static constexpr int kBarOffset =
      TC ? (kAuxOffset + kAuxFloats * 4 + 7) / 8 * 8 : (kRingBytes + kRecvFloats * 4 + 7) / 8 * 8;
  static constexpr int kBars = 2 * kStages + 1 + (TC ? 4 : 0);
  // (+ 1024 bytes of slack for aligning the ring to the 128-byte swizzle atoms)
  static constexpr int kSmemBytes = kBarOffset + kBars * 8 + 16 + (TC ? 1024 : 0);
  // Tensor-core weighted sum of V: a row is read by D/8 threads (16 bytes
  // each); the 128 threads of a group form 128 / (D/8) row groups of
  // kTileRows / (128 / (D/8)) rows each.
  static constexpr int kVThreadsPerRow = D / 8;
  static constexpr int kRowGroups = 128 / kVThreadsPerRow;
  static constexpr int kRowsPerThread = kTileRows / kRowGroups;
  static constexpr int kPerThread = (G * D + kConsumerThreads - 1) / kConsumerThreads;
  static_assert(DPL == 8 || DPL == 16, "8 or 16 elements per lane");
  static_assert(G <= kLanesPerRow, "the score reduction gives each head its own lanes");
  static_assert(kRowsPerWarp % kRowsPerStep == 0 && kSteps >= 1, "tile rows must split evenly over warps");
  static_assert(kMergeFloats * 4 <= kRingBytes, "the per-warp states fit the ring");
  static_assert(kBarOffset % 8 == 0, "mbarriers need 8-byte alignment");
  static_assert(kVecs == 1, "one 16-byte vector per lane (rotary embedding pairs lanes c and c ^ D/16)");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory of one CTA");
  static_assert(!TC || (CW == 8 && G <= 16 && D % 64 == 0 && kTileRows % 32 == 0 && kTileRows <= 128),
                "tensor-core scores: two groups of four consumer warps, at most 16 heads, whole 64-column halves");
  static_assert(!TC || kRowsPerThread * kRowGroups == kTileRows, "V rows split evenly over the row groups");
  static_assert(!TC || 2 * kRowGroups * G * D * 4 <= kRingBytes, "the group partials fit the ring");
};

// Consumer warps, elements per lane and ring depth of each instance. With
// one or two query heads per KV head, scores take one mixed-precision FMA
// per element and head on the raw 16-bit q and K (packed fp32x2 products on
// converted K measured no faster), and a 3-stage ring of 32 KiB stages
// (96 KiB) per CTA covers the loaded HBM latency and leaves room for two
// CTAs per SM: thread-block clusters of up to 13 CTAs then fit once per
// group for 16 groups, and the next launch's CTAs can be resident while this
// one drains. Eight elements per lane (one 16-byte vector of a row) give each
// warp more independent rows per tile than sixteen, and fewer registers for
// the G query slices. With four or more the scores run on the tensor cores
// and the CTA takes an SM to itself with a 5-stage ring (4 and 6 stages
// measured slower on long single-sequence prefixes and the layers call).
template <int D, int G>
struct DecodeConfig {
  static constexpr int kWarps = 8;
  static constexpr int kPerLane = 8;
  static constexpr int kStages = G >= 4 ? 5 : 3;
  // Four or more query heads per KV head: the scores on the tensor cores
  // (the CUDA-core score loop is instruction-bound there: about 560
  // warp-instructions per consumer warp per 64-row tile, 48 GB/s per CTA;
  // with tensor-core scores one CTA streams 70 GB/s, and a 5-stage ring
  // keeps more bytes in flight behind the longer per-tile path).
  static constexpr bool kTensorScores = G >= 4;
};

// Flavours of an instance with four or more query heads per KV head. The
// default runs the scores on the tensor cores with one CTA per SM and a
// 5-stage ring. kFlavorPair is the same with a 3-stage ring and a register
// bound of two CTAs per SM (four heads per KV head only): a launch whose
// groups already fill the GPU one CTA per group (the layers call) then runs
// in one wave instead of two. kFlavorCudaCores keeps the scores on the CUDA
// cores (4-stage ring): it reaches the first tile's output sooner, which
// wins when each CTA streams only a few tiles. Instances with fewer heads per
// KV head ignore the flavour (the same kernel). (kFlavor*: common.cuh.)
template <int D, int G, int F>
struct InstanceConfig {
  static constexpr bool kTensorScores = DecodeConfig<D, G>::kTensorScores && F != kFlavorCudaCores;
  static constexpr bool kTwoPerSm = F == kFlavorPair && kTensorScores && G <= 4;
  static constexpr int kStages = kTwoPerSm ? 3 : kTensorScores ? DecodeConfig<D, G>::kStages : G >= 4 ? 4 : 3;
  static constexpr int kMinBlocks = kTwoPerSm ? 2 : 1;
  // The flavour this instance actually is (the kernel shared by flavours that coincide).
  static constexpr int kFlavor = kTwoPerSm ? kFlavorPair : (G >= 4 && !kTensorScores) ? kFlavorCudaCores : kFlavorWide;
};

// Merge the per-warp (m, l, acc) states kept in shared memory for head g,
// element d: returns the common max, the rescaled sum and accumulator.
template <int D, int G, int CW>
__device__ __forceinline__ void merge_warps(const float* red, int g, int d, float* mm_out, float* ls_out,
                                            float* as_out) {
  float mm = -INFINITY;
#pragma unroll
  for (int w = 0; w < CW; ++w) mm = fmaxf(mm, red[(w * G + g) * (D + 2) + D]);
  float ls = 0.f, as = 0.f;
#pragma unroll
  for (int w = 0; w < CW; ++w) {
    const float* src = red + (w * G + g) * (D + 2);
    const float mw = src[D];
    const float f = (mw == -INFINITY) ? 0.f : fast_exp2(mw - mm);
    ls = fmaf(src[D + 1], f, ls);
    as = fmaf(src[d], f, as);
  }
  *mm_out = mm;
  *ls_out = ls;
  *as_out = as;
}

// Arrival counter of one (b, g) group: zero before the call, each CTA of the
// group adds one, the arrival that completes the count is the last one and
// puts the counter back to zero for the next call. Returns 1 for the last.
// The add is acquire-release at GPU scope: called by one thread after a CTA
// barrier, it publishes every partial the CTA wrote before the barrier and,
// for the last arrival, makes every other CTA's partials visible to the
// threads that pass the next barrier (no separate fences).
// A count already at or past `arrivals` means the counter was not zero when
// the call started: that is reported as kErrWorkspace and returns -1, and the
// caller writes NaN rows for the group (its merge cannot be trusted). The
// counter is left as it is, so that every later call on it fails the same
// visible way until the caller zero-fills it.
__device__ __forceinline__ int arrive_count(unsigned int* counter, int arrivals, int32_t* err_flag) {
  unsigned int before;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(before) : "l"(counter) : "memory");
  if (before + 1u < (unsigned int)arrivals) return 0;
  if (before + 1u > (unsigned int)arrivals) {
    if (err_flag) atomicOr(err_flag, kErrWorkspace);
    return -1;
  }
  atomicExch(counter, 0u);
  return 1;
}

template <typename T>
__device__ __forceinline__ void store_out(const DecodeParams& p, int64_t idx, float v) {
  reinterpret_cast<uint16_t*>(p.out)[idx] = Storage<T>::round(v);
}

// A running max may lag the true max by up to 2^kLazyRescale (in base-2
// units) before the accumulators are rescaled: the weights then stay below
// 2^8, far from fp32 overflow, and rescales become rare.
constexpr float kLazyRescale = 8.f;

// One tile of K and V rows for one warp: scores of this lane group's rows
// (mixed-precision FMAs on the raw 16-bit q and K, reduced over the lanes of
// a row, then scaled), the lazily rescaled online-softmax update, and the
// weighted V accumulation (packed fp32x2 FMAs). `kt`/`vt` point at this lane
// group's first row of the tile; with kFull false only rows whose offset
// from it is below `left` (in lane-group steps) are valid.
template <typename S, typename Shape, int G, bool kFull>
__device__ __forceinline__ void consume_tile(const uint8_t* kt, const uint8_t* vt, int left,
                                             const uint4 (&q)[G][Shape::kVecs], float qscale,
                                             int c, int swap, float (&m)[G], float& l_own,
                                             float2 (&acc)[G][Shape::kVecs][4]) {
  constexpr int NV = Shape::kVecs;
  constexpr int LPR = Shape::kLanesPerRow;
  constexpr int RS = Shape::kRowsPerStep * Shape::kRowBytes;  // bytes between a lane group's rows
  float own[Shape::kSteps];  // this lane's head's score of each step's row
#pragma unroll
  for (int u = 0; u < Shape::kSteps; ++u) {
    const bool valid = kFull || u * Shape::kRowsPerStep < left;
    float part[G];
    float a0[G], a1[G];
#pragma unroll
    for (int g = 0; g < G; ++g) a0[g] = a1[g] = 0.f;
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      uint4 kv = make_uint4(0u, 0u, 0u, 0u);
      if (valid) kv = *reinterpret_cast<const uint4*>(kt + u * RS + (c + LPR * (j ^ swap)) * 16);
#pragma unroll
      for (int g = 0; g < G; ++g) {
        S::dot2(q[g][j].x, kv.x, a0[g], a1[g]);
        S::dot2(q[g][j].y, kv.y, a0[g], a1[g]);
        S::dot2(q[g][j].z, kv.z, a0[g], a1[g]);
        S::dot2(q[g][j].w, kv.w, a0[g], a1[g]);
      }
    }
#pragma unroll
    for (int g = 0; g < G; ++g) part[g] = a0[g] + a1[g];
    // Sum over the LPR lanes of the row. With one head this is a butterfly.
    // With several, each halving step sends the half of the heads this lane
    // gives up and adds the partner's half of the ones it keeps; after
    // log2(G) steps lane c holds head c / (LPR / G) alone, and the remaining
    // steps add that one value.
    if (G == 1) {
      float v = part[0];
#pragma unroll
      for (int off = LPR / 2; off >= 1; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
      own[u] = valid ? v * qscale : -INFINITY;
    } else {
#pragma unroll
      for (int n = G, off = LPR / 2; n > 1; n >>= 1, off >>= 1) {
        const bool upper = (c & off) != 0;
#pragma unroll
        for (int i = 0; i < n / 2; ++i) {
          const float send = upper ? part[i] : part[i + n / 2];
          const float keep = upper ? part[i + n / 2] : part[i];
          part[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
        }
      }
      float v = part[0];
#pragma unroll
      for (int off = LPR / (2 * G); off >= 1; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
      own[u] = valid ? v * qscale : -INFINITY;
    }
  }

  // Online softmax, one head per lane: the lane owns head `h` (all heads when
  // G = 1), exponentiates only its head's scores and hands the weights to
  // the other lanes of its row. The running max of every head is kept by
  // every lane (the accumulators of all heads live in every lane); one vote
  // per tile decides a (rare) lazy rescale of all heads.
  const int h = G == 1 ? 0 : c / (LPR / G);
  const int base = (threadIdx.x & 31) & ~(LPR - 1);
  float mx = own[0];
#pragma unroll
  for (int u = 1; u < Shape::kSteps; ++u) mx = fmaxf(mx, own[u]);
  float m_own = m[0];
#pragma unroll
  for (int g = 1; g < G; ++g) m_own = (h == g) ? m[g] : m_own;
  if (__any_sync(0xffffffffu, mx > m_own + kLazyRescale)) {
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float mxg = G == 1 ? mx : __shfl_sync(0xffffffffu, mx, base + g * (LPR / G));
      const float mnew = fmaxf(m[g], mxg);
      const float alpha = (m[g] == -INFINITY) ? 0.f : fast_exp2(m[g] - mnew);
      const float2 alpha2 = make_float2(alpha, alpha);
#pragma unroll
      for (int j = 0; j < NV; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[g][j][e] = __fmul2_rn(acc[g][j][e], alpha2);
      if (g == h) l_own *= alpha;
      m[g] = mnew;
    }
    m_own = m[0];
#pragma unroll
    for (int g = 1; g < G; ++g) m_own = (h == g) ? m[g] : m_own;
  }
  const bool none = (m_own == -INFINITY);  // no visible row yet for this head in this lane group
  float pown[Shape::kSteps];
#pragma unroll
  for (int u = 0; u < Shape::kSteps; ++u) {
    pown[u] = none ? 0.f : fast_exp2(own[u] - m_own);
    l_own += pown[u];
  }

#pragma unroll
  for (int u = 0; u < Shape::kSteps; ++u) {
    const bool valid = kFull || u * Shape::kRowsPerStep < left;
    float pb[G];
#pragma unroll
    for (int g = 0; g < G; ++g) pb[g] = G == 1 ? pown[u] : __shfl_sync(0xffffffffu, pown[u], base + g * (LPR / G));
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      uint4 vv = make_uint4(0u, 0u, 0u, 0u);
      if (valid) vv = *reinterpret_cast<const uint4*>(vt + u * RS + (c + LPR * (j ^ swap)) * 16);
      float2 vf[4];
      S::unpack2(vv, vf);
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float2 p2 = make_float2(pb[g], pb[g]);
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[g][j][e] = __ffma2_rn(p2, vf[e], acc[g][j][e]);
      }
    }
  }
}

// Final merge of the per-cluster partials of one group by the last CTA to
// arrive: out = sum_k 2^(m_k - M) acc_k / sum_k 2^(m_k - M) l_k over the P
// clusters. When the CTA has more threads than the group has outputs, R
// threads share an output and each takes every R-th partial; otherwise each
// thread takes KPT outputs. A thread loads a batch of partials of all its
// outputs at once, (m, l) together with acc, and folds the batch into a
// running (max, sum, acc): up to kBatch * R partials cost a single round trip
// to L2. The R shares are combined through shared memory (`buf`, 3 * R * E
// floats).
template <typename T, int D, int G, int NT>
__device__ __forceinline__ void merge_partials(const DecodeParams& p, int64_t head0, int P, int nc, float* buf) {
  constexpr int E = G * D;
  constexpr int R = E >= NT ? 1 : NT / E;              // threads per output
  constexpr int KPT = R > 1 ? 1 : (E + NT - 1) / NT;  // outputs per thread
  constexpr int kBatch = KPT >= 4 ? 8 : 16;            // partials per output per round trip
  const int r = R > 1 ? (int)threadIdx.x / E : 0;      // this thread's share of the partials
  const bool active = r < R;
  float mm[KPT], ls[KPT], as[KPT];
#pragma unroll
  for (int q = 0; q < KPT; ++q) {
    mm[q] = -INFINITY;
    ls[q] = 0.f;
    as[q] = 0.f;
  }
  for (int k0 = r; active && k0 < P; k0 += kBatch * R) {
    float mv[KPT][kBatch], lv[KPT][kBatch], av[KPT][kBatch];
#pragma unroll
    for (int q = 0; q < KPT; ++q) {
      const int i = R > 1 ? (int)threadIdx.x % E : (int)threadIdx.x + q * NT;
      const int g = min(i, E - 1) / D;
      const float* ml = p.ws_ml + (head0 + g) * nc * 2;
      const float* part = p.ws_acc + (head0 + g) * nc * D + (min(i, E - 1) % D);
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        const int k = k0 + j * R;
        const bool ok = i < E && k < P;
        mv[q][j] = ok ? __ldcg(ml + 2 * k) : -INFINITY;
        lv[q][j] = ok ? __ldcg(ml + 2 * k + 1) : 0.f;
        av[q][j] = ok ? __ldcg(part + (int64_t)k * D) : 0.f;
      }
    }
#pragma unroll
    for (int q = 0; q < KPT; ++q) {
      float mb = mm[q];
#pragma unroll
      for (int j = 0; j < kBatch; ++j) mb = fmaxf(mb, mv[q][j]);
      const float f = (mm[q] == -INFINITY) ? 0.f : fast_exp2(mm[q] - mb);
      ls[q] *= f;
      as[q] *= f;
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        const float w = (mv[q][j] == -INFINITY) ? 0.f : fast_exp2(mv[q][j] - mb);
        ls[q] = fmaf(lv[q][j], w, ls[q]);
        as[q] = fmaf(av[q][j], w, as[q]);
      }
      mm[q] = mb;
    }
  }
  if constexpr (R > 1) {
    float* rm = buf;
    float* rl = buf + R * E;
    float* ra = buf + 2 * R * E;
    if (active) {
      const int i = (int)threadIdx.x % E;
      rm[r * E + i] = mm[0];
      rl[r * E + i] = ls[0];
      ra[r * E + i] = as[0];
    }
    __syncthreads();
    if ((int)threadIdx.x < E) {
      const int i = threadIdx.x;
      float M = -INFINITY;
#pragma unroll
      for (int q = 0; q < R; ++q) M = fmaxf(M, rm[q * E + i]);
      float L = 0.f, A = 0.f;
#pragma unroll
      for (int q = 0; q < R; ++q) {
        const float mq = rm[q * E + i];
        const float w = (mq == -INFINITY) ? 0.f : fast_exp2(mq - M);
        L = fmaf(rl[q * E + i], w, L);
        A = fmaf(ra[q * E + i], w, A);
      }
      store_out<T>(p, head0 * D + i, A / L);
    }
  } else {
#pragma unroll
    for (int q = 0; q < KPT; ++q) {
      const int i = (int)threadIdx.x + q * NT;
      if (i < E) store_out<T>(p, head0 * D + i, as[q] / ls[q]);
    }
  }
}

// Partials merge_partials folds in one round trip to L2 (a batch of each
// thread's share).
template <int D, int G, int NT>
__host__ __device__ constexpr int merge_one_trip() {
  constexpr int E = G * D;
  constexpr int R = E >= NT ? 1 : NT / E;
  constexpr int KPT = R > 1 ? 1 : (E + NT - 1) / NT;
  return (KPT >= 4 ? 8 : 16) * R;
}

// The same merge with the partials brought into shared memory first (when
// there are more than merge_one_trip of them and the G x P partials fit
// the idle ring): thread 0 copies each head's P
// accumulator rows with one bulk copy while the threads load the (m, l)
// pairs; the weights 2^(m_k - M) and the denominators are computed once per
// (head, partial), and each output is then a P-term weighted sum read from
// shared memory. One round trip to L2 whatever P is.
template <typename T, int D, int G, int NT>
__device__ __forceinline__ void merge_partials_smem(const DecodeParams& p, int64_t head0, int P, int nc,
                                                    uint8_t* smem, uint64_t* bar) {
  constexpr int E = G * D;
  float* acc_s = reinterpret_cast<float*>(smem);  // [G][P][D]
  float* ml_s = acc_s + G * P * D;                // [G][P][2]
  float* w_s = ml_s + G * P * 2;                  // [G][P] weights, then [G] denominators
  float* den_s = w_s + G * P;
  if (threadIdx.x == 0) {
    // The partials were written by other CTAs and acquired by this thread's
    // arrival; the bulk copies read them through the async proxy.
    fence_proxy_async_global();
    mbar_arrive_expect_tx(bar, (uint32_t)(G * P * D * 4));
#pragma unroll
    for (int g = 0; g < G; ++g)
      bulk_load_plain(acc_s + g * P * D, p.ws_acc + (head0 + g) * nc * D, (uint32_t)(P * D * 4), bar);
  }
  for (int t = threadIdx.x; t < G * P; t += NT) {
    const int g = t / P, k = t - (t / P) * P;
    const float* ml = p.ws_ml + ((head0 + g) * nc + k) * 2;
    ml_s[2 * t] = __ldcg(ml);
    ml_s[2 * t + 1] = __ldcg(ml + 1);
  }
  __syncthreads();
  for (int t = threadIdx.x; t < G * P; t += NT) {
    const int g = t / P;
    float M = -INFINITY;
    for (int k = 0; k < P; ++k) M = fmaxf(M, ml_s[2 * (g * P + k)]);
    const float m = ml_s[2 * t];
    w_s[t] = (m == -INFINITY) ? 0.f : fast_exp2(m - M);
  }
  __syncthreads();
  if ((int)threadIdx.x < G) {
    const int g = threadIdx.x;
    float den = 0.f;
    for (int k = 0; k < P; ++k) den = fmaf(ml_s[2 * (g * P + k) + 1], w_s[g * P + k], den);
    den_s[g] = den;
  }
  const bool landed = mbar_wait(bar, 0);
  __syncthreads();
  if (!landed) {
    if (threadIdx.x == 0 && p.err_flag) atomicOr(p.err_flag, kErrTimeout);
    for (int i = threadIdx.x; i < E; i += NT) reinterpret_cast<uint16_t*>(p.out)[head0 * D + i] = Storage<T>::kNaN;
    return;
  }
  for (int i = threadIdx.x; i < E; i += NT) {
    const int g = i / D, d = i - (i / D) * D;
    const float* a = acc_s + g * P * D + d;
    const float* w = w_s + g * P;
    float A = 0.f;
    for (int k = 0; k < P; ++k) A = fmaf(w[k], a[k * D], A);
    store_out<T>(p, head0 * D + i, A / den_s[g]);
  }
}

template <typename T, int D, int G, int CW, int DPL, int NS, bool RP, bool TC, int MB>
__global__ void __launch_bounds__(DecodeShape<D, G, CW, DPL, NS, TC>::kThreads, MB)
    decode_split_kernel(const __grid_constant__ DecodeParams p) {
  using Shape = DecodeShape<D, G, CW, DPL, NS, TC>;
  constexpr int kStages = NS;
  using S = Storage<T>;
  constexpr int LPR = Shape::kLanesPerRow;
  constexpr int NV = Shape::kVecs;
  constexpr int CT = Shape::kConsumerThreads;
  constexpr int E = G * D;  // outputs of a group

  extern __shared__ __align__(128) uint8_t smem_base[];
  // With tensor-core scores the ring starts on a 1024-byte boundary (the
  // atoms of the 128-byte swizzle the K tiles arrive in).
  uint8_t* smem = TC ? smem_base + ((1024u - (smem_addr(smem_base) & 1023u)) & 1023u) : smem_base;
  float* red = reinterpret_cast<float*>(smem);  // per-warp states, once the ring is idle
  float* recv = reinterpret_cast<float*>(smem + Shape::kRingBytes);  // receive area of the cluster merge
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + Shape::kBarOffset);
  uint64_t* empty = full + kStages;
  uint64_t* merge_bar = empty + kStages;  // the partials' bulk copies of the workspace merge
  uint64_t* sready = merge_bar + 1;       // tensor-core scores of a group's tile are in tensor memory [2]
  uint64_t* sfree = sready + 2;           // a group has read them [2]
  int* abort_flag = reinterpret_cast<int*>(merge_bar + 1 + (TC ? 4 : 0));
  int* last_flag = abort_flag + 1;
  // Tensor-core scores (unused otherwise).
  uint8_t* q_op = smem + Shape::kQOffset;                                  // the B operand
  float* pw = reinterpret_cast<float*>(smem + Shape::kPOffset);            // [2][kTileRows][G] weights
  float* gmax = reinterpret_cast<float*>(smem + Shape::kAuxOffset);        // [2][4][G]
  float* lsum = gmax + 8 * G;                                              // [2][4][G]
  float* mgrp = lsum + 8 * G;                                              // [2][G]
  float* snew = mgrp + 2 * G;                                              // [G]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(snew + G);
  constexpr uint32_t kTmemCols = 32;  // two 16-column score buffers

  const int s = blockIdx.x;
  const int g_kv = blockIdx.y;
  const int b = blockIdx.z;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int H = p.n_head;
  const int CS = p.cluster;    // CTAs per cluster along the split axis
  const int rank = s % CS;     // rank of this CTA in its cluster
  const int cid = s / CS;      // which cluster of the group
  const int64_t head0 = (int64_t)b * H + (int64_t)g_kv * G;
  const int64_t kv_row0 = ((int64_t)b * p.n_kv_head + g_kv) * p.capacity;  // first cache row of this (b, g)

  uint64_t policy = 0;  // L2 eviction policy of the tile copies (producer lane)
  enum : int { kSlotAll = 0, kSlotCached = 1, kSlotNew = 2 };
  const bool fused = p.k_new != nullptr;
  const bool rope = RP && fused && p.rope_cos != nullptr;  // instances with RP serve the rotary step
  const int64_t new_row = ((int64_t)b * p.n_kv_head + g_kv) * D;  // element offset into k_new
  // Ring slot u takes rows [tr0, tr0 + rows) of this CTA's K and V, the row
  // at Lx - 1 from k_new/v_new in the fused step (producer lane only).
  // `part` may split that in two: kSlotCached arms the slot's barrier for all
  // of its bytes and copies the cached rows, kSlotNew copies the new row.
  auto issue = [&](int u, int tr0, int rows, int Lx, int part) {
    // Test hook: leave one slot of one CTA unfilled (its waits then time out).
    if (u == p.skip_slot && s == 0 && b == 0 && g_kv == 0) return;
    const int stage = u % kStages;
    const bool new_last = fused && (tr0 + rows == Lx);
    const int cached = new_last ? rows - 1 : rows;
    uint8_t* kdst = smem + stage * Shape::kStageBytes;
    uint8_t* vdst = kdst + kTileBytes;
    if constexpr (TC) {
      // K arrives by tensor copies in the swizzled operand layout, whole
      // tiles in one box per 64-column half, a partial tile in 8-row boxes
      // (rows past the chunk are read but never weighted; the new row's
      // score is computed apart, so the cache row L - 1 may hold anything).
      // V arrives as in the other instances.
      if (part != kSlotNew) {
        // With rotary embedding the producer warp has already stored the new
        // V row into this stage (rope_row): only the cached V rows arrive by TMA.
        const int krows = rows == Shape::kTileRows ? rows : (rows + 7) / 8 * 8;
        const int vrows = new_last && rope ? cached : rows;
        mbar_arrive_expect_tx(&full[stage], (uint32_t)(krows + vrows) * Shape::kRowBytes);
        const int z = b * p.n_kv_head + g_kv;
        if (rows == Shape::kTileRows) {
#pragma unroll
          for (int h = 0; h < D / 64; ++h)
            tensor_load_3d(kdst + h * Shape::kTileRows * 128, &p.k_tiles, h * 64, tr0, z, &full[stage], policy);
        } else {
          for (int j = 0; j < krows / 8; ++j)
#pragma unroll
            for (int h = 0; h < D / 64; ++h)
              tensor_load_3d(kdst + h * Shape::kTileRows * 128 + j * 1024, &p.k_rows8, h * 64, tr0 + 8 * j, z,
                             &full[stage], policy);
        }
        if (cached > 0)
          bulk_load(vdst, p.v_cache + (kv_row0 + tr0) * Shape::kRowBytes, cached * Shape::kRowBytes, &full[stage],
                    policy);
      }
      if (new_last && !rope && part != kSlotCached)
        bulk_load(vdst + cached * Shape::kRowBytes, p.v_new + new_row * 2, Shape::kRowBytes, &full[stage], policy);
      return;
    }
    if (part != kSlotNew) {
      // With rotary embedding the producer warp has already stored the new row
      // into this stage (rope_row): only the cached rows arrive by TMA.
      mbar_arrive_expect_tx(&full[stage], 2u * (new_last && rope ? cached : rows) * Shape::kRowBytes);
      if (cached > 0) {
        const int64_t off = (kv_row0 + tr0) * Shape::kRowBytes;
        bulk_load(kdst, p.k_cache + off, cached * Shape::kRowBytes, &full[stage], policy);
        bulk_load(vdst, p.v_cache + off, cached * Shape::kRowBytes, &full[stage], policy);
      }
    }
    if (new_last && !rope && part != kSlotCached) {
      const int64_t off = new_row * 2;
      bulk_load(kdst + cached * Shape::kRowBytes, p.k_new + off, Shape::kRowBytes, &full[stage], policy);
      bulk_load(vdst + cached * Shape::kRowBytes, p.v_new + off, Shape::kRowBytes, &full[stage], policy);
    }
  };

  // Fused step with rotary embedding: the whole producer warp rotates the new
  // key row for position `pos` (lanes < D/8 hold one 16-byte vector each;
  // lane c pairs with lane c ^ D/16, the same columns in the other half) and
  // stores it, with the V row, as row `at` of the (free) stage of ring slot
  // u, before lane 0 issues that slot: the __syncwarp and lane 0's mbarrier
  // arrive (release) order these stores before the consumers' wait. With
  // tensor-core scores only the V row goes into the stage (the new key's
  // scores are computed apart). With `to_cache` it also writes the rows into
  // the cache at `pos`; without `to_stage` it writes only the cache.
  auto rope_row = [&](int pos, int u, int at, bool to_cache, bool to_stage = true) {
    uint4 kx = make_uint4(0u, 0u, 0u, 0u), vx = kx;
    float cs[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f}, sn[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    if (lane < D / 8) {
      kx = ld_global_nc_v4(p.k_new + (new_row + lane * 8) * 2);
      vx = ld_global_nc_v4(p.v_new + (new_row + lane * 8) * 2);
      load_f32x8(p.rope_cos, pos, D, lane * 8, cs);
      load_f32x8(p.rope_sin, pos, D, lane * 8, sn);
    }
    const uint4 ky = shfl_xor_v4(kx, D / 16);
    if (lane < D / 8) {
      const uint4 kr = rope_vec8<T>(kx, ky, cs, sn, lane < D / 16);
      uint8_t* kdst = smem + (u % kStages) * Shape::kStageBytes + at * Shape::kRowBytes + lane * 16;
      if (to_stage) {
        if (!TC) *reinterpret_cast<uint4*>(kdst) = kr;
        *reinterpret_cast<uint4*>(kdst + kTileBytes) = vx;
      }
      if (to_cache) {
        const int64_t dst = (kv_row0 + pos) * Shape::kRowBytes + lane * 16;
        *reinterpret_cast<uint4*>(p.k_cache_w + dst) = kr;
        *reinterpret_cast<uint4*>(p.v_cache_w + dst) = vx;
      }
    }
    __syncwarp();
  };

  // Early tiles: when the host's bound is expected to be the exact length
  // (p.speculate), the producer issues this CTA's first tiles for that length
  // before the length itself has been read: slots 0..spec-1 take rows
  // [r0h, r1h) of the bound's split. They are kept if the length matches,
  // else left to land and discarded.
  const int lh = p.len_hint;
  const int chh = split_chunk(lh, p.splits, Shape::kTileRows);
  const int r0h = min(s * chh, lh);
  const int r1h = min(lh, r0h + chh);
  const int spec = p.speculate ? min((r1h - r0h + Shape::kTileRows - 1) / Shape::kTileRows, kStages) : 0;
  // With a ready prefix, the early tiles are copied before the grid wait when
  // they are every CTA's whole chunk (short chunks, where the wait
  // dominates); launches with longer chunks keep the L2 prefetch, since
  // copies into shared memory then slow the previous kernel's streaming more
  // than they gain.
  const bool pre = p.prefix_ready && chh <= kStages * Shape::kTileRows;

  // Everything before pdl_wait() touches no memory the previous kernel on the
  // stream may still write, except for L2 prefetches (L2 is coherent) and,
  // when the caller has declared the cached prefix ready (p.prefix_ready:
  // no kernel still running writes rows [0, len_hint) of these caches other
  // than the new row) and `pre` holds, the cached rows of the early tiles.
  if (threadIdx.x == CT) {
    policy = evict_first_policy();
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], Shape::kEmptyArrivals);
    }
    mbar_init(merge_bar, 1);
    if constexpr (TC) {
      for (int i = 0; i < 2; ++i) {
        mbar_init(&sready[i], 1);
        mbar_init(&sfree[i], 1);
      }
    }
    *abort_flag = 0;
    fence_mbar_init();
    const int ch = chh;
    const int pr0 = s * ch;
    if (pre) {
      // The early tiles' cached rows go straight into the ring; a slot whose
      // new row is rotated first (rope) waits for the grid in full.
      for (int t = 0; t < spec; ++t) {
        const int tr0 = r0h + t * Shape::kTileRows;
        const int rows = min(Shape::kTileRows, r1h - tr0);
        if (!(rope && tr0 + rows == lh)) issue(t, tr0, rows, lh, kSlotCached);
      }
    } else if (pr0 < lh && p.speculate) {
      // Pull the first tiles this CTA will read into L2, with rows from the
      // host's length bound, when that bound is expected to be the length
      // (one length and an explicit bound: otherwise rows past a sequence's
      // prefix would be fetched from DRAM for nothing): when one sequence
      // gives each CTA a short chunk, one tile for chunks of at most two and
      // two for chunks of at most six (every CTA's first tiles then land
      // sooner and compete less with the previous kernel's streaming; the
      // rest streams behind them); two as well for the long chunks of the
      // 4-stage instances (several query heads per KV head); else a ring's
      // worth.
      const int ahead = (p.B == 1 && ch <= 2 * Shape::kTileRows) ? 1
                        : (p.B == 1 && (ch <= 6 * Shape::kTileRows || kStages == 4)) ? min(2, kStages)
                                                                                    : kStages;
      const int rows = min(min(ch, lh - pr0), ahead * Shape::kTileRows);
      for (int t0 = 0; t0 < rows; t0 += Shape::kTileRows) {
        const int n = min(Shape::kTileRows, rows - t0);
        const int64_t off = (kv_row0 + pr0 + t0) * Shape::kRowBytes;
        prefetch_l2(p.k_cache + off, n * Shape::kRowBytes);
        prefetch_l2(p.v_cache + off, n * Shape::kRowBytes);
      }
    }
  }
  if constexpr (TC) {
    if (warp == CW + 1) {
      tmem_alloc(tmem_slot, kTmemCols);
      tc_fence_before();
    }
  }
  __syncthreads();
  uint32_t tmem = 0;
  if constexpr (TC) {
    tc_fence_after();
    tmem = *tmem_slot;
  }
  // The warp that allocated the tensor memory frees it before the CTA leaves.
  auto free_tmem = [&]() {
    if constexpr (TC) {
      if (warp == CW + 1) tmem_free(tmem, kTmemCols);
    }
  };
  pdl_wait();
  // The next grid may be scheduled from here on: once it runs, every grid
  // before this one has completed. CTAs with more than two tiles to stream
  // (by the host's bound) signal it only when their streaming is done, so
  // that the next grid's early CTAs prefetch while this one folds and merges
  // rather than while it streams (measured: MHA kv 4096 / 8192 and long-context
  // GQA kv 32768 0.08 / 0.15 / 0.28 us faster per call, MHA kv 1024 with its
  // two-tile chunks 0.11 us slower, hence the early signal there).
  const bool late_trigger = chh > 2 * Shape::kTileRows;
  if (!late_trigger) pdl_trigger();

  // Early tiles after the wait: all of them, or with a ready prefix the new
  // rows of the slots issued above and the rotated slot.
  int spec_new = -1;  // early slot holding the rotated row of the bound's last position
  if (warp == CW) {
    for (int t = 0; t < spec; ++t) {
      const int tr0 = r0h + t * Shape::kTileRows;
      const int rows = min(Shape::kTileRows, r1h - tr0);
      const bool has_new = fused && tr0 + rows == lh;
      if (pre && !(rope && has_new)) {
        if (has_new && lane == 0) issue(t, tr0, rows, lh, kSlotNew);
        continue;
      }
      if (rope && has_new) {
        rope_row(lh - 1, t, rows - 1, false);  // not into the cache before the length is known
        spec_new = t;
      }
      if (lane == 0) issue(t, tr0, rows, lh, kSlotAll);
    }
  }
  // A CTA leaving before its pipeline runs first lets the early tiles land.
  auto drain_early = [&]() {
    if (threadIdx.x == CT)
      for (int t = 0; t < spec; ++t) mbar_wait(&full[t], 0);
  };

  // Lane layout of the consumers: lane group `lrow` of a step takes one row;
  // within it, lane c holds vectors c + LPR * j (j < NV) of the row, slot j
  // visiting vector c + LPR * (j ^ swap).
  const int c = lane % LPR;
  const int lrow = lane / LPR;
  const int swap = Shape::kSwap ? (lrow & 1) : 0;
  uint4 qraw[G][NV];
  uint4 q_chunk = make_uint4(0u, 0u, 0u, 0u);  // tensor-core scores: this thread's 16 bytes of the q operand
  constexpr int kQChunks = D / 8;               // 16-byte chunks of a q row
  if constexpr (TC) {
    if (warp < CW && (int)threadIdx.x < 16 * kQChunks && (int)threadIdx.x / kQChunks < G)
      q_chunk = ld_global_nc_v4(p.q + ((head0 + threadIdx.x / kQChunks) * D + (threadIdx.x % kQChunks) * 8) * 2);
  } else if (warp < CW) {  // q loads overlap the length load below
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
      for (int j = 0; j < NV; ++j)
        qraw[g][j] = ld_global_nc_v4(p.q + ((head0 + g) * D + (c + LPR * (j ^ swap)) * 8) * 2);
  }
  // Rotary embedding of q: the consumers fetch cos and sin of their columns
  // for the bound's position now, and again below if the length differs.
  float qcos[8], qsin[8];
  int qpos = -1;
  if (rope && warp < CW && p.speculate) {
    qpos = p.len_hint - 1;
    load_f32x8(p.rope_cos, qpos, D, c * 8, qcos);
    load_f32x8(p.rope_sin, qpos, D, c * 8, qsin);
  }

  int32_t err_bits = 0;
  const int L = sequence_length(p, b, &err_bits);
  if (L < 0) {
    // Invalid input (the same for every CTA of the group, so whole clusters
    // leave here): split 0 writes NaN rows for the group's heads.
    if (s == 0) {
      for (int i = threadIdx.x; i < E; i += Shape::kThreads)
        reinterpret_cast<uint16_t*>(p.out)[head0 * D + i] = S::kNaN;
      if (threadIdx.x == 0 && p.err_flag) atomicOr(p.err_flag, err_bits);
    }
    drain_early();
    free_tmem();
    return;
  }
  const int chunk = split_chunk(L, p.splits, Shape::kTileRows);
  const int nsplit = active_splits(L, chunk);
  const int nclusters = (nsplit + CS - 1) / CS;  // clusters with at least one active split
  if (cid >= nclusters) {  // the whole cluster is idle
    drain_early();
    free_tmem();
    return;
  }
  // Splits past nsplit in an active cluster read nothing and contribute an
  // empty state (m = -inf, l = 0), but take part in the cluster barriers.
  const int r0 = min(s * chunk, L);
  const int r1 = min(L, r0 + chunk);
  const int ntiles = (r1 - r0 + Shape::kTileRows - 1) / Shape::kTileRows;
  // Tile t sits in ring slot t + slot0: the early tiles are tiles 0..spec-1
  // when the length matched the bound, else they occupy the first slots.
  const bool keep = spec > 0 && L == p.len_hint;
  const int slot0 = keep ? 0 : spec;
  if (rope && warp < CW) {
    if (qpos != L - 1) {
      qpos = L - 1;
      load_f32x8(p.rope_cos, qpos, D, c * 8, qcos);
      load_f32x8(p.rope_sin, qpos, D, c * 8, qsin);
    }
    if constexpr (TC) {
      // This thread's chunk of the q operand: chunk c of its row (c = lane % LPR).
      q_chunk = rope_vec8<T>(q_chunk, shfl_xor_v4(q_chunk, LPR / 2), qcos, qsin, c < LPR / 2);
    } else {
#pragma unroll
      for (int g = 0; g < G; ++g)
        qraw[g][0] = rope_vec8<T>(qraw[g][0], shfl_xor_v4(qraw[g][0], LPR / 2), qcos, qsin, c < LPR / 2);
    }
  }

  // Cluster merge geometry: rank k of the cluster merges outputs
  // [k * per, (k + 1) * per); its receive area holds every rank's (m, l) and
  // every rank's share of that slice.
  const int per = (E + CS - 1) / CS;
  float* ml_in = recv;                 // [CS][2G]
  float* acc_in = recv + CS * 2 * G;   // [CS][per]

  // Output i of the group, merged over this cluster: into `out` when one
  // cluster holds the group, else as this cluster's partial in the workspace.
  auto emit = [&](int i, float mm, float ls, float as) {
    const int g = i / D;
    const int d = i % D;
    if (nclusters == 1) {
      store_out<T>(p, head0 * D + i, as / ls);
    } else {
      const int64_t base = (head0 + g) * (p.splits / CS) + cid;
      p.ws_acc[base * D + d] = as;
      if (d == 0) {
        p.ws_ml[base * 2] = mm;
        p.ws_ml[base * 2 + 1] = ls;
      }
    }
  };

  if constexpr (TC) {
    // The q operand: row h holds head h of the group (rows G..15 zero), in
    // the 128-byte swizzle (16-byte chunk c of row r at chunk c ^ (r & 7)).
    if (warp < CW) {
      if ((int)threadIdx.x < 16 * kQChunks) {
        const int row = threadIdx.x / kQChunks, ch = threadIdx.x % kQChunks;
        *reinterpret_cast<uint4*>(q_op + (ch / 8) * 2048 + row * 128 + (((ch % 8) ^ (row & 7)) * 16)) = q_chunk;
      }
      if (warp == 0 && fused && r0 < r1 && r1 == L) {
        // The new row is attended from k_new (the cache row L - 1 is being
        // written by this launch): its scores on the CUDA cores, one 16-byte
        // vector of k_new and q per lane (lane = chunk; with rotary
        // embedding both rotated as above, lane c pairing with c ^ LPR / 2).
        const bool in_row = lane < kQChunks;
        const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
        uint4 kn = in_row ? ld_global_nc_v4(p.k_new + (new_row + lane * 8) * 2) : zero;
        if (rope) kn = rope_vec8<T>(kn, shfl_xor_v4(kn, LPR / 2), qcos, qsin, c < LPR / 2);
        float part[G];
#pragma unroll
        for (int g = 0; g < G; ++g) {
          uint4 qv = in_row ? ld_global_nc_v4(p.q + ((head0 + g) * D + lane * 8) * 2) : zero;
          if (rope) qv = rope_vec8<T>(qv, shfl_xor_v4(qv, LPR / 2), qcos, qsin, c < LPR / 2);
          float a0 = 0.f, a1 = 0.f;
          S::dot2(qv.x, kn.x, a0, a1);
          S::dot2(qv.y, kn.y, a0, a1);
          S::dot2(qv.z, kn.z, a0, a1);
          S::dot2(qv.w, kn.w, a0, a1);
          part[g] = in_row ? a0 + a1 : 0.f;
        }
#pragma unroll
        for (int g = 0; g < G; ++g) {
#pragma unroll
          for (int off = 16; off >= 1; off >>= 1) part[g] += __shfl_xor_sync(0xffffffffu, part[g], off);
        }
        if (lane == 0) {
#pragma unroll
          for (int g = 0; g < G; ++g) snew[g] = part[g] * p.qscale;
        }
      }
      fence_proxy_async_shared();
    }
    if (warp != CW) named_barrier_sync<4, CT + 32>();  // consumers and the MMA warp: q operand staged
  }

  // Publication of this CTA's folded outputs (va, vm, vl per output
  // threadIdx.x + k * CT): pushed to the cluster ranks, or emitted at once by
  // a lone CTA. A CTA whose pipeline timed out publishes NaN, which poisons
  // every output of its group.
  auto publish = [&](const float (&va)[Shape::kPerThread], const float (&vm)[Shape::kPerThread],
                     const float (&vl)[Shape::kPerThread], bool failed) {
    const float nan = __int_as_float(0x7fc00000);
    if (CS > 1) {
      // Cluster plans: each folded value goes straight to the rank that
      // merges it (distributed shared-memory stores), (m, l) of each head to
      // every rank: the thread folding column r of the head sends them to
      // rank r (every thread of a head holds that head's m and l).
#pragma unroll
      for (int k = 0; k < Shape::kPerThread; ++k) {
        const int i = threadIdx.x + k * CT;
        if (i < E) {
          const int kk = i / per;
          st_cluster_f32(acc_in + rank * per + (i - kk * per), kk, failed ? nan : va[k]);
          const int g = i / D, r = i - g * D;
          if (r < CS) {
            st_cluster_f32(ml_in + rank * 2 * G + g, r, failed ? nan : vm[k]);
            st_cluster_f32(ml_in + rank * 2 * G + G + g, r, vl[k]);
          }
        }
      }
    } else {
      // A lone CTA: each folded output goes out (or into the workspace) at once.
#pragma unroll
      for (int k = 0; k < Shape::kPerThread; ++k) {
        const int i = threadIdx.x + k * CT;
        if (i < E) emit(i, failed ? nan : vm[k], vl[k], failed ? nan : va[k]);
      }
    }
  };

  if (warp == CW) {
    // ---------------- producer warp ----------------
    if (fused && !rope && s == 0 && lane < D / 8) {
      // The new row goes into the cache; no CTA of this launch reads it back
      // from there (the CTA owning row L-1 takes it from k_new/v_new).
      const int64_t dst = (kv_row0 + (L - 1)) * Shape::kRowBytes + lane * 16;
      const int64_t src = new_row * 2 + lane * 16;
      *reinterpret_cast<uint4*>(p.k_cache_w + dst) = ld_global_nc_v4(p.k_new + src);
      *reinterpret_cast<uint4*>(p.v_cache_w + dst) = ld_global_nc_v4(p.v_new + src);
    }
    if (lane == 0 && !keep) {
      // Discarded early tiles: wait for them to land, then free their stages.
      for (int t = 0; t < spec; ++t) {
        if (!mbar_wait(&full[t], 0)) atomicOr(abort_flag, 1);
        for (int w = 0; w < Shape::kEmptyArrivals; ++w) mbar_arrive(&empty[t]);
      }
    }
    __syncwarp();
    if (TC && keep && spec_new >= 0) {
      // The kept early slot spec_new holds the new V row but not the key
      // row: both go into the cache from k_new / v_new again (rotated).
      rope_row(L - 1, spec_new, 0, true, false);
    } else if (keep && spec_new >= 0 && lane < D / 8) {
      // The kept early slot spec_new holds the rotated row of position L - 1
      // (its stage is not reused before the loop below): it goes into the
      // cache now. No CTA of this launch reads that row back from the cache.
      const uint8_t* src = smem + (spec_new % kStages) * Shape::kStageBytes +
                           ((L - 1) - (r0 + spec_new * Shape::kTileRows)) * Shape::kRowBytes + lane * 16;
      const int64_t dst = (kv_row0 + (L - 1)) * Shape::kRowBytes + lane * 16;
      *reinterpret_cast<uint4*>(p.k_cache_w + dst) = *reinterpret_cast<const uint4*>(src);
      *reinterpret_cast<uint4*>(p.v_cache_w + dst) = *reinterpret_cast<const uint4*>(src + kTileBytes);
    }
    int next = keep ? spec : slot0;  // next ring slot to fill
    if (RP && rope && r1 == L) {
      // The CTA whose chunk ends at the new row: the whole warp walks the
      // slots (lane 0 waits and issues) so that it can store the rotated row
      // into a stage right before it is issued.
      for (int t = keep ? spec : 0; t < ntiles; ++t) {
        const int u = t + slot0;
        const int stage = u % kStages;
        int ok = 1;
        if (lane == 0) {
          if (u >= kStages && !mbar_wait(&empty[stage], ((u / kStages) & 1) ^ 1)) atomicOr(abort_flag, 1);
          ok = *reinterpret_cast<volatile int*>(abort_flag) == 0;
        }
        __syncwarp();
        if (!__shfl_sync(0xffffffffu, ok, 0)) break;
        const int tr0 = r0 + t * Shape::kTileRows;
        const int rows = min(Shape::kTileRows, r1 - tr0);
        if (rope && tr0 + rows == L) rope_row(L - 1, u, rows - 1, true);
        if (lane == 0) issue(u, tr0, rows, L, kSlotAll);
        next = u + 1;
      }
    } else if (lane == 0) {
      for (int t = keep ? spec : 0; t < ntiles; ++t) {
        const int u = t + slot0;
        const int stage = u % kStages;
        if (u >= kStages) {
          if (!mbar_wait(&empty[stage], ((u / kStages) & 1) ^ 1)) {
            atomicOr(abort_flag, 1);
            break;
          }
        }
        if (*reinterpret_cast<volatile int*>(abort_flag)) break;
        const int tr0 = r0 + t * Shape::kTileRows;
        issue(u, tr0, min(Shape::kTileRows, r1 - tr0), L, kSlotAll);
        next = u + 1;
      }
    }
    // After an abort, let copies already in flight land before the CTA
    // exits (bounded): the last slot filled in each stage.
    if (lane == 0 && *reinterpret_cast<volatile int*>(abort_flag)) {
      for (int u = max(0, next - kStages); u < next; ++u) mbar_wait(&full[u % kStages], (u / kStages) & 1);
    }
    __syncwarp();
  } else if (warp == CW + 1) {
    if constexpr (TC) {
      // ---------------- MMA warp (tensor-core scores) ----------------
      // Lane 0 issues the scores of tile t into buffer t & 1 once the tile
      // has landed and the group that read the buffer's previous tile has
      // released it: S^T = K q^T over D / 16 steps of 16 columns, then one
      // commit that arrives on sready[t & 1] when the products are in
      // tensor memory.
      constexpr uint32_t idesc = mma_idesc_m128_n16(S::kBf16);
      // Descriptors of the ring's first byte and of the q operand; an
      // operand at byte offset o from them is the descriptor + o / 16 (the
      // start-address field; every address stays below 256 KiB).
      const uint64_t a_base = sw128_desc(smem);
      const uint64_t b_base = sw128_desc(q_op);
      int issued = 0;
      if (lane == 0) {
        bool ok = true;
        for (int t = 0; t < slot0 && ok; ++t) ok = mbar_wait(&full[t], 0);  // discarded early tiles
        for (int t = 0; t < ntiles && ok; ++t) {
          const int u = t + slot0;
          const int stage = u % kStages;
          ok = mbar_wait(&full[stage], (u / kStages) & 1);
          if (ok && t >= 2) ok = mbar_wait(&sfree[t & 1], ((t - 2) >> 1) & 1);
          if (!ok || *reinterpret_cast<volatile int*>(abort_flag)) break;
          tc_fence_after();
          const uint64_t a_stage = a_base + (uint64_t)((stage * Shape::kStageBytes) >> 4);
          const uint32_t dcol = tmem + (uint32_t)(t & 1) * 16u;
#pragma unroll
          for (int k = 0; k < D / 16; ++k) {
            const int h = k / 4, kk = k % 4;
            mma_f16_ss(dcol, a_stage + (uint64_t)((h * Shape::kTileRows * 128 + kk * 32) >> 4),
                       b_base + (uint64_t)((h * 2048 + kk * 32) >> 4), idesc, k > 0);
          }
          mma_commit(&sready[t & 1]);
          issued = t + 1;
        }
        if (!ok) atomicOr(abort_flag, 1);
      }
      __syncwarp();
      named_barrier_sync<4, CT + 32>();  // every consumer is done with the tensor memory
      if (lane == 0) {
        // Products still in flight after an abort land before the memory is freed.
        for (int t = max(0, issued - 2); t < issued; ++t) mbar_wait(&sready[t & 1], (t >> 1) & 1);
      }
      __syncwarp();
      tc_fence_after();
      tmem_free(tmem, kTmemCols);
    }
  } else if constexpr (TC) {
    // ---------------- consumer warps (tensor-core scores) ----------------
    // Two groups of four warps take the tiles in turn (group t & 1 takes
    // tile t), each with its own online-softmax state. In a tile, the
    // group's first kTileRows threads each own one row (TMEM lane = row):
    // they read its G scores from tensor memory, scale and mask them, and
    // turn them into weights against the group's running max (raised, and
    // the group's state rescaled, only when a score passes it by more than
    // 2^kLazyRescale, decided by one barrier-reduction). The weights go
    // through shared memory; then every thread of the group adds its rows'
    // weighted V to its slice of the accumulators (D/8 threads per row, 16
    // bytes of V each, packed fp32x2 FMAs), and the group releases the stage.
    constexpr int TR = Shape::kTileRows;
    constexpr int SW = TR / 32;                     // scoring warps of a group
    constexpr int TPR = Shape::kVThreadsPerRow;
    constexpr int RPT = Shape::kRowsPerThread;
    constexpr int RG = Shape::kRowGroups;
    const int grp = warp >> 2, gw = warp & 3, gt = (int)threadIdx.x & 127;
    const bool scorer = gw < SW;
    const int sw = gw;
    const int vc = gt % TPR, rg = gt / TPR;
    const uint32_t tcol = tmem + (uint32_t)grp * 16u + ((uint32_t)(gw * 32) << 16);
    float* pg = pw + grp * TR * G;                  // this group's weights [TR][G]
    // The group's barriers (IDs 2 and 3, 128 threads each).
    auto group_sync = [&]() {
      if (grp == 0) named_barrier_sync<2, 128>();
      else named_barrier_sync<3, 128>();
    };
    auto group_or = [&](bool v) { return grp == 0 ? named_barrier_or<2, 128>(v) : named_barrier_or<3, 128>(v); };
    float m[G], l_own[G];
    float2 acc[G][4];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      m[g] = -INFINITY;
      l_own[g] = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[g][e] = make_float2(0.f, 0.f);
    }
    // The tile whose last row is the new row (scores computed apart).
    const int new_tile = (fused && r0 < r1 && r1 == L) ? ntiles - 1 : -1;
    // Discarded early tiles: their copies must have landed (phase 0 of their
    // stages) before a later phase of the same stages is waited for.
    bool ok_pre = true;
    for (int t = 0; t < slot0; ++t) ok_pre = mbar_wait(&full[t], 0) && ok_pre;
    bool aborted = false;
    volatile int* grp_abort = reinterpret_cast<volatile int*>(last_flag + 1 + grp);  // a wait of the group gave up
    if (gt == 0) *grp_abort = 0;
    group_sync();
    for (int t = grp; t < ntiles; t += 2) {
      const int u = t + slot0;
      const int stage = u % kStages;
      bool ok = ok_pre && mbar_wait(&full[stage], (u / kStages) & 1);
      ok = ok && mbar_wait(&sready[grp], (t >> 1) & 1);
      ok_pre = true;
      // A warp reads the scores only if all its lanes' waits succeeded (the
      // load is warp-wide); the group learns of a failed wait after the
      // barrier below, which also decides the raise.
      const bool warp_ok = __all_sync(0xffffffffu, ok);
      if (!warp_ok && lane == 0) *grp_abort = 1;
      const int rows = min(TR, r1 - (r0 + t * TR));
      float sc[G];
      bool over = false;
      if (scorer && warp_ok) {
        tc_fence_after();
        uint32_t raw[G];
        tmem_load<G>(tcol, raw);
        tc_fence_before();
        const bool valid = gt < rows;
#pragma unroll
        for (int g = 0; g < G; ++g) sc[g] = valid ? __uint_as_float(raw[g]) * p.qscale : -INFINITY;
        if (t == new_tile && gt == rows - 1) {
#pragma unroll
          for (int g = 0; g < G; ++g) sc[g] = snew[g];
        }
#pragma unroll
        for (int g = 0; g < G; ++g) over = over || sc[g] > m[g] + kLazyRescale;
      }
      const bool raise = group_or(over);
      if (*grp_abort) {
        aborted = true;
        break;
      }
      if (gt == 0) mbar_arrive(&sfree[grp]);  // the MMA warp may overwrite this buffer
      if (raise) {
        if (scorer) {
#pragma unroll
          for (int g = 0; g < G; ++g) {
            float x = sc[g];
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, off));
            if (lane == 0) gmax[(grp * 4 + sw) * G + g] = x;
          }
        }
        group_sync();
#pragma unroll
        for (int g = 0; g < G; ++g) {
          float tm = gmax[(grp * 4) * G + g];
#pragma unroll
          for (int w = 1; w < SW; ++w) tm = fmaxf(tm, gmax[(grp * 4 + w) * G + g]);
          const float mnew = fmaxf(m[g], tm);
          const float alpha = (m[g] == -INFINITY) ? 0.f : fast_exp2(m[g] - mnew);
          const float2 alpha2 = make_float2(alpha, alpha);
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[g][e] = __fmul2_rn(acc[g][e], alpha2);
          l_own[g] *= alpha;
          m[g] = mnew;
        }
      }
      if (scorer) {
        float w[G];
#pragma unroll
        for (int g = 0; g < G; ++g) {
          w[g] = (m[g] == -INFINITY) ? 0.f : fast_exp2(sc[g] - m[g]);
          l_own[g] += w[g];
        }
#pragma unroll
        for (int g = 0; g < G; g += 4)
          *reinterpret_cast<float4*>(pg + gt * G + g) = make_float4(w[g], w[g + 1], w[g + 2], w[g + 3]);
      }
      group_sync();
      // This thread's rows: [rg * RPT, (rg + 1) * RPT) of the tile.
      const uint8_t* vt = smem + stage * Shape::kStageBytes + kTileBytes + vc * 16;
      auto add_row = [&](int r) {
        const uint4 vv = *reinterpret_cast<const uint4*>(vt + r * Shape::kRowBytes);
        float2 vf[4];
        S::unpack2(vv, vf);
        float wr[G];
#pragma unroll
        for (int g = 0; g < G; g += 4) {
          const float4 w4 = *reinterpret_cast<const float4*>(pg + r * G + g);
          wr[g] = w4.x;
          wr[g + 1] = w4.y;
          wr[g + 2] = w4.z;
          wr[g + 3] = w4.w;
        }
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float2 w2 = make_float2(wr[g], wr[g]);
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[g][e] = __ffma2_rn(w2, vf[e], acc[g][e]);
        }
      };
      if (rows == TR) {
#pragma unroll
        for (int j = 0; j < RPT; ++j) add_row(rg * RPT + j);
      } else {
        for (int j = 0; j < RPT && rg * RPT + j < rows; ++j) add_row(rg * RPT + j);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[stage]);
    }
    if (aborted) atomicOr(abort_flag, 1);
    tc_fence_before();
    named_barrier_sync<4, CT + 32>();  // the MMA warp may free the tensor memory

    // Fold: the weight sums of each group's scoring threads, each group's
    // running max, and the row groups' accumulators (over the idle ring).
    if (scorer) {
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float x = l_own[g];
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
        if (lane == 0) lsum[(grp * 4 + sw) * G + g] = x;
      }
    }
    if (gt == 0) {
#pragma unroll
      for (int g = 0; g < G; ++g) mgrp[grp * G + g] = m[g];
    }
    named_barrier_sync<1, CT>();  // every consumer is done with the ring
#pragma unroll
    for (int g = 0; g < G; ++g) {
      float* dst = red + ((grp * RG + rg) * G + g) * D + vc * 8;
      *reinterpret_cast<float4*>(dst) = make_float4(acc[g][0].x, acc[g][0].y, acc[g][1].x, acc[g][1].y);
      *reinterpret_cast<float4*>(dst + 4) = make_float4(acc[g][2].x, acc[g][2].y, acc[g][3].x, acc[g][3].y);
    }
    named_barrier_sync<1, CT>();
    const bool failed = *reinterpret_cast<volatile int*>(abort_flag) != 0;
    if (failed && threadIdx.x == 0 && p.err_flag) atomicOr(p.err_flag, kErrTimeout);
    float va[Shape::kPerThread], vm[Shape::kPerThread], vl[Shape::kPerThread];
#pragma unroll
    for (int k = 0; k < Shape::kPerThread; ++k) {
      const int i = threadIdx.x + k * CT;
      if (i < E) {
        const int g = i / D, d = i % D;
        float mg[2], lg[2], ag[2];
#pragma unroll
        for (int q2 = 0; q2 < 2; ++q2) {
          mg[q2] = mgrp[q2 * G + g];
          float ls = 0.f, as = 0.f;
#pragma unroll
          for (int w = 0; w < SW; ++w) ls += lsum[(q2 * 4 + w) * G + g];
#pragma unroll
          for (int j = 0; j < RG; ++j) as += red[((q2 * RG + j) * G + g) * D + d];
          lg[q2] = ls;
          ag[q2] = as;
        }
        const float mm = fmaxf(mg[0], mg[1]);
        const float f0 = (mg[0] == -INFINITY) ? 0.f : fast_exp2(mg[0] - mm);
        const float f1 = (mg[1] == -INFINITY) ? 0.f : fast_exp2(mg[1] - mm);
        vm[k] = mm;
        vl[k] = lg[0] * f0 + lg[1] * f1;
        va[k] = ag[0] * f0 + ag[1] * f1;
      }
    }
    publish(va, vm, vl, failed);
  } else {
    // ---------------- consumer warps ----------------
    float m[G], l_own = 0.f;  // running max of every head; weight sum of this lane's head
    float2 acc[G][NV][4];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      m[g] = -INFINITY;
#pragma unroll
      for (int j = 0; j < NV; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[g][j][e] = make_float2(0.f, 0.f);
    }
    const int lane_off = (warp * Shape::kRowsPerWarp + lrow) * Shape::kRowBytes;
    bool aborted = false;
    // Discarded early tiles: their copies must have landed (phase 0 of their
    // stages) before this warp waits on a later phase of the same stages; a
    // parity wait tells only the current phase from the one before it.
    for (int t = 0; t < slot0; ++t) {
      if (__any_sync(0xffffffffu, !mbar_wait(&full[t], 0))) aborted = true;
    }
    for (int t = 0; t < ntiles && !aborted; ++t) {
      const int u = t + slot0;
      const int stage = u % kStages;
      const bool ok_wait = mbar_wait(&full[stage], (u / kStages) & 1);
      if (__any_sync(0xffffffffu, !ok_wait)) {
        aborted = true;
        break;
      }
      const uint8_t* kt = smem + stage * Shape::kStageBytes + lane_off;
      const uint8_t* vt = kt + kTileBytes;
      const int rows = min(Shape::kTileRows, r1 - (r0 + t * Shape::kTileRows));
      if (rows == Shape::kTileRows) {
        consume_tile<S, Shape, G, true>(kt, vt, 0, qraw, p.qscale, c, swap, m, l_own, acc);
      } else {
        consume_tile<S, Shape, G, false>(kt, vt, rows - (warp * Shape::kRowsPerWarp + lrow), qraw, p.qscale, c,
                                         swap, m, l_own, acc);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[stage]);
    }
    if (aborted) atomicOr(abort_flag, 1);

    // Back to the canonical slot order (slot j = vector c + LPR * j).
    if (Shape::kSwap) {
#pragma unroll
      for (int g = 0; g < G; ++g)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 a0 = acc[g][0][e], a1 = acc[g][NV - 1][e];
          acc[g][0][e] = swap ? a1 : a0;
          acc[g][NV - 1][e] = swap ? a0 : a1;
        }
    }

    // Weight sums of all heads (each lane kept its own head's).
    float l[G];
#pragma unroll
    for (int g = 0; g < G; ++g)
      l[g] = G == 1 ? l_own : __shfl_sync(0xffffffffu, l_own, (lane & ~(LPR - 1)) + g * (LPR / G));

    // Merge the lane groups of the warp that hold the same vectors.
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
        for (int j = 0; j < NV; ++j)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float ax = __shfl_xor_sync(0xffffffffu, acc[g][j][e].x, off);
            const float ay = __shfl_xor_sync(0xffffffffu, acc[g][j][e].y, off);
            acc[g][j][e] = make_float2(acc[g][j][e].x * fa + ax * fb, acc[g][j][e].y * fa + ay * fb);
          }
        m[g] = mm;
      }
    }

    // Per-warp states to shared memory, over the ring once every consumer
    // warp is done with it: red[warp][g][0..D) = acc, [D] = m, [D+1] = l.
    asm volatile("bar.sync 1, %0;" ::"n"(CT) : "memory");
    if (lrow == 0) {
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float* dst = red + (warp * G + g) * (D + 2);
#pragma unroll
        for (int j = 0; j < NV; ++j)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            dst[(c + LPR * j) * 8 + 2 * e] = acc[g][j][e].x;
            dst[(c + LPR * j) * 8 + 2 * e + 1] = acc[g][j][e].y;
          }
        if (c == 0) {
          dst[D] = m[g];
          dst[D + 1] = l[g];
        }
      }
    }
    asm volatile("bar.sync 1, %0;" ::"n"(CT) : "memory");

    // Fold the warps into one state per output. A CTA whose pipeline timed out
    // publishes NaN, which poisons every output of its group.
    const bool failed = *reinterpret_cast<volatile int*>(abort_flag) != 0;
    if (failed && threadIdx.x == 0 && p.err_flag) atomicOr(p.err_flag, kErrTimeout);
    float va[Shape::kPerThread], vm[Shape::kPerThread], vl[Shape::kPerThread];
#pragma unroll
    for (int k = 0; k < Shape::kPerThread; ++k) {
      const int i = threadIdx.x + k * CT;
      if (i < E) merge_warps<D, G, CW>(red, i / D, i % D, &vm[k], &vl[k], &va[k]);
    }
    publish(va, vm, vl, failed);
  }

  if (late_trigger) pdl_trigger();
  // ---------------- merge over the cluster ----------------
  // Rank k of the cluster merges outputs [k * per, (k + 1) * per). Every CTA
  // has pushed its (m, l) and, for each rank, the slice of its accumulator
  // that rank merges into that rank's receive area (distributed shared-memory
  // stores made by the fold above); after one cluster barrier each CTA merges its
  // slice from its own shared memory: a narrow slice one output per 16 lanes
  // (lane r holds rank r; the max and the sums are shuffle reductions), a
  // wide one one output per thread. Nothing is read remotely, so a CTA may
  // leave as soon as it has merged.
  const int e0 = rank * per;
  const int e1 = min(E, e0 + per);
  if (CS > 1) {
    cluster_arrive_release();
    cluster_wait_acquire();
  }
  constexpr int kLaneOutputs = 2 * (Shape::kThreads / 32);  // outputs per pass of the 16-lane merge
  if (CS == 1) {
    // emitted by the fold above
  } else if (e1 - e0 > 2 * kLaneOutputs) {
    // A wide slice over few ranks: one thread per output, ranks in turn.
    for (int i = e0 + (int)threadIdx.x; i < e1; i += Shape::kThreads) {
      const int g = i / D;
      float mm = -INFINITY;
#pragma unroll
      for (int r = 0; r < kMaxCluster; ++r)
        if (r < CS) mm = fmaxf(mm, ml_in[r * 2 * G + g]);
      float ls = 0.f, as = 0.f;
#pragma unroll
      for (int r = 0; r < kMaxCluster; ++r) {
        if (r < CS) {
          const float mr = ml_in[r * 2 * G + g];
          const float f = (mr == -INFINITY) ? 0.f : fast_exp2(mr - mm);
          ls = fmaf(ml_in[r * 2 * G + G + g], f, ls);
          as = fmaf(acc_in[r * per + (i - e0)], f, as);
        }
      }
      emit(i, mm, ls, as);
    }
  } else {
    // A narrow slice (at most two passes): 16 lanes per output, lane r
    // holding rank r; the max and the two sums are xor-shuffle reductions
    // over those lanes (all loads independent).
    static_assert(kMaxCluster <= 16, "16 lanes per output cover every rank of a cluster");
    const int r = lane & 15;
    const int n_out = e1 - e0;
    for (int j0 = warp * 2; j0 < n_out; j0 += kLaneOutputs) {
      const int j = j0 + (lane >> 4);
      const bool ok = r < CS && j < n_out;
      const int i = e0 + min(j, n_out - 1);
      const int g = i / D;
      const float mr = ok ? ml_in[r * 2 * G + g] : -INFINITY;
      const float lr = ok ? ml_in[r * 2 * G + G + g] : 0.f;
      const float ar = ok ? acc_in[r * per + (i - e0)] : 0.f;
      float mm = mr;
#pragma unroll
      for (int off = 8; off >= 1; off >>= 1) mm = fmaxf(mm, __shfl_xor_sync(0xffffffffu, mm, off));
      const float w = (mr == -INFINITY) ? 0.f : fast_exp2(mr - mm);
      float ls = lr * w, as = ar * w;
#pragma unroll
      for (int off = 8; off >= 1; off >>= 1) {
        ls += __shfl_xor_sync(0xffffffffu, ls, off);
        as += __shfl_xor_sync(0xffffffffu, as, off);
      }
      if (r == 0 && j < n_out) emit(i, mm, ls, as);
    }
  }

  if (nclusters > 1) {
    // Several clusters: the last CTA of the group to arrive merges the
    // cluster partials (written by other SMs, so read from L2).
    __syncthreads();
    if (threadIdx.x == 0) {
      const int last = arrive_count(p.counters + (int64_t)b * p.n_kv_head + g_kv, nclusters * CS, p.err_flag);
      *reinterpret_cast<volatile int*>(last_flag) = last;
    }
    __syncthreads();
    const int last = *reinterpret_cast<volatile int*>(last_flag);
    if (last > 0) {
      // the ring is idle now
      if (nclusters > merge_one_trip<D, G, Shape::kThreads>() &&
          (int64_t)G * (nclusters * (D + 3) + 1) * 4 <= Shape::kRingBytes) {
        merge_partials_smem<T, D, G, Shape::kThreads>(p, head0, nclusters, p.splits / CS, smem, merge_bar);
      } else {
        merge_partials<T, D, G, Shape::kThreads>(p, head0, nclusters, p.splits / CS, reinterpret_cast<float*>(smem));
      }
    } else if (last < 0) {
      for (int i = threadIdx.x; i < E; i += Shape::kThreads)
        reinterpret_cast<uint16_t*>(p.out)[head0 * D + i] = S::kNaN;
    }
  }
}

}  // namespace da
