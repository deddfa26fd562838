// Shared device helpers of the decode-attention library (sm_103a).
//
// Inline PTX wrappers for the mbarrier / bulk-copy (TMA) pipeline, the
// programmatic-dependent-launch controls, fp16/bf16 <-> fp32 conversion and
// the split geometry of the decode kernel.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace da {

// Bits of the device error word (mirrors DA_DEVERR_* of the public header).
constexpr int32_t kErrKvLen = 1;
constexpr int32_t kErrPosition = 2;
constexpr int32_t kErrTimeout = 4;
constexpr int32_t kErrWorkspace = 8;

// A pipeline wait gives up after this long and reports kErrTimeout.
constexpr unsigned long long kWaitLimitNs = 1000ull * 1000ull * 1000ull;  // 1 s

// Decode kernel pipeline: one stage holds kTileBytes of K rows and as many
// bytes of V rows.
constexpr int kTileBytes = 16384;
constexpr int kMaxSplits = 128;
// Largest thread-block cluster of split CTAs (the non-portable hardware limit).
constexpr int kMaxClusterSize = 16;
// A group whose splits would stream at most this many tiles each (twice as
// many for instances that run one CTA per SM) is served by one thread-block
// cluster (on-chip merge); longer prefixes are split over every resident CTA
// and merged through the workspace.
constexpr int kClusterTilesPerSplit = 4;
// Kernel flavours of the instances with four or more query heads per KV
// head (InstanceConfig in decode_kernel.cuh): tensor-core scores with one CTA
// per SM, the same with two CTAs per SM, and CUDA-core scores.
constexpr int kFlavorWide = 0;
constexpr int kFlavorPair = 1;
constexpr int kFlavorCudaCores = 2;
// The workspace starts with one 32-bit arrival counter per (sequence, KV
// head) group, in a fixed region so that calls of any shape find their
// counters at the same place; split decoding is used only for at most
// kMaxCounterGroups groups (more groups fill the GPU without splitting).
constexpr int kMaxCounterGroups = 1024;
constexpr int kCounterBytes = kMaxCounterGroups * 4;

__host__ __device__ constexpr int tile_rows(int head_dim) { return kTileBytes / (2 * head_dim); }

// Rows per split for a sequence of L active rows cut into at most S splits:
// an even share rounded up to whole tiles.
__host__ __device__ inline int split_chunk(int L, int S, int rows_per_tile) {
  const int share = (L + S - 1) / S;
  return ((share + rows_per_tile - 1) / rows_per_tile) * rows_per_tile;
}

__host__ __device__ inline int active_splits(int L, int chunk) { return (L + chunk - 1) / chunk; }

// ---------------------------------------------------------------------------
// PTX wrappers.

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Wait for the phase of the given parity to complete; false after
// kWaitLimitNs without completion.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_ns() - t0 > kWaitLimitNs) return false;
  }
  return true;
}

// L2 policy for data streamed once.
__device__ __forceinline__ uint64_t evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// Bulk (non-tensor) TMA copy global -> shared, completing on `bar`.
// Both addresses 16-byte aligned, bytes a positive multiple of 16.
__device__ __forceinline__ void bulk_load(void* smem_dst, const void* gmem_src, uint32_t bytes, uint64_t* bar,
                                          uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::
          "r"(smem_addr(smem_dst)),
      "l"(gmem_src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

// The same without a cache hint.
__device__ __forceinline__ void bulk_load_plain(void* smem_dst, const void* gmem_src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_addr(smem_dst)),
               "l"(gmem_src), "r"(bytes), "r"(smem_addr(bar))
               : "memory");
}

// Orders this thread's earlier generic-proxy view of global memory (for
// instance data acquired from other CTAs) before its later bulk copies.
__device__ __forceinline__ void fence_proxy_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }

// Bulk prefetch of global memory into L2 (no completion tracking). Address
// 16-byte aligned, bytes a positive multiple of 16.
__device__ __forceinline__ void prefetch_l2(const void* gmem, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(gmem), "r"(bytes) : "memory");
}

// Thread-block cluster barrier (every thread of every CTA of the cluster
// arrives once per phase; release/acquire order the shared-memory writes
// before it against the distributed reads after it).
__device__ __forceinline__ void cluster_arrive_release() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Store a float at the same shared-memory offset as `local` in the CTA of
// the given rank in this cluster (distributed shared memory).
__device__ __forceinline__ void st_cluster_f32(float* local, int rank, float v) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_addr(local)), "r"(rank));
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(remote), "f"(v) : "memory");
}

// ---------------------------------------------------------------------------
// Tensor-memory scores (fifth-generation tensor cores, sm_100 family).
//
// The score tile S^T = K q^T of the instances with several query heads per
// KV head runs as tcgen05.mma (kind::f16: fp16 or bf16 operands, fp32
// accumulation) with the K tile (A, M = 128 rows) and the q operand (B,
// N = 16 rows: the group's heads, the rest zero) in shared memory, both
// K-major with the 128-byte swizzle that TMA tensor copies write, and the
// accumulator in tensor memory (row i of S^T in lane i).

// Opaque copy of a CUtensorMap (a 128-byte, 64-byte aligned descriptor that
// the host encodes with cuTensorMapEncodeTiled).
struct alignas(64) TensorMap {
  unsigned long long words[16];
};

// 3-D tiled TMA copy global -> shared: the box at element coordinates
// (x, y, z) of `map`, completing on `bar`. x * element size must be a
// multiple of 16 bytes.
__device__ __forceinline__ void tensor_load_3d(void* smem_dst, const TensorMap* map, int x, int y, int z,
                                               uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_addr(smem_dst)),
      "l"(map), "r"(x), "r"(y), "r"(z), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

// Orders this thread's generic-proxy shared-memory writes before later
// async-proxy reads of them (the tensor core reading an operand).
__device__ __forceinline__ void fence_proxy_async_shared() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Tensor-memory allocation of `cols` columns (a power of two >= 32) by one
// whole warp; the base address is written to *slot.
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t cols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(slot)), "r"(cols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_free(uint32_t base, uint32_t cols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(base), "r"(cols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor of a K-major operand in the 128-byte
// swizzle layout: 8-row atoms of 128-byte rows, 1024 bytes apart (stride
// byte offset); the leading byte offset is unused in this layout.
__device__ __forceinline__ uint64_t sw128_desc(const void* smem_ptr) {
  const uint32_t a = smem_addr(smem_ptr);
  return (uint64_t)((a & 0x3FFFFu) >> 4) | (1ull << 16) | ((uint64_t)(1024 >> 4) << 32) | (1ull << 46) |
         (2ull << 61);
}

// Instruction descriptor of kind::f16 with fp32 accumulation, both operands
// K-major, M = 128 and N = 16; `bf16` selects bf16 operands (else fp16).
__host__ __device__ constexpr uint32_t mma_idesc_m128_n16(bool bf16) {
  return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) | ((16u >> 3) << 17) | ((128u >> 4) << 24);
}

// D (tensor memory) = A B^T (+ D when `accumulate`), issued by one thread.
__device__ __forceinline__ void mma_f16_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          bool accumulate) {
  asm volatile(
      "{\n\t.reg .pred acc;\n\tsetp.ne.b32 acc, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, acc;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"((uint32_t)accumulate)
      : "memory");
}

// Arrive once on `bar` when every tcgen05.mma this thread issued before has completed.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
               : "memory");
}

// This warp's 32 lanes of tensor memory (the lanes of its subpartition),
// N consecutive 32-bit columns from `taddr`, then wait for the load.
template <int N>
__device__ __forceinline__ void tmem_load(uint32_t taddr, uint32_t (&r)[N]) {
  static_assert(N == 4 || N == 8, "4 or 8 columns");
  if constexpr (N == 4) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(taddr)
                 : "memory");
  } else {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr)
                 : "memory");
  }
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Named barrier ID over COUNT threads (whole warps).
template <int ID, int COUNT>
__device__ __forceinline__ void named_barrier_sync() {
  asm volatile("bar.sync %0, %1;" ::"n"(ID), "n"(COUNT) : "memory");
}

// Named barrier ID over COUNT threads that also returns whether any of them
// passed true.
template <int ID, int COUNT>
__device__ __forceinline__ bool named_barrier_or(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred pi, po;\n\tsetp.ne.u32 pi, %1, 0;\n\t"
      "bar.red.or.pred po, %2, %3, pi;\n\tselp.u32 %0, 1, 0, po;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v), "n"(ID), "n"(COUNT)
      : "memory");
  return r != 0;
}

// Programmatic dependent launch: wait for the preceding grid's memory, and
// allow the following grid to be scheduled.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint4 ld_shared_v4(const void* p) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(smem_addr(p)));
  return v;
}

__device__ __forceinline__ uint4 ld_global_nc_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// ---------------------------------------------------------------------------
// Storage types.

template <typename T>
struct Storage;

template <>
struct Storage<__nv_bfloat16> {
  // a0 += q.lo * k.lo, a1 += q.hi * k.hi for two packed bf16 pairs, each
  // product exact in fp32 and the sum rounded once (mixed-precision FMA).
  static __device__ __forceinline__ void dot2(uint32_t q2, uint32_t k2, float& a0, float& a1) {
    asm("{\n\t.reg .b16 ql, qh, kl, kh;\n\t"
        "mov.b32 {ql, qh}, %2;\n\t"
        "mov.b32 {kl, kh}, %3;\n\t"
        "fma.rn.f32.bf16 %0, ql, kl, %0;\n\t"
        "fma.rn.f32.bf16 %1, qh, kh, %1;\n\t}"
        : "+f"(a0), "+f"(a1)
        : "r"(q2), "r"(k2));
  }
  // 8 packed bf16 -> fp32 (exact: bf16 is the top half of an fp32).
  static __device__ __forceinline__ void unpack(const uint4& v, float (&f)[8]) {
    f[0] = __uint_as_float(v.x << 16);
    f[1] = __uint_as_float(v.x & 0xffff0000u);
    f[2] = __uint_as_float(v.y << 16);
    f[3] = __uint_as_float(v.y & 0xffff0000u);
    f[4] = __uint_as_float(v.z << 16);
    f[5] = __uint_as_float(v.z & 0xffff0000u);
    f[6] = __uint_as_float(v.w << 16);
    f[7] = __uint_as_float(v.w & 0xffff0000u);
  }
  // 8 packed bf16 -> 4 fp32 pairs.
  static __device__ __forceinline__ void unpack2(const uint4& v, float2 (&f)[4]) {
    f[0] = make_float2(__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xffff0000u));
    f[1] = make_float2(__uint_as_float(v.y << 16), __uint_as_float(v.y & 0xffff0000u));
    f[2] = make_float2(__uint_as_float(v.z << 16), __uint_as_float(v.z & 0xffff0000u));
    f[3] = make_float2(__uint_as_float(v.w << 16), __uint_as_float(v.w & 0xffff0000u));
  }
  static __device__ __forceinline__ uint16_t round(float x) { return __bfloat16_as_ushort(__float2bfloat16_rn(x)); }
  static constexpr uint16_t kNaN = 0x7FC0;
  static constexpr bool kBf16 = true;
};

template <>
struct Storage<__half> {
  static __device__ __forceinline__ void dot2(uint32_t q2, uint32_t k2, float& a0, float& a1) {
    asm("{\n\t.reg .b16 ql, qh, kl, kh;\n\t"
        "mov.b32 {ql, qh}, %2;\n\t"
        "mov.b32 {kl, kh}, %3;\n\t"
        "fma.rn.f32.f16 %0, ql, kl, %0;\n\t"
        "fma.rn.f32.f16 %1, qh, kh, %1;\n\t}"
        : "+f"(a0), "+f"(a1)
        : "r"(q2), "r"(k2));
  }
  static __device__ __forceinline__ float2 pair(uint32_t u) {
    __half2 h = *reinterpret_cast<__half2*>(&u);
    return __half22float2(h);
  }
  static __device__ __forceinline__ void unpack(const uint4& v, float (&f)[8]) {
    float2 a = pair(v.x), b = pair(v.y), c = pair(v.z), d = pair(v.w);
    f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
    f[4] = c.x; f[5] = c.y; f[6] = d.x; f[7] = d.y;
  }
  static __device__ __forceinline__ void unpack2(const uint4& v, float2 (&f)[4]) {
    f[0] = pair(v.x);
    f[1] = pair(v.y);
    f[2] = pair(v.z);
    f[3] = pair(v.w);
  }
  static __device__ __forceinline__ uint16_t round(float x) { return __half_as_ushort(__float2half_rn(x)); }
  static constexpr uint16_t kNaN = 0x7E00;
  static constexpr bool kBf16 = false;
};

// Rotary position embedding of one 16-byte vector x (8 elements at columns
// [8c, 8c + 8) of a head) given the vector y at the same place in the other
// half of the head, and that row's cos and sin: x * cos - y * sin in the
// first half, x * cos + y * sin in the second (x * cos + rotate_half(x) *
// sin). Each product and the sum are rounded to fp32 separately (no fused
// multiply-add), and the result once to the storage type.
template <typename T>
__device__ __forceinline__ uint4 rope_vec8(const uint4& x, const uint4& y, const float (&cs)[8], const float (&sn)[8],
                                           bool first_half) {
  float xf[8], yf[8];
  Storage<T>::unpack(x, xf);
  Storage<T>::unpack(y, yf);
  uint16_t r[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const float a = __fmul_rn(xf[e], cs[e]);
    const float b = __fmul_rn(yf[e], sn[e]);
    r[e] = Storage<T>::round(first_half ? __fsub_rn(a, b) : __fadd_rn(a, b));
  }
  uint4 v;
  v.x = (uint32_t)r[0] | ((uint32_t)r[1] << 16);
  v.y = (uint32_t)r[2] | ((uint32_t)r[3] << 16);
  v.z = (uint32_t)r[4] | ((uint32_t)r[5] << 16);
  v.w = (uint32_t)r[6] | ((uint32_t)r[7] << 16);
  return v;
}

__device__ __forceinline__ uint4 shfl_xor_v4(const uint4& v, int mask) {
  uint4 r;
  r.x = __shfl_xor_sync(0xffffffffu, v.x, mask);
  r.y = __shfl_xor_sync(0xffffffffu, v.y, mask);
  r.z = __shfl_xor_sync(0xffffffffu, v.z, mask);
  r.w = __shfl_xor_sync(0xffffffffu, v.w, mask);
  return r;
}

// The 8 fp32 values at columns [col, col + 8) of row `row` of a table with
// `width` columns (16-byte aligned).
__device__ __forceinline__ void load_f32x8(const float* table, int64_t row, int width, int col, float (&out)[8]) {
  const uint8_t* p = reinterpret_cast<const uint8_t*>(table + row * width + col);
  const uint4 a = ld_global_nc_v4(p);
  const uint4 b = ld_global_nc_v4(p + 16);
  out[0] = __uint_as_float(a.x);
  out[1] = __uint_as_float(a.y);
  out[2] = __uint_as_float(a.z);
  out[3] = __uint_as_float(a.w);
  out[4] = __uint_as_float(b.x);
  out[5] = __uint_as_float(b.y);
  out[6] = __uint_as_float(b.z);
  out[7] = __uint_as_float(b.w);
}

// Parameters of one decode-kernel launch.
struct alignas(64) DecodeParams {
  // Instances with tensor-memory scores: the K cache as a 3-D tensor
  // [B * n_kv_head][capacity][D] with a box of one tile's rows (k_tiles) and
  // of 8 rows (k_rows8, for the last partial tile), 64 columns wide, 128-byte
  // swizzle. Unused by the other instances.
  TensorMap k_tiles;
  TensorMap k_rows8;
  const uint8_t* q;        // [B, n_head, D]
  const uint8_t* k_cache;  // [B, n_kv_head, capacity, D]
  const uint8_t* v_cache;
  uint8_t* k_cache_w;      // fused step: caches to write the new row into (else null)
  uint8_t* v_cache_w;
  const uint8_t* k_new;    // fused step: [B, n_kv_head, D] (else null)
  const uint8_t* v_new;
  const int32_t* lens;     // kv_len, or position_ids when lens_are_positions
  int lens_are_positions;
  int lens_period;         // entries of `lens`: sequence b reads lens[b % lens_period]
  int B, n_head, n_kv_head, capacity, splits;
  const float* rope_cos;   // fused step with rotary embedding: tables [rope_rows, D] (else null)
  const float* rope_sin;
  int rope_rows;
  int len_hint;            // host bound on the active lengths (<= capacity): L2 prefetch, early tiles
  int skip_slot;           // test hook: ring slot left unfilled in one CTA (< 0: none)
  int speculate;           // 1: len_hint is expected to be the exact length (early tiles are issued)
  int prefix_ready;        // with speculate: the early tiles' cached rows may be read before the grid wait
  int cluster;             // CTAs per thread-block cluster along the split axis (divides splits)
  float qscale;            // softmax scale * log2(e)
  uint8_t* out;            // [B, n_head, D]
  float* ws_acc;           // [B, n_head, splits / cluster, D]: one partial per cluster
  float* ws_ml;            // [B, n_head, splits / cluster, 2]: running max (log2 units), sum
  unsigned int* counters;  // [B, n_kv_head] arrival counters of the split groups
  int32_t* err_flag;       // may be null
};

// Active length of sequence b, or -1 when its input is out of range
// (setting the matching error bit in *err).
__device__ __forceinline__ int sequence_length(const DecodeParams& p, int b, int32_t* err_bits) {
  const int v = p.lens[p.lens_period == p.B ? b : b % p.lens_period];
  if (p.lens_are_positions) {
    if (v < 0 || v >= p.capacity) {
      *err_bits = kErrPosition | kErrKvLen;
      return -1;
    }
    return v + 1;
  }
  if (v < 1 || v > p.capacity) {
    *err_bits = kErrKvLen;
    return -1;
  }
  return v;
}

}  // namespace da
