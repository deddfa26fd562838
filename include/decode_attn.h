/*
 * decode_attn.h — C ABI of the GB300 (sm_103a) decode-attention library.
 *
 * One autoregressive decode step of one attention layer over a STATIC,
 * preallocated KV cache: the new key/value row is written in place at
 * position_id, and a single query token per head attends to the active prefix
 * [0, kv_len) of the cache only, with kv_len = position_id + 1. Grouped-query
 * heads are served straight from their shared KV head (no expansion).
 *
 * The operation follows:
 *  - VoxCPM issue #395, "MiniCPM4 MiniCPMAttention.forward_step Attention
 *    Performance Fix", section 3 (attend to the slice [0, position_id] only;
 *    position 0 attends to one row and returns V[0]) and section 4.1 (the
 *    patched forward_step: in-place write key_cache[:, :, position_id, :],
 *    then SDPA on the slice with enable_gqa=True);
 *  - fish-speech issue #1310, "Optimize native AR decoding by attending only
 *    to the active KV-cache prefix", section 2 (the cache keeps its physical
 *    max_seq_len size; only k[:, :, :kv_len], v[:, :, :kv_len] are consumed);
 *  - Cuda-Compute-OSS issue #343, "one-token decode fast path", section
 *    "Proposed implementation" (softmax(q K^T / sqrt(d)) V, max-subtracted
 *    softmax accumulated in fp32, result cast back to the input dtype).
 *
 * Conventions for every entry point:
 *  - All tensor pointers are DEVICE pointers to contiguous row-major arrays
 *    owned by the caller, 16-byte aligned. The library never allocates,
 *    frees or synchronises; work is enqueued on `stream` (a cudaStream_t;
 *    NULL is the legacy default stream) and the call returns at once.
 *  - Layouts: q and out [B, n_head, head_dim]; k_cache and v_cache
 *    [B, n_kv_head, capacity, head_dim]; k_new and v_new
 *    [B, n_kv_head, head_dim]; kv_len and position_ids int32 [B].
 *    Query head h reads KV head h / (n_head / n_kv_head).
 *  - dtype is DA_F16 or DA_BF16 and applies to q, out and both caches.
 *    Arithmetic is fp32; out is rounded to nearest even.
 *  - Supported: head_dim in {64, 128}; n_head / n_kv_head in {1, 2, 4, 8}.
 *  - Errors the host can see (null pointers, bad sizes, misalignment, a
 *    small workspace, an unsupported shape) return a negative da_status
 *    before anything is enqueued. Facts only the device knows (a kv_len
 *    outside [1, capacity], a position outside [0, capacity)) never fault:
 *    the affected output rows become NaN, the affected cache write is
 *    skipped, and the DA_DEVERR_* bit is OR-ed into *err_flag (a device
 *    int32, may be NULL). A launch failure returns DA_ERR_CUDA.
 */
#ifndef DECODE_ATTN_H_
#define DECODE_ATTN_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define DA_API __attribute__((visibility("default")))
#else
#define DA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { DA_F16 = 0, DA_BF16 = 1 } da_dtype;

typedef enum {
  DA_OK = 0,
  DA_ERR_NULL = -1,        /* a required pointer is NULL */
  DA_ERR_SHAPE = -2,       /* a size is out of range or inconsistent */
  DA_ERR_UNSUPPORTED = -3, /* valid but not built: head_dim or group size */
  DA_ERR_WORKSPACE = -4,   /* workspace NULL or smaller than required */
  DA_ERR_CUDA = -5,        /* a CUDA runtime call or launch failed */
  DA_ERR_ALIGN = -6,       /* a pointer is not 16-byte aligned */
  DA_ERR_DTYPE = -7        /* unknown dtype code */
} da_status;

/* Bits OR-ed into *err_flag by the kernels. */
#define DA_DEVERR_KV_LEN 1u   /* some kv_len[b] outside [1, capacity]: rows of b are NaN */
#define DA_DEVERR_POSITION 2u /* some position_ids[b] outside [0, capacity): write skipped */
#define DA_DEVERR_TIMEOUT 4u  /* a pipeline wait hit its time limit: rows are NaN */
#define DA_DEVERR_WORKSPACE 8u /* the workspace counters were not zero: rows of the group are NaN */

/* Human-readable name of a da_status value (static string). */
DA_API const char* da_status_string(int status);

/* Library ABI version (major * 10000 + minor * 100 + patch). */
DA_API int da_version(void);

/*
 * Split plan of the decode kernel, a pure host computation (no CUDA call):
 * the number of KV splits S per (sequence, KV head) group for B sequences,
 * n_kv_head KV heads, head_dim and a bound max_kv_len on the active length,
 * on a GPU with num_sms multiprocessors holding ctas_per_sm decode CTAs each,
 * where one thread-block cluster of up to cluster_max CTAs per group can be
 * resident. Flat plan: S is as many splits as fit one wave of resident CTAs
 * (two waves when B > 1, since most sequences of a batch are shorter than the
 * bound), at most one per tile of max_kv_len rows and at most 128; the
 * partials go through the workspace (*cluster_size = 1). Cluster plans, where
 * the S splits of a group form one cluster of *cluster_size = S CTAs that
 * merge their partial softmax states through distributed shared memory:
 * (a) one sequence whose clusters of c = min(cluster_max, 16) CTAs cover every
 * SM (B * n_kv_head * c >= num_sms) over at least 2c tiles: S = c;
 * (b) a short prefix: S = min(c, num_sms / (B * n_kv_head), tiles /
 * ctas_per_sm rounded up) when each split then streams at most 4 tiles, and
 * no split at all (S = 1) when that S is below 2.
 * (*cluster_size is written when non-NULL.) Each sequence b then splits its
 * own kv_len[b] rows evenly over at most S CTAs, in whole tiles.
 * Returns S >= 1, or a negative da_status.
 */
DA_API int decode_attn_plan_splits(int B, int n_kv_head, int head_dim, int max_kv_len, int num_sms,
                                   int ctas_per_sm, int cluster_max, int* cluster_size);

/*
 * Bytes of scratch memory decode_attn_fwd / decode_step_fwd need for these
 * sizes on the current device, for any max_kv_len_hint <= capacity.
 * Returns 0 when no scratch is needed (one cluster serves each group), or
 * (size_t)-1 for invalid sizes or a failed device query. Otherwise the
 * workspace starts with a 4 KiB region of 32-bit arrival counters (one per
 * sequence and KV head), followed by fp32 per-cluster partials
 * [B, n_head, S / cluster, head_dim + 2]. It must be zero-filled once before
 * its first use (decode_attn_workspace_init, or any memset); every call that
 * completes leaves it ready for the next call of any shape. Calls that
 * overlap on one workspace can leave a counter non-zero: a later call then
 * merges that group early or writes NaN rows with DA_DEVERR_WORKSPACE. After
 * a DA_DEVERR_TIMEOUT or DA_DEVERR_WORKSPACE, or an overlap, zero it again.
 */
DA_API size_t decode_attn_workspace_size(int B, int n_head, int n_kv_head, int head_dim, int capacity);

/* Zero-fill a workspace on `stream` (cudaMemsetAsync; allocates nothing). */
DA_API int decode_attn_workspace_init(void* workspace, size_t workspace_bytes, void* stream);

/*
 * The split count S that decode_attn_fwd / decode_step_fwd will use for
 * these arguments on the current device, and (when cluster_size is non-NULL)
 * the cluster size. S == 1: one CTA per group writes out directly; S equal
 * to the cluster size: one cluster per group merges in distributed shared
 * memory, no workspace; S larger: one partial per cluster goes through the
 * workspace and the last CTA of each group merges them, in the same launch.
 * The plan is decode_attn_plan_splits with this device's occupancy (the
 * largest cluster size of which one cluster per group is co-resident).
 * Returns S >= 1 or a negative da_status.
 */
DA_API int decode_attn_splits_for(int B, int n_head, int n_kv_head, int head_dim, int capacity,
                                  int max_kv_len_hint, int dtype, int* cluster_size);

/* Kernels decode_attn_kernel_for reports. */
#define DA_KERNEL_CUDA_CORES 0        /* scores on the CUDA cores (every group size) */
#define DA_KERNEL_TENSOR_CORES 1      /* >= 4 query heads per KV head: scores on the tensor cores, one CTA per SM */
#define DA_KERNEL_TENSOR_CORES_PAIRED 2 /* the same with two CTAs per SM (one CTA per group filling the GPU) */

/*
 * The decode kernel that decode_attn_fwd / decode_step_fwd / the layers call
 * (rotary == 0) or decode_step_rope_fwd (rotary != 0) will launch for these
 * arguments on the current device (for the layers call pass layers * B as
 * B). With four or more query heads per KV head the scores of a K tile,
 * q K^T, are a small dense product: the library runs it on the tensor cores
 * when each CTA streams more than 4 tiles or when the groups fill the GPU one
 * CTA each, and on the CUDA cores otherwise (shorter per-tile path). Every
 * kernel computes the same softmax(q K^T * scale) V within the stated
 * tolerance (the operation of decode_attn_fwd: Cuda-Compute-OSS issue #343,
 * "Proposed implementation"); results of different kernels may differ in
 * the last bits. Sizes are validated as in decode_attn_fwd (DA_ERR_SHAPE,
 * DA_ERR_UNSUPPORTED, DA_ERR_DTYPE before any device query). Returns a
 * DA_KERNEL_* value or a negative da_status.
 */
DA_API int decode_attn_kernel_for(int B, int n_head, int n_kv_head, int head_dim, int capacity,
                                  int max_kv_len_hint, int dtype, int rotary);

/*
 * Profiling hook. When both are non-NULL, every later decode_attn_fwd /
 * decode_step_fwd call made by this host thread records event_before (a
 * cudaEvent_t) on its stream immediately before its split-KV decode kernel
 * and event_after immediately after it, so that cudaEventElapsedTime gives
 * that kernel's device time. Under stream capture the records become graph
 * nodes. NULL, NULL turns the hook off. Returns DA_OK.
 */
DA_API int da_set_timing_events(void* event_before, void* event_after);

/*
 * Ordering promise for the decode calls of this host thread (default off).
 * Every decode kernel waits, by programmatic dependent launch, for the
 * kernel before it on the stream to complete before it reads its inputs.
 * With on != 0 the caller promises, for every later call of this thread with
 * B == 1 and max_kv_len_hint > 0, that no kernel that may still be running
 * when the call's kernel starts writes the cache rows the call will read:
 * rows [0, max_kv_len_hint) of k_cache and v_cache for decode_attn_fwd, rows
 * [0, max_kv_len_hint - 1) for the fused steps (whose last row comes from
 * k_new and v_new). The kernel then copies those rows of its first tiles into
 * shared memory before that wait; q, the lengths, k_new, v_new and the rotary
 * tables are still read after it. A decode loop meets the promise when the
 * only kernels between two calls on the same caches complete before the next
 * one starts: for instance the previous layer's call and the projections
 * (kernels on this stream release their dependents only after their own wait,
 * as this library's do). Back-to-back calls on the SAME caches (one layer,
 * nothing in between) do not: the first writes row position into the rows the
 * second reads. Breaking the promise gives wrong results, never a fault.
 * Returns DA_OK.
 */
DA_API int da_set_prefix_ready(int on);

/*
 * Failure-detection test hook. With slot >= 0, every later decode call made
 * by this host thread leaves ring slot `slot` of the first split of sequence
 * 0, KV head 0 unfilled: that CTA's pipeline waits run into their time limit
 * (about one second), the CTA publishes NaN and the call sets
 * DA_DEVERR_TIMEOUT; nothing faults and the context stays usable. Zero the
 * workspace afterwards (as after any DA_DEVERR_TIMEOUT). slot < 0 turns the
 * hook off (the default). Returns DA_OK.
 */
DA_API int da_test_skip_slot(int slot);

/*
 * In-place append: k_cache[b, g, position_ids[b], :] = k_new[b, g, :] and the
 * same for V, for every sequence b and KV head g, copied bit for bit.
 * (VoxCPM issue #395, section 4.1.) A position outside [0, capacity) skips
 * that sequence and sets DA_DEVERR_POSITION.
 */
DA_API int kvcache_append(void* k_cache, void* v_cache, const void* k_new, const void* v_new,
                   const int32_t* position_ids, int B, int n_kv_head, int head_dim, int capacity,
                   int dtype, int32_t* err_flag, void* stream);

/*
 * Decode attention over the active prefix:
 *   out[b, h, :] = softmax_j(scale * <q[b, h, :], K[b, g, j, :]>) V[b, g, j, :]
 * for j in [0, kv_len[b]) and g = h / (n_head / n_kv_head). Cache rows at or
 * beyond kv_len[b] are never read. kv_len is a DEVICE array, so no host
 * synchronisation is needed; max_kv_len_hint (> 0) is an optional host bound
 * on max_b kv_len[b] that only sizes the launch (<= 0 means capacity). A
 * kv_len above the hint but within capacity is still computed correctly.
 * workspace/workspace_bytes: caller-owned device scratch of at least
 * decode_attn_workspace_size(...) bytes (may be NULL when that is 0); calls
 * that share one workspace must not overlap on the GPU.
 * (Cuda-Compute-OSS issue #343, "Proposed implementation"; VoxCPM issue
 * #395, section 4.1.)
 */
DA_API int decode_attn_fwd(const void* q, const void* k_cache, const void* v_cache, const int32_t* kv_len,
                    int B, int n_head, int n_kv_head, int head_dim, int capacity, float scale,
                    void* out, void* workspace, size_t workspace_bytes, int max_kv_len_hint,
                    int dtype, int32_t* err_flag, void* stream);

/*
 * One fused decode step: the append of kvcache_append followed by
 * decode_attn_fwd with kv_len[b] = position_ids[b] + 1, in a single pass
 * over the cache. The attended row position_ids[b] is taken from k_new/v_new
 * and also written into the cache. Same arguments, layouts and error
 * behaviour as the two calls it replaces (VoxCPM issue #395, section 4.1:
 * write at position_id, then attend over [0, position_id]).
 */
DA_API int decode_step_fwd(const void* q, void* k_cache, void* v_cache, const void* k_new,
                    const void* v_new, const int32_t* position_ids, int B, int n_head,
                    int n_kv_head, int head_dim, int capacity, float scale, void* out,
                    void* workspace, size_t workspace_bytes, int max_kv_len_hint, int dtype,
                    int32_t* err_flag, void* stream);

/*
 * decode_step_fwd with the rotary position embedding the patched
 * forward_step applies to the query and the new key before the append
 * (VoxCPM issue #395, section 4.1: apply_rotary_pos_emb(query_states,
 * key_states, cos, sin), then the write at position_id and the attention).
 * q and k_new are the vectors before rotation; for sequence b with
 * p = position_ids[b], every query head and the new key row become
 *   x * cos[p] + rotate_half(x) * sin[p],  rotate_half(x) = [-x[D/2:], x[:D/2]]
 * with each product and the sum rounded to fp32 (no fused multiply-add) and
 * the result rounded to nearest even in the storage type; the rotated key row
 * is what the cache receives. v_new is appended unchanged.
 *   rope_cos, rope_sin  device fp32 tables [rope_rows, head_dim], row p
 *                       holding the embedding of position p; 16-byte
 *                       aligned; rope_rows >= capacity (else DA_ERR_SHAPE)
 * Everything else as decode_step_fwd. NULL tables give DA_ERR_NULL.
 */
DA_API int decode_step_rope_fwd(const void* q, void* k_cache, void* v_cache, const void* k_new,
                    const void* v_new, const float* rope_cos, const float* rope_sin, int rope_rows,
                    const int32_t* position_ids, int B, int n_head, int n_kv_head, int head_dim,
                    int capacity, float scale, void* out, void* workspace, size_t workspace_bytes,
                    int max_kv_len_hint, int dtype, int32_t* err_flag, void* stream);

/*
 * decode_step_fwd for `layers` layers of one model in one call: layer l
 * reads q[l], k_new[l], v_new[l] and appends to and attends over its own
 * caches k_cache[l], v_cache[l], writing out[l]:
 *   q, out          [layers, B, n_head, head_dim]
 *   k_cache, v_cache [layers, B, n_kv_head, capacity, head_dim]
 *   k_new, v_new    [layers, B, n_kv_head, head_dim]
 * all contiguous; position_ids [B] (the same step for every layer).
 * Every layer's inputs are given at once, so no layer depends on another:
 * the stacks are one batch of layers * B sequences (sequence l * B + b has
 * position position_ids[b]) and the whole call is ONE launch of the decode
 * kernel, with no per-layer launch cost. For a caller that holds every
 * layer's inputs at once (replays, benchmarks, several independent models or
 * requests stacked on a leading axis); in a model whose layer l + 1 query
 * depends on layer l's output, call decode_step_fwd per layer instead.
 * Results equal decode_step_fwd on the flattened [layers * B, ...] batch with
 * position_ids repeated per layer, bit for bit.
 *   workspace   at least decode_attn_workspace_size(layers * B, n_head,
 *               n_kv_head, head_dim, capacity) bytes
 * Validation as decode_step_fwd, all of it before the launch: an invalid
 * argument enqueues nothing, and a launch failure (DA_ERR_CUDA) leaves every
 * layer untouched. layers < 0 or layers * B > 65535 gives DA_ERR_SHAPE,
 * layers == 0 does nothing.
 */
DA_API int decode_step_layers_fwd(const void* q, void* k_cache, void* v_cache, const void* k_new,
                    const void* v_new, const int32_t* position_ids, int layers, int B, int n_head,
                    int n_kv_head, int head_dim, int capacity, float scale, void* out, void* workspace,
                    size_t workspace_bytes, int max_kv_len_hint, int dtype, int32_t* err_flag, void* stream);

/*
 * KV-head partition of one attention layer over `world` ranks (one GPU
 * each), a pure host computation. Every (sequence, KV head) group is
 * independent (its G = n_head / n_kv_head query heads read only that KV
 * head), so rank r can own a contiguous block of KV heads with their query
 * heads and run the decode calls of this header on its block alone, with no
 * exchange of data: its caches are [B, n_kv_local, capacity, head_dim] for KV
 * heads [kv_head0, kv_head0 + n_kv_local), its q and out [B, n_head_local,
 * head_dim] for query heads [head0, head0 + n_head_local) (n_head_local =
 * G * n_kv_local), and the ranks' outputs laid side by side on the head axis,
 * in rank order, are the layer's output. KV heads are dealt as evenly as
 * possible: the first n_kv_head % world ranks hold one more; a rank holds
 * none when world > n_kv_head. (fish-speech issue #1310, section 2: the GQA
 * head map h -> h / G; the pages run on one GPU, so this partition is this
 * library's own.) Returns DA_OK, DA_ERR_SHAPE for inconsistent sizes or a
 * rank outside [0, world), DA_ERR_NULL for a NULL output pointer.
 */
DA_API int decode_attn_shard_heads(int n_head, int n_kv_head, int world, int rank, int* kv_head0,
                                   int* n_kv_local, int* head0, int* n_head_local);

/* Size of the library-owned scratch array used by
 * decode_attn_fwd_static_scratch (1 MiB per GPU that loads the library). */
#define DA_STATIC_SCRATCH_BYTES (1u << 20)

/*
 * decode_attn_fwd for callers that must not allocate GPU memory. This entry
 * point is an addition of this library; the pages have no counterpart.
 *
 * Some callers only receive input and output buffers from the framework that
 * hosts them (a plugin inside an inference server or a real-time audio
 * engine, for instance) and are not allowed to call cudaMalloc, or cannot
 * reach the memory pool that owns the device memory. This variant takes the
 * same arguments as decode_attn_fwd minus the workspace: its split partials
 * live in a file-scope device array of DA_STATIC_SCRATCH_BYTES that the
 * library holds on every GPU that loads it, until the process exits. Nothing
 * is allocated or freed by the call.
 *
 * - The first call on a device that needs scratch looks up that array's
 *   device address (cudaGetSymbolAddress, with that device current) and keeps
 *   it for the life of the process; make that first call before any stream
 *   capture on the device (a first call made while `stream` is capturing
 *   returns DA_ERR_CUDA). A device reset (cudaDeviceReset) is not supported
 *   afterwards.
 * - Arguments whose split plan needs more scratch than
 *   DA_STATIC_SCRATCH_BYTES (decode_attn_workspace_size-style need for this
 *   call's max_kv_len_hint) are rejected with DA_ERR_SHAPE before anything is
 *   enqueued; use decode_attn_fwd with your own workspace for those.
 * - Every call on a device shares the one array and leaves its partials in
 *   it. A call that needs scratch first zero-fills its own arrival counters
 *   on `stream` (a cudaMemsetAsync of 4 * B * n_kv_head bytes), and its
 *   kernels write every partial they later read, so each call is correct
 *   whatever an earlier call left in the array. Calls that overlap on the GPU
 *   (different streams without ordering, or different host threads) race on
 *   the array: their outputs may be wrong, NaN (with DA_DEVERR_WORKSPACE) or
 *   left unwritten. Keep such calls ordered; the first ordered call after an
 *   overlap is correct again, with nothing to reset.
 * Otherwise identical to decode_attn_fwd, including results bit for bit.
 */
DA_API int decode_attn_fwd_static_scratch(const void* q, const void* k_cache, const void* v_cache,
                                          const int32_t* kv_len, int B, int n_head, int n_kv_head,
                                          int head_dim, int capacity, float scale, void* out,
                                          int max_kv_len_hint, int dtype, int32_t* err_flag,
                                          void* stream);

#ifdef __cplusplus
}
#endif

#endif /* DECODE_ATTN_H_ */
