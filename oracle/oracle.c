/*
 * Decode-attention oracle: the plain fp64 CPU definition of one single-query
 * (q_len = 1) attention step over the active prefix of a static KV cache, and
 * of the in-place append of one K/V row per (sequence, KV head).
 *
 * TEST INFRASTRUCTURE. This file is the checker, not the product: only the
 * test suite, the smoke check and the benchmark's CPU-baseline leg may load
 * it. It shares no code, header, table or helper with the CUDA library, and
 * the CUDA library never calls it.
 *
 * What it follows:
 *  - fish-speech issue #1310, "Optimize native AR decoding by attending only
 *    to the active KV-cache prefix", section 2 ("What is your suggested
 *    solution?"): the cache keeps its physical size max_seq_len, attention
 *    reads only k[:, :, :kv_len] and v[:, :, :kv_len], and query heads are
 *    served by KV heads through repeat_interleave on the head axis.
 *  - VoxCPM issue #395, "MiniCPM4 MiniCPMAttention.forward_step Attention
 *    Performance Fix", section 3 (the fix) and section 4.1 (the patched
 *    forward_step): the new row is written in place at position_id, then
 *    attention runs on [0, position_id] with enable_gqa, so kv_len =
 *    position_id + 1, and position 0 reduces to returning V[0].
 *  - Cuda-Compute-OSS issue #343, "one-token decode fast path", section
 *    "Proposed implementation": out = softmax(q K^T / sqrt(d)) V with the
 *    softmax max-subtracted; the caller passes the scale (1/sqrt(d) there).
 *
 * Everything is computed in double precision from the decoded 16-bit inputs;
 * nothing is blocked, fused or reordered beyond the definition.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORACLE_F16 = 0, ORACLE_BF16 = 1 };

enum {
  ORACLE_OK = 0,
  ORACLE_ERR_ARGS = -1,
  ORACLE_ERR_NOMEM = -2
};

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
static double decode_f16(uint16_t h) {
  int sign = (h >> 15) & 1;
  int expo = (h >> 10) & 0x1f;
  int frac = h & 0x3ff;
  double mag;
  if (expo == 0) {
    mag = ldexp((double)frac, -24); /* subnormal: frac * 2^-24 */
  } else if (expo == 31) {
    mag = frac ? NAN : INFINITY;
  } else {
    mag = ldexp((double)(1024 + frac), expo - 25); /* (1 + frac/1024) * 2^(expo-15) */
  }
  return sign ? -mag : mag;
}

/* bfloat16: 1 sign bit, 8 exponent bits (bias 127), 7 fraction bits. */
static double decode_bf16(uint16_t h) {
  int sign = (h >> 15) & 1;
  int expo = (h >> 7) & 0xff;
  int frac = h & 0x7f;
  double mag;
  if (expo == 0) {
    mag = ldexp((double)frac, -133); /* subnormal: frac * 2^-133 */
  } else if (expo == 255) {
    mag = frac ? NAN : INFINITY;
  } else {
    mag = ldexp((double)(128 + frac), expo - 134); /* (1 + frac/128) * 2^(expo-127) */
  }
  return sign ? -mag : mag;
}

static double decode(uint16_t h, int dtype) {
  return dtype == ORACLE_BF16 ? decode_bf16(h) : decode_f16(h);
}

/* Decode n raw 16-bit values to double (exposed so that the decoders can be
 * checked against other implementations of the two formats). */
int oracle_decode_bits(const uint16_t* bits, int64_t n, int dtype, double* out) {
  if (!bits || !out || n < 0 || (dtype != ORACLE_F16 && dtype != ORACLE_BF16))
    return ORACLE_ERR_ARGS;
  for (int64_t i = 0; i < n; ++i) out[i] = decode(bits[i], dtype);
  return ORACLE_OK;
}

/*
 * One decode-attention step.
 *
 *   q        [B, n_head, head_dim]                 raw 16-bit values
 *   k_cache  [B, n_kv_head, capacity, head_dim]    raw 16-bit values
 *   v_cache  [B, n_kv_head, capacity, head_dim]    raw 16-bit values
 *   kv_len   [B]                                   active prefix length per sequence
 *   out      [B, n_head, head_dim]                 double
 *
 * For every sequence b and query head h, with G = n_head / n_kv_head and the
 * KV head g = h / G that repeat_interleave assigns to h, and L = kv_len[b]:
 *   x_j    = scale * sum_d q[b,h,d] * K[b,g,j,d]         for j in [0, L)
 *   m      = max_j x_j
 *   w_j    = exp(x_j - m)
 *   out[d] = sum_j w_j * V[b,g,j,d] / sum_j w_j
 * Rows j >= L are never read. A kv_len outside [1, capacity] is a caller
 * error; that output row is NaN.
 *
 * n_threads > 1 runs the independent (b, h) rows on that many OpenMP threads
 * (when built with OpenMP); each row's arithmetic is unchanged.
 */
int oracle_decode_attn(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                       const int32_t* kv_len, int B, int n_head, int n_kv_head, int head_dim,
                       int capacity, int dtype, double scale, double* out, int n_threads) {
  if (!q || !k_cache || !v_cache || !kv_len || !out) return ORACLE_ERR_ARGS;
  if (B < 0 || n_head < 1 || n_kv_head < 1 || head_dim < 1 || capacity < 1) return ORACLE_ERR_ARGS;
  if (n_head % n_kv_head != 0) return ORACLE_ERR_ARGS;
  if (dtype != ORACLE_F16 && dtype != ORACLE_BF16) return ORACLE_ERR_ARGS;
  const int G = n_head / n_kv_head;
  const int64_t rows = (int64_t)B * n_head;
  int status = ORACLE_OK;
  if (n_threads < 1) n_threads = 1;

#pragma omp parallel for schedule(dynamic, 1) num_threads(n_threads)
  for (int64_t bh = 0; bh < rows; ++bh) {
    const int b = (int)(bh / n_head);
    const int h = (int)(bh % n_head);
    const int g = h / G;
    const int L = kv_len[b];
    double* o = out + bh * head_dim;
    if (L < 1 || L > capacity) {
      for (int d = 0; d < head_dim; ++d) o[d] = NAN;
      continue;
    }
    const uint16_t* qr = q + bh * head_dim;
    const uint16_t* K = k_cache + ((int64_t)b * n_kv_head + g) * capacity * head_dim;
    const uint16_t* V = v_cache + ((int64_t)b * n_kv_head + g) * capacity * head_dim;
    double* x = (double*)malloc(sizeof(double) * (size_t)L);
    if (!x) {
#pragma omp atomic write
      status = ORACLE_ERR_NOMEM;
      for (int d = 0; d < head_dim; ++d) o[d] = NAN;
      continue;
    }
    for (int j = 0; j < L; ++j) {
      double dot = 0.0;
      for (int d = 0; d < head_dim; ++d)
        dot += decode(qr[d], dtype) * decode(K[(int64_t)j * head_dim + d], dtype);
      x[j] = scale * dot;
    }
    double m = x[0];
    for (int j = 1; j < L; ++j)
      if (x[j] > m) m = x[j];
    double Z = 0.0;
    for (int j = 0; j < L; ++j) {
      x[j] = exp(x[j] - m); /* x now holds the weights w_j */
      Z += x[j];
    }
    for (int d = 0; d < head_dim; ++d) {
      double acc = 0.0;
      for (int j = 0; j < L; ++j) acc += x[j] * decode(V[(int64_t)j * head_dim + d], dtype);
      o[d] = acc / Z;
    }
    free(x);
  }
  return status;
}

/*
 * In-place append of the new K/V rows (VoxCPM issue #395, section 4.1:
 * key_cache[:, :, position_id, :] = key_states, and the same for V).
 *
 *   k_new, v_new  [B, n_kv_head, head_dim]   raw 16-bit values
 *   position_ids  [B]
 * The row is copied bit for bit. A position outside [0, capacity) is a
 * caller error: that sequence's rows are left untouched and the returned
 * count includes it.
 * Returns the number of sequences whose position was out of range, or a
 * negative error for bad arguments.
 */
int oracle_kvcache_append(uint16_t* k_cache, uint16_t* v_cache, const uint16_t* k_new,
                          const uint16_t* v_new, const int32_t* position_ids, int B,
                          int n_kv_head, int head_dim, int capacity) {
  if (!k_cache || !v_cache || !k_new || !v_new || !position_ids) return ORACLE_ERR_ARGS;
  if (B < 0 || n_kv_head < 1 || head_dim < 1 || capacity < 1) return ORACLE_ERR_ARGS;
  int bad = 0;
  for (int b = 0; b < B; ++b) {
    const int p = position_ids[b];
    if (p < 0 || p >= capacity) {
      ++bad;
      continue;
    }
    for (int g = 0; g < n_kv_head; ++g) {
      const int64_t src = ((int64_t)b * n_kv_head + g) * head_dim;
      const int64_t dst = (((int64_t)b * n_kv_head + g) * capacity + p) * head_dim;
      memcpy(k_cache + dst, k_new + src, sizeof(uint16_t) * (size_t)head_dim);
      memcpy(v_cache + dst, v_new + src, sizeof(uint16_t) * (size_t)head_dim);
    }
  }
  return bad;
}

/* Number of OpenMP threads a parallel region would use (1 without OpenMP). */
int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
