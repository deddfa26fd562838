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

/*
 * Rotary position embedding of the query and of the new key row, as the
 * patched forward_step applies it before the append (VoxCPM issue #395,
 * section 4.1: query_states, key_states = apply_rotary_pos_emb(query_states,
 * key_states, cos, sin), with (cos, sin) the position embedding of the
 * current position). The pages do not print apply_rotary_pos_emb; this takes
 * the usual half-rotation form of the MiniCPM / Llama family:
 *
 *   out = x * cos + rotate_half(x) * sin,  rotate_half(x) = [-x[D/2:], x[:D/2]]
 *
 * with cos and sin given as rows of two tables [rows, head_dim] indexed by
 * the sequence's position. The rotated vector is rounded to the storage type
 * (round to nearest even), as the pages' tensors are. Because that rounding
 * decides stored bits, the arithmetic is fixed exactly: the 16-bit x is
 * widened to fp32 (exact), each product is rounded to fp32, their sum (or
 * difference) is rounded to fp32 (no fused multiply-add), and that fp32 value
 * is rounded once to fp16 or bf16.
 */

/* fp32 -> IEEE 754 binary16, round to nearest even, overflow to infinity.
 * NaN becomes the quiet NaN 0x7E00. */
static uint16_t encode_f16(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  const uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
  const uint32_t expo = (u >> 23) & 0xffu;
  uint32_t mant = u & 0x7fffffu;
  if (expo == 0xffu) return (uint16_t)(sign | (mant ? 0x7e00u : 0x7c00u));
  /* value = (1.mant) * 2^(expo - 127) for normal fp32; binary16 has bias 15 */
  const int e = (int)expo - 127;
  if (e > 15) return (uint16_t)(sign | 0x7c00u);
  if (e >= -14) {
    /* normal half: keep 10 of the 23 fraction bits */
    uint32_t h = ((uint32_t)(e + 15) << 10) | (mant >> 13);
    const uint32_t rest = mant & 0x1fffu; /* 13 dropped bits */
    if (rest > 0x1000u || (rest == 0x1000u && (h & 1u))) h += 1u; /* may carry into the exponent: fine */
    return (uint16_t)(sign | h);
  }
  /* subnormal half (or zero): value / 2^-24 rounded to an integer */
  if (expo == 0) return sign; /* fp32 zero or subnormal: far below half's smallest subnormal */
  mant |= 0x800000u;          /* 24-bit significand, value = mant * 2^(e - 23) */
  const int shift = -e - 1;   /* value / 2^-24 = mant * 2^(e + 1) = mant >> (-e - 1) */
  if (shift > 24) return sign;
  const uint32_t q = mant >> shift;
  const uint32_t rem = mant & ((1u << shift) - 1u);
  const uint32_t half = 1u << (shift - 1);
  uint32_t h = q;
  if (rem > half || (rem == half && (q & 1u))) h += 1u; /* 0x400 carries into the smallest normal */
  return (uint16_t)(sign | h);
}

/* fp32 -> bfloat16 (the top half of an fp32), round to nearest even.
 * NaN becomes the quiet NaN 0x7FC0. */
static uint16_t encode_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x7fffffu)) return (uint16_t)(((u >> 16) & 0x8000u) | 0x7fc0u);
  const uint32_t lower = u & 0xffffu;
  uint32_t upper = u >> 16;
  if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u))) upper += 1u;
  return (uint16_t)upper;
}

static uint16_t encode(float f, int dtype) { return dtype == ORACLE_F16 ? encode_f16(f) : encode_bf16(f); }

/* fp32 -> 16-bit storage, exported for the tests of the encoders. */
int oracle_encode_f32(const float* in, int64_t n, int dtype, uint16_t* out) {
  if (!in || !out || n < 0 || (dtype != ORACLE_F16 && dtype != ORACLE_BF16)) return ORACLE_ERR_ARGS;
  for (int64_t i = 0; i < n; ++i) out[i] = encode(in[i], dtype);
  return ORACLE_OK;
}

/*
 *   x            [B, heads, head_dim]   raw 16-bit values (head_dim even)
 *   cos_table    [rows, head_dim]       fp32
 *   sin_table    [rows, head_dim]       fp32
 *   position_ids [B]                    row of the tables for sequence b
 *   out          [B, heads, head_dim]   raw 16-bit values
 * A position outside [0, rows) leaves that sequence's rows of `out`
 * untouched and is counted. Returns that count, or a negative error.
 */
int oracle_rope(const uint16_t* x, const float* cos_table, const float* sin_table, const int32_t* position_ids,
                int B, int heads, int head_dim, int rows, int dtype, uint16_t* out) {
  if (!x || !cos_table || !sin_table || !position_ids || !out) return ORACLE_ERR_ARGS;
  if (B < 0 || heads < 1 || head_dim < 2 || (head_dim & 1) || rows < 1) return ORACLE_ERR_ARGS;
  if (dtype != ORACLE_F16 && dtype != ORACLE_BF16) return ORACLE_ERR_ARGS;
  const int half = head_dim / 2;
  int bad = 0;
  for (int b = 0; b < B; ++b) {
    const int p = position_ids[b];
    if (p < 0 || p >= rows) {
      ++bad;
      continue;
    }
    const float* c = cos_table + (int64_t)p * head_dim;
    const float* s = sin_table + (int64_t)p * head_dim;
    for (int h = 0; h < heads; ++h) {
      const uint16_t* xr = x + ((int64_t)b * heads + h) * head_dim;
      uint16_t* o = out + ((int64_t)b * heads + h) * head_dim;
      for (int d = 0; d < head_dim; ++d) {
        const float xv = (float)decode(xr[d], dtype);
        float r;
        if (d < half) {
          const float yv = (float)decode(xr[d + half], dtype); /* rotate_half: -x[d + D/2] */
          const float a = xv * c[d];
          const float bb = yv * s[d];
          r = a - bb;
        } else {
          const float yv = (float)decode(xr[d - half], dtype); /* rotate_half: +x[d - D/2] */
          const float a = xv * c[d];
          const float bb = yv * s[d];
          r = a + bb;
        }
        o[d] = encode(r, dtype);
      }
    }
  }
  return bad;
}
