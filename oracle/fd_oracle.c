/*
 * fd_oracle.c -- plain CPU fp64 oracle for decode-step (single query token)
 * attention over a contiguous or paged KV cache.
 *
 * TEST INFRASTRUCTURE.  Only the test suite, the package smoke check and the
 * benchmark's CPU-baseline leg load this file.  It shares no code, header,
 * table or constant with the CUDA library; the two only read the same input
 * arrays.
 *
 * What it computes is the plain definition of softmax attention for one query
 * row per (sequence, query head), with a full two-pass softmax and no
 * blocking, splitting or online rescaling:
 *
 *   kvh      = qh / (num_q_heads / num_kv_heads)        (consecutive query
 *                                                        heads share a KV head)
 *   row(t)   = kv_start_idx[b] + t                       (contiguous cache)
 *            = block_table[b][t / P] * P + t % P         (paged cache)
 *   k_t[d]   = k_scale * ks(t) * dec(K[row(t)][kvh][d])
 *   v_t[d]   = v_scale * vs(t) * dec(V[row(t)][kvh][d])
 *   ks(t), vs(t) = 1                                     (per-tensor scales only)
 *            = k_scales[kvh], v_scales[kvh]              (per KV head)
 *            = k_scales[row(t) * KVH + kvh], v_scales[..] (per token and KV head)
 *   s_t      = softmax_scale * sum_d q[b][qh][d] * k_t[d]
 *   M        = max_t s_t,  w_t = exp(s_t - M),  Z = sum_t w_t
 *   out[d]   = sum_t (w_t / Z) * v_t[d]
 *   lse      = M + ln Z           (natural log of sum_t exp(s_t))
 *
 * With q_len > 1 query tokens per sequence (fdo_decode_attention_q: a
 * speculative-decoding verify batch, "Learn CUDA from scratch, chapter 15",
 * section 15.21), the last q_len tokens of each sequence are the new ones:
 * query token j (q[b][qh][j], j < q_len) sits at position T_b - q_len + j and
 * attends over t = 0 .. T_b - q_len + j (its own and every earlier key), with
 * the same definition; a query with no key gets out = 0 and lse = -inf.
 *
 * Sources, by page and section:
 *  - scaled dot product, softmax and the weighted sum of V rows: "SGLang
 *    Prefill optimisation: dissecting FlashAttention kernel bottlenecks with
 *    GPU Trace", section 2.2 (the score is dot(q, k) times a scale; the
 *    weights are the exponentials normalised by their sum; the output is
 *    the weighted sum of V);
 *  - per-sequence start index and length of a variable-length batch: "From
 *    SGLang kernel source to GPU trace: DeepSeek V4.1 Flash-Decode",
 *    section 3.1 (kernel arguments kv_start_idx and seq_len);
 *  - page addressing: "Learn CUDA from scratch, chapter 15: GPU profiling and
 *    LLM inference", section 15.26 (physical page from the block table, then
 *    (page * page_size + offset) rows into a [page, offset, head, dim] pool);
 *  - GQA grouping (group = QH / KVH query heads per KV head): same chapter,
 *    section 15.12;
 *  - FP8 and INT8 scales: the decoded code times a fp32 scale, the KV
 *    quantisation of section 15.11 of the same chapter (FP8 or INT8 K/V
 *    payloads with scale metadata read next to them), which names the scale
 *    granularity (one per tensor, per head or per token) as part of the method.
 *
 * Readings where the pages are silent: the contiguous cache is token-major
 * [rows, KVH, D] with kv_start_idx in rows; LSE is in natural log of the
 * scaled scores (softmax_scale and k_scale included); seq_len = 0 gives
 * out = 0 and lse = -inf.  FP8 is OCP e4m3fn (bias 7, no infinities, S.1111.111
 * is NaN and is rejected).  INT8 is a symmetric signed code: the value is the
 * two's-complement integer (-128 .. 127) itself, with no zero point.
 *
 * All attention arithmetic is IEEE fp64 (build without -ffast-math).
 *
 * KV append (fdo_append_kv): the write of one new token per sequence into the
 * cache before the attention read ("Learn CUDA from scratch, chapter 15",
 * section 15.9: contiguous and paged cache write layouts, and its exercise on
 * a single-token decode append; quantisation with scales as in section
 * 15.11).  For each sequence b with positions[b] >= 0, each of its n_new new
 * tokens i (n_new > 1: the drafted tokens of a speculative verify step) and
 * each KV head h:
 *
 *   row       = row(b, positions[b] + i)        (as above)
 *   x_d       = new[b][i][h][d]                  (f16 or bf16, exact in fp32)
 *   16-bit cache: the element is stored as it is (the cache has new's dtype);
 *   8-bit cache, with QMAX = 448 (e4m3) or 127 (int8):
 *     s = k_scale                                (per tensor)
 *       = fl32(k_scale * k_scales[h])            (per KV head)
 *       = fl32(k_scale * ks), ks = fl32(amax / fl32(QMAX * k_scale)) written to
 *         k_scales[row * KVH + h], amax = max_d |x_d| (ks = 1 if amax = 0)
 *                                                (per token: scale from the row)
 *     code_d = enc(fl32(x_d / s))
 *   enc: e4m3 -- the nearest finite code, ties to the even code, magnitudes
 *        above 448 saturate to 448; int8 -- the nearest integer, ties to even,
 *        clamped to [-127, 127].
 * V likewise with v_scale and v_scales.  The scale products and the quotient
 * are taken in IEEE fp32, the precision of the device path, because they
 * decide integer codes.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { FDO_F16 = 0, FDO_BF16 = 1, FDO_E4M3 = 2, FDO_I8 = 3 };
enum { FDO_SCALE_TENSOR = 0, FDO_SCALE_HEAD = 1, FDO_SCALE_TOKEN = 2 };

enum {
  FDO_OK = 0,
  FDO_BAD_ARG = 1,
  FDO_ROW_OUT_OF_RANGE = 2,
  FDO_NAN_CODE = 3,
  FDO_NO_MEMORY = 4,
};

/* OCP 8-bit floating point, E4M3 ("e4m3fn"): 1 sign bit, 4 exponent bits with
 * bias 7, 3 mantissa bits.  Exponent field 0 holds subnormals m/8 * 2^-6;
 * S.1111.111 is NaN and there is no infinity. */
double fdo_e4m3_value(uint8_t code) {
  int s = (code >> 7) & 1;
  int e = (code >> 3) & 0xF;
  int m = code & 0x7;
  double mag;
  if (e == 0xF && m == 0x7) return NAN;
  if (e == 0)
    mag = ldexp((double)m / 8.0, -6);
  else
    mag = ldexp(1.0 + (double)m / 8.0, e - 7);
  return s ? -mag : mag;
}

/* Signed 8-bit integer, two's complement: codes 0x80 .. 0xFF are -128 .. -1. */
double fdo_i8_value(uint8_t code) {
  int v = code;
  if (v >= 128) v -= 256;
  return (double)v;
}

/* IEEE 754 binary16: 1 sign, 5 exponent bits with bias 15, 10 mantissa bits. */
double fdo_f16_value(uint16_t bits) {
  int s = (bits >> 15) & 1;
  int e = (bits >> 10) & 0x1F;
  int m = bits & 0x3FF;
  double mag;
  if (e == 0x1F) mag = m ? NAN : INFINITY;
  else if (e == 0) mag = ldexp((double)m / 1024.0, -14);
  else mag = ldexp(1.0 + (double)m / 1024.0, e - 15);
  return s ? -mag : mag;
}

/* bfloat16: the upper 16 bits of an IEEE binary32 (8 exponent bits, bias 127,
 * 7 mantissa bits). */
double fdo_bf16_value(uint16_t bits) {
  int s = (bits >> 15) & 1;
  int e = (bits >> 7) & 0xFF;
  int m = bits & 0x7F;
  double mag;
  if (e == 0xFF) mag = m ? NAN : INFINITY;
  else if (e == 0) mag = ldexp((double)m / 128.0, -126);
  else mag = ldexp(1.0 + (double)m / 128.0, e - 127);
  return s ? -mag : mag;
}

static double decode_elem(const void *base, int dtype, size_t idx) {
  if (dtype == FDO_E4M3) return fdo_e4m3_value(((const uint8_t *)base)[idx]);
  if (dtype == FDO_I8) return fdo_i8_value(((const uint8_t *)base)[idx]);
  if (dtype == FDO_BF16) return fdo_bf16_value(((const uint16_t *)base)[idx]);
  return fdo_f16_value(((const uint16_t *)base)[idx]);
}

/* Nearest e4m3 code to x (finite), ties to the even code, |x| > 448 -> 448.
 * Found by search over the 127 non-negative finite codes; sign kept (so -0
 * and negative values that round to zero give 0x80). */
uint8_t fdo_e4m3_encode(float x) {
  const int neg = signbit(x) != 0;
  double a = fabs((double)x);
  if (a > 448.0) a = 448.0;
  int best = 0;
  double best_err = a;   /* code 0 is 0.0 */
  for (int c = 1; c <= 0x7E; ++c) {
    double err = fabs(fdo_e4m3_value((uint8_t)c) - a);
    if (err < best_err || (err == best_err && (c & 1) == 0 && (best & 1) == 1)) {
      best = c;
      best_err = err;
    }
  }
  return (uint8_t)(best | (neg ? 0x80 : 0));
}

/* Nearest integer to x, ties to even, clamped to [-127, 127]; two's complement. */
uint8_t fdo_i8_encode(float x) {
  double r = floor((double)x);
  double f = (double)x - r;
  if (f > 0.5 || (f == 0.5 && fmod(r, 2.0) != 0.0)) r += 1.0;
  if (r > 127.0) r = 127.0;
  if (r < -127.0) r = -127.0;
  return (uint8_t)(int8_t)(int)r;
}

/* Row of the cache holding token t of sequence b, or -1 if out of range. */
static int64_t cache_row(const int32_t *kv_start_idx, const int32_t *block_table,
                         int block_table_stride, int page_size, int b, int t,
                         int64_t kv_rows) {
  int64_t row;
  if (block_table) {
    int64_t phys = block_table[(int64_t)b * block_table_stride + t / page_size];
    row = phys * page_size + t % page_size;
  } else {
    row = (int64_t)kv_start_idx[b] + t;
  }
  if (row < 0 || row >= kv_rows) return -1;
  return row;
}

/* The finer scale of a K or V element: 1, per KV head, or per (row, KV head). */
static double scale_at(int kind, const float *arr, int64_t row, int num_kv_heads, int kvh) {
  if (kind == FDO_SCALE_HEAD) return (double)arr[kvh];
  if (kind == FDO_SCALE_TOKEN) return (double)arr[(size_t)row * num_kv_heads + kvh];
  return 1.0;
}

/*
 * Computes out[B][QH][D] and lse[B][QH] in fp64.
 *
 * q: [B][QH][D] 16-bit patterns of q_dtype.
 * k_cache, v_cache: [rows][KVH][D] (contiguous) or [pages][P][KVH][D] (paged)
 *   elements of kv_dtype; kv_rows = number of token rows they hold.
 * Exactly one of kv_start_idx / block_table is non-NULL.
 * scale_kind: FDO_SCALE_TENSOR (k_scales, v_scales unused), FDO_SCALE_HEAD
 *   (k_scales, v_scales: [KVH]) or FDO_SCALE_TOKEN ([kv_rows][KVH], indexed by
 *   cache row like the caches); they multiply k_scale, v_scale.
 * pairs: NULL for every (b, qh), else n_pairs entries of (b, qh) to compute;
 *   the other outputs are left untouched.
 * weights: NULL, or [B][QH][weights_stride] receiving w_t / Z.
 * threads_used: NULL, or receives the number of threads that ran.
 */
int fdo_decode_attention_q(const void *q, int q_dtype, const void *k_cache, const void *v_cache,
                           int kv_dtype, const int32_t *kv_start_idx, const int32_t *block_table,
                           int block_table_stride, const int32_t *seq_len, int64_t kv_rows,
                           int batch, int q_len, int num_q_heads, int num_kv_heads, int head_dim,
                           int page_size, double softmax_scale, double k_scale, double v_scale,
                           int scale_kind, const float *k_scales, const float *v_scales,
                           const int32_t *pairs, int n_pairs, int nthreads, double *out,
                           double *lse, double *weights, int weights_stride, int *threads_used) {
  if (q_len < 1) return FDO_BAD_ARG;
  if (!q || !k_cache || !v_cache || !seq_len || !out || !lse) return FDO_BAD_ARG;
  if ((kv_start_idx == NULL) == (block_table == NULL)) return FDO_BAD_ARG;
  if (batch < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0) return FDO_BAD_ARG;
  if (num_q_heads % num_kv_heads != 0) return FDO_BAD_ARG;
  if (block_table && page_size <= 0) return FDO_BAD_ARG;
  if (q_dtype != FDO_F16 && q_dtype != FDO_BF16) return FDO_BAD_ARG;
  if (kv_dtype != FDO_F16 && kv_dtype != FDO_BF16 && kv_dtype != FDO_E4M3 && kv_dtype != FDO_I8)
    return FDO_BAD_ARG;
  if (scale_kind < FDO_SCALE_TENSOR || scale_kind > FDO_SCALE_TOKEN) return FDO_BAD_ARG;
  if (scale_kind != FDO_SCALE_TENSOR && (!k_scales || !v_scales)) return FDO_BAD_ARG;

  const int group = num_q_heads / num_kv_heads;
  const int n_work = pairs ? n_pairs : batch * num_q_heads;
  int status = FDO_OK;
  int used = 1;

#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel
  {
#pragma omp single
    used = omp_get_num_threads();
  }
#endif

#pragma omp parallel for schedule(dynamic, 1)
  for (int w = 0; w < n_work; ++w) {
    int b = pairs ? pairs[2 * w] : w / num_q_heads;
    int qh = pairs ? pairs[2 * w + 1] : w % num_q_heads;
    if (b < 0 || b >= batch || qh < 0 || qh >= num_q_heads) {
#pragma omp atomic write
      status = FDO_BAD_ARG;
      continue;
    }
    int kvh = qh / group;
    for (int j = 0; j < q_len; ++j) {
      /* query token j sits at position seq_len - q_len + j and sees the keys up
         to and including its own position */
      int T = seq_len[b] - (q_len - 1 - j);
      const size_t qi = ((size_t)b * num_q_heads + qh) * q_len + j;   /* [B][QH][q_len] */
      double *o = out + qi * head_dim;
      double *l = lse + qi;
      if (T <= 0) {
        for (int d = 0; d < head_dim; ++d) o[d] = 0.0;
        *l = -INFINITY;
        continue;
      }
      double *s = (double *)malloc(sizeof(double) * (size_t)T);
      int64_t *rows = (int64_t *)malloc(sizeof(int64_t) * (size_t)T);
      double *qv = (double *)malloc(sizeof(double) * (size_t)head_dim);
      if (!s || !rows || !qv) {
        free(s); free(rows); free(qv);
#pragma omp atomic write
        status = FDO_NO_MEMORY;
        continue;
      }
      int bad = 0;
      for (int d = 0; d < head_dim; ++d)
        qv[d] = decode_elem(q, q_dtype, qi * head_dim + d);

      /* scores s_t = softmax_scale * q . (k_scale * ks(t) * dec(k_t)) */
      for (int t = 0; t < T && !bad; ++t) {
        rows[t] = cache_row(kv_start_idx, block_table, block_table_stride, page_size, b, t, kv_rows);
        if (rows[t] < 0) { bad = FDO_ROW_OUT_OF_RANGE; break; }
        size_t base = ((size_t)rows[t] * num_kv_heads + kvh) * head_dim;
        const double ks = k_scale * scale_at(scale_kind, k_scales, rows[t], num_kv_heads, kvh);
        double dot = 0.0;
        for (int d = 0; d < head_dim; ++d) {
          double kd = decode_elem(k_cache, kv_dtype, base + d);
          if (isnan(kd)) { bad = FDO_NAN_CODE; break; }
          dot += qv[d] * (ks * kd);
        }
        s[t] = softmax_scale * dot;
      }
      if (!bad) {
        /* two-pass softmax: max, then normalised exponentials */
        double M = s[0];
        for (int t = 1; t < T; ++t) if (s[t] > M) M = s[t];
        double Z = 0.0;
        for (int t = 0; t < T; ++t) { s[t] = exp(s[t] - M); Z += s[t]; }
        for (int d = 0; d < head_dim; ++d) o[d] = 0.0;
        for (int t = 0; t < T && !bad; ++t) {
          double wt = s[t] / Z;
          if (weights) weights[qi * weights_stride + t] = wt;
          size_t base = ((size_t)rows[t] * num_kv_heads + kvh) * head_dim;
          const double vs = v_scale * scale_at(scale_kind, v_scales, rows[t], num_kv_heads, kvh);
          for (int d = 0; d < head_dim; ++d) {
            double vd = decode_elem(v_cache, kv_dtype, base + d);
            if (isnan(vd)) { bad = FDO_NAN_CODE; break; }
            o[d] += wt * (vs * vd);
          }
        }
        *l = M + log(Z);
      }
      if (bad) {
#pragma omp atomic write
        status = bad;
      }
      free(s); free(rows); free(qv);
    }
  }
  if (threads_used) *threads_used = used;
  return status;
}

/* One query token per sequence (q_len = 1): q, out [B][QH][D], lse [B][QH]. */
int fdo_decode_attention(const void *q, int q_dtype, const void *k_cache, const void *v_cache,
                         int kv_dtype, const int32_t *kv_start_idx, const int32_t *block_table,
                         int block_table_stride, const int32_t *seq_len, int64_t kv_rows,
                         int batch, int num_q_heads, int num_kv_heads, int head_dim,
                         int page_size, double softmax_scale, double k_scale, double v_scale,
                         int scale_kind, const float *k_scales, const float *v_scales,
                         const int32_t *pairs, int n_pairs, int nthreads, double *out,
                         double *lse, double *weights, int weights_stride, int *threads_used) {
  return fdo_decode_attention_q(q, q_dtype, k_cache, v_cache, kv_dtype, kv_start_idx,
                                block_table, block_table_stride, seq_len, kv_rows, batch, 1,
                                num_q_heads, num_kv_heads, head_dim, page_size, softmax_scale,
                                k_scale, v_scale, scale_kind, k_scales, v_scales, pairs, n_pairs,
                                nthreads, out, lse, weights, weights_stride, threads_used);
}

/* fp32 value of a 16-bit element (f16 or bf16 bits); exact. */
static float elem16_to_f32(const uint16_t *base, int dtype, size_t idx) {
  return (float)(dtype == FDO_BF16 ? fdo_bf16_value(base[idx]) : fdo_f16_value(base[idx]));
}

/* One tensor (K or V) of the append; see the file comment. */
static int append_one(const uint16_t *x_new, int new_dtype, void *cache, int kv_dtype,
                      const int32_t *kv_start_idx, const int32_t *block_table,
                      int block_table_stride, const int32_t *positions, int64_t kv_rows,
                      int batch, int n_new, int num_kv_heads, int head_dim, int page_size,
                      float scale, int scale_kind, float *scales) {
  int status = FDO_OK;
  const float qmax = kv_dtype == FDO_I8 ? 127.0f : 448.0f;
  for (int b = 0; b < batch; ++b) {
    if (positions[b] < 0) continue;
    for (int i = 0; i < n_new; ++i) {
      int64_t row = cache_row(kv_start_idx, block_table, block_table_stride, page_size, b,
                              positions[b] + i, kv_rows);
      if (row < 0) { status = FDO_ROW_OUT_OF_RANGE; continue; }
      for (int h = 0; h < num_kv_heads; ++h) {
        const size_t src = (((size_t)b * n_new + i) * num_kv_heads + h) * head_dim;
        const size_t dst = ((size_t)row * num_kv_heads + h) * head_dim;
        if (kv_dtype == FDO_F16 || kv_dtype == FDO_BF16) {
          for (int d = 0; d < head_dim; ++d) ((uint16_t *)cache)[dst + d] = x_new[src + d];
          continue;
        }
        float s = scale;
        if (scale_kind == FDO_SCALE_HEAD) {
          s = scale * scales[h];
        } else if (scale_kind == FDO_SCALE_TOKEN) {
          float amax = 0.0f;
          for (int d = 0; d < head_dim; ++d) {
            float a = fabsf(elem16_to_f32(x_new, new_dtype, src + d));
            if (a > amax) amax = a;
          }
          const float denom = qmax * scale;
          const float ks = amax > 0.0f ? amax / denom : 1.0f;
          scales[(size_t)row * num_kv_heads + h] = ks;
          s = scale * ks;
        }
        for (int d = 0; d < head_dim; ++d) {
          const float q = elem16_to_f32(x_new, new_dtype, src + d) / s;
          ((uint8_t *)cache)[dst + d] = kv_dtype == FDO_I8 ? fdo_i8_encode(q) : fdo_e4m3_encode(q);
        }
      }
    }
  }
  return status;
}

/*
 * Writes the n_new new tokens of every sequence into k_cache / v_cache (see
 * the file comment).  k_new, v_new: [batch][n_new][KVH][D] 16-bit patterns
 * of new_dtype.  positions: [batch] token index of the first new token (< 0:
 * no append).
 * k_scales / v_scales: read (per KV head) or written (per token).
 */
int fdo_append_kv(const void *k_new, const void *v_new, int new_dtype, void *k_cache,
                  void *v_cache, int kv_dtype, const int32_t *kv_start_idx,
                  const int32_t *block_table, int block_table_stride, const int32_t *positions,
                  int64_t kv_rows, int batch, int n_new, int num_kv_heads, int head_dim,
                  int page_size, float k_scale, float v_scale, int scale_kind, float *k_scales,
                  float *v_scales) {
  if (n_new < 1) return FDO_BAD_ARG;
  if (!k_new || !v_new || !k_cache || !v_cache || !positions) return FDO_BAD_ARG;
  if ((kv_start_idx == NULL) == (block_table == NULL)) return FDO_BAD_ARG;
  if (new_dtype != FDO_F16 && new_dtype != FDO_BF16) return FDO_BAD_ARG;
  if ((kv_dtype == FDO_F16 || kv_dtype == FDO_BF16) && kv_dtype != new_dtype) return FDO_BAD_ARG;
  if (kv_dtype != FDO_F16 && kv_dtype != FDO_BF16 && kv_dtype != FDO_E4M3 && kv_dtype != FDO_I8)
    return FDO_BAD_ARG;
  if (scale_kind != FDO_SCALE_TENSOR && (!k_scales || !v_scales)) return FDO_BAD_ARG;
  if (block_table && page_size <= 0) return FDO_BAD_ARG;
  int a = append_one((const uint16_t *)k_new, new_dtype, k_cache, kv_dtype, kv_start_idx,
                     block_table, block_table_stride, positions, kv_rows, batch, n_new,
                     num_kv_heads, head_dim, page_size, k_scale, scale_kind, k_scales);
  int b = append_one((const uint16_t *)v_new, new_dtype, v_cache, kv_dtype, kv_start_idx,
                     block_table, block_table_stride, positions, kv_rows, batch, n_new,
                     num_kv_heads, head_dim, page_size, v_scale, scale_kind, v_scales);
  return a != FDO_OK ? a : b;
}
