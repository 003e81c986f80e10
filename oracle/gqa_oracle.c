/*
 * gqa_oracle.c -- plain, slow, fp64 CPU oracle for grouped-query attention over a
 * KV cache with a sliding window, a sink logit, softcap and RoPE+append.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and bench.py's CPU
 * baseline may load this library.  It shares no code, header, table or constant with
 * the CUDA library under sliding_window_gb300/, and it imports nothing from it.
 *
 * Sources (the pages this follows):
 *   [P1] OpenVINO PR #37423 "[NPUW] Support GQA sliding-window and smooth-softmax in
 *        DecomposeGQA", sections "Sliding window" and "smooth_softmax / head_sink".
 *   [P2] tract PR #2645 "onnx: import GroupQueryAttention decode steps and its internal
 *        rotary", section "What changed" (KV cache concat, do_rotary, bottom-right band).
 *   [P3] ExecuTorch PR #21901 "Add sliding windows to the off-graph KV-cache reference",
 *        Summary (per-layer window, mask rather than evict).
 *   [P4] onnx-light-cpu "Attention Kernel Design", sections "Layouts and semantics",
 *        "Compute paths" and "Scheduling, precision, and invariants".
 *
 * Every attention output here is the plain definition: for each query row, the set of
 * visible cache slots is enumerated, every score is materialized in fp64, and the softmax
 * (with the optional extra sink logit in its denominator) is taken over that set.  This
 * is the shape of [P4]'s materialized path, carried out in double precision.
 *
 * Layouts (the library's boundary uses the same ones, [P4] "Layouts and semantics"):
 *   q, out        [B, curr, Hq*D]     (rank-3, heads packed in the last dimension)
 *   k, v (new)    [B, curr, Hkv*D]
 *   past/present  [B, Hkv, cap, D]    (rank-4)
 *   cos/sin cache [rope_len, D/2]
 *   seqlens_k     [B] int32 = number of valid past tokens of each sequence
 *   head_sink     [Hq] float, or NULL
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fno-fast-math -fPIC -shared [-fopenmp].
 * -ffp-contract=off matters: the RoPE emulation rounds every product and every sum to
 * fp32 separately, exactly as the kernel does.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ODT_F32 0
#define ODT_F16 1
#define ODT_BF16 2
#define ODT_F64 3 /* internal: dequantized rows of a quantized cache */

/* ------------------------------------------------------------------------------------
 * Number formats.  Decoding and RNE rounding written from the IEEE-754 definitions of
 * binary16 (1 sign, 5 exponent, 10 fraction bits, bias 15) and bfloat16 (1 sign,
 * 8 exponent, 7 fraction bits, bias 127, i.e. the top half of a binary32).
 * ---------------------------------------------------------------------------------- */

static double decode_f16(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 0x1f;
  int f = h & 0x3ff;
  double mag;
  if (e == 0)
    mag = ldexp((double)f, -24); /* subnormal: f * 2^-24 */
  else if (e == 31)
    mag = f ? NAN : INFINITY;
  else
    mag = ldexp((double)(1024 + f), e - 25); /* (1 + f/1024) * 2^(e-15) */
  return sign ? -mag : mag;
}

static double decode_bf16(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float x;
  memcpy(&x, &u, 4);
  return (double)x;
}

/* Round a finite or non-finite double (which here always holds an fp32 value) to the
 * nearest value of a binary format with `fbits` fraction bits, exponent bias `bias`
 * and `ebits` exponent bits, ties to even, and return its encoding. */
static uint32_t encode_rne(double x, int fbits, int ebits, int bias) {
  uint32_t sign = signbit(x) ? 1u : 0u;
  uint32_t emax_field = (1u << ebits) - 1u;
  uint32_t out_sign = sign << (fbits + ebits);
  if (isnan(x)) return out_sign | (emax_field << fbits) | (1u << (fbits - 1)); /* quiet NaN */
  double a = fabs(x);
  if (isinf(a)) return out_sign | (emax_field << fbits);
  int emin = 1 - bias;                       /* exponent of the smallest normal */
  double quantum_sub = ldexp(1.0, emin - fbits); /* spacing of subnormals */
  if (a < ldexp(1.0, emin)) {
    /* subnormal range: integer multiple of the quantum, RNE via rint (default mode) */
    double n = rint(a / quantum_sub);
    return out_sign | (uint32_t)n; /* n == 2^fbits encodes the smallest normal */
  }
  int e2;
  double m = frexp(a, &e2);               /* a = m * 2^e2, m in [0.5, 1) */
  int E = e2 - 1;                          /* a = (2m) * 2^E, 2m in [1, 2) */
  double n = rint(ldexp(m, 1 + fbits));    /* 2m * 2^fbits rounded, in [2^fbits, 2^(fbits+1)] */
  if (n == ldexp(1.0, fbits + 1)) {
    n = ldexp(1.0, fbits);
    E += 1;
  }
  if (E + bias >= (int)emax_field) return out_sign | (emax_field << fbits); /* overflow -> inf */
  uint32_t frac = (uint32_t)(n - ldexp(1.0, fbits));
  return out_sign | ((uint32_t)(E + bias) << fbits) | frac;
}

uint16_t oracle_encode_f16(float x) { return (uint16_t)encode_rne((double)x, 10, 5, 15); }
uint16_t oracle_encode_bf16(float x) { return (uint16_t)encode_rne((double)x, 7, 8, 127); }
double oracle_decode_f16(uint16_t h) { return decode_f16(h); }
double oracle_decode_bf16(uint16_t h) { return decode_bf16(h); }

/* Element idx of an array of the given dtype, as a double (exact for all three). */
static double load_elem(const void *base, size_t idx, int dtype) {
  if (dtype == ODT_F64) return ((const double *)base)[idx];
  if (dtype == ODT_F32) return (double)((const float *)base)[idx];
  uint16_t h = ((const uint16_t *)base)[idx];
  return dtype == ODT_F16 ? decode_f16(h) : decode_bf16(h);
}

static float load_f32(const void *base, size_t idx, int dtype) {
  /* every f16/bf16 value is exactly representable in fp32 */
  return (float)load_elem(base, idx, dtype);
}

static void store_from_f32(void *base, size_t idx, int dtype, float x) {
  if (dtype == ODT_F32)
    ((float *)base)[idx] = x;
  else if (dtype == ODT_F16)
    ((uint16_t *)base)[idx] = oracle_encode_f16(x);
  else
    ((uint16_t *)base)[idx] = oracle_encode_bf16(x);
}

static size_t elem_size(int dtype) { return dtype == ODT_F32 ? 4 : 2; }

/* ------------------------------------------------------------------------------------
 * Per-sequence validity.  A sequence whose past length is negative, whose past plus the
 * new tokens do not fit the present capacity (or, when past and present are separate
 * buffers, whose past does not fit the past capacity), or whose last RoPE position lies
 * beyond the cos/sin cache, is rejected: its outputs are zeros and nothing of it is
 * appended.  Bit 1 = bad seqlens_k, bit 2 = RoPE position out of range.  ([P4]
 * "Scheduling, precision, and invariants": invalid combinations fail explicitly.)
 * ---------------------------------------------------------------------------------- */
int32_t oracle_sequence_status(int32_t past, int32_t curr, int32_t cap_past, int32_t cap_present,
                               int32_t past_is_separate, int32_t do_rotary, int32_t rope_len) {
  int32_t st = 0;
  if (past < 0 || (int64_t)past + curr > cap_present || (past_is_separate && past > cap_past))
    st |= 1;
  else if (do_rotary && (int64_t)past + curr > rope_len)
    st |= 2;
  return st;
}

/* ------------------------------------------------------------------------------------
 * RoPE + append, emulated bit for bit.
 *
 * [P2] "What changed": RoPE runs on the cos/sin cache halves widened to the head size,
 * positions are 0..S-1 for a first prompt and start at seqlens_k for generated tokens,
 * and K is rotated before it enters the cache; past_key/past_value are concatenated
 * with the step and returned as present_key/present_value.
 *
 * Rotation (non-interleaved half split), for d in [0, D/2):
 *     y[d]       = x[d] * c[d] - x[d + D/2] * s[d]
 *     y[d + D/2] = x[d + D/2] * c[d] + x[d] * s[d]
 * with c, s = cos/sin_cache[pos, d].  Each product and each sum is rounded to fp32, and
 * the result is rounded to the storage dtype with ties to even.
 *
 * present rows [past_b, past_b + curr) receive the (rotated) new keys and the new values;
 * when past is a separate buffer, rows [0, past_b) are copied from it; other rows are not
 * touched.  q_rot (may be NULL) receives the rotated queries in q's layout.
 * ---------------------------------------------------------------------------------- */
static void rotate_row(const void *x, size_t xoff, const void *cosc, const void *sinc, size_t coff,
                       int D, int dtype, void *y, size_t yoff) {
  int half = D / 2;
  for (int d = 0; d < half; ++d) {
    float x1 = load_f32(x, xoff + d, dtype);
    float x2 = load_f32(x, xoff + d + half, dtype);
    float c = load_f32(cosc, coff + d, dtype);
    float s = load_f32(sinc, coff + d, dtype);
    float a = x1 * c;
    float b = x2 * s;
    float y1 = a - b;
    float e = x2 * c;
    float f = x1 * s;
    float y2 = e + f;
    store_from_f32(y, yoff + d, dtype, y1);
    store_from_f32(y, yoff + d + half, dtype, y2);
  }
}

void oracle_rope_append(int32_t B, int32_t Hq, int32_t Hkv, int32_t D, int32_t Dv, int32_t curr, int32_t cap_past,
                        int32_t cap_present, int32_t rope_len, int32_t dtype, int32_t do_rotary,
                        const void *q, const void *k, const void *v, const void *past_k,
                        const void *past_v, const int32_t *seqlens_k, const void *cos_cache,
                        const void *sin_cache, void *q_rot, void *present_k, void *present_v,
                        int32_t *status_out) {
  size_t es = elem_size(dtype);
  int separate = past_k != NULL && past_k != present_k;
  int32_t status_all = 0;
  for (int b = 0; b < B; ++b) {
    int32_t past = seqlens_k[b];
    int32_t st = oracle_sequence_status(past, curr, cap_past, cap_present, separate, do_rotary, rope_len);
    status_all |= st;
    if (st) continue;
    for (int h = 0; h < Hkv; ++h) {
      size_t dst_base = ((size_t)b * Hkv + h) * (size_t)cap_present * D;
      size_t dst_base_v = ((size_t)b * Hkv + h) * (size_t)cap_present * Dv;
      if (separate) {
        size_t src_base = ((size_t)b * Hkv + h) * (size_t)cap_past * D;
        size_t src_base_v = ((size_t)b * Hkv + h) * (size_t)cap_past * Dv;
        memcpy((char *)present_k + dst_base * es, (const char *)past_k + src_base * es, (size_t)past * D * es);
        memcpy((char *)present_v + dst_base_v * es, (const char *)past_v + src_base_v * es,
               (size_t)past * Dv * es);
      }
      for (int i = 0; i < curr; ++i) {
        size_t src = (((size_t)b * curr + i) * Hkv + h) * D;
        size_t dst = dst_base + (size_t)(past + i) * D;
        if (do_rotary)
          rotate_row(k, src, cos_cache, sin_cache, (size_t)(past + i) * (D / 2), D, dtype, present_k, dst);
        else
          memcpy((char *)present_k + dst * es, (const char *)k + src * es, (size_t)D * es);
        size_t src_v = (((size_t)b * curr + i) * Hkv + h) * Dv;
        size_t dst_v = dst_base_v + (size_t)(past + i) * Dv;
        memcpy((char *)present_v + dst_v * es, (const char *)v + src_v * es, (size_t)Dv * es);
      }
    }
    if (q_rot) {
      for (int i = 0; i < curr; ++i)
        for (int h = 0; h < Hq; ++h) {
          size_t off = (((size_t)b * curr + i) * Hq + h) * D;
          if (do_rotary)
            rotate_row(q, off, cos_cache, sin_cache, (size_t)(past + i) * (D / 2), D, dtype, q_rot, off);
          else
            memcpy((char *)q_rot + off * es, (const char *)q + off * es, (size_t)D * es);
        }
    }
  }
  if (status_out) *status_out = status_all;
}

/* ------------------------------------------------------------------------------------
 * The band predicate ([P1] "Sliding window", [P2] "What changed", [P3] Summary, [P4]
 * "Compute paths").  Slot j of the present buffer holds absolute position j (the step is
 * appended contiguously after the past).  A query at absolute position q_abs sees slot j
 * iff
 *     j < total                         (slots at or past seqlens_k + curr are stale)
 *   and (not causal or j <= q_abs)      (bottom-right aligned causal band)
 *   and (window < 0 or q_abs - j < window)   (masked when q_abs - k_abs >= window)
 * ---------------------------------------------------------------------------------- */
int32_t oracle_visible(int64_t q_abs, int64_t j, int64_t total, int32_t causal, int32_t window) {
  if (j < 0 || j >= total) return 0;
  if (causal && j > q_abs) return 0;
  if (window >= 0 && q_abs - j >= window) return 0;
  return 1;
}

/* ------------------------------------------------------------------------------------
 * One query row over an explicit visibility mask (and, optionally, an additive bias).
 *   s_j = scale * <q, k_j> [+ bias_j];  if softcap > 0: s_j = softcap * tanh(s_j / softcap)
 *   the sink z (when present) is one more logit in the denominator only, not scaled and
 *   not capped ([P1] "smooth_softmax / head_sink": the extra logit joins the softmax
 *   denominator and is sliced out);
 *   out = sum_j exp(s_j - M) v_j / (exp(z - M) [if sink] + sum_j exp(s_j - M)),
 *   M = max over the visible s_j and z;  a row with no visible slot gives zeros
 *   ([P4] "A fully masked query row produces zeros rather than NaN").  A score of -inf
 *   (an additive mask value of -inf without a softcap) has weight exactly zero, so a row
 *   whose scores are all -inf is fully masked and gives zeros too, not 0/0.
 * q is D doubles; k points at `n` rows of D elements of `dtype`, v at `n` rows of Dv
 * ([P4] "Layouts and semantics": the V head dimension may differ from the Q/K one); out
 * holds Dv doubles.
 * ---------------------------------------------------------------------------------- */
void oracle_attend_row_bias(const double *q, const void *k, const void *v, int64_t row0, int64_t n,
                            const uint8_t *visible, const double *bias, int32_t D, int32_t Dv, int32_t dtype,
                            double scale, double softcap, int32_t has_sink, double sink, double *out) {
  double *s = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
  double M = -INFINITY;
  int any = 0;
  for (int64_t j = 0; j < n; ++j) {
    if (!visible[j]) continue;
    double dot = 0.0;
    for (int d = 0; d < D; ++d) dot += q[d] * load_elem(k, (size_t)(row0 + j) * D + d, dtype);
    double sj = scale * dot;
    if (bias) sj += bias[j];
    if (softcap > 0.0) sj = softcap * tanh(sj / softcap);
    s[j] = sj;
    if (sj == -INFINITY) continue;  /* an additive -inf removes the key: weight exp(-inf) = 0 */
    if (sj > M) M = sj;
    any = 1;
  }
  for (int d = 0; d < Dv; ++d) out[d] = 0.0;
  if (!any) {
    free(s);
    return;
  }
  if (has_sink && sink > M) M = sink;
  double den = has_sink ? exp(sink - M) : 0.0;
  for (int64_t j = 0; j < n; ++j) {
    if (!visible[j]) continue;
    double w = exp(s[j] - M);
    den += w;
    for (int d = 0; d < Dv; ++d) out[d] += w * load_elem(v, (size_t)(row0 + j) * Dv + d, dtype);
  }
  for (int d = 0; d < Dv; ++d) out[d] /= den;
  free(s);
}

void oracle_attend_row(const double *q, const void *k, const void *v, int64_t row0, int64_t n,
                       const uint8_t *visible, int32_t D, int32_t Dv, int32_t dtype, double scale, double softcap,
                       int32_t has_sink, double sink, double *out) {
  oracle_attend_row_bias(q, k, v, row0, n, visible, NULL, D, Dv, dtype, scale, softcap, has_sink, sink, out);
}

/* ------------------------------------------------------------------------------------
 * Whole attention over the present cache, for a list of rows (or all rows).
 * Row index r = ((b * curr) + i) * Hq + hq; out holds Dv doubles per listed row.
 * Head mapping ([P4] "Layouts and semantics"): group_size G = Hq / Hkv and q head hq
 * reads kv head hq / G, with no copy of K or V.
 * q is the query as it enters the scores (already rotated when do_rotary).
 * scale == 0 means 1/sqrt(D).  sink: head_sink[hq] when head_sink != NULL, else 0 when
 * smooth_softmax, else none.
 * Rejected sequences (oracle_sequence_status != 0) give zeros.
 * ---------------------------------------------------------------------------------- */
void oracle_attention(int32_t B, int32_t Hq, int32_t Hkv, int32_t D, int32_t Dv, int32_t curr, int32_t cap_past,
                      int32_t cap_present, int32_t rope_len, int32_t dtype, double scale,
                      double softcap, int32_t window, int32_t causal, int32_t do_rotary,
                      int32_t smooth_softmax, int32_t past_is_separate, const void *q,
                      const void *present_k, const void *present_v, const int32_t *seqlens_k,
                      const float *head_sink, const int64_t *rows, int64_t nrows, double *out) {
  int G = Hq / Hkv;
  if (scale == 0.0) scale = 1.0 / sqrt((double)D);
  int64_t count = rows ? nrows : (int64_t)B * curr * Hq;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1)
#endif
  for (int64_t t = 0; t < count; ++t) {
    int64_t r = rows ? rows[t] : t;
    int hq = (int)(r % Hq);
    int i = (int)((r / Hq) % curr);
    int b = (int)(r / ((int64_t)Hq * curr));
    double *o = out + (size_t)t * Dv;
    int32_t past = seqlens_k[b];
    if (oracle_sequence_status(past, curr, cap_past, cap_present, past_is_separate, do_rotary, rope_len)) {
      for (int d = 0; d < Dv; ++d) o[d] = 0.0;
      continue;
    }
    int hk = hq / G;
    int64_t total = (int64_t)past + curr;
    int64_t q_abs = (int64_t)past + i;
    double *qv = (double *)malloc(sizeof(double) * (size_t)D);
    for (int d = 0; d < D; ++d) qv[d] = load_elem(q, (size_t)r * D + d, dtype);
    uint8_t *vis = (uint8_t *)malloc((size_t)cap_present);
    for (int64_t j = 0; j < cap_present; ++j) vis[j] = (uint8_t)oracle_visible(q_abs, j, total, causal, window);
    int has_sink = head_sink != NULL || smooth_softmax;
    double z = head_sink ? (double)head_sink[hq] : 0.0;
    int64_t row0 = ((int64_t)b * Hkv + hk) * cap_present;
    oracle_attend_row(qv, present_k, present_v, row0, cap_present, vis, D, Dv, dtype, scale, softcap, has_sink, z,
                      o);
    free(vis);
    free(qv);
  }
}

/* ------------------------------------------------------------------------------------
 * A K/V cache with padding ([P4] "Layouts and semantics": the opset-24 nonpad_kv_seqlen
 * input; "Compute paths": padding frontiers).  Sequence b has n = nonpad_kv_seqlen[b]
 * valid keys, rows [0, n) of the cache; rows at or past n are padding and never seen.  The
 * curr queries are the last curr of the n valid tokens (bottom-right alignment, as for the
 * causal band), so query i sits at absolute position n - curr + i, and the band predicate
 * is oracle_visible's with total = n.  A sequence with n < curr or n > cap cannot hold its
 * own queries and gives zeros (the caller reports it).
 * ---------------------------------------------------------------------------------- */
void oracle_attention_nonpad(int32_t B, int32_t Hq, int32_t Hkv, int32_t D, int32_t Dv, int32_t curr, int32_t cap,
                             int32_t dtype, double scale, double softcap, int32_t window, int32_t causal,
                             int32_t smooth_softmax, const void *q, const void *k_cache, const void *v_cache,
                             const int64_t *nonpad, const float *head_sink, const int64_t *rows, int64_t nrows,
                             double *out) {
  int G = Hq / Hkv;
  if (scale == 0.0) scale = 1.0 / sqrt((double)D);
  int64_t count = rows ? nrows : (int64_t)B * curr * Hq;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1)
#endif
  for (int64_t t = 0; t < count; ++t) {
    int64_t r = rows ? rows[t] : t;
    int hq = (int)(r % Hq);
    int i = (int)((r / Hq) % curr);
    int b = (int)(r / ((int64_t)Hq * curr));
    double *o = out + (size_t)t * Dv;
    int64_t n = nonpad[b];
    if (n < curr || n > cap) {
      for (int d = 0; d < Dv; ++d) o[d] = 0.0;
      continue;
    }
    int hk = hq / G;
    int64_t q_abs = n - curr + i;
    double *qv = (double *)malloc(sizeof(double) * (size_t)D);
    for (int d = 0; d < D; ++d) qv[d] = load_elem(q, (size_t)r * D + d, dtype);
    uint8_t *vis = (uint8_t *)malloc((size_t)cap);
    for (int64_t j = 0; j < cap; ++j) vis[j] = (uint8_t)oracle_visible(q_abs, j, n, causal, window);
    int has_sink = head_sink != NULL || smooth_softmax;
    double z = head_sink ? (double)head_sink[hq] : 0.0;
    int64_t row0 = ((int64_t)b * Hkv + hk) * cap;
    oracle_attend_row(qv, k_cache, v_cache, row0, cap, vis, D, Dv, dtype, scale, softcap, has_sink, z, o);
    free(vis);
    free(qv);
  }
}

/* ------------------------------------------------------------------------------------
 * Ring layout of the present cache ([P1] "Sliding window": sliding_window_cache, the
 * physical rolling KV buffer whose memory is bounded by the window; [P3] Summary: a window
 * is a per-layer setting).  The cache has cap slots and absolute position p lives in slot
 * p mod cap, so only the last cap positions are resident.  It is valid only with a window
 * W >= 1 such that W + curr - 1 <= cap: every key that a query of the step can see is then
 * still resident after the step's own rows were written (the oldest key the first query
 * sees, past - W + 1, is at least total - cap).  The band predicate is unchanged; only the
 * slot of a position differs.  The append has no separate past (the ring is updated in
 * place) and no capacity limit on the past length.
 * ---------------------------------------------------------------------------------- */
int32_t oracle_ring_valid(int32_t curr, int32_t cap, int32_t window) {
  return window >= 1 && curr >= 1 && (int64_t)window + curr - 1 <= cap;
}

int32_t oracle_ring_status(int32_t past, int32_t curr, int32_t do_rotary, int32_t rope_len) {
  if (past < 0) return 1;
  if (do_rotary && (int64_t)past + curr > rope_len) return 2;
  return 0;
}

void oracle_rope_append_ring(int32_t B, int32_t Hq, int32_t Hkv, int32_t D, int32_t curr, int32_t cap,
                             int32_t rope_len, int32_t dtype, int32_t do_rotary, const void *q, const void *k,
                             const void *v, const int32_t *seqlens_k, const void *cos_cache,
                             const void *sin_cache, void *q_rot, void *present_k, void *present_v,
                             int32_t *status_out) {
  size_t es = elem_size(dtype);
  int32_t status_all = 0;
  for (int b = 0; b < B; ++b) {
    int32_t past = seqlens_k[b];
    int32_t st = oracle_ring_status(past, curr, do_rotary, rope_len);
    status_all |= st;
    if (st) continue;
    for (int h = 0; h < Hkv; ++h) {
      size_t base = ((size_t)b * Hkv + h) * (size_t)cap * D;
      for (int i = 0; i < curr; ++i) {
        int64_t pos = (int64_t)past + i;
        size_t src = (((size_t)b * curr + i) * Hkv + h) * D;
        size_t dst = base + (size_t)(pos % cap) * D;
        if (do_rotary)
          rotate_row(k, src, cos_cache, sin_cache, (size_t)pos * (D / 2), D, dtype, present_k, dst);
        else
          memcpy((char *)present_k + dst * es, (const char *)k + src * es, (size_t)D * es);
        memcpy((char *)present_v + dst * es, (const char *)v + src * es, (size_t)D * es);
      }
    }
    if (q_rot) {
      for (int i = 0; i < curr; ++i)
        for (int h = 0; h < Hq; ++h) {
          size_t off = (((size_t)b * curr + i) * Hq + h) * D;
          if (do_rotary)
            rotate_row(q, off, cos_cache, sin_cache, (size_t)(past + i) * (D / 2), D, dtype, q_rot, off);
          else
            memcpy((char *)q_rot + off * es, (const char *)q + off * es, (size_t)D * es);
        }
    }
  }
  if (status_out) *status_out = status_all;
}

/* Attention over a ring cache: the resident positions [max(0, total - cap), total) are
 * gathered into position order (position p from slot p mod cap) and each row is the same
 * oracle_attend_row over them, with the same band predicate as the linear layout.  Rows of
 * rejected sequences, and every row when the ring cannot hold the band, are zeros. */
void oracle_attention_ring(int32_t B, int32_t Hq, int32_t Hkv, int32_t D, int32_t curr, int32_t cap,
                           int32_t rope_len, int32_t dtype, double scale, double softcap, int32_t window,
                           int32_t causal, int32_t do_rotary, int32_t smooth_softmax, const void *q,
                           const void *present_k, const void *present_v, const int32_t *seqlens_k,
                           const float *head_sink, const int64_t *rows, int64_t nrows, double *out) {
  int G = Hq / Hkv;
  size_t es = elem_size(dtype);
  if (scale == 0.0) scale = 1.0 / sqrt((double)D);
  int valid = oracle_ring_valid(curr, cap, window);
  int64_t count = rows ? nrows : (int64_t)B * curr * Hq;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1)
#endif
  for (int64_t t = 0; t < count; ++t) {
    int64_t r = rows ? rows[t] : t;
    int hq = (int)(r % Hq);
    int i = (int)((r / Hq) % curr);
    int b = (int)(r / ((int64_t)Hq * curr));
    double *o = out + (size_t)t * D;
    int32_t past = seqlens_k[b];
    if (!valid || oracle_ring_status(past, curr, do_rotary, rope_len)) {
      for (int d = 0; d < D; ++d) o[d] = 0.0;
      continue;
    }
    int hk = hq / G;
    int64_t total = (int64_t)past + curr;
    int64_t q_abs = (int64_t)past + i;
    int64_t first = total > cap ? total - cap : 0;  /* oldest resident position */
    int64_t n = total - first;
    char *kg = (char *)malloc((size_t)n * D * es);
    char *vg = (char *)malloc((size_t)n * D * es);
    uint8_t *vis = (uint8_t *)malloc((size_t)n);
    size_t base = ((size_t)b * Hkv + hk) * (size_t)cap * D;
    for (int64_t j = 0; j < n; ++j) {
      int64_t pos = first + j;
      size_t src = base + (size_t)(pos % cap) * D;
      memcpy(kg + (size_t)j * D * es, (const char *)present_k + src * es, (size_t)D * es);
      memcpy(vg + (size_t)j * D * es, (const char *)present_v + src * es, (size_t)D * es);
      vis[j] = (uint8_t)oracle_visible(q_abs, pos, total, causal, window);
    }
    double *qv = (double *)malloc(sizeof(double) * (size_t)D);
    for (int d = 0; d < D; ++d) qv[d] = load_elem(q, (size_t)r * D + d, dtype);
    int has_sink = head_sink != NULL || smooth_softmax;
    double z = head_sink ? (double)head_sink[hq] : 0.0;
    oracle_attend_row(qv, kg, vg, 0, n, vis, D, D, dtype, scale, softcap, has_sink, z, o);
    free(qv);
    free(vis);
    free(vg);
    free(kg);
  }
}

/* ------------------------------------------------------------------------------------
 * Paged layout of the present cache ([P3] Summary: a cell cache whose slots belong to
 * sequences through a per-step occupancy/membership plan, masked rather than evicted).
 * Here the cache is a pool of pages of `page` positions, [num_pages][Hkv][page][D], and a
 * block table [B][max_pages] names the page that holds positions [n*page, (n+1)*page) of
 * sequence b.  The logical capacity is max_pages * page; the band predicate is unchanged.
 * A sequence whose table entries for the positions it reads or writes ([lo, total) with lo
 * the band's first position, rounded down to a page) fall outside [0, num_pages) is
 * rejected like a bad seqlens_k: bit 8, zeros, nothing written.
 * ---------------------------------------------------------------------------------- */
int32_t oracle_paged_status(int32_t past, int32_t curr, int32_t cap, int32_t do_rotary, int32_t rope_len,
                            int32_t window, const int32_t *table_row, int32_t page, int32_t num_pages) {
  int32_t st = oracle_sequence_status(past, curr, 0, cap, 0, do_rotary, rope_len);
  if (st) return st;
  int64_t total = (int64_t)past + curr;
  int64_t lo = window > 0 ? (past - window + 1 > 0 ? past - window + 1 : 0) : 0;
  for (int64_t n = lo / page; n * page < total; ++n)
    if (table_row[n] < 0 || table_row[n] >= num_pages) return 8;
  return 0;
}

static size_t paged_row(int32_t b, int32_t h, int64_t pos, int32_t Hkv, int32_t page, const int32_t *table,
                        int32_t max_pages) {
  int32_t pg = table[(size_t)b * max_pages + pos / page];
  return ((size_t)pg * Hkv + h) * page + (size_t)(pos % page);
}

void oracle_rope_append_paged(int32_t B, int32_t Hq, int32_t Hkv, int32_t D, int32_t curr, int32_t page,
                              int32_t max_pages, int32_t num_pages, int32_t rope_len, int32_t dtype,
                              int32_t do_rotary, int32_t window, const int32_t *table, const void *q, const void *k,
                              const void *v, const int32_t *seqlens_k, const void *cos_cache, const void *sin_cache,
                              void *q_rot, void *pool_k, void *pool_v, int32_t *status_out) {
  size_t es = elem_size(dtype);
  int32_t status_all = 0;
  int32_t cap = max_pages * page;
  for (int b = 0; b < B; ++b) {
    int32_t past = seqlens_k[b];
    int32_t st = oracle_paged_status(past, curr, cap, do_rotary, rope_len, window, table + (size_t)b * max_pages,
                                     page, num_pages);
    status_all |= st;
    if (st) continue;
    for (int h = 0; h < Hkv; ++h)
      for (int i = 0; i < curr; ++i) {
        int64_t pos = (int64_t)past + i;
        size_t src = (((size_t)b * curr + i) * Hkv + h) * D;
        size_t dst = paged_row(b, h, pos, Hkv, page, table, max_pages) * D;
        if (do_rotary)
          rotate_row(k, src, cos_cache, sin_cache, (size_t)pos * (D / 2), D, dtype, pool_k, dst);
        else
          memcpy((char *)pool_k + dst * es, (const char *)k + src * es, (size_t)D * es);
        memcpy((char *)pool_v + dst * es, (const char *)v + src * es, (size_t)D * es);
      }
    if (q_rot) {
      for (int i = 0; i < curr; ++i)
        for (int h = 0; h < Hq; ++h) {
          size_t off = (((size_t)b * curr + i) * Hq + h) * D;
          if (do_rotary)
            rotate_row(q, off, cos_cache, sin_cache, (size_t)(past + i) * (D / 2), D, dtype, q_rot, off);
          else
            memcpy((char *)q_rot + off * es, (const char *)q + off * es, (size_t)D * es);
        }
    }
  }
  if (status_out) *status_out = status_all;
}

/* Attention over a paged cache: positions [0, total) gathered in order from their pages,
 * then the same oracle_attend_row and band predicate as the contiguous layout. */
void oracle_attention_paged(int32_t B, int32_t Hq, int32_t Hkv, int32_t D, int32_t curr, int32_t page,
                            int32_t max_pages, int32_t num_pages, int32_t rope_len, int32_t dtype, double scale,
                            double softcap, int32_t window, int32_t causal, int32_t do_rotary,
                            int32_t smooth_softmax, const int32_t *table, const void *q, const void *pool_k,
                            const void *pool_v, const int32_t *seqlens_k, const float *head_sink,
                            const int64_t *rows, int64_t nrows, double *out) {
  int G = Hq / Hkv;
  size_t es = elem_size(dtype);
  int32_t cap = max_pages * page;
  if (scale == 0.0) scale = 1.0 / sqrt((double)D);
  int64_t count = rows ? nrows : (int64_t)B * curr * Hq;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1)
#endif
  for (int64_t t = 0; t < count; ++t) {
    int64_t r = rows ? rows[t] : t;
    int hq = (int)(r % Hq);
    int i = (int)((r / Hq) % curr);
    int b = (int)(r / ((int64_t)Hq * curr));
    double *o = out + (size_t)t * D;
    int32_t past = seqlens_k[b];
    if (oracle_paged_status(past, curr, cap, do_rotary, rope_len, window, table + (size_t)b * max_pages, page,
                            num_pages)) {
      for (int d = 0; d < D; ++d) o[d] = 0.0;
      continue;
    }
    int hk = hq / G;
    int64_t total = (int64_t)past + curr;
    int64_t q_abs = (int64_t)past + i;
    int64_t first = window > 0 ? ((past - window + 1 > 0 ? past - window + 1 : 0) / page) * page : 0;
    int64_t n = total - first;  /* positions before `first` are never visible */
    char *kg = (char *)malloc((size_t)n * D * es);
    char *vg = (char *)malloc((size_t)n * D * es);
    uint8_t *vis = (uint8_t *)malloc((size_t)n);
    for (int64_t j = 0; j < n; ++j) {
      int64_t pos = first + j;
      size_t src = paged_row(b, hk, pos, Hkv, page, table, max_pages) * D;
      memcpy(kg + (size_t)j * D * es, (const char *)pool_k + src * es, (size_t)D * es);
      memcpy(vg + (size_t)j * D * es, (const char *)pool_v + src * es, (size_t)D * es);
      vis[j] = (uint8_t)oracle_visible(q_abs, pos, total, causal, window);
    }
    double *qv = (double *)malloc(sizeof(double) * (size_t)D);
    for (int d = 0; d < D; ++d) qv[d] = load_elem(q, (size_t)r * D + d, dtype);
    int has_sink = head_sink != NULL || smooth_softmax;
    double z = head_sink ? (double)head_sink[hq] : 0.0;
    oracle_attend_row(qv, kg, vg, 0, n, vis, D, D, dtype, scale, softcap, has_sink, z, o);
    free(qv);
    free(vis);
    free(vg);
    free(kg);
  }
}

/* ------------------------------------------------------------------------------------
 * Attention masks ([P4] "Layouts and semantics": boolean and FLOAT additive broadcast masks
 * next to the bottom-right causal band; [P2] "What changed": attention_bias is summed with
 * the causal band).  The mask is indexed [b][hq][i][j] with element strides stride_b,
 * stride_h, stride_i (0 broadcasts that dimension) and contiguous keys j = absolute
 * position (slot) in [0, keys).  kind 1: uint8, nonzero keeps the key, zero removes it
 * from the row's softmax like the band does.  kind 2: values of the dtype added to the
 * scaled score before the softcap (matmul, mask, softcap, softmax).  The band, the sink and
 * the fully-masked-row rule are unchanged; the contiguous layout only.
 * ---------------------------------------------------------------------------------- */
void oracle_attention_masked(int32_t B, int32_t Hq, int32_t Hkv, int32_t D, int32_t Dv, int32_t curr,
                             int32_t cap_present,
                             int32_t rope_len, int32_t dtype, double scale, double softcap, int32_t window,
                             int32_t causal, int32_t do_rotary, int32_t smooth_softmax, int32_t mask_kind,
                             const void *mask, int64_t stride_b, int64_t stride_h, int64_t stride_i, int32_t keys,
                             const void *q, const void *present_k, const void *present_v, const int32_t *seqlens_k,
                             const float *head_sink, const int64_t *rows, int64_t nrows, double *out) {
  int G = Hq / Hkv;
  if (scale == 0.0) scale = 1.0 / sqrt((double)D);
  int64_t count = rows ? nrows : (int64_t)B * curr * Hq;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1)
#endif
  for (int64_t t = 0; t < count; ++t) {
    int64_t r = rows ? rows[t] : t;
    int hq = (int)(r % Hq);
    int i = (int)((r / Hq) % curr);
    int b = (int)(r / ((int64_t)Hq * curr));
    double *o = out + (size_t)t * Dv;
    int32_t past = seqlens_k[b];
    if (oracle_sequence_status(past, curr, 0, cap_present, 0, do_rotary, rope_len) ||
        (int64_t)past + curr > keys) {
      for (int d = 0; d < Dv; ++d) o[d] = 0.0;
      continue;
    }
    int hk = hq / G;
    int64_t total = (int64_t)past + curr;
    int64_t q_abs = (int64_t)past + i;
    size_t mrow = (size_t)(b * stride_b + hq * stride_h + i * stride_i);
    double *qv = (double *)malloc(sizeof(double) * (size_t)D);
    for (int d = 0; d < D; ++d) qv[d] = load_elem(q, (size_t)r * D + d, dtype);
    uint8_t *vis = (uint8_t *)malloc((size_t)cap_present);
    double *bias = mask_kind == 2 ? (double *)malloc(sizeof(double) * (size_t)cap_present) : NULL;
    for (int64_t j = 0; j < cap_present; ++j) {
      vis[j] = (uint8_t)oracle_visible(q_abs, j, total, causal, window);
      if (!vis[j]) continue;
      if (mask_kind == 1) vis[j] = ((const uint8_t *)mask)[mrow + (size_t)j] != 0;
      if (mask_kind == 2) bias[j] = load_elem(mask, mrow + (size_t)j, dtype);
    }
    int has_sink = head_sink != NULL || smooth_softmax;
    double z = head_sink ? (double)head_sink[hq] : 0.0;
    int64_t row0 = ((int64_t)b * Hkv + hk) * cap_present;
    oracle_attend_row_bias(qv, present_k, present_v, row0, cap_present, vis, bias, D, Dv, dtype, scale, softcap,
                           has_sink, z, o);
    free(bias);
    free(vis);
    free(qv);
  }
}

/* ------------------------------------------------------------------------------------
 * Quantized KV cache.  The pages leave a quantized cache out of their own designs ([P1]
 * puts i8/i4/f8 KV out of its scope at the end of "smooth_softmax / head_sink"; [P2] "What
 * changed" rejects quantized KV); the reading taken here is the plainest one for an f8
 * cache: present K and V hold 8-bit floating-point codes of the E4M3
 * kind (1 sign, 4 exponent bits with bias 7, 3 fraction bits; no infinities; the code
 * S.1111.111 is NaN, so the largest magnitude is 1.75 * 2^8 = 448), one float scale per kv
 * head for K and one for V.  The stored value of an element is code * scale.
 *
 * Append: the row is first formed in the storage dtype exactly as in oracle_rope_append
 * (K rotated and rounded to the dtype), then each element x becomes
 *     code = e4m3(fp32(x) / fp32(scale))      (IEEE fp32 division)
 * rounded to nearest, ties to even, saturating: a magnitude beyond 448 (including one
 * that rounds past it, and infinity) gives the code of +-448, NaN gives NaN.
 * Attention is oracle_attention's definition over the dequantized rows code * scale,
 * computed in fp64.  The cache is updated in place (no separate past).
 * ---------------------------------------------------------------------------------- */
double oracle_decode_e4m3(uint8_t c) {
  int sign = (c >> 7) & 1;
  int e = (c >> 3) & 0xf;
  int f = c & 7;
  double mag;
  if (e == 15 && f == 7)
    mag = NAN;
  else if (e == 0)
    mag = ldexp((double)f, -9); /* subnormal: f/8 * 2^(1-7) */
  else
    mag = ldexp((double)(8 + f), e - 10); /* (1 + f/8) * 2^(e-7) */
  return sign ? -mag : mag;
}

uint8_t oracle_encode_e4m3(float x) {
  uint8_t sign = signbit(x) ? 0x80 : 0;
  if (isnan(x)) return (uint8_t)(sign | 0x7f);
  double a = fabs((double)x);
  if (a >= 464.0) return (uint8_t)(sign | 0x7e); /* 464 is the tie 448 | 480: saturate */
  if (a < ldexp(1.0, -6)) {                       /* subnormal range, quantum 2^-9 */
    double n = rint(a / ldexp(1.0, -9));         /* n == 8 is the smallest normal */
    return (uint8_t)(sign | (uint8_t)n);
  }
  int e2;
  double m = frexp(a, &e2); /* a = m * 2^e2, m in [0.5, 1) */
  int E = e2 - 1;
  double n = rint(ldexp(m, 4)); /* 2m * 8 rounded, in [8, 16] */
  if (n == 16.0) {
    n = 8.0;
    E += 1;
  }
  return (uint8_t)(sign | (uint8_t)((E + 7) << 3) | (uint8_t)(n - 8.0));
}

/* The second quantized reading: an int8 cache.  Each element holds a two's-complement code
 * in [-128, 127] with the same per-kv-head scales; the stored value is code * scale.  The
 * code follows the ONNX QuantizeLinear convention with a zero point of 0:
 *     code = saturate(round(fp32(x) / fp32(scale)))
 * rounded half to even and saturated at -128 and 127 (infinities too); NaN, which that
 * convention leaves undefined, gives 0. */
int8_t oracle_encode_i8(float x) {
  if (isnan(x)) return 0;
  double r = rint((double)x); /* the default rounding mode: nearest, ties to even */
  if (r > 127.0) r = 127.0;
  if (r < -128.0) r = -128.0;
  return (int8_t)r;
}
double oracle_decode_i8(int8_t c) { return (double)c; }

/* fmt 0: E4M3 codes; fmt 1: int8 codes */
static uint8_t encode_code(float x, int32_t fmt) {
  return fmt == 1 ? (uint8_t)oracle_encode_i8(x) : oracle_encode_e4m3(x);
}
static double decode_code(uint8_t c, int32_t fmt) {
  return fmt == 1 ? oracle_decode_i8((int8_t)c) : oracle_decode_e4m3(c);
}

void oracle_rope_append_q8(int32_t B, int32_t Hq, int32_t Hkv, int32_t D, int32_t Dv, int32_t curr, int32_t cap,
                           int32_t rope_len, int32_t dtype, int32_t do_rotary, const void *q, const void *k,
                           const void *v, const int32_t *seqlens_k, const void *cos_cache, const void *sin_cache,
                           const float *k_scale, const float *v_scale, void *q_rot, uint8_t *present_k,
                           uint8_t *present_v, int32_t *status_out, int32_t fmt) {
  size_t es = elem_size(dtype);
  int32_t status_all = 0;
  void *row = malloc(es * (size_t)(D > Dv ? D : Dv));
  for (int b = 0; b < B; ++b) {
    int32_t past = seqlens_k[b];
    int32_t st = oracle_sequence_status(past, curr, 0, cap, 0, do_rotary, rope_len);
    status_all |= st;
    if (st) continue;
    for (int h = 0; h < Hkv; ++h)
      for (int i = 0; i < curr; ++i) {
        size_t src = (((size_t)b * curr + i) * Hkv + h) * D;
        size_t dst = (((size_t)b * Hkv + h) * cap + (size_t)(past + i)) * D;
        if (do_rotary)
          rotate_row(k, src, cos_cache, sin_cache, (size_t)(past + i) * (D / 2), D, dtype, row, 0);
        else
          memcpy(row, (const char *)k + src * es, (size_t)D * es);
        for (int d = 0; d < D; ++d) present_k[dst + d] = encode_code(load_f32(row, d, dtype) / k_scale[h], fmt);
        size_t src_v = (((size_t)b * curr + i) * Hkv + h) * Dv;
        size_t dst_v = (((size_t)b * Hkv + h) * cap + (size_t)(past + i)) * Dv;
        for (int d = 0; d < Dv; ++d)
          present_v[dst_v + d] = encode_code(load_f32(v, src_v + d, dtype) / v_scale[h], fmt);
      }
    if (q_rot) {
      for (int i = 0; i < curr; ++i)
        for (int h = 0; h < Hq; ++h) {
          size_t off = (((size_t)b * curr + i) * Hq + h) * D;
          if (do_rotary)
            rotate_row(q, off, cos_cache, sin_cache, (size_t)(past + i) * (D / 2), D, dtype, q_rot, off);
          else
            memcpy((char *)q_rot + off * es, (const char *)q + off * es, (size_t)D * es);
        }
    }
  }
  free(row);
  if (status_out) *status_out = status_all;
}

void oracle_attention_q8(int32_t B, int32_t Hq, int32_t Hkv, int32_t D, int32_t Dv, int32_t curr, int32_t cap,
                         int32_t rope_len, int32_t dtype, double scale, double softcap, int32_t window,
                         int32_t causal, int32_t do_rotary, int32_t smooth_softmax, const void *q,
                         const uint8_t *present_k, const uint8_t *present_v, const float *k_scale,
                         const float *v_scale, const int32_t *seqlens_k, const float *head_sink,
                         const int64_t *rows, int64_t nrows, double *out, int32_t fmt) {
  int G = Hq / Hkv;
  if (scale == 0.0) scale = 1.0 / sqrt((double)D);
  int64_t count = rows ? nrows : (int64_t)B * curr * Hq;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1)
#endif
  for (int64_t t = 0; t < count; ++t) {
    int64_t r = rows ? rows[t] : t;
    int hq = (int)(r % Hq);
    int i = (int)((r / Hq) % curr);
    int b = (int)(r / ((int64_t)Hq * curr));
    double *o = out + (size_t)t * Dv;
    int32_t past = seqlens_k[b];
    if (oracle_sequence_status(past, curr, 0, cap, 0, do_rotary, rope_len)) {
      for (int d = 0; d < Dv; ++d) o[d] = 0.0;
      continue;
    }
    int hk = hq / G;
    int64_t total = (int64_t)past + curr;
    int64_t q_abs = (int64_t)past + i;
    /* the dequantized rows of slots [0, total) of this kv head */
    double *kd = (double *)malloc(sizeof(double) * (size_t)(total * D));
    double *vd = (double *)malloc(sizeof(double) * (size_t)(total * Dv));
    size_t kb = ((size_t)b * Hkv + hk) * (size_t)cap * D, vb = ((size_t)b * Hkv + hk) * (size_t)cap * Dv;
    for (int64_t j = 0; j < total * D; ++j) kd[j] = decode_code(present_k[kb + (size_t)j], fmt) * (double)k_scale[hk];
    for (int64_t j = 0; j < total * Dv; ++j) vd[j] = decode_code(present_v[vb + (size_t)j], fmt) * (double)v_scale[hk];
    double *qv = (double *)malloc(sizeof(double) * (size_t)D);
    for (int d = 0; d < D; ++d) qv[d] = load_elem(q, (size_t)r * D + d, dtype);
    uint8_t *vis = (uint8_t *)malloc((size_t)total);
    for (int64_t j = 0; j < total; ++j) vis[j] = (uint8_t)oracle_visible(q_abs, j, total, causal, window);
    int has_sink = head_sink != NULL || smooth_softmax;
    double z = head_sink ? (double)head_sink[hq] : 0.0;
    oracle_attend_row(qv, kd, vd, 0, total, vis, D, Dv, ODT_F64, scale, softcap, has_sink, z, o);
    free(vis);
    free(qv);
    free(vd);
    free(kd);
  }
}

int32_t oracle_has_openmp(void) {
#ifdef _OPENMP
  return 1;
#else
  return 0;
#endif
}
