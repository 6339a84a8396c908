/*
 * extkv_oracle.c -- plain, slow fp64 CPU oracle for biased grouped-query
 * attention over an external static KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, the smoke check and the bench's CPU
 * baseline may load this file's library.  It shares no code, header or
 * constant with the CUDA path; it is written from the pages' text:
 *
 *   [I366]  "Emit bias-aware external-KV (TensorScatter + nonpad_kv_seqlen)
 *           attention for float-bias decoders" (mobius issue #366):
 *           Problem, Mobius-side deliverable, Acceptance criteria.
 *   [ORT]   "ONNX Domain Attention (Opset 23/24) CUDA Patterns"
 *           (onnxruntime cuda-attention-kernel-patterns skill): section 1
 *           (unified unfused, reshape-Q GQA), 4 (op order), 6 (fully-masked
 *           rows and batches), 8 (cross-EP consistency, CPU sentinel),
 *           11 (causal alignment with an external cache), 12 (signed offsets).
 *   [SKILL] "Skill: Attention Optimization" (mobius attention-optimization):
 *           "In-place KV for ONNX Attention via TensorScatter (static cache)",
 *           "GQA sliding window via local_window_size".
 *   [PR]    "[GQA] Support KV-shared layers with empty K/V inputs"
 *           (onnxruntime PR #28242): Design, Changes.
 *
 * Element types: code 0 = fp32, code 1 = bf16 (stored as raw uint16 bits).
 * Inputs are widened exactly to double; all arithmetic is fp64; the
 * attention output is fp64.  Every loop walks indices in ascending order, and
 * rows are independent, so the result does not depend on the thread count.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_F32 0
#define ORC_BF16 1

/* ---- element access --------------------------------------------------- */

static size_t orc_elem_size(int dt) { return dt == ORC_F32 ? 4u : 2u; }

/* Exact widening of one element of type dt to double. */
static double orc_load(const void *base, int64_t idx, int dt) {
  if (dt == ORC_F32) return (double)((const float *)base)[idx];
  uint32_t bits = (uint32_t)((const uint16_t *)base)[idx] << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

/* The CPU reference masks with numeric_limits<T>::lowest(), a finite value,
 * not -inf ([ORT] section 8).  Bit patterns: fp32 0xFF7FFFFF, bf16 0xFF7F. */
static double orc_lowest(int dt) {
  uint32_t bits = dt == ORC_F32 ? 0xFF7FFFFFu : 0xFF7F0000u;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

static void orc_store_lowest(void *base, int64_t idx, int dt) {
  if (dt == ORC_F32) {
    uint32_t bits = 0xFF7FFFFFu;
    memcpy((char *)base + idx * 4, &bits, 4);
  } else {
    ((uint16_t *)base)[idx] = 0xFF7Fu;
  }
}

static void orc_store_zero(void *base, int64_t idx, int dt) {
  memset((char *)base + idx * (int64_t)orc_elem_size(dt), 0, orc_elem_size(dt));
}

static void orc_copy_elem(void *dst, int64_t di, const void *src, int64_t si, int dt) {
  size_t es = orc_elem_size(dt);
  memcpy((char *)dst + di * (int64_t)es, (const char *)src + si * (int64_t)es, es);
}

/* ---- step 1: TensorScatter into the static cache ---------------------- */
/*
 * [SKILL] "In-place KV ... via TensorScatter (static cache)": the new K/V rows
 * are written into the preallocated buffer at write_indices, in place.
 * Layout: cache (B,Hkv,max_seq,D), update (B,Hkv,S_new,D); the scatter runs
 * along the sequence axis (the cache is BNSH).  Row s of batch b lands in slot
 * write_idx[b] + s.  A batch whose rows would leave [0,max_seq) is skipped and
 * counted.  Returns the number of skipped batches.
 */
int64_t oracle_scatter(void *k_cache, void *v_cache, const void *k_new, const void *v_new,
                       const int64_t *write_idx, int64_t B, int64_t Hkv, int64_t S_new,
                       int64_t max_seq, int64_t D, int dt) {
  int64_t bad = 0;
  for (int64_t b = 0; b < B; ++b) {
    int64_t w = write_idx[b];
    if (w < 0 || w > max_seq - S_new) { ++bad; continue; }
    for (int64_t h = 0; h < Hkv; ++h)
      for (int64_t s = 0; s < S_new; ++s)
        for (int64_t d = 0; d < D; ++d) {
          int64_t src = ((b * Hkv + h) * S_new + s) * D + d;
          int64_t dst = ((b * Hkv + h) * max_seq + (w + s)) * D + d;
          orc_copy_elem(k_cache, dst, k_new, src, dt);
          orc_copy_elem(v_cache, dst, v_new, src, dt);
        }
  }
  return bad;
}

/* ---- step 2: the static-cache additive bias --------------------------- */
/*
 * [I366] deliverable: a (B,1,S_q,max_seq) additive bias keyed on absolute
 * query positions, combining causal, sliding window, bidirectional block
 * overlay and padding, valid only where slot < nonpad_kv_seqlen[b].
 *
 * Query positions ([ORT] section 11, external cache): bottom-right alignment,
 * offset[b] = nonpad[b] - S_q clamped to >= 0, query i at offset[b] + i.  The
 * difference is formed in signed 64-bit arithmetic ([ORT] section 12).  An
 * explicit q_start[b] replaces the offset when given.
 *
 * Sliding window ([SKILL] "GQA sliding window"): the query at position p sees
 * keys p-W+1 .. p, i.e. p - j < W.  window <= 0 means no window.
 *
 * Block overlay: tokens of one image span see every token of that span, past
 * or future.  Spans are (start, len) pairs in absolute positions, grouped per
 * batch by span_offsets (length B+1).  Composition (the pages name the overlay
 * but give no formula; the reading used is the OR-overlay):
 *     allowed = j < nonpad && ((causal_ok && window_ok) || same_span)
 * Value: allowed ? extra[b,0,i,j] (or 0 without extra) : lowest(T).
 * A batch with nonpad outside [0,max_seq] is skipped and counted.
 */
static int orc_same_span(const int64_t *span_offsets, const int64_t *spans, int64_t b, int64_t p,
                         int64_t j) {
  if (!span_offsets || !spans) return 0;
  for (int64_t s = span_offsets[b]; s < span_offsets[b + 1]; ++s) {
    int64_t lo = spans[2 * s], hi = spans[2 * s] + spans[2 * s + 1];
    if (p >= lo && p < hi && j >= lo && j < hi) return 1;
  }
  return 0;
}

static int orc_allowed(int causal, int64_t window, const int64_t *span_offsets, const int64_t *spans,
                int64_t b, int64_t nonpad, int64_t p, int64_t j) {
  if (j >= nonpad) return 0;
  int causal_ok = !causal || j <= p;
  int window_ok = window <= 0 || p - j < window;
  return (causal_ok && window_ok) || orc_same_span(span_offsets, spans, b, p, j);
}

int64_t oracle_bias(void *bias, int causal, int64_t window, const int64_t *span_offsets,
                    const int64_t *spans, const void *extra, const int64_t *q_start,
                    const int64_t *nonpad, int64_t B, int64_t S_q, int64_t max_seq, int dt) {
  int64_t bad = 0;
  for (int64_t b = 0; b < B; ++b) {
    int64_t np = nonpad[b];
    if (np < 0 || np > max_seq) { ++bad; continue; }
    int64_t qs = q_start ? q_start[b] : (np - S_q > 0 ? np - S_q : 0);
    for (int64_t i = 0; i < S_q; ++i) {
      int64_t p = qs + i;
      for (int64_t j = 0; j < max_seq; ++j) {
        int64_t idx = (b * S_q + i) * max_seq + j;
        if (orc_allowed(causal, window, span_offsets, spans, b, np, p, j)) {
          if (extra) orc_copy_elem(bias, idx, extra, idx, dt);
          else orc_store_zero(bias, idx, dt);
        } else {
          orc_store_lowest(bias, idx, dt);
        }
      }
    }
  }
  return bad;
}

/* ---- a boolean attention mask as the additive bias ---------------------- */
/*
 * [ORT] section 6, "Additive-bias path", and the attention-mask skill ("Bool
 * mask vs float additive bias"): a boolean mask is turned into an additive
 * bias -- an attended slot (mask != 0) gets 0, a masked slot the sentinel,
 * here lowest(T) as for every other masked slot of this path ([ORT] section
 * 8).  n elements of (B,1,S_q,max_seq), element by element.
 */
void oracle_bias_from_mask(void *bias, const unsigned char *mask, int64_t n, int dt) {
  for (int64_t i = 0; i < n; ++i) {
    if (mask[i]) orc_store_zero(bias, i, dt);
    else orc_store_lowest(bias, i, dt);
  }
}

/* ---- steps 3-6: scores, bias, softmax, PV ----------------------------- */
/*
 * One query row (b, h, i), written out as the plain definition:
 *   kv head  = h / (Hq/Hkv)          (contiguous groups; the reshape-Q GQA of
 *                                     [ORT] section 1 shares one KV head among
 *                                     Hq/Hkv consecutive query heads)
 *   U        = { j < nonpad[b] : bias[b,0,i,j] > lowest(T) }   ([ORT] section 6:
 *              a key is unmasked iff it is inside the nonpad frontier and its
 *              bias is above the sentinel; a finite very negative bias stays
 *              unmasked)
 *   U empty  -> y = 0                ([ORT] section 6, rows and whole batches)
 *   s_j      = c(scale * (q . k_j)) + bias_j      ([ORT] section 4 op order:
 *              c(x) = cap * tanh(x / cap) when the softcap cap > 0, else x;
 *              the cap acts before the bias, so a masked slot stays masked)
 *   y        = sum_{j in U} exp(s_j - m) v_j / sum_{j in U} exp(s_j - m),
 *              m = max_{j in U} s_j  (max-subtracted softmax, [ORT] section 8)
 * Without a bias, U = { j < nonpad[b] } and bias_j = 0.
 * q and k rows have Dk elements, v rows and y rows Dv: the query-key head
 * size and the value head size may differ (the "ORT CUDA Attention Kernel
 * Dispatch" section of the attention-optimization skill: a KV-shared layer
 * borrowing K/V from a layer of another head size has head_size !=
 * v_head_size); the scores use the Dk-long dot products, the output is a
 * weighted sum of Dv-long value rows.
 * Returns 0, or 1 when nonpad[b] is outside [0,max_seq] (the row is zeroed).
 */
static int orc_row(double *y, const void *q, const void *k_cache, const void *v_cache,
                   const void *bias, const int64_t *nonpad, double scale, double softcap, int64_t Hq,
                   int64_t Hkv, int64_t S_q, int64_t max_seq, int64_t Dk, int64_t Dv, int dt, int64_t b,
                   int64_t h, int64_t i, double *s, unsigned char *in_u) {
  int64_t np = nonpad[b];
  for (int64_t d = 0; d < Dv; ++d) y[d] = 0.0;
  if (np < 0 || np > max_seq) return 1;
  int64_t kv = h / (Hq / Hkv);
  const int64_t q_off = ((b * Hq + h) * S_q + i) * Dk;
  const int64_t kv_base = (b * Hkv + kv) * max_seq;
  const double lowest = orc_lowest(dt);
  int any = 0;
  double m = -INFINITY;
  for (int64_t j = 0; j < np; ++j) {
    double bj = bias ? orc_load(bias, (b * S_q + i) * max_seq + j, dt) : 0.0;
    in_u[j] = (unsigned char)(!bias || bj > lowest);
    if (!in_u[j]) continue;
    double dot = 0.0;
    for (int64_t d = 0; d < Dk; ++d)
      dot += orc_load(q, q_off + d, dt) * orc_load(k_cache, (kv_base + j) * Dk + d, dt);
    double t = scale * dot;
    if (softcap > 0.0) t = softcap * tanh(t / softcap);
    s[j] = t + bj;
    if (!any || s[j] > m) m = s[j];
    any = 1;
  }
  if (!any) return 0;
  double denom = 0.0;
  for (int64_t j = 0; j < np; ++j) {
    if (!in_u[j]) continue;
    double w = exp(s[j] - m);
    denom += w;
    for (int64_t d = 0; d < Dv; ++d) y[d] += w * orc_load(v_cache, (kv_base + j) * Dv + d, dt);
  }
  for (int64_t d = 0; d < Dv; ++d) y[d] /= denom;
  return 0;
}

/*
 * Attention over the external cache for all rows (rows == NULL, y is
 * (B,Hq,S_q,Dv)) or for the n_rows flat row indices r = (b*Hq + h)*S_q + i
 * listed in rows (y is (n_rows,Dv)).  q is (B,Hq,S_q,Dk), the caches
 * (B,Hkv,max_seq,Dk) and (B,Hkv,max_seq,Dv); bias is NULL or
 * (B,1,S_q,max_seq).  A KV-shared layer ([PR] Design) is this same call on a
 * borrowed cache with no preceding scatter.  Returns the number of rows whose
 * batch had an out-of-range nonpad.
 */
int64_t oracle_attention_dv(double *y, const void *q, const void *k_cache, const void *v_cache, const void *bias,
                            const int64_t *nonpad, float scale, float softcap, int64_t B, int64_t Hq, int64_t Hkv,
                            int64_t S_q, int64_t max_seq, int64_t Dk, int64_t Dv, int dt, const int64_t *rows,
                            int64_t n_rows) {
  int64_t total = rows ? n_rows : B * Hq * S_q;
  int64_t bad = 0;
#pragma omp parallel reduction(+ : bad)
  {
    double *s = (double *)malloc(sizeof(double) * (size_t)(max_seq > 0 ? max_seq : 1));
    unsigned char *in_u = (unsigned char *)malloc((size_t)(max_seq > 0 ? max_seq : 1));
#pragma omp for schedule(dynamic, 4)
    for (int64_t t = 0; t < total; ++t) {
      int64_t r = rows ? rows[t] : t;
      int64_t i = r % S_q, bh = r / S_q;
      int64_t h = bh % Hq, b = bh / Hq;
      bad += orc_row(y + t * Dv, q, k_cache, v_cache, bias, nonpad, (double)scale, (double)softcap, Hq, Hkv,
                     S_q, max_seq, Dk, Dv, dt, b, h, i, s, in_u);
    }
    free(s);
    free(in_u);
  }
  return bad;
}

/* One head size for queries, keys and values. */
int64_t oracle_attention_softcap(double *y, const void *q, const void *k_cache, const void *v_cache,
                                 const void *bias, const int64_t *nonpad, float scale, float softcap,
                                 int64_t B, int64_t Hq, int64_t Hkv, int64_t S_q, int64_t max_seq, int64_t D,
                                 int dt, const int64_t *rows, int64_t n_rows) {
  return oracle_attention_dv(y, q, k_cache, v_cache, bias, nonpad, scale, softcap, B, Hq, Hkv, S_q, max_seq, D, D,
                             dt, rows, n_rows);
}

/* The attention without a softcap. */
int64_t oracle_attention(double *y, const void *q, const void *k_cache, const void *v_cache,
                         const void *bias, const int64_t *nonpad, float scale, int64_t B,
                         int64_t Hq, int64_t Hkv, int64_t S_q, int64_t max_seq, int64_t D, int dt,
                         const int64_t *rows, int64_t n_rows) {
  return oracle_attention_softcap(y, q, k_cache, v_cache, bias, nonpad, scale, 0.0f, B, Hq, Hkv, S_q, max_seq, D,
                                  dt, rows, n_rows);
}

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
