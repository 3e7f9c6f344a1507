/*
 * fp64 CPU oracle for multi-head scaled dot-product attention (forward and
 * backward).
 *
 * TEST INFRASTRUCTURE ONLY.  This file is compiled into a host library that
 * the tests, the package's smoke check and the bench's CPU-baseline leg load to
 * check the CUDA path.  The product path never links, loads or calls it, and it
 * shares no code, header or constant with the CUDA sources.
 *
 * What it computes, per (batch b, head h, query row i), following
 * "Attention Is All You Need" as explained on the pages
 *   - trishampatil.com, "Scaled Dot-Product Attention: Step by Step"
 *     (Attention(Q,K,V) = softmax(QK^T / sqrt(d_k)) V, steps 1-4) and
 *     "Why Masking Is Required" (illegal logits set to -inf, exp(-inf) = 0);
 *   - aicomputerinstitute.com, "Worked example: attention weights and
 *     outputs by hand" (the same four steps on numbers);
 *   - alexdo.xyz, "Decoder block" (causal: position i sees positions <= i;
 *     cross-attention T x S) and "Two masks, not one" (padded slots get -inf);
 *   - aicassindra.com, "Pitfalls when reproducing the paper" (padding masks
 *     keys, not queries; a row with every key masked would be NaN).
 *
 *   0. len_b = clamp(key_lengths[b], 0, Lk) when a padding bit is set.
 *   1. QUERY_PADDING and i >= len_b: the row is padding, output +0.  Stop.
 *   2. Allowed keys A_i = { j < Lk : (!CAUSAL or j <= i) and
 *                                    (!KEY_PADDING or j < len_b) and
 *                                    (!CAUSAL_TAIL or j <= len_b - Lq + i) }.
 *      CAUSAL_TAIL is generation with a key/value cache (alexdo.xyz, "How
 *      predictions are generated": the keys and values of earlier positions
 *      are cached, only the new positions are computed): the Lq queries are
 *      the last Lq positions len_b - Lq .. len_b - 1 of a sequence whose
 *      len_b keys are in the cache (len_b = Lk without KEY_PADDING), and each
 *      sees the keys up to its own position.
 *   3. A_i empty: output +0 (the pages leave this row undefined -- NaN -- and
 *      ask that no query attend to nothing; zero is the convention here).
 *   4. s_j = scale * sum_c q[i,c] k[j,c]                (step 1 and step 2)
 *   5. w_j = exp(s_j - m) / sum_{j' in A_i} exp(s_j' - m),  m = max s_j
 *      (step 3; subtracting the row max leaves the quotient unchanged).
 *      Keys outside A_i have weight exactly 0 (exp(-inf) = 0).
 *   6. out[i,c] = sum_{j in A_i} w_j v[j,c]             (step 4)
 *
 * Every product and sum is in IEEE double, in index order, one row at a time.
 * Inputs are read in their stored type (double, float or bfloat16 bits) and
 * widened exactly to double.  Rows are independent; OpenMP spreads them over
 * host threads without changing any row's arithmetic.
 *
 * Layouts (contiguous): layout 0 ("BHSD", the per-head layout after the head
 * split): q [B,H,Lq,dk], k [B,Hkv,Lk,dk], v [B,Hkv,Lk,dv]; layout 1 ("BSHD",
 * the layout before the split): q [B,Lq,H,dk], k [B,Lk,Hkv,dk],
 * v [B,Lk,Hkv,dv].  Hkv key/value heads serve H query heads, Hkv dividing H:
 * query head h reads key/value head h / (H / Hkv) (zeroshotmind.com, "Many
 * heads, many subspaces": grouped- and multi-query attention share or
 * collapse the key/value heads).  Hkv == H is plain multi-head attention.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORACLE_IN_F64 = 0, ORACLE_IN_F32 = 1, ORACLE_IN_BF16 = 2 };
enum { ORACLE_CAUSAL = 1, ORACLE_KEY_PADDING = 2, ORACLE_QUERY_PADDING = 4, ORACLE_CAUSAL_TAIL = 8 };

static double widen(const void *base, int in_dtype, int64_t idx) {
  if (in_dtype == ORACLE_IN_F64) return ((const double *)base)[idx];
  if (in_dtype == ORACLE_IN_F32) return (double)((const float *)base)[idx];
  /* bfloat16: the upper half of a float32 */
  uint32_t u = (uint32_t)((const uint16_t *)base)[idx] << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* element offset of (b, head, position, c) in a tensor of `heads` heads,
   `len` positions and `d` columns */
static int64_t offset(int layout, int64_t b, int64_t head, int64_t pos, int64_t c, int64_t heads,
                      int64_t len, int64_t d) {
  if (layout == 0) return ((b * heads + head) * len + pos) * d + c;
  return ((b * len + pos) * heads + head) * d + c;
}

/*
 * Computes the rows listed in `rows` (logical index (b*H + h)*Lq + i,
 * whatever the layout), or every row in that order when rows == NULL (then
 * nrows must be B*H*Lq).
 *   out     [nrows, dv]           attention output rows
 *   weights [nrows, Lk] or NULL   softmax weights (0 outside A_i)
 *   scores  [nrows, Lk] or NULL   scaled logits s_j (-inf outside A_i)
 * Returns 0 on success, 1 on an invalid argument.
 */
int oracle_mha_rows_ex_f64(const void *q, const void *k, const void *v, int in_dtype,
                           int B, int H, int Hkv, int Lq, int Lk, int dk, int dv, int layout,
                           int mask_kind, const int32_t *key_lengths, double scale,
                           const int64_t *rows, int64_t nrows,
                           double *out, double *weights, double *scores, int nthreads) {
  if (B < 0 || H < 0 || Lq < 0 || Lk < 0 || dk < 0 || dv < 0) return 1;
  if (Hkv <= 0 ? H > 0 : (H % Hkv) != 0) return 1;
  if (layout != 0 && layout != 1) return 1;
  if (in_dtype < ORACLE_IN_F64 || in_dtype > ORACLE_IN_BF16) return 1;
  if (mask_kind & ~(ORACLE_CAUSAL | ORACLE_KEY_PADDING | ORACLE_QUERY_PADDING | ORACLE_CAUSAL_TAIL))
    return 1;
  if ((mask_kind & (ORACLE_CAUSAL | ORACLE_QUERY_PADDING)) && Lq != Lk) return 1;
  if ((mask_kind & ORACLE_CAUSAL_TAIL) && (mask_kind & (ORACLE_CAUSAL | ORACLE_QUERY_PADDING)))
    return 1;
  if ((mask_kind & (ORACLE_KEY_PADDING | ORACLE_QUERY_PADDING)) && key_lengths == NULL && B > 0)
    return 1;
  const int64_t total = (int64_t)B * H * Lq;
  if (rows == NULL && nrows != total) return 1;
  if (nrows < 0) return 1;
  for (int64_t r = 0; rows != NULL && r < nrows; ++r)
    if (rows[r] < 0 || rows[r] >= total) return 1;
  if (nthreads <= 0) nthreads = oracle_max_threads();

  int bad = 0;
#pragma omp parallel num_threads(nthreads)
  {
    double *s = (double *)malloc(sizeof(double) * (size_t)(Lk > 0 ? Lk : 1));
    char *allowed = (char *)malloc((size_t)(Lk > 0 ? Lk : 1));
    if (s == NULL || allowed == NULL) {
#pragma omp atomic write
      bad = 1;
    }
#pragma omp for schedule(dynamic, 8)
    for (int64_t r = 0; r < nrows; ++r) {
      if (s == NULL || allowed == NULL) continue;
      const int64_t row = rows ? rows[r] : r;
      const int64_t bh = row / Lq;
      const int i = (int)(row % Lq);
      const int b = (int)(bh / H);
      double *o = out + r * dv;
      double *w = weights ? weights + r * Lk : NULL;
      double *sc = scores ? scores + r * Lk : NULL;

      /* step 0 */
      int len_b = Lk;
      if (mask_kind & (ORACLE_KEY_PADDING | ORACLE_QUERY_PADDING)) {
        int32_t l = key_lengths[b];
        len_b = l < 0 ? 0 : (l > Lk ? Lk : (int)l);
      }
      for (int c = 0; c < dv; ++c) o[c] = 0.0;
      for (int j = 0; j < Lk; ++j) {
        if (w) w[j] = 0.0;
        if (sc) sc[j] = -INFINITY;
      }
      /* step 1 */
      if ((mask_kind & ORACLE_QUERY_PADDING) && i >= len_b) continue;
      /* step 2 */
      int n_allowed = 0;
      for (int j = 0; j < Lk; ++j) {
        int ok = 1;
        if ((mask_kind & ORACLE_CAUSAL) && j > i) ok = 0;
        if ((mask_kind & ORACLE_KEY_PADDING) && j >= len_b) ok = 0;
        if ((mask_kind & ORACLE_CAUSAL_TAIL) && j > len_b - Lq + i) ok = 0;
        allowed[j] = (char)ok;
        n_allowed += ok;
      }
      /* step 3 */
      if (n_allowed == 0) continue;
      /* step 4 */
      const int h = (int)(bh % H);
      const int hk = h / (H / Hkv);
      for (int j = 0; j < Lk; ++j) {
        if (!allowed[j]) continue;
        double dot = 0.0;
        for (int c = 0; c < dk; ++c)
          dot += widen(q, in_dtype, offset(layout, b, h, i, c, H, Lq, dk)) *
                 widen(k, in_dtype, offset(layout, b, hk, j, c, Hkv, Lk, dk));
        s[j] = scale * dot;
        if (sc) sc[j] = s[j];
      }
      /* step 5 */
      double m = -INFINITY;
      for (int j = 0; j < Lk; ++j)
        if (allowed[j] && s[j] > m) m = s[j];
      double denom = 0.0;
      for (int j = 0; j < Lk; ++j)
        if (allowed[j]) {
          s[j] = exp(s[j] - m);
          denom += s[j];
        }
      /* step 6 */
      for (int j = 0; j < Lk; ++j) {
        if (!allowed[j]) continue;
        const double wj = s[j] / denom;
        if (w) w[j] = wj;
        for (int c = 0; c < dv; ++c)
          o[c] += wj * widen(v, in_dtype, offset(layout, b, hk, j, c, Hkv, Lk, dv));
      }
    }
    free(s);
    free(allowed);
  }
  return bad ? 1 : 0;
}

/* multi-head attention in the per-head layout (Hkv == H, layout 0) */
int oracle_mha_rows_f64(const void *q, const void *k, const void *v, int in_dtype,
                        int B, int H, int Lq, int Lk, int dk, int dv,
                        int mask_kind, const int32_t *key_lengths, double scale,
                        const int64_t *rows, int64_t nrows,
                        double *out, double *weights, double *scores, int nthreads) {
  return oracle_mha_rows_ex_f64(q, k, v, in_dtype, B, H, H, Lq, Lk, dk, dv, 0, mask_kind,
                                key_lengths, scale, rows, nrows, out, weights, scores, nthreads);
}

/*
 * Backward pass: the gradients of a scalar loss L through the forward above,
 * for training (trishampatil.com, "Training (Teacher Forcing + Masking)": the
 * whole target sequence goes through one parallel forward pass under the
 * causal mask and the gradients flow back through every layer at once;
 * aicomputerinstitute.com, "The core idea: attention as a lookup, not a
 * summary": the gradient through a saturated softmax vanishes, which is why
 * the scores are scaled).  The pages print no backward formulas; these are
 * the derivatives of steps 4-6 as written, by the chain rule.  Given
 * dout = dL/dout, for each computed row i of query head h (key/value head g):
 *
 *   g_j = sum_c dout[i,c] v[j,c]              dL/dw_j            (step 6)
 *   D   = sum_{j in A_i} w_j g_j
 *   t_j = w_j (g_j - D)                       dL/ds_j, from the softmax
 *                                              Jacobian dw_j/ds_l =
 *                                              w_j (delta_jl - w_l) (step 5)
 *   dq[i,c]  = scale sum_{j in A_i} t_j k[j,c]                     (step 4)
 *   dk[j,c] += scale t_j q[i,c]
 *   dv[j,c] += w_j dout[i,c]                                       (step 6)
 *
 * Rows whose output is fixed at +0 (steps 1 and 3) depend on no input: they
 * contribute nothing and their dq is 0.  Keys outside A_i get nothing from
 * row i.  With shared key/value heads, dk and dv of head g sum over the query
 * heads that read g.  Sums run in index order (heads, then rows, then keys),
 * in IEEE double.
 *
 * Work is split by (batch element, key/value head) units, so each unit's dk
 * and dv are written by one thread.  units / nunits: the logical units
 * b * Hkv + g to compute (NULL: all B * Hkv); [i_lo, i_hi): the query rows
 * taken in each (a timing sample; 0, Lq for the whole pass).  dq, dk, dv are
 * full tensors in the inputs' layout; only the listed units' parts are
 * written.  Returns 0, or 1 on an invalid argument.
 */
int oracle_mha_bwd_f64(const void *q, const void *k, const void *v, const void *dout,
                       int in_dtype, int B, int H, int Hkv, int Lq, int Lk, int dk, int dv,
                       int layout, int mask_kind, const int32_t *key_lengths, double scale,
                       const int64_t *units, int64_t nunits, int i_lo, int i_hi, double *dq,
                       double *dk_out, double *dv_out, int nthreads) {
  if (B < 0 || H < 0 || Lq < 0 || Lk < 0 || dk < 0 || dv < 0) return 1;
  if (Hkv <= 0 ? H > 0 : (H % Hkv) != 0) return 1;
  if (layout != 0 && layout != 1) return 1;
  if (in_dtype < ORACLE_IN_F64 || in_dtype > ORACLE_IN_BF16) return 1;
  if (mask_kind & ~(ORACLE_CAUSAL | ORACLE_KEY_PADDING | ORACLE_QUERY_PADDING | ORACLE_CAUSAL_TAIL))
    return 1;
  if ((mask_kind & (ORACLE_CAUSAL | ORACLE_QUERY_PADDING)) && Lq != Lk) return 1;
  if ((mask_kind & ORACLE_CAUSAL_TAIL) && (mask_kind & (ORACLE_CAUSAL | ORACLE_QUERY_PADDING)))
    return 1;
  if ((mask_kind & (ORACLE_KEY_PADDING | ORACLE_QUERY_PADDING)) && key_lengths == NULL && B > 0)
    return 1;
  if (i_lo < 0 || i_hi > Lq || i_lo > i_hi) return 1;
  const int64_t total_units = Hkv > 0 ? (int64_t)B * Hkv : 0;
  if (units == NULL && nunits != total_units) return 1;
  if (nunits < 0) return 1;
  for (int64_t u = 0; units != NULL && u < nunits; ++u)
    if (units[u] < 0 || units[u] >= total_units) return 1;
  if (nthreads <= 0) nthreads = oracle_max_threads();
  const int group = Hkv > 0 ? H / Hkv : 0;

  int bad = 0;
#pragma omp parallel num_threads(nthreads)
  {
    const size_t n = (size_t)(Lk > 0 ? Lk : 1);
    double *w = (double *)malloc(sizeof(double) * n);
    double *g = (double *)malloc(sizeof(double) * n);
    char *allowed = (char *)malloc(n);
    if (w == NULL || g == NULL || allowed == NULL) {
#pragma omp atomic write
      bad = 1;
    }
#pragma omp for schedule(dynamic, 1)
    for (int64_t u = 0; u < nunits; ++u) {
      if (w == NULL || g == NULL || allowed == NULL) continue;
      const int64_t unit = units ? units[u] : u;
      const int b = (int)(unit / Hkv), hk = (int)(unit % Hkv);
      /* this unit's gradients start at zero */
      for (int j = 0; j < Lk; ++j) {
        for (int c = 0; c < dk; ++c) dk_out[offset(layout, b, hk, j, c, Hkv, Lk, dk)] = 0.0;
        for (int c = 0; c < dv; ++c) dv_out[offset(layout, b, hk, j, c, Hkv, Lk, dv)] = 0.0;
      }
      for (int h = hk * group; h < (hk + 1) * group; ++h)
        for (int i = 0; i < Lq; ++i)
          for (int c = 0; c < dk; ++c) dq[offset(layout, b, h, i, c, H, Lq, dk)] = 0.0;
      int len_b = Lk;
      if (mask_kind & (ORACLE_KEY_PADDING | ORACLE_QUERY_PADDING)) {
        int32_t l = key_lengths[b];
        len_b = l < 0 ? 0 : (l > Lk ? Lk : (int)l);
      }
      for (int h = hk * group; h < (hk + 1) * group; ++h) {
        for (int i = i_lo; i < i_hi; ++i) {
          /* steps 1-3: rows whose output is fixed contribute nothing */
          if ((mask_kind & ORACLE_QUERY_PADDING) && i >= len_b) continue;
          int n_allowed = 0;
          for (int j = 0; j < Lk; ++j) {
            int ok = 1;
            if ((mask_kind & ORACLE_CAUSAL) && j > i) ok = 0;
            if ((mask_kind & ORACLE_KEY_PADDING) && j >= len_b) ok = 0;
            if ((mask_kind & ORACLE_CAUSAL_TAIL) && j > len_b - Lq + i) ok = 0;
            allowed[j] = (char)ok;
            n_allowed += ok;
          }
          if (n_allowed == 0) continue;
          /* steps 4-5 again: the weights w_j */
          double m = -INFINITY;
          for (int j = 0; j < Lk; ++j) {
            if (!allowed[j]) continue;
            double dot = 0.0;
            for (int c = 0; c < dk; ++c)
              dot += widen(q, in_dtype, offset(layout, b, h, i, c, H, Lq, dk)) *
                     widen(k, in_dtype, offset(layout, b, hk, j, c, Hkv, Lk, dk));
            w[j] = scale * dot;
            if (w[j] > m) m = w[j];
          }
          double denom = 0.0;
          for (int j = 0; j < Lk; ++j)
            if (allowed[j]) {
              w[j] = exp(w[j] - m);
              denom += w[j];
            }
          for (int j = 0; j < Lk; ++j) w[j] = allowed[j] ? w[j] / denom : 0.0;
          /* g_j and D */
          double D = 0.0;
          for (int j = 0; j < Lk; ++j) {
            if (!allowed[j]) continue;
            double gj = 0.0;
            for (int c = 0; c < dv; ++c)
              gj += widen(dout, in_dtype, offset(layout, b, h, i, c, H, Lq, dv)) *
                    widen(v, in_dtype, offset(layout, b, hk, j, c, Hkv, Lk, dv));
            g[j] = gj;
            D += w[j] * gj;
          }
          /* t_j, then the three gradients */
          for (int j = 0; j < Lk; ++j) {
            if (!allowed[j]) continue;
            const double t = w[j] * (g[j] - D);
            for (int c = 0; c < dk; ++c) {
              dq[offset(layout, b, h, i, c, H, Lq, dk)] +=
                  scale * t * widen(k, in_dtype, offset(layout, b, hk, j, c, Hkv, Lk, dk));
              dk_out[offset(layout, b, hk, j, c, Hkv, Lk, dk)] +=
                  scale * t * widen(q, in_dtype, offset(layout, b, h, i, c, H, Lq, dk));
            }
            for (int c = 0; c < dv; ++c)
              dv_out[offset(layout, b, hk, j, c, Hkv, Lk, dv)] +=
                  w[j] * widen(dout, in_dtype, offset(layout, b, h, i, c, H, Lq, dv));
          }
        }
      }
    }
    free(w);
    free(g);
    free(allowed);
  }
  return bad ? 1 : 0;
}
