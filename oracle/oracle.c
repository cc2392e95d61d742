/*
 * oracle.c -- plain, slow CPU oracle for one decode step of grouped-query
 * attention over a paged KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file: only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg do.  It shares no code, header, table or helper with the
 * CUDA library; it is written from the definitions on the source pages:
 *
 *  [S1] "LLM inference from smollm3.go" (zhuyie.github.io), section
 *       "Self-attention: how the current token looks back": score of a cached
 *       position = dot(q, k) * attScale; softmax over positions 0..pos (the
 *       current token included); output = sum of softmax-weighted V rows.
 *  [S2] same page, section "Positional encoding: why the model knows order":
 *       RoPE rotates pairs of q/k coordinates by a position-dependent angle;
 *       the cos/sin depend on (position, headSize, RopeTheta).
 *  [S3] same page, section "Multi-head attention": query head h reads KV head
 *       h / kvMul (consecutive query heads share one KV head).
 *  [S4] same page, section "KV cache: the link between the two": the new K/V
 *       are written at the current position, then attention covers [0, pos].
 *  [S5] same page, section "int8 weight-only quantization": a row is stored
 *       as int8 codes plus one fp32 scale max(abs(row)) / 127.
 *  [S6] "C17 CPU-first LLM inference engine" (nxmr.cn), section 4.4
 *       "Attention: GQA + RoPE": RoPE splits the vector into two halves
 *       (half-split, not interleaved).
 *  [S7] "Qwen3-8B inference engine from scratch in C++/CUDA" (jh158.com),
 *       section 4.3.1 "Paged KV cache": fixed-size blocks, the last block of
 *       a sequence receives the appended token; section 4.4.2 "GQA grouped
 *       decode": scores are dot(q_h, K_g) / sqrt(d_head), one KV group serves
 *       all query heads of the group.
 *  [S8] "lightLLM, a pure-Python inference framework" (haoling.cc), section 1
 *       "Overview": Int8KV cache; the cache write around attention.
 *
 * Readings taken where the pages are silent:
 *  - frequency i of a head of size d is theta^(-2i/d), i < d/2; pair (i, i+d/2);
 *  - cached K are stored after RoPE; only q and the new k are rotated here;
 *  - seq_lens[b] = tokens cached before the step = slot of the new token;
 *    positions[b] = RoPE position of the new token;
 *  - page layout [page][kv_head][slot][d]; int8 scales [page][kv_head][slot];
 *  - storage recipe of the appended k: cos/sin computed in double, rounded to
 *    fp32; rotation with fp32 products and sums (each rounded, no fused
 *    multiply-add); bf16 round-to-nearest-even, or int8 with scale
 *    fl32(max|x| / 127), code = clamp(rint(fl32(x / scale)), -127, 127),
 *    an all-zero row gives scale 0 and codes 0;
 *  - a sequence whose length is out of range is skipped (its output row is
 *    left untouched); a page index outside [0, num_pages) makes the tokens of
 *    that page invisible (and no append happens there); a sequence with no
 *    visible token gets a zero output row.
 *
 * Everything that is not the storage recipe is computed in IEEE double.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* status bits, same meaning as the device status word of the library */
#define ORC_BAD_LEN 1u  /* seq_lens[b] < 0 or seq_lens[b] + 1 > max_pages*page */
#define ORC_BAD_PAGE 2u /* a block-table entry used by the step is out of range */

/* ---------------------------------------------------------------- bf16 --- */

static double bf16_to_double(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

static float bf16_to_float(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

/* IEEE round-to-nearest-even of an fp32 value to bf16 (NaN kept quiet). */
static uint16_t float_to_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu) != 0)
    return (uint16_t)((u >> 16) | 0x0040u);
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7fffu + lsb;
  return (uint16_t)(u >> 16);
}

/* ---------------------------------------------------------------- RoPE --- */

/* Inverse frequency of rotation pair i for a head of size d [S2][S6]. */
static double rope_inv_freq(double theta, int i, int d) {
  return pow(theta, -(2.0 * i) / d);
}

/*
 * Half-split RoPE in double [S2][S6]: for i < d/2, with phi = pos * theta^(-2i/d),
 *   y[i]       = x[i] cos(phi) - x[i+d/2] sin(phi)
 *   y[i+d/2]   = x[i+d/2] cos(phi) + x[i] sin(phi)
 * theta <= 0 means "no RoPE on this layer" (y = x).
 */
void oracle_rope_f64(const double *x, int d, double pos, double theta, double *y) {
  int h = d / 2;
  if (!(theta > 0.0)) {
    for (int i = 0; i < d; ++i) y[i] = x[i];
    return;
  }
  for (int i = 0; i < h; ++i) {
    double phi = pos * rope_inv_freq(theta, i, d);
    double c = cos(phi), s = sin(phi);
    double lo = x[i], hi = x[i + h];
    y[i] = lo * c - hi * s;
    y[i + h] = hi * c + lo * s;
  }
}

/*
 * Storage recipe of the appended key (fp32): the rotation of [S2][S6] with
 * c = (float)cos(phi), s = (float)sin(phi), phi = (double)pos * theta^(-2i/d)
 * computed in double, and every product and sum rounded to fp32 on its own.
 * The volatile temporaries keep the compiler from fusing a multiply and an add.
 */
void oracle_rope_store_f32(const uint16_t *x_bf16, int d, int pos, float theta,
                           float *y) {
  int h = d / 2;
  if (!(theta > 0.0f)) {
    for (int i = 0; i < d; ++i) y[i] = bf16_to_float(x_bf16[i]);
    return;
  }
  for (int i = 0; i < h; ++i) {
    double phi = (double)pos * rope_inv_freq((double)theta, i, d);
    float c = (float)cos(phi), s = (float)sin(phi);
    float lo = bf16_to_float(x_bf16[i]), hi = bf16_to_float(x_bf16[i + h]);
    volatile float lc = lo * c, hs = hi * s, hc = hi * c, ls = lo * s;
    volatile float a = lc - hs, b = hc + ls;
    y[i] = a;
    y[i + h] = b;
  }
}

/*
 * Symmetric int8 quantisation of one row [S5] (per token and KV head):
 * scale = fl32(max|x| / 127); code = clamp(rint(fl32(x / scale)), -127, 127),
 * rint rounding half to even; a zero row gives scale 0 and codes 0.
 */
void oracle_quant_int8(const float *x, int d, int8_t *codes, float *scale) {
  float a = 0.0f;
  for (int i = 0; i < d; ++i) {
    float m = fabsf(x[i]);
    if (m > a) a = m;
  }
  if (a == 0.0f) {
    *scale = 0.0f;
    for (int i = 0; i < d; ++i) codes[i] = 0;
    return;
  }
  volatile float sc = a / 127.0f;
  *scale = sc;
  for (int i = 0; i < d; ++i) {
    volatile float t = x[i] / sc;
    float r = rintf(t);
    if (r > 127.0f) r = 127.0f;
    if (r < -127.0f) r = -127.0f;
    codes[i] = (int8_t)r;
  }
}

/* ------------------------------------------------------------- layout --- */

typedef struct {
  int n_seq, n_qh, n_kvh, d, page, max_pages, num_pages, kv_int8;
} geom_t;

static size_t slot_index(const geom_t *g, int page, int j, int off) {
  return (((size_t)page * g->n_kvh + j) * g->page + off);
}

static int seq_len_ok(const geom_t *g, int L) {
  return L >= 0 && (long long)L + 1 <= (long long)g->max_pages * g->page;
}

/* physical page of token t of sequence b, or -1 if the entry is out of range */
static int page_of(const geom_t *g, const int32_t *block_table, int b, int t) {
  int p = block_table[(size_t)b * g->max_pages + t / g->page];
  return (p >= 0 && p < g->num_pages) ? p : -1;
}

/* value of element i of cached token t (head j), dequantised to double */
static double kv_value(const geom_t *g, const void *pool, const float *scales,
                       int page, int j, int off, int i) {
  size_t s = slot_index(g, page, j, off);
  if (g->kv_int8) {
    const int8_t *p = (const int8_t *)pool;
    return (double)p[s * g->d + i] * (double)scales[s];
  }
  const uint16_t *p = (const uint16_t *)pool;
  return bf16_to_double(p[s * g->d + i]);
}

/* -------------------------------------------------------------- append --- */

/*
 * Write the new token of every valid sequence into slot seq_lens[b] of its
 * pages [S4][S7]: page = block_table[b][L / page], offset L % page; the key is
 * rotated by the storage recipe, the value is stored as given (bf16) or both
 * are quantised [S5][S8].  Returns the status bits.
 */
unsigned oracle_append(const uint16_t *k_new, const uint16_t *v_new, void *k_pages,
                       void *v_pages, float *k_scales, float *v_scales,
                       const int32_t *block_table, const int32_t *seq_lens,
                       const int32_t *positions, int n_seq, int n_kvh, int d,
                       int page, float rope_theta, int kv_int8, int max_pages,
                       int num_pages) {
  geom_t g = {n_seq, 0, n_kvh, d, page, max_pages, num_pages, kv_int8};
  unsigned st = 0;
  float *kr = (float *)malloc(sizeof(float) * (size_t)d);
  float *vr = (float *)malloc(sizeof(float) * (size_t)d);
  int8_t *codes = (int8_t *)malloc((size_t)d);
  for (int b = 0; b < n_seq; ++b) {
    int L = seq_lens[b];
    if (!seq_len_ok(&g, L)) {
      st |= ORC_BAD_LEN;
      continue;
    }
    int pg = page_of(&g, block_table, b, L);
    if (pg < 0) {
      st |= ORC_BAD_PAGE;
      continue;
    }
    int off = L % page;
    for (int j = 0; j < n_kvh; ++j) {
      const uint16_t *kx = k_new + ((size_t)b * n_kvh + j) * d;
      const uint16_t *vx = v_new + ((size_t)b * n_kvh + j) * d;
      size_t s = slot_index(&g, pg, j, off);
      oracle_rope_store_f32(kx, d, positions[b], rope_theta, kr);
      if (!kv_int8) {
        uint16_t *kp = (uint16_t *)k_pages, *vp = (uint16_t *)v_pages;
        for (int i = 0; i < d; ++i) {
          kp[s * d + i] = float_to_bf16_rne(kr[i]);
          vp[s * d + i] = vx[i];
        }
      } else {
        for (int i = 0; i < d; ++i) vr[i] = bf16_to_float(vx[i]);
        oracle_quant_int8(kr, d, codes, &k_scales[s]);
        memcpy((int8_t *)k_pages + s * d, codes, (size_t)d);
        oracle_quant_int8(vr, d, codes, &v_scales[s]);
        memcpy((int8_t *)v_pages + s * d, codes, (size_t)d);
      }
    }
  }
  free(kr);
  free(vr);
  free(codes);
  return st;
}

/* ------------------------------------------------------------- attend --- */

/*
 * Softmax attention of one query head over n cached rows [S1][S7], in double:
 *   s_t = scale * sum_i qh[i] k_t[i];  m = max_t s_t;  w_t = exp(s_t - m);
 *   out = sum_t w_t v_t / sum_t w_t.
 * The rows are given as arrays of row pointers prepared by the caller; a NULL
 * row is an invisible token.  No visible row -> zero output.
 */
static void attend_rows(const double *qh, int d, double scale, int n,
                        const double *const *krow, const double *const *vrow,
                        double *sc, double *out) {
  int any = 0;
  double m = -INFINITY;
  for (int t = 0; t < n; ++t) {
    if (!krow[t]) continue;
    double acc = 0.0;
    for (int i = 0; i < d; ++i) acc += qh[i] * krow[t][i];
    sc[t] = scale * acc;
    if (!any || sc[t] > m) m = sc[t];
    any = 1;
  }
  for (int i = 0; i < d; ++i) out[i] = 0.0;
  if (!any) return;
  double l = 0.0;
  for (int t = 0; t < n; ++t) {
    if (!krow[t]) continue;
    double w = exp(sc[t] - m);
    l += w;
    for (int i = 0; i < d; ++i) out[i] += w * vrow[t][i];
  }
  for (int i = 0; i < d; ++i) out[i] /= l;
}

/*
 * Attention of every query head of the valid sequences over the paged cache
 * (after the append), in double.  out is [n_seq][n_qh][d] double; rows of
 * invalid sequences, and of sequences with seq_mask[b] == 0 when seq_mask is
 * given, are left untouched.  q is rotated in double at positions[b] [S2][S6];
 * query head h reads KV head h / (n_qh / n_kvh) [S3].
 */
unsigned oracle_attend_paged(const uint16_t *q, const void *k_pages,
                             const void *v_pages, const float *k_scales,
                             const float *v_scales, const int32_t *block_table,
                             const int32_t *seq_lens, const int32_t *positions,
                             double *out, int n_seq, int n_qh, int n_kvh, int d,
                             int page, float rope_theta, float scale, int kv_int8,
                             int max_pages, int num_pages,
                             const uint8_t *seq_mask, int n_threads) {
  geom_t g = {n_seq, n_qh, n_kvh, d, page, max_pages, num_pages, kv_int8};
  unsigned st = 0;
  int grp = n_qh / n_kvh;
  for (int b = 0; b < n_seq; ++b) {
    if (!seq_len_ok(&g, seq_lens[b])) {
      st |= ORC_BAD_LEN;
      continue;
    }
    for (int t = 0; t <= seq_lens[b]; t += page)
      if (page_of(&g, block_table, b, t) < 0) st |= ORC_BAD_PAGE;
  }
  int total = n_seq * n_kvh;
#ifdef _OPENMP
  if (n_threads <= 0) n_threads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(n_threads)
#endif
  for (int w = 0; w < total; ++w) {
    int b = w / n_kvh, j = w % n_kvh;
    int L = seq_lens[b];
    if (!seq_len_ok(&g, L)) continue;
    if (seq_mask && !seq_mask[b]) continue;
    int n = L + 1;
    /* dequantised K/V rows of this (sequence, KV head), gathered via the table */
    double *kv = (double *)malloc(sizeof(double) * (size_t)n * d * 2);
    const double **kr = (const double **)malloc(sizeof(double *) * (size_t)n);
    const double **vr = (const double **)malloc(sizeof(double *) * (size_t)n);
    double *sc = (double *)malloc(sizeof(double) * (size_t)n);
    double *xq = (double *)malloc(sizeof(double) * (size_t)d * 2);
    for (int t = 0; t < n; ++t) {
      int pg = page_of(&g, block_table, b, t);
      if (pg < 0) {
        kr[t] = vr[t] = NULL;
        continue;
      }
      double *kk = kv + (size_t)t * d * 2, *vv = kk + d;
      for (int i = 0; i < d; ++i) {
        kk[i] = kv_value(&g, k_pages, k_scales, pg, j, t % page, i);
        vv[i] = kv_value(&g, v_pages, v_scales, pg, j, t % page, i);
      }
      kr[t] = kk;
      vr[t] = vv;
    }
    for (int hh = 0; hh < grp; ++hh) {
      int h = j * grp + hh;
      const uint16_t *qx = q + ((size_t)b * n_qh + h) * d;
      for (int i = 0; i < d; ++i) xq[i] = bf16_to_double(qx[i]);
      oracle_rope_f64(xq, d, (double)positions[b], (double)rope_theta, xq + d);
      attend_rows(xq + d, d, (double)scale, n, kr, vr, sc,
                  out + ((size_t)b * n_qh + h) * d);
    }
    free(kv);
    free(kr);
    free(vr);
    free(sc);
    free(xq);
  }
  return st;
}

/*
 * Contiguous twin [S4]: the cache of sequence b is a plain [L_b + 1][n_kvh][d]
 * array of doubles (the layout [position][kvDim] of the smollm3.go cache),
 * concatenated over b in batch order; no block table.  Summation order is the
 * same as in oracle_attend_paged, so on the same data the two agree exactly.
 */
void oracle_attend_contiguous(const uint16_t *q, const double *k_cache,
                              const double *v_cache, const int32_t *seq_lens,
                              const int32_t *positions, double *out, int n_seq,
                              int n_qh, int n_kvh, int d, float rope_theta,
                              float scale) {
  int grp = n_qh / n_kvh;
  size_t base = 0;
  for (int b = 0; b < n_seq; ++b) {
    int n = seq_lens[b] + 1;
    const double **kr = (const double **)malloc(sizeof(double *) * (size_t)n);
    const double **vr = (const double **)malloc(sizeof(double *) * (size_t)n);
    double *sc = (double *)malloc(sizeof(double) * (size_t)n);
    double xq[2 * 512];
    for (int j = 0; j < n_kvh; ++j) {
      for (int t = 0; t < n; ++t) {
        kr[t] = k_cache + ((base + t) * n_kvh + j) * d;
        vr[t] = v_cache + ((base + t) * n_kvh + j) * d;
      }
      for (int hh = 0; hh < grp; ++hh) {
        int h = j * grp + hh;
        const uint16_t *qx = q + ((size_t)b * n_qh + h) * d;
        for (int i = 0; i < d; ++i) xq[i] = bf16_to_double(qx[i]);
        oracle_rope_f64(xq, d, (double)positions[b], (double)rope_theta, xq + d);
        attend_rows(xq + d, d, (double)scale, n, kr, vr, sc,
                    out + ((size_t)b * n_qh + h) * d);
      }
    }
    base += (size_t)n;
    free(kr);
    free(vr);
    free(sc);
  }
}

/* One whole decode step on host arrays: append, then attend. */
unsigned oracle_decode(const uint16_t *q, const uint16_t *k_new, const uint16_t *v_new,
                       void *k_pages, void *v_pages, float *k_scales, float *v_scales,
                       const int32_t *block_table, const int32_t *seq_lens,
                       const int32_t *positions, double *out, int n_seq, int n_qh,
                       int n_kvh, int d, int page, float rope_theta, float scale,
                       int kv_int8, int max_pages, int num_pages,
                       const uint8_t *seq_mask, int n_threads) {
  unsigned st = oracle_append(k_new, v_new, k_pages, v_pages, k_scales, v_scales,
                              block_table, seq_lens, positions, n_seq, n_kvh, d, page,
                              rope_theta, kv_int8, max_pages, num_pages);
  st |= oracle_attend_paged(q, k_pages, v_pages, k_scales, v_scales, block_table,
                            seq_lens, positions, out, n_seq, n_qh, n_kvh, d, page,
                            rope_theta, scale, kv_int8, max_pages, num_pages,
                            seq_mask, n_threads);
  return st;
}

/* Number of threads an OpenMP region of this library uses by default. */
int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
