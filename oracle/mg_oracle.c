/*
 * mg_oracle.c -- plain fp64 CPU oracle for hybrid local/global grouped-query
 * attention with a narrow KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library calls, links or
 * includes this file; only the tests, the package smoke check and the
 * benchmark's CPU-baseline leg use it.  It shares no code, header, table or
 * helper with the CUDA library.
 *
 * Sources (web pages, cited by title and section):
 *   [P1] "深度拆解Muse Glimmer，24 GB显存跑30 B Agent，Meta到底做了什么？"
 *        (shishifenxi.com) -- section 01 "128K 上下文怎么压进 24GB 显存",
 *        section 04 "一前一后的两个问题".
 *   [P2] "Tomas Koutsky 解释了 Meta 如何在 24 GB 的容量内容纳 Muse Glimmer"
 *        (runtimewire.com) -- sections "窄缓存为长上下文留出空间" and
 *        "长上下文仍然带来计算开销".
 *   [P4] "Meta开源30B模型Muse Glimmer：一张显卡跑本地Agent的实战解析"
 *        (kongchang.com) -- "第二招：混合注意力机制节省显存开销",
 *        "第三招：D-Flash投机解码实现3倍提速".
 *
 * What it computes is the plain definition of softmax attention: the pages
 * say memory-efficient kernels avoid storing the attention matrix but still
 * compute full attention [P2 "长上下文仍然带来计算开销"], so every fast
 * variant (flash, split-KV, chunked prefill, block verify) must reach this
 * same value up to rounding.
 *
 * Shape fixed by the pages: 32 query heads, 2 KV heads, head dim 128
 * [P1 §01], so 16 query heads share each KV head (head h reads KV group
 * h / 16 -- contiguous grouping, a reading).  Local layers attend a sliding
 * window of 2048 tokens with RoPE, global layers attend the full causal
 * history without RoPE [P1 §01; P2 "长上下文仍然带来计算开销"].
 *
 * Readings where the pages are silent (chosen parameters):
 *   - the window includes the query itself: keys j in [p-W+1, p];
 *   - RoPE pairs dimension i with i+64 ("rotate half"), frequency
 *     w_i = theta^(-2i/128), theta = 10000;
 *   - softmax scale 1/sqrt(128);
 *   - the cache stores K and V verbatim (un-rotated), slot = pos mod 2048 for
 *     a local layer ("cyclically reuse stale entries" [P2
 *     "窄缓存为长上下文留出空间"]) and slot = pos for a global layer.
 *
 * Arithmetic: bf16 inputs are widened exactly to double; everything after
 * that is IEEE double with libm exp/sin/cos/pow.  OpenMP splits independent
 * (query, head) rows only; each row is computed exactly as written below.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define OR_HQ 32
#define OR_HKV 2
#define OR_D 128
#define OR_HALF 64
#define OR_GROUP (OR_HQ / OR_HKV)

enum { OR_LOCAL = 0, OR_GLOBAL = 1 };

/* Layer description used by the oracle.  `rope` is separate from `kind` only
 * so that tests can switch RoPE off to check that a local layer whose window
 * covers the whole history equals a global layer. */
typedef struct {
  int32_t kind;   /* OR_LOCAL or OR_GLOBAL */
  int32_t window; /* W for a local layer (2048); ignored for global */
  int32_t rope;   /* 1: rotate q and k by their absolute positions */
  int32_t pad;
  double theta;   /* RoPE base */
  double scale;   /* softmax scale */
} or_layer;

/* bf16 bit pattern -> double (exact). */
static double bf16_bits_to_double(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* RoPE, rotate-half pairing: (x_i, x_{i+64}) is rotated by angle t*w_i.
 * RoPE itself is named by [P2 "长上下文仍然带来计算开销"] (global layers omit
 * it, so local layers carry it); pairing and theta are readings. */
static void rope_rotate(double *x, double t, double theta) {
  for (int i = 0; i < OR_HALF; ++i) {
    double w = pow(theta, -2.0 * (double)i / (double)OR_D);
    double a = t * w;
    double c = cos(a), s = sin(a);
    double x0 = x[i], x1 = x[i + OR_HALF];
    x[i] = x0 * c - x1 * s;
    x[i + OR_HALF] = x0 * s + x1 * c;
  }
}

/* First key position a query at position p may attend [P1 §01: local layers
 * only see the nearby 2048 tokens; global layers see the full causal
 * history]. */
static int64_t key_lo(const or_layer *L, int64_t p) {
  if (L->kind == OR_LOCAL) {
    int64_t lo = p - (int64_t)L->window + 1;
    return lo < 0 ? 0 : lo;
  }
  return 0;
}

/* Exported: RoPE of one 128-vector at position t, in place (used by the pins
 * that check R(0) = I and norm preservation). */
void mg_oracle_rope(double *x, double t, double theta) { rope_rotate(x, t, theta); }

/* Exported: softmax-attention probabilities of one (query, head) against a
 * linear history.  probs[j] is set for every j < T (zero outside the key
 * set).  Returns 0, or -1 on bad arguments. */
int mg_oracle_probs(const or_layer *L, int32_t T, const uint16_t *k_hist,
                    int32_t p, const uint16_t *q_row /* [128] */, int32_t head,
                    double *probs /* [T] */) {
  if (!L || T <= 0 || p < 0 || p >= T || head < 0 || head >= OR_HQ) return -1;
  int g = head / OR_GROUP;
  double q[OR_D], k[OR_D];
  for (int d = 0; d < OR_D; ++d) q[d] = bf16_bits_to_double(q_row[d]);
  if (L->rope) rope_rotate(q, (double)p, L->theta);
  int64_t lo = key_lo(L, p);
  for (int64_t j = 0; j < T; ++j) probs[j] = 0.0;
  double m = -INFINITY;
  for (int64_t j = lo; j <= p; ++j) {
    const uint16_t *kr = k_hist + ((size_t)j * OR_HKV + g) * OR_D;
    for (int d = 0; d < OR_D; ++d) k[d] = bf16_bits_to_double(kr[d]);
    if (L->rope) rope_rotate(k, (double)j, L->theta);
    double s = 0.0;
    for (int d = 0; d < OR_D; ++d) s += q[d] * k[d];
    s *= L->scale;
    probs[j] = s;
    if (s > m) m = s;
  }
  double z = 0.0;
  for (int64_t j = lo; j <= p; ++j) {
    probs[j] = exp(probs[j] - m);
    z += probs[j];
  }
  for (int64_t j = lo; j <= p; ++j) probs[j] /= z;
  return 0;
}

/* Exported: attention of nq query tokens (all 32 heads each) against one
 * linear key/value history of T positions.
 *   k_hist, v_hist : [T][2][128] bf16 bits (position t holds the K/V of t)
 *   q              : [nq][32][128] bf16 bits, query i sits at q_pos[i] < T
 *   o              : [nq][32][128] double
 * For query position p and head h (KV group g = h/16), with the key set
 * J(p) = {key_lo(p) .. p}:
 *   s_j = scale * <R(p) q, R(j) k_j>   (R = identity when rope == 0)
 *   o   = sum_j softmax(s)_j v_j.
 * Returns 0, or -1 on bad arguments. */
int mg_oracle_attention(const or_layer *L, int32_t T, const uint16_t *k_hist,
                        const uint16_t *v_hist, int32_t nq, const int32_t *q_pos,
                        const uint16_t *q, double *o) {
  if (!L || T <= 0 || nq < 0) return -1;
  if (L->kind != OR_LOCAL && L->kind != OR_GLOBAL) return -1;
  if (L->kind == OR_LOCAL && L->window <= 0) return -1;
  int64_t jmin = T, jmax = -1;
  for (int32_t i = 0; i < nq; ++i) {
    if (q_pos[i] < 0 || q_pos[i] >= T) return -1;
    int64_t lo = key_lo(L, q_pos[i]);
    if (lo < jmin) jmin = lo;
    if (q_pos[i] > jmax) jmax = q_pos[i];
  }
  if (nq == 0) return 0;
  /* Keys (rotated when RoPE is on) and values widened to double for the
   * positions any query can see. */
  int64_t nk = jmax - jmin + 1;
  double *kd = (double *)malloc((size_t)nk * OR_HKV * OR_D * sizeof(double));
  double *vd = (double *)malloc((size_t)nk * OR_HKV * OR_D * sizeof(double));
  if (!kd || !vd) { free(kd); free(vd); return -2; }
#pragma omp parallel for schedule(static)
  for (int64_t jj = 0; jj < nk; ++jj) {
    int64_t j = jmin + jj;
    for (int g = 0; g < OR_HKV; ++g) {
      const uint16_t *kr = k_hist + ((size_t)j * OR_HKV + g) * OR_D;
      const uint16_t *vr = v_hist + ((size_t)j * OR_HKV + g) * OR_D;
      double *kk = kd + ((size_t)jj * OR_HKV + g) * OR_D;
      double *vv = vd + ((size_t)jj * OR_HKV + g) * OR_D;
      for (int d = 0; d < OR_D; ++d) {
        kk[d] = bf16_bits_to_double(kr[d]);
        vv[d] = bf16_bits_to_double(vr[d]);
      }
      if (L->rope) rope_rotate(kk, (double)j, L->theta);
    }
  }
  int64_t rows = (int64_t)nq * OR_HQ;
  int fail = 0;
#pragma omp parallel
  {
    double *s = (double *)malloc((size_t)nk * sizeof(double));
    if (!s) {
#pragma omp atomic write
      fail = 1;
    }
#pragma omp for schedule(dynamic, 4)
    for (int64_t r = 0; r < rows; ++r) {
      if (!s) continue;
      int32_t i = (int32_t)(r / OR_HQ);
      int h = (int)(r % OR_HQ);
      int g = h / OR_GROUP;
      int64_t p = q_pos[i];
      double qv[OR_D];
      const uint16_t *qr = q + ((size_t)i * OR_HQ + h) * OR_D;
      for (int d = 0; d < OR_D; ++d) qv[d] = bf16_bits_to_double(qr[d]);
      if (L->rope) rope_rotate(qv, (double)p, L->theta);
      int64_t lo = key_lo(L, p);
      double m = -INFINITY;
      for (int64_t j = lo; j <= p; ++j) {
        const double *kk = kd + ((size_t)(j - jmin) * OR_HKV + g) * OR_D;
        double acc = 0.0;
        for (int d = 0; d < OR_D; ++d) acc += qv[d] * kk[d];
        acc *= L->scale;
        s[j - jmin] = acc;
        if (acc > m) m = acc;
      }
      double z = 0.0;
      for (int64_t j = lo; j <= p; ++j) {
        double e = exp(s[j - jmin] - m);
        s[j - jmin] = e;
        z += e;
      }
      double out[OR_D];
      for (int d = 0; d < OR_D; ++d) out[d] = 0.0;
      for (int64_t j = lo; j <= p; ++j) {
        double w = s[j - jmin] / z;
        const double *vv = vd + ((size_t)(j - jmin) * OR_HKV + g) * OR_D;
        for (int d = 0; d < OR_D; ++d) out[d] += w * vv[d];
      }
      double *orow = o + ((size_t)i * OR_HQ + h) * OR_D;
      for (int d = 0; d < OR_D; ++d) orow[d] = out[d];
    }
    free(s);
  }
  free(kd);
  free(vd);
  return fail ? -2 : 0;
}

/* Exported: the cache after appending positions pos0 .. pos0+n-1 of one
 * sequence, replayed one token at a time in order.  A local layer writes
 * slot pos mod slots (a ring that reuses the oldest entry), a global layer
 * writes slot pos [P2 "窄缓存为长上下文留出空间"].  K and V are stored
 * verbatim.
 *   k_cache, v_cache : [2][slots][128] bf16 bits (one sequence), updated
 *   k_new, v_new     : [n][2][128] bf16 bits
 * Returns 0, or -1 if a global position is beyond the cache. */
int mg_oracle_cache_append(int32_t kind, int32_t slots, uint16_t *k_cache,
                           uint16_t *v_cache, int32_t pos0, int32_t n,
                           const uint16_t *k_new, const uint16_t *v_new) {
  if (slots <= 0 || pos0 < 0 || n < 0) return -1;
  for (int32_t t = 0; t < n; ++t) {
    int64_t pos = (int64_t)pos0 + t;
    int64_t slot;
    if (kind == OR_LOCAL) slot = pos % slots;
    else if (kind == OR_GLOBAL) {
      if (pos >= slots) return -1;
      slot = pos;
    } else return -1;
    for (int g = 0; g < OR_HKV; ++g) {
      memcpy(k_cache + ((size_t)g * slots + slot) * OR_D,
             k_new + ((size_t)t * OR_HKV + g) * OR_D, OR_D * sizeof(uint16_t));
      memcpy(v_cache + ((size_t)g * slots + slot) * OR_D,
             v_new + ((size_t)t * OR_HKV + g) * OR_D, OR_D * sizeof(uint16_t));
    }
  }
  return 0;
}

/* Exported: decode attention for one query token read straight from a cache
 * in slot layout (ring for local, linear for global), the way a serving
 * engine holds it.  Slot s of a local ring holds the largest position j <= p
 * with j = s (mod slots); it is attended if j >= 0 and j is in the window.
 * This is the "ring buffer + mask" form; a pin checks it against
 * mg_oracle_attention on the linear history.
 *   k_cache, v_cache : [2][slots][128] bf16 bits (one sequence)
 *   q                : [32][128] bf16 bits at position p
 *   o                : [32][128] double */
int mg_oracle_decode_from_cache(const or_layer *L, int32_t slots,
                                const uint16_t *k_cache, const uint16_t *v_cache,
                                int32_t p, const uint16_t *q, double *o) {
  if (!L || slots <= 0 || p < 0) return -1;
  if (L->kind == OR_GLOBAL && p >= slots) return -1;
  if (L->kind == OR_LOCAL && L->window > slots) return -1;
  int64_t lo = key_lo(L, p);
#pragma omp parallel for schedule(static)
  for (int h = 0; h < OR_HQ; ++h) {
    int g = h / OR_GROUP;
    double qv[OR_D], kk[OR_D];
    for (int d = 0; d < OR_D; ++d) qv[d] = bf16_bits_to_double(q[(size_t)h * OR_D + d]);
    if (L->rope) rope_rotate(qv, (double)p, L->theta);
    double *s = (double *)malloc((size_t)slots * sizeof(double));
    int64_t *js = (int64_t *)malloc((size_t)slots * sizeof(int64_t));
    int64_t cnt = 0;
    double m = -INFINITY;
    for (int64_t sl = 0; sl < slots; ++sl) {
      int64_t j;
      if (L->kind == OR_LOCAL) j = (int64_t)p - ((((int64_t)p - sl) % slots + slots) % slots);
      else j = sl;
      if (j < lo || j > p) continue;
      const uint16_t *kr = k_cache + ((size_t)g * slots + sl) * OR_D;
      for (int d = 0; d < OR_D; ++d) kk[d] = bf16_bits_to_double(kr[d]);
      if (L->rope) rope_rotate(kk, (double)j, L->theta);
      double acc = 0.0;
      for (int d = 0; d < OR_D; ++d) acc += qv[d] * kk[d];
      acc *= L->scale;
      s[cnt] = acc;
      js[cnt] = sl;
      ++cnt;
      if (acc > m) m = acc;
    }
    double z = 0.0;
    for (int64_t c = 0; c < cnt; ++c) { s[c] = exp(s[c] - m); z += s[c]; }
    double out[OR_D];
    for (int d = 0; d < OR_D; ++d) out[d] = 0.0;
    for (int64_t c = 0; c < cnt; ++c) {
      const uint16_t *vr = v_cache + ((size_t)g * slots + js[c]) * OR_D;
      double w = s[c] / z;
      for (int d = 0; d < OR_D; ++d) out[d] += w * bf16_bits_to_double(vr[d]);
    }
    for (int d = 0; d < OR_D; ++d) o[(size_t)h * OR_D + d] = out[d];
    free(s);
    free(js);
  }
  return 0;
}

/* Exported: threads OpenMP will use (for reporting the CPU baseline). */
int mg_oracle_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
