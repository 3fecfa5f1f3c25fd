/*
 * cpthd_oracle.c -- plain fp64 CPU oracle for causal varlen self-attention
 * over THD-packed documents.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link or call
 * this file; only the tests, the smoke check and the CPU-baseline leg of the
 * benchmark use it.  It shares no code with the CUDA library.
 *
 * What it computes (the plain definition, no blocking, no fusion, no
 * reordering beyond the definition):
 *
 *   Layout "THD": a packed tensor [T, H, D], row-major; documents are the row
 *   ranges delimited by cu_seqlens_padded (cup, int32 [n+1]).  Document i
 *   holds L_i real tokens (L_i = cu[i+1]-cu[i] when pad_between_seqs is set,
 *   else L_i = cup[i+1]-cup[i]) at rows [cup[i], cup[i]+L_i); the remaining
 *   rows of its padded range are padding.
 *
 *   Causal self-attention without a sliding window, bounded by document
 *   boundaries ("[PyTorch] Add no-load-balance THD all-gather CP",
 *   §Scope and constraints: causal, window_size=(-1, 0); §What changed:
 *   logical document boundaries are kept in the THD metadata):
 *     a valid query row g of document i attends the keys j in [cup[i], g];
 *     s_gj   = scale * sum_d q[g,h,d] k[j,h,d]
 *     LSE_g  = m + ln sum_j exp(s_gj - m),  m = max_j s_gj   (natural log)
 *     O_g    = sum_j exp(s_gj - LSE_g) v[j,h,:]
 *   A padding row attends nothing: O = 0, LSE = -inf.
 *
 *   Backward of the same function for an upstream gradient dO:
 *     Delta_g = sum_d dO[g,h,d] O[g,h,d]
 *     P_gj    = exp(s_gj - LSE_g),  dP_gj = sum_d dO[g,h,d] v[j,h,d]
 *     dS_gj   = P_gj (dP_gj - Delta_g)
 *     dQ_g = scale sum_j dS_gj k_j,  dK_j = scale sum_g dS_gj q_g,
 *     dV_j = sum_g P_gj dO_g
 *   An optional query mask restricts every sum to the masked-in queries, which
 *   gives one context-parallel rank's partial dK/dV.
 *
 * All arithmetic is fp64.  OpenMP parallelises over independent outputs only
 * (one query row, or one key row, per iteration), so there are no reductions
 * across threads.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Document containing physical row g: the i with cup[i] <= g < cup[i+1]. */
static int doc_of(int64_t g, int n, const int32_t* cup) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) / 2;
    if (cup[mid] <= g) lo = mid; else hi = mid - 1;
  }
  return lo;
}

static int64_t doc_len(int i, const int32_t* cu, const int32_t* cup, int pad) {
  return pad ? (int64_t)cu[i + 1] - cu[i] : (int64_t)cup[i + 1] - cup[i];
}

/* Keys of query row g: [*lo, *hi]; returns 0 for a padding row. */
static int key_range(int64_t g, int n, const int32_t* cu, const int32_t* cup, int pad,
                     int64_t* lo, int64_t* hi) {
  int i = doc_of(g, n, cup);
  if (g < cup[i] || g >= cup[i + 1]) return 0;
  if (g - cup[i] >= doc_len(i, cu, cup, pad)) return 0;
  *lo = cup[i];
  *hi = g;
  return 1;
}

static double dot(const double* a, const double* b, int D) {
  double s = 0.0;
  for (int d = 0; d < D; ++d) s += a[d] * b[d];
  return s;
}

/* Forward.  q,k,v: [T,H,D]; o: [T,H,D]; lse: [H,T].  Only the listed heads
 * and (when qmask != NULL) the masked-in query rows are written. */
void oracle_attn_fwd(int64_t T, int H, int D, int n, const int32_t* cu, const int32_t* cup,
                     int pad, double scale, const double* q, const double* k, const double* v,
                     const uint8_t* qmask, const int32_t* heads, int n_heads,
                     double* o, double* lse) {
  int64_t work = (int64_t)n_heads * T;
#pragma omp parallel
  {
    double* s = (double*)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1));
#pragma omp for schedule(dynamic, 64)
    for (int64_t w = 0; w < work; ++w) {
      int h = heads[w / T];
      int64_t g = w % T;
      if (qmask && !qmask[g]) continue;
      double* og = o + (g * H + h) * D;
      int64_t lo, hi;
      if (!key_range(g, n, cu, cup, pad, &lo, &hi)) {
        for (int d = 0; d < D; ++d) og[d] = 0.0;
        lse[(int64_t)h * T + g] = -INFINITY;
        continue;
      }
      const double* qg = q + (g * H + h) * D;
      double m = -INFINITY;
      for (int64_t j = lo; j <= hi; ++j) {
        s[j - lo] = scale * dot(qg, k + (j * H + h) * D, D);
        if (s[j - lo] > m) m = s[j - lo];
      }
      double sum = 0.0;
      for (int64_t j = lo; j <= hi; ++j) sum += exp(s[j - lo] - m);
      double L = m + log(sum);
      lse[(int64_t)h * T + g] = L;
      for (int d = 0; d < D; ++d) og[d] = 0.0;
      for (int64_t j = lo; j <= hi; ++j) {
        double p = exp(s[j - lo] - L);
        const double* vj = v + (j * H + h) * D;
        for (int d = 0; d < D; ++d) og[d] += p * vj[d];
      }
    }
    free(s);
  }
}

/* Backward.  Uses the caller's O and LSE (normally the oracle's own fp64
 * forward).  dq is written for masked-in queries; dk/dv are written for every
 * key row of the listed heads (zero where no masked-in query attends). */
void oracle_attn_bwd(int64_t T, int H, int D, int n, const int32_t* cu, const int32_t* cup,
                     int pad, double scale, const double* q, const double* k, const double* v,
                     const double* o, const double* lse, const double* dout,
                     const uint8_t* qmask, const int32_t* heads, int n_heads,
                     double* dq, double* dk, double* dv) {
  int64_t work = (int64_t)n_heads * T;
  /* Delta_g = dO_g . O_g  (per head, per query) */
  double* delta = (double*)malloc(sizeof(double) * (size_t)(work > 0 ? work : 1));
#pragma omp parallel for schedule(static)
  for (int64_t w = 0; w < work; ++w) {
    int h = heads[w / T];
    int64_t g = w % T;
    delta[w] = dot(dout + (g * H + h) * D, o + (g * H + h) * D, D);
  }
  /* dQ: one query row per iteration */
#pragma omp parallel for schedule(dynamic, 64)
  for (int64_t w = 0; w < work; ++w) {
    int hi_idx = (int)(w / T);
    int h = heads[hi_idx];
    int64_t g = w % T;
    if (qmask && !qmask[g]) continue;
    double* dqg = dq + (g * H + h) * D;
    for (int d = 0; d < D; ++d) dqg[d] = 0.0;
    int64_t lo, hi;
    if (!key_range(g, n, cu, cup, pad, &lo, &hi)) continue;
    const double* qg = q + (g * H + h) * D;
    const double* dog = dout + (g * H + h) * D;
    double Lg = lse[(int64_t)h * T + g];
    for (int64_t j = lo; j <= hi; ++j) {
      const double* kj = k + (j * H + h) * D;
      double p = exp(scale * dot(qg, kj, D) - Lg);
      double dp = dot(dog, v + (j * H + h) * D, D);
      double ds = p * (dp - delta[w]);
      for (int d = 0; d < D; ++d) dqg[d] += scale * ds * kj[d];
    }
  }
  /* dK, dV: one key row per iteration; the queries attending key j are the
   * valid rows g >= j of j's document. */
#pragma omp parallel for schedule(dynamic, 64)
  for (int64_t w = 0; w < work; ++w) {
    int hi_idx = (int)(w / T);
    int h = heads[hi_idx];
    int64_t j = w % T;
    double* dkj = dk + (j * H + h) * D;
    double* dvj = dv + (j * H + h) * D;
    for (int d = 0; d < D; ++d) { dkj[d] = 0.0; dvj[d] = 0.0; }
    int i = doc_of(j, n, cup);
    if (j < cup[i] || j >= cup[i + 1]) continue;
    int64_t valid_end = (int64_t)cup[i] + doc_len(i, cu, cup, pad);
    const double* kj = k + (j * H + h) * D;
    const double* vj = v + (j * H + h) * D;
    for (int64_t g = j; g < valid_end; ++g) {
      if (qmask && !qmask[g]) continue;
      const double* qg = q + (g * H + h) * D;
      const double* dog = dout + (g * H + h) * D;
      double p = exp(scale * dot(qg, kj, D) - lse[(int64_t)h * T + g]);
      double dp = dot(dog, vj, D);
      double ds = p * (dp - delta[(int64_t)hi_idx * T + g]);
      for (int d = 0; d < D; ++d) {
        dkj[d] += scale * ds * qg[d];
        dvj[d] += p * dog[d];
      }
    }
  }
  free(delta);
}

int oracle_num_threads(void) {
  int nt = 1;
#pragma omp parallel
  {
#pragma omp single
    {
#ifdef _OPENMP
      extern int omp_get_num_threads(void);
      nt = omp_get_num_threads();
#endif
    }
  }
  return nt;
}
