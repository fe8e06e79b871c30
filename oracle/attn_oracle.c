/*
 * attn_oracle.c -- plain, slow, fp64 CPU reference for attention forward.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file: it is used by the tests, by the package's smoke check and
 * by the timed CPU baseline of bench.py.  It shares no code, header, table or
 * helper with the CUDA library; the two meet only on the seeded inputs.
 *
 * What it computes (sources are the pages this project is built from):
 *
 *  - MHA forward, "FP32 CUDA-core FlashAttention-2 v2" blog (dandandamowang,
 *    post_1787450400), sections 1.3 and 3.3: for every query row i,
 *        s_j = scale * <q_i, k_j>               for every visible key j
 *        O_i = sum_j softmax(s)_j * v_j
 *    The blog reaches this with an online softmax and a deferred 1/l; this
 *    oracle instead writes the plain definition out: S is materialised for
 *    the row and the softmax takes two passes (max, then exp/sum).  Both are
 *    the same value up to rounding.
 *  - Causal visibility, same blog section 3.4: key j is visible to query i
 *    iff j <= i (square case only; the blog treats no other).
 *  - Out-of-range keys get weight zero (blog section 3.2, the zero-fill and
 *    -inf rule), which here simply means they are never visited.
 *  - LSE: the blog keeps m and l but never outputs them.  Reading used here:
 *    the natural-log logsumexp of the scaled, masked scores,
 *        LSE_i = m_i + ln(sum_j exp(s_j - m_i)).
 *  - MLA absorbed decode, "MLA x FlashAttention-3 fusion" article (hnwysp
 *    news 119127), sections on the latent layout and on in-place absorption:
 *    each cached token is one 576-wide row [c_kv (512) | k_rope (64)]; the
 *    absorbed query is [q_nope W_UK (512) | q_rope (64)], so
 *        s_t = scale * <q, C_t>    (one 576-deep dot product)
 *        O   = sum_t softmax(s)_t * C_t[0:512]   (V is the c_kv slice)
 *    Rows are gathered through a block table of 64-token pages.  A sequence
 *    of length 0 gives O = 0 and LSE = -inf (reading; no page covers it).
 *
 * Inputs are float32 arrays (bf16 data is widened to fp32 exactly before the
 * call); every product and sum is taken in double.  exp and log are libm's.
 * OpenMP spreads independent rows over threads; each row is computed by one
 * thread in key order, so results do not depend on the thread count.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_EINVAL -1
#define ORACLE_ENOMEM -2
#define ORACLE_EBADTABLE -3

/* One attention row by the plain definition: s materialised, two passes. */
static void attention_row(const float* q, const float* const* krows,
                          const float* const* vrows, int64_t nkeys, int64_t dk,
                          int64_t dv, double scale, double* s, double* o_out,
                          double* lse_out) {
  int64_t j, d;
  if (nkeys == 0) {
    for (d = 0; d < dv; d++) o_out[d] = 0.0;
    *lse_out = -INFINITY;
    return;
  }
  /* scores */
  for (j = 0; j < nkeys; j++) {
    double acc = 0.0;
    const float* kr = krows[j];
    for (d = 0; d < dk; d++) acc += (double)q[d] * (double)kr[d];
    s[j] = scale * acc;
  }
  /* pass 1: row maximum */
  double m = -INFINITY;
  for (j = 0; j < nkeys; j++)
    if (s[j] > m) m = s[j];
  /* pass 2: normaliser and weighted sum of values */
  double l = 0.0;
  for (d = 0; d < dv; d++) o_out[d] = 0.0;
  for (j = 0; j < nkeys; j++) {
    double p = exp(s[j] - m);
    l += p;
    const float* vr = vrows[j];
    for (d = 0; d < dv; d++) o_out[d] += p * (double)vr[d];
  }
  for (d = 0; d < dv; d++) o_out[d] /= l;
  *lse_out = m + log(l);
}

static int pick_threads(int nthreads) {
#ifdef _OPENMP
  return nthreads > 0 ? nthreads : omp_get_max_threads();
#else
  (void)nthreads;
  return 1;
#endif
}

int oracle_num_threads(int nthreads) { return pick_threads(nthreads); }

/*
 * Multi-head attention forward.
 *   q, k : [B, H, N, Dk] float32, contiguous
 *   v    : [B, H, N, Dv] float32, contiguous
 *   rows : flat row ids (b*H + h)*N + i to compute, or NULL for all B*H*N
 *   o    : [nrows, Dv] double (row order of `rows`), lse : [nrows] double
 */
int oracle_mha(const float* q, const float* k, const float* v, int64_t B,
               int64_t H, int64_t N, int64_t Dk, int64_t Dv, int causal,
               double scale, const int64_t* rows, int64_t nrows, double* o,
               double* lse, int nthreads) {
  if (!q || !k || !v || !o || !lse || B < 0 || H < 0 || N < 0 || Dk <= 0 ||
      Dv <= 0)
    return ORACLE_EINVAL;
  int64_t total = B * H * N;
  if (!rows) nrows = total;
  if (nrows < 0) return ORACLE_EINVAL;
  if (rows)
    for (int64_t r = 0; r < nrows; r++)
      if (rows[r] < 0 || rows[r] >= total) return ORACLE_EINVAL;
  if (nrows == 0 || N == 0) return ORACLE_OK;

  int err = ORACLE_OK;
  int nt = pick_threads(nthreads);
#pragma omp parallel num_threads(nt)
  {
    double* s = (double*)malloc(sizeof(double) * (size_t)N);
    const float** kr = (const float**)malloc(sizeof(float*) * (size_t)N);
    const float** vr = (const float**)malloc(sizeof(float*) * (size_t)N);
    if (!s || !kr || !vr) {
#pragma omp atomic write
      err = ORACLE_ENOMEM;
    } else {
#pragma omp for schedule(dynamic, 8)
      for (int64_t r = 0; r < nrows; r++) {
        int64_t flat = rows ? rows[r] : r;
        int64_t bh = flat / N, i = flat % N;
        int64_t nkeys = causal ? (i + 1) : N; /* j <= i when causal */
        for (int64_t j = 0; j < nkeys; j++) {
          kr[j] = k + (bh * N + j) * Dk;
          vr[j] = v + (bh * N + j) * Dv;
        }
        attention_row(q + (bh * N + i) * Dk, kr, vr, nkeys, Dk, Dv, scale, s,
                      o + r * Dv, lse + r);
      }
    }
    free(s);
    free((void*)kr);
    free((void*)vr);
  }
  return err;
}

/*
 * Softmax probabilities of MHA, for tiny inputs only: P [B, H, N, N] double,
 * P[b,h,i,j] = exp(s_ij - LSE_i) for visible j and 0 for masked j.
 */
int oracle_mha_probs(const float* q, const float* k, int64_t B, int64_t H,
                     int64_t N, int64_t Dk, int causal, double scale,
                     double* P) {
  if (!q || !k || !P || B < 0 || H < 0 || N < 0 || Dk <= 0)
    return ORACLE_EINVAL;
  double* s = (double*)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
  if (!s) return ORACLE_ENOMEM;
  for (int64_t bh = 0; bh < B * H; bh++) {
    for (int64_t i = 0; i < N; i++) {
      int64_t nkeys = causal ? (i + 1) : N;
      double m = -INFINITY;
      for (int64_t j = 0; j < nkeys; j++) {
        double acc = 0.0;
        for (int64_t d = 0; d < Dk; d++)
          acc += (double)q[(bh * N + i) * Dk + d] *
                 (double)k[(bh * N + j) * Dk + d];
        s[j] = scale * acc;
        if (s[j] > m) m = s[j];
      }
      double l = 0.0;
      for (int64_t j = 0; j < nkeys; j++) l += exp(s[j] - m);
      double* prow = P + (bh * N + i) * N;
      for (int64_t j = 0; j < N; j++)
        prow[j] = (j < nkeys) ? exp(s[j] - m) / l : 0.0;
    }
  }
  free(s);
  return ORACLE_OK;
}

/*
 * MLA absorbed decode (one query token per sequence).
 *   q           : [B, Hq, Dk] float32 (absorbed query, Dk = 576 in the model)
 *   kv          : [num_blocks, page, Dk] float32 latent pool
 *   block_table : [B, max_blocks] int32, page j of sequence b is
 *                 kv[block_table[b*max_blocks + j]]
 *   seqlens     : [B] int32, tokens t < seqlens[b] are visible
 *   rows        : flat ids b*Hq + h to compute, or NULL for all
 *   o           : [nrows, Dv] double, V row t = C_t[0:Dv]; lse : [nrows]
 * Returns ORACLE_EBADTABLE if a needed table entry or a length is out of
 * range (nothing is read out of bounds).
 */
int oracle_mla(const float* q, const float* kv, const int32_t* block_table,
               const int32_t* seqlens, int64_t B, int64_t Hq, int64_t Dk,
               int64_t Dv, int64_t page, int64_t max_blocks,
               int64_t num_blocks, double scale, const int64_t* rows,
               int64_t nrows, double* o, double* lse, int nthreads) {
  if (!q || !kv || !block_table || !seqlens || !o || !lse || B < 0 ||
      Hq <= 0 || Dk <= 0 || Dv <= 0 || Dv > Dk || page <= 0 ||
      max_blocks < 0 || num_blocks < 0)
    return ORACLE_EINVAL;
  int64_t total = B * Hq;
  if (!rows) nrows = total;
  if (nrows < 0) return ORACLE_EINVAL;
  if (rows)
    for (int64_t r = 0; r < nrows; r++)
      if (rows[r] < 0 || rows[r] >= total) return ORACLE_EINVAL;
  /* validate every sequence that a requested row touches */
  for (int64_t b = 0; b < B; b++) {
    int64_t L = seqlens[b];
    if (L < 0 || L > max_blocks * page) return ORACLE_EBADTABLE;
    for (int64_t j = 0; j * page < L; j++) {
      int32_t blk = block_table[b * max_blocks + j];
      if (blk < 0 || blk >= num_blocks) return ORACLE_EBADTABLE;
    }
  }
  if (nrows == 0) return ORACLE_OK;
  int64_t maxlen = max_blocks * page;

  int err = ORACLE_OK;
  int nt = pick_threads(nthreads);
#pragma omp parallel num_threads(nt)
  {
    size_t cap = (size_t)(maxlen > 0 ? maxlen : 1);
    double* s = (double*)malloc(sizeof(double) * cap);
    const float** cr = (const float**)malloc(sizeof(float*) * cap);
    if (!s || !cr) {
#pragma omp atomic write
      err = ORACLE_ENOMEM;
    } else {
#pragma omp for schedule(dynamic, 4)
      for (int64_t r = 0; r < nrows; r++) {
        int64_t flat = rows ? rows[r] : r;
        int64_t b = flat / Hq;
        int64_t L = seqlens[b];
        /* gather the sequence's rows through the block table */
        for (int64_t t = 0; t < L; t++) {
          int64_t blk = block_table[b * max_blocks + t / page];
          cr[t] = kv + (blk * page + t % page) * Dk;
        }
        /* V rows are the first Dv entries of the same cached rows */
        attention_row(q + flat * Dk, cr, cr, L, Dk, Dv, scale, s, o + r * Dv,
                      lse + r);
      }
    }
    free(s);
    free((void*)cr);
  }
  return err;
}
