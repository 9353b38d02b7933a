/*
 * oracle.c -- plain CPU oracle for exact brute-force top-K retrieval.
 *
 * TEST INFRASTRUCTURE. Only the tests, the package's smoke check and the
 * bench's CPU-baseline leg load this library. The CUDA library never links,
 * includes or calls it, and this file includes nothing of the CUDA side.
 *
 * What it computes is the plain definition of the result, written out with no
 * blocking, fusion or reordering:
 *
 *   Exact top-K inner-product retrieval (GPU-Resident Top-K for Agentic RAG,
 *   section 2 "why top-K retrieval exists"): score a query of D floats against
 *   each of N corpus rows and return the K rows with the highest similarity,
 *   best first. Inner product = one multiply-add per dimension.
 *
 *   The ordering rule (same article, section 3, problem B, "the tie rule"):
 *   a higher score is better; on an exact score tie the lower row index is
 *   better.
 *
 *   Cosine similarity (same article, section 4 step 2, the scoring kernel's
 *   cosine mode, and the later section on the two flavours of similarity):
 *   the inner product divided by the product of the query's and the row's L2
 *   norms; a row whose denominator is not positive scores -infinity.
 *
 *   The flat int32 formulation (CUDA programming model series 9, sections 1
 *   and 2.1): the K largest values of an int32 array. Positions are returned
 *   too and the lower position wins ties (that page tracks no positions; the
 *   tie rule is carried over from the retrieval article).
 *
 * Readings taken where the pages are silent:
 *   - Scores are accumulated in double, in index order d = 0..D-1. Each
 *     fp32 x fp32 product is exact in double. Cosine norms are the square
 *     roots of double sums of squares in the same order, and the quotient is
 *     taken in double.
 *   - A NaN score ranks as -infinity (the tie rule is not a strict order with
 *     NaN). -0.0 and +0.0 compare equal, so they tie and the index decides.
 *   - The selection is a full sort of all (score, index) pairs by the rule,
 *     keeping the first K.
 *
 * Build: gcc -O2 -fopenmp -ffp-contract=off -fPIC -shared (no fast-math).
 * Scoring is parallel over rows; each row's sum is sequential, so results do
 * not depend on the thread count.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

typedef struct {
  double score;
  int64_t index;
} oracle_pair;

/* Best-first order of (score, index) pairs: higher score first, then lower
 * index first. Indices are distinct, so this is a strict total order. */
static int oracle_pair_cmp(const void* a, const void* b) {
  const oracle_pair* x = (const oracle_pair*)a;
  const oracle_pair* y = (const oracle_pair*)b;
  if (x->score != y->score) return (x->score > y->score) ? -1 : 1;
  if (x->index != y->index) return (x->index < y->index) ? -1 : 1;
  return 0;
}

typedef struct {
  int32_t value;
  int64_t position;
} oracle_ipair;

/* Largest value first, then lower position first. */
static int oracle_ipair_cmp(const void* a, const void* b) {
  const oracle_ipair* x = (const oracle_ipair*)a;
  const oracle_ipair* y = (const oracle_ipair*)b;
  if (x->value != y->value) return (x->value > y->value) ? -1 : 1;
  if (x->position != y->position) return (x->position < y->position) ? -1 : 1;
  return 0;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

void oracle_set_num_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

/* sigma_i = sum_{d=0}^{D-1} c[i, d] * q[d] in double, for every row i.
 * corpus is row-major N x D fp32; out has N doubles. */
int oracle_scores(const float* corpus, int64_t n, int32_t d, const float* query, double* out) {
  if (!corpus || !query || !out || n < 0 || d < 1) return 1;
  int64_t i;
#pragma omp parallel for schedule(static)
  for (i = 0; i < n; ++i) {
    const float* row = corpus + i * (int64_t)d;
    double acc = 0.0;
    for (int32_t j = 0; j < d; ++j) acc += (double)row[j] * (double)query[j];
    if (isnan(acc)) acc = -INFINITY;
    out[i] = acc;
  }
  return 0;
}

/* cos_i = (sum_d c[i, d] * q[d]) / (||c_i|| * ||q||) in double, for every
 * row i, with ||x|| = sqrt(sum_d x[d]^2). A denominator that is not positive
 * (a zero row or a zero query) gives -infinity, as does a NaN quotient. */
int oracle_scores_cosine(const float* corpus, int64_t n, int32_t d, const float* query, double* out) {
  if (!corpus || !query || !out || n < 0 || d < 1) return 1;
  double qq = 0.0;
  for (int32_t j = 0; j < d; ++j) qq += (double)query[j] * (double)query[j];
  const double qnorm = sqrt(qq);
  int64_t i;
#pragma omp parallel for schedule(static)
  for (i = 0; i < n; ++i) {
    const float* row = corpus + i * (int64_t)d;
    double dot = 0.0, cc = 0.0;
    for (int32_t j = 0; j < d; ++j) {
      dot += (double)row[j] * (double)query[j];
      cc += (double)row[j] * (double)row[j];
    }
    const double denom = qnorm * sqrt(cc);
    double cosv = denom > 0.0 ? dot / denom : -INFINITY;
    if (isnan(cosv)) cosv = -INFINITY;
    out[i] = cosv;
  }
  return 0;
}

/* Sort all N (score, index) pairs best-first under the rule and keep K. */
static int select_topk(const double* sigma, int64_t n, int32_t k, int64_t* out_idx, double* out_score) {
  oracle_pair* pairs = (oracle_pair*)malloc(sizeof(oracle_pair) * (size_t)n);
  if (!pairs) return 2;
  for (int64_t i = 0; i < n; ++i) {
    pairs[i].score = sigma[i];
    pairs[i].index = i;
  }
  qsort(pairs, (size_t)n, sizeof(oracle_pair), oracle_pair_cmp);
  for (int32_t j = 0; j < k; ++j) {
    out_idx[j] = pairs[j].index;
    out_score[j] = pairs[j].score;
  }
  free(pairs);
  return 0;
}

/* Top-K of one query: score every row, sort all N pairs best-first, keep K.
 * out_idx gets K row indices, out_score their double scores. cosine != 0
 * scores by cosine similarity instead of the inner product. */
static int topk_metric(const float* corpus, int64_t n, int32_t d, const float* query, int32_t k, int cosine,
                       int64_t* out_idx, double* out_score) {
  if (!corpus || !query || !out_idx || !out_score || n < 1 || d < 1 || k < 1 || k > n) return 1;
  double* sigma = (double*)malloc(sizeof(double) * (size_t)n);
  if (!sigma) return 2;
  if (cosine)
    oracle_scores_cosine(corpus, n, d, query, sigma);
  else
    oracle_scores(corpus, n, d, query, sigma);
  const int rc = select_topk(sigma, n, k, out_idx, out_score);
  free(sigma);
  return rc;
}

int oracle_topk(const float* corpus, int64_t n, int32_t d, const float* query, int32_t k,
                int64_t* out_idx, double* out_score) {
  return topk_metric(corpus, n, d, query, k, 0, out_idx, out_score);
}

int oracle_topk_cosine(const float* corpus, int64_t n, int32_t d, const float* query, int32_t k,
                       int64_t* out_idx, double* out_score) {
  return topk_metric(corpus, n, d, query, k, 1, out_idx, out_score);
}

/* B queries (row-major B x D), one top-K each: out arrays are B x K. */
int oracle_topk_batch(const float* corpus, int64_t n, int32_t d, const float* queries, int32_t b,
                      int32_t k, int64_t* out_idx, double* out_score) {
  if (b < 1) return 1;
  for (int32_t q = 0; q < b; ++q) {
    int rc = oracle_topk(corpus, n, d, queries + (int64_t)q * d, k, out_idx + (int64_t)q * k,
                         out_score + (int64_t)q * k);
    if (rc) return rc;
  }
  return 0;
}

/* The K largest values of x with their positions, largest first, lower
 * position first among equal values. */
int oracle_topk_int32(const int32_t* x, int64_t n, int32_t k, int32_t* out_val, int64_t* out_pos) {
  if (!x || !out_val || !out_pos || n < 1 || k < 1 || k > n) return 1;
  oracle_ipair* pairs = (oracle_ipair*)malloc(sizeof(oracle_ipair) * (size_t)n);
  if (!pairs) return 2;
  for (int64_t i = 0; i < n; ++i) {
    pairs[i].value = x[i];
    pairs[i].position = i;
  }
  qsort(pairs, (size_t)n, sizeof(oracle_ipair), oracle_ipair_cmp);
  for (int32_t j = 0; j < k; ++j) {
    out_val[j] = pairs[j].value;
    out_pos[j] = pairs[j].position;
  }
  free(pairs);
  return 0;
}

/* fp32 -> bf16 -> fp32 with round-to-nearest, ties to even: keep the top 16
 * bits of the fp32 pattern after adding half an ulp of the kept part, with the
 * tie going to the even kept pattern. NaN stays NaN (quiet). This is the
 * conversion the batched path applies to its inputs; the oracle uses it only
 * to score the rounded inputs for the tighter bf16 check. */
int oracle_round_bf16(const float* in, float* out, int64_t n) {
  if (!in || !out || n < 0) return 1;
  for (int64_t i = 0; i < n; ++i) {
    uint32_t bits;
    memcpy(&bits, &in[i], 4);
    if ((bits & 0x7F800000u) == 0x7F800000u && (bits & 0x007FFFFFu) != 0) {
      bits |= 0x00400000u;
      bits &= 0xFFFF0000u;
    } else {
      uint32_t lsb = (bits >> 16) & 1u;
      bits += 0x7FFFu + lsb;
      bits &= 0xFFFF0000u;
    }
    memcpy(&out[i], &bits, 4);
  }
  return 0;
}
