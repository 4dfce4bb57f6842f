/*
 * Oracle for row-wise top-k selection (RTop-K) and the MaxK layer.
 *
 * TEST INFRASTRUCTURE ONLY. This file is plain, slow, obviously-correct C that
 * the tests, the smoke check and the CPU-baseline leg of the benchmark use to
 * check the CUDA path. The product path never links, loads or calls it, and it
 * shares no code, header, table or helper with the CUDA sources.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fPIC -shared (no -ffast-math):
 * every float operation below is one IEEE binary32 operation rounded to
 * nearest-even, with no contraction into fused multiply-add.
 *
 * Sources (page titles and sections):
 *  [RTopK]  "RTop-K: Ultra-Fast Row-Wise Top-K Selection for Neural Network
 *           Acceleration on GPUs" (summary page), sections "Problem",
 *           "Approach", "Key results", "Surprising findings".
 *  [MaxK]   "MaxK-GNN: Extremely Fast GPU Kernel Design for Accelerating Graph
 *           Neural Networks Training", sections "How MaxK-GNN works" ("The
 *           idea", "Asymmetric passes, one mask") and "Why it works".
 *
 * Readings of points the pages leave open:
 *  - count with ">=": c(t) = #{j : x_j >= t};
 *  - midpoint (lo + hi) * 0.5f in binary32, two roundings, no FMA;
 *  - eps is absolute and tested as (hi - lo) > eps in binary32 before the
 *    midpoint is formed; max_iter counts midpoint passes, < 0 means no cap;
 *  - when c(max) >= k the threshold is the row maximum and the k lowest
 *    indices among the maximum's ties are kept (no search is run);
 *  - the "second pass using the minimum" keeps {x >= hi} outright and fills
 *    the remainder from [lo, hi) in ascending index order;
 *  - the output row lists the kept indices in ascending order;
 *  - inputs must be finite with |x| <= 1e38 (so lo + hi cannot overflow);
 *    the functions return ORACLE_EINPUT for any other row.
 *
 * Parity pins (tests under tests/ that do not need a GPU): brute force over
 * all k-subsets for tiny rows, hand-worked examples in tests/golden/,
 * closed forms for max_iter = 0 and max_iter = 1, exact-mode equality of the
 * replay with the sort definition, invariants, and torch.topk's value
 * multiset.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_EARG (-1)
#define ORACLE_EINPUT (-2)
#define ORACLE_ENOMEM (-3)

/* Input precondition: finite and |x| <= 1e38 (NaN fails both compares). */
static int row_is_valid(const float* x, int32_t M) {
  for (int32_t j = 0; j < M; ++j) {
    if (!(x[j] >= -1e38f && x[j] <= 1e38f)) return 0;
  }
  return 1;
}

/* --------------------------------------------------------------------- */
/* Definition: exact top-k under the lowest-index tie rule.                */
/* [RTopK] "Problem": top-k of every row; ties at the k-th value are       */
/* broken by lowest index (the reading), output in ascending index order.  */
/* --------------------------------------------------------------------- */

typedef struct {
  float v;
  int32_t j;
} entry_t;

/* value descending (compared as binary32, so -0 == +0), index ascending */
static int cmp_value_desc_index_asc(const void* a, const void* b) {
  const entry_t* p = (const entry_t*)a;
  const entry_t* q = (const entry_t*)b;
  if (p->v > q->v) return -1;
  if (p->v < q->v) return 1;
  return (p->j > q->j) - (p->j < q->j);
}

static int cmp_int32_asc(const void* a, const void* b) {
  int32_t p = *(const int32_t*)a, q = *(const int32_t*)b;
  return (p > q) - (p < q);
}

int oracle_sort_topk(const float* x, int64_t N, int32_t M, int32_t k, int32_t* idx) {
  if (N < 0 || M < 1 || k < 1 || k > M) return ORACLE_EARG;
  entry_t* e = (entry_t*)malloc(sizeof(entry_t) * (size_t)M);
  if (!e) return ORACLE_ENOMEM;
  int rc = ORACLE_OK;
  for (int64_t r = 0; r < N; ++r) {
    const float* row = x + r * (int64_t)M;
    int32_t* out = idx + r * (int64_t)k;
    if (!row_is_valid(row, M)) { rc = ORACLE_EINPUT; break; }
    for (int32_t j = 0; j < M; ++j) { e[j].v = row[j]; e[j].j = j; }
    qsort(e, (size_t)M, sizeof(entry_t), cmp_value_desc_index_asc);
    for (int32_t i = 0; i < k; ++i) out[i] = e[i].j;
    qsort(out, (size_t)k, sizeof(int32_t), cmp_int32_asc);
  }
  free(e);
  return rc;
}

/* --------------------------------------------------------------------- */
/* Brute force for tiny rows, independent of the sort above: among all    */
/* k-subsets pick the one whose values, listed in descending order, are    */
/* lexicographically largest; among those, the one whose ascending index   */
/* list is lexicographically smallest. Only for M <= 20.                   */
/* --------------------------------------------------------------------- */

static void subset_desc_values(const float* row, uint32_t mask, int32_t M, float* out) {
  int32_t n = 0;
  for (int32_t j = 0; j < M; ++j)
    if (mask & (1u << j)) out[n++] = row[j];
  /* insertion sort, descending */
  for (int32_t a = 1; a < n; ++a) {
    float v = out[a];
    int32_t b = a - 1;
    while (b >= 0 && out[b] < v) { out[b + 1] = out[b]; --b; }
    out[b + 1] = v;
  }
}

/* returns <0 if subset a is better than b, >0 if worse, 0 if identical */
static int compare_subsets(const float* row, int32_t M, int32_t k, uint32_t a, uint32_t b) {
  float va[32], vb[32];
  subset_desc_values(row, a, M, va);
  subset_desc_values(row, b, M, vb);
  for (int32_t i = 0; i < k; ++i) {
    if (va[i] > vb[i]) return -1;
    if (va[i] < vb[i]) return 1;
  }
  /* equal value lists: the lexicographically smaller ascending index list */
  for (int32_t j = 0; j < M; ++j) {
    int ia = (a >> j) & 1, ib = (b >> j) & 1;
    if (ia != ib) return ia ? -1 : 1; /* a lists j first: a is smaller */
  }
  return 0;
}

int oracle_brute_topk(const float* x, int64_t N, int32_t M, int32_t k, int32_t* idx) {
  if (N < 0 || M < 1 || M > 20 || k < 1 || k > M) return ORACLE_EARG;
  for (int64_t r = 0; r < N; ++r) {
    const float* row = x + r * (int64_t)M;
    if (!row_is_valid(row, M)) return ORACLE_EINPUT;
    uint32_t best = 0;
    int have = 0;
    for (uint32_t m = 0; m < (1u << M); ++m) {
      if (__builtin_popcount(m) != k) continue;
      if (!have || compare_subsets(row, M, k, m, best) < 0) { best = m; have = 1; }
    }
    int32_t n = 0;
    for (int32_t j = 0; j < M; ++j)
      if (best & (1u << j)) idx[r * (int64_t)k + n++] = j;
  }
  return ORACLE_OK;
}

/* --------------------------------------------------------------------- */
/* Replay of the method, step by step ([RTopK] "Approach"): a binary       */
/* search over the row's value range [min, max] for a threshold that       */
/* selects k elements, capped at max_iter passes (early stopping) and      */
/* stopped at precision eps, then a second pass that keeps everything at   */
/* or above the upper bound and fills the borderline ties from the lower   */
/* bound upward, lowest index first.                                       */
/* --------------------------------------------------------------------- */

static int32_t count_at_least(const float* row, int32_t M, float t) {
  int32_t c = 0;
  for (int32_t j = 0; j < M; ++j)
    if (row[j] >= t) ++c;
  return c;
}

static void replay_row(const float* row, int32_t M, int32_t k, int32_t max_iter, float eps,
                       int32_t* out, int32_t* iters_out) {
  /* value range */
  float lo = row[0], hi = row[0];
  for (int32_t j = 1; j < M; ++j) {
    if (row[j] < lo) lo = row[j];
    if (row[j] > hi) hi = row[j];
  }

  /* ties at the maximum already fill k: keep the k lowest-index ties */
  if (count_at_least(row, M, hi) >= k) {
    int32_t n = 0;
    for (int32_t j = 0; j < M && n < k; ++j)
      if (row[j] >= hi) out[n++] = j;
    *iters_out = 0;
    return;
  }

  /* bisection; invariant: c(lo) >= k and c(hi) < k */
  int32_t it = 0;
  while ((max_iter < 0 || it < max_iter) && (hi - lo) > eps) {
    float mid = (lo + hi) * 0.5f;
    if (!(lo < mid && mid < hi)) break; /* no binary32 value strictly between */
    int32_t cnt = count_at_least(row, M, mid);
    ++it;
    if (cnt == k) { lo = mid; break; }
    if (cnt > k) lo = mid;
    else hi = mid;
  }

  /* second pass: keep x >= hi, fill from [lo, hi) by ascending index */
  int32_t need = k - count_at_least(row, M, hi);
  int32_t n = 0;
  for (int32_t j = 0; j < M; ++j) {
    if (row[j] >= hi) {
      out[n++] = j;
    } else if (row[j] >= lo && need > 0) {
      out[n++] = j;
      --need;
    }
  }
  *iters_out = it;
}

int oracle_replay(const float* x, int64_t N, int32_t M, int32_t k, int32_t max_iter, float eps,
                  int32_t* idx, int32_t* iters) {
  if (N < 0 || M < 1 || k < 1 || k > M || !(eps >= 0.0f)) return ORACLE_EARG;
  for (int64_t r = 0; r < N; ++r) {
    const float* row = x + r * (int64_t)M;
    if (!row_is_valid(row, M)) return ORACLE_EINPUT;
    int32_t it = 0;
    replay_row(row, M, k, max_iter, eps, idx + r * (int64_t)k, &it);
    if (iters) iters[r] = it;
  }
  return ORACLE_OK;
}

/* --------------------------------------------------------------------- */
/* MaxK backward ([MaxK] "Asymmetric passes, one mask"): only the kept     */
/* features carry gradient, at the positions the forward pass recorded.    */
/* The dense gradient row is zero except grad[r, idx[r, j]] = dy[r, j].    */
/* Values are moved as raw 16-bit patterns (bf16), never rounded.          */
/* --------------------------------------------------------------------- */

int oracle_maxk_backward_u16(const uint16_t* dy, const int16_t* idx, int64_t N, int32_t M,
                             int32_t k, uint16_t* grad) {
  if (N < 0 || M < 1 || k < 1 || k > M) return ORACLE_EARG;
  memset(grad, 0, sizeof(uint16_t) * (size_t)N * (size_t)M);
  for (int64_t r = 0; r < N; ++r) {
    for (int32_t j = 0; j < k; ++j) {
      int32_t c = idx[r * (int64_t)k + j];
      if (c < 0 || c >= M) return ORACLE_EINPUT;
      grad[r * (int64_t)M + c] = dy[r * (int64_t)k + j];
    }
  }
  return ORACLE_OK;
}
