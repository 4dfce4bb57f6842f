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

/* --------------------------------------------------------------------- */
/* MaxK-GNN aggregation over CBSR ([MaxK] "How MaxK-GNN works": forward    */
/* feature aggregation as a row-wise-product SpGEMM over the compressed    */
/* rows; "Asymmetric passes, one mask" and "Why it works": the backward   */
/* pass is a sampled product evaluated only at the forward sp_index).     */
/*                                                                         */
/* Forward: out[i, m] = sum over the edges e of destination row i, in      */
/* edge order, of w_e * v, where (v, m) runs over the CBSR entries          */
/* (value, index) of source row col[e]; w_e = 1 when no weights are given.  */
/* binary32: each product and each running sum rounded, no FMA, starting   */
/* from +0. A source row's indices are distinct, so each out[i, m] gets at */
/* most one term per edge and the order of terms is the edge order.        */
/* --------------------------------------------------------------------- */

static float bf16_to_f32(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

int oracle_spgemm_cbsr(const int64_t* row_ptr, const int32_t* col, const float* w, int64_t n_dst,
                       int64_t n_src, const uint16_t* sp_data, const int16_t* sp_index, int32_t M,
                       int32_t k, float* out) {
  if (n_dst < 0 || n_src < 0 || M < 1 || k < 1 || k > M) return ORACLE_EARG;
  for (int64_t i = 0; i < n_dst; ++i) {
    float* o = out + i * (int64_t)M;
    for (int32_t m = 0; m < M; ++m) o[m] = 0.0f;
    for (int64_t e = row_ptr[i]; e < row_ptr[i + 1]; ++e) {
      const int64_t j = col[e];
      if (j < 0 || j >= n_src) return ORACLE_EINPUT;
      const float we = w ? w[e] : 1.0f;
      for (int32_t t = 0; t < k; ++t) {
        const int32_t m = sp_index[j * k + t];
        if (m < 0 || m >= M) return ORACLE_EINPUT;
        const float p = we * bf16_to_f32(sp_data[j * k + t]);
        o[m] = o[m] + p;
      }
    }
  }
  return ORACLE_OK;
}

/* Backward: d_sp[j, t] = sum over the edges e of source row j in the     */
/* transposed graph (destination t_row[e], weight t_w[e]), in that order,   */
/* of w_e * dout[t_row[e], sp_index[j, t]]. binary32, no FMA, from +0.     */
int oracle_sspmm_cbsr(const int64_t* t_ptr, const int32_t* t_row, const float* t_w, int64_t n_src,
                      int64_t n_dst, const float* dout, const int16_t* sp_index, int32_t M, int32_t k,
                      float* d_sp) {
  if (n_dst < 0 || n_src < 0 || M < 1 || k < 1 || k > M) return ORACLE_EARG;
  for (int64_t j = 0; j < n_src; ++j) {
    for (int32_t t = 0; t < k; ++t) {
      const int32_t m = sp_index[j * k + t];
      if (m < 0 || m >= M) return ORACLE_EINPUT;
      float acc = 0.0f;
      for (int64_t e = t_ptr[j]; e < t_ptr[j + 1]; ++e) {
        const int64_t i = t_row[e];
        if (i < 0 || i >= n_dst) return ORACLE_EINPUT;
        const float we = t_w ? t_w[e] : 1.0f;
        const float p = we * dout[i * (int64_t)M + m];
        acc = acc + p;
      }
      d_sp[j * k + t] = acc;
    }
  }
  return ORACLE_OK;
}
