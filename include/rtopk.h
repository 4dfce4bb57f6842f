/*
 * rtopk.h -- C ABI of librtopk.so: row-wise top-k selection (RTop-K) and the
 * MaxK sparse-activation layer on NVIDIA GB300 (sm_103a).
 *
 * Sources (page titles and sections):
 *  [RTopK] "RTop-K: Ultra-Fast Row-Wise Top-K Selection for Neural Network
 *          Acceleration on GPUs" (summary page): "Problem" (row-wise top-k of
 *          a large batch of short vectors, output need not be sorted),
 *          "Approach" (binary search over the value range for a threshold
 *          selecting k, early stop by capping iterations, second pass filling
 *          borderline ties), "Surprising findings" (precision epsilon),
 *          "Limitations" (the method stops at M = 8192; rtopk_select goes on
 *          to 65536 with one CTA cluster per row, same arithmetic).
 *  [MaxK]  "MaxK-GNN: Extremely Fast GPU Kernel Design for Accelerating Graph
 *          Neural Networks Training": "How MaxK-GNN works" ("The idea": exactly
 *          k survivors per row stored as two dense arrays; "Asymmetric passes,
 *          one mask": the forward sp_index is reused by the backward pass),
 *          "Why it works".
 *
 * Conventions shared by every entry point:
 *  - All array pointers are caller-owned memory the device can address:
 *    device memory (e.g. torch tensors), or pinned / registered host memory,
 *    which the kernels then read and write in place over the host link
 *    (NVLink-C2C on Grace-Blackwell) with no staging copy. Arrays are dense
 *    and row-major: inputs have row stride M, CBSR outputs row stride k.
 *    The library allocates no memory and keeps no state between calls, except
 *    a per-device cache of the SM count and occupancy used to size grids.
 *  - Every call is asynchronous on `stream` (0 = legacy default stream).
 *  - Argument errors return a negative code synchronously and launch nothing.
 *    A failed launch returns RTOPK_ECUDA. Problems found in the data on the
 *    device are reported through the optional `status` word (see below).
 *  - N == 0 is a no-op that returns RTOPK_OK.
 *  - Input values must be finite with |x| <= 1e38, so that the binary32
 *    midpoint (lo + hi) * 0.5 cannot overflow. Rows that break this set a
 *    status bit; their outputs are unspecified but every write stays inside
 *    the row.
 *
 * Semantics of the selection (identical for every entry point that selects):
 *  lo = min(row), hi = max(row), c(t) = #{j : x_j >= t}.
 *  1. If c(hi) >= k: keep the k lowest indices whose value equals the maximum;
 *     no search pass runs (iters = 0).
 *  2. Otherwise repeat while (max_iter < 0 or iters < max_iter) and
 *     (hi - lo) > eps:  mid = (lo + hi) * 0.5 (binary32, no FMA); stop if no
 *     binary32 value lies strictly between lo and hi; cnt = c(mid); iters++;
 *     cnt == k: lo = mid and stop; cnt > k: lo = mid; cnt < k: hi = mid.
 *  3. Keep every x >= hi, then fill up to exactly k from lo <= x < hi in
 *     ascending index order.
 *  4. Write the k kept (value, index) pairs of the row in ascending index
 *     order; values are bit copies of the input.
 *  With max_iter < 0 and eps == 0 (exact mode) the result is the exact top-k
 *  with ties at the k-th value broken by the lowest index.
 *
 * Device status word bits (OR-ed with atomicOr; the caller zeroes the word
 * before the call and reads it after synchronising the stream):
 */
#ifndef RTOPK_H_
#define RTOPK_H_

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define RTOPK_STATUS_NONFINITE  0x1u /* a row holds NaN or +-Inf */
#define RTOPK_STATUS_RANGE      0x2u /* a row holds a finite value with |x| > 1e38 */
#define RTOPK_STATUS_SAFETY_CAP 0x4u /* a search reached 512 passes (cannot happen for valid rows) */
#define RTOPK_STATUS_BAD_INDEX  0x8u /* an sp_index entry outside [0, M) was skipped */
#define RTOPK_STATUS_BAD_EDGE   0x10u /* aggregation: an edge endpoint outside its row range was skipped */

#define RTOPK_MAX_M 8192 /* [RTopK] "Limitations": the method's row limit; all entry points but rtopk_select */
#define RTOPK_SELECT_MAX_M 65536 /* rtopk_select / _stats: longer rows run one CTA cluster per row */
#define RTOPK_GNN_MAX_K 256 /* largest k of the aggregation entry points */

typedef enum {
  RTOPK_F32 = 0,  /* IEEE binary32 */
  RTOPK_BF16 = 1  /* bfloat16, passed as 16-bit patterns */
} rtopk_dtype;

typedef enum {
  RTOPK_OK = 0,
  RTOPK_EINVAL_SHAPE = -1, /* N < 0, M < 1 or M above the entry point's limit */
  RTOPK_EINVAL_K = -2,     /* k < 1 or k > M */
  RTOPK_EINVAL_PTR = -3,   /* a required pointer is NULL (with N > 0) */
  RTOPK_EINVAL_DTYPE = -4, /* dtype is not an rtopk_dtype value */
  RTOPK_ECUDA = -5,        /* a CUDA runtime call or launch failed */
  RTOPK_EINVAL_ARG = -6,   /* eps < 0 or NaN; buckets not dividing M and k */
  RTOPK_EDEVICE = -7       /* rtopk_status_read: the device status word is non-zero */
} rtopk_status;

/*
 * rtopk_select -- row-wise top-k of an N x M matrix into CBSR.
 * [RTopK] "Problem", "Approach"; [MaxK] "The idea" (CBSR = two dense N x k arrays).
 *
 *  in        device, N x M, dtype elements (fp32 or bf16 bit patterns), read only
 *  N, M, k   rows, row length (1..65536), kept per row (1..M). Rows up to 8192
 *            elements are the pages' range; longer rows (beyond the limit the
 *            pages state in "Limitations") run the same search with one
 *            cluster of 2, 4 or 8 CTAs per row, exchanging pass counts through
 *            distributed shared memory -- same results as the scalar definition
 *  max_iter  cap on counted bisection passes; < 0 = no cap (early stop off)
 *  eps       absolute precision: the search stops once (hi - lo) <= eps; >= 0
 *  dtype     RTOPK_F32 or RTOPK_BF16
 *  vals      device, N x k, same dtype as `in`: the kept values (bit copies)
 *  idx       device, N x k int32: the kept column indices, ascending per row
 *  stream    CUDA stream to launch on
 * Returns RTOPK_OK or a negative rtopk_status.
 */
int rtopk_select(const void* in, int64_t N, int32_t M, int32_t k, int32_t max_iter, float eps,
                 int32_t dtype, void* vals, int32_t* idx, cudaStream_t stream);

/*
 * rtopk_select_stats -- rtopk_select plus diagnostics (same kernel, same outputs).
 * [RTopK] "Surprising findings" (the exact search usually ends after a small,
 * bounded number of passes) -- `iters` gives that pass count for every row.
 *
 *  iters   device, N int32 or NULL: counted bisection passes of each row
 *  status  device, one uint32 or NULL: OR of RTOPK_STATUS_* bits over all rows
 * Performance note: with iters != NULL in exact mode every row runs the
 * binary32 search whose passes are counted. In exact mode with iters == NULL
 * (and in rtopk_select / maxk_forward) rows of 128..1024 elements (one warp per
 * row) and of 2048 / 4096 / 8192 elements (a team of warps per row) may
 * instead run a search counted on packed 16-bit images of the row, finished in
 * binary32 where needed: same outputs, fewer instructions. Early stop and eps
 * on rows of 128..1024 follow the same binary32 trajectory on a kernel that
 * streams rows through shared memory.
 */
int rtopk_select_stats(const void* in, int64_t N, int32_t M, int32_t k, int32_t max_iter,
                       float eps, int32_t dtype, void* vals, int32_t* idx, int32_t* iters,
                       uint32_t* status, cudaStream_t stream);

/*
 * rtopk_select_bucketed -- bucketed approximate row-wise top-k.
 * "Approximate Top-k for Increased Parallelism" (abstract): split each vector
 * into buckets and take many smaller top-k selections independently.
 *
 * Each row is split into `buckets` contiguous buckets of M / buckets columns;
 * bucket b keeps the top-(k / buckets) of its columns under the selection of
 * rtopk_select (max_iter / eps apply per bucket). Output as rtopk_select: k
 * (value, index) pairs per row, indices in [0, M), ascending. buckets = 1 is
 * rtopk_select. Requires buckets to divide both M and k (else
 * RTOPK_EINVAL_ARG). Other arguments as for rtopk_select.
 */
int rtopk_select_bucketed(const void* in, int64_t N, int32_t M, int32_t k, int32_t buckets, int32_t max_iter,
                          float eps, int32_t dtype, void* vals, int32_t* idx, cudaStream_t stream);

/*
 * maxk_forward -- the MaxK nonlinearity: keep the top-k features of each row of
 * a bf16 activation matrix, written as CBSR with 16-bit indices.
 * [MaxK] "The idea" (exactly k survivors per node, dense data + sp_index arrays).
 *
 *  in_bf16    device, N x M bf16 bit patterns
 *  vals_bf16  device, N x k bf16: sp_data
 *  idx        device, N x k int16: sp_index, ascending per row (M <= 8192 < 2^15)
 *  other arguments as for rtopk_select; exact mode by default (max_iter = -1, eps = 0)
 */
int maxk_forward(const void* in_bf16, int64_t N, int32_t M, int32_t k, int32_t max_iter,
                 float eps, void* vals_bf16, int16_t* idx, cudaStream_t stream);

/*
 * maxk_backward_scatter -- MaxK backward: gradient flows only to the kept
 * features, at the positions the forward pass recorded.
 * [MaxK] "Asymmetric passes, one mask"; "Why it works" (only MaxK survivors
 * carry gradients).
 *
 *  dy_bf16    device, N x k bf16: upstream gradient w.r.t. the CBSR values
 *  idx        device, N x k int16: the forward sp_index (distinct per row)
 *  grad_bf16  device, N x M bf16: written in full -- dy at the kept positions,
 *             +0.0 everywhere else (no separate zero-fill is needed)
 *  status     device uint32 or NULL: RTOPK_STATUS_BAD_INDEX if an index was
 *             outside [0, M) (that entry is skipped)
 * Indices repeated within a row leave which of their values lands unspecified.
 */
int maxk_backward_scatter(const void* dy_bf16, const int16_t* idx, int64_t N, int32_t M,
                          int32_t k, void* grad_bf16, uint32_t* status, cudaStream_t stream);

/*
 * maxk_spgemm_forward -- MaxK-GNN forward feature aggregation over CBSR: a
 * row-wise-product SpGEMM of the graph with the compressed feature rows.
 * [MaxK] "How MaxK-GNN works" (row-wise product with shared-memory
 * scatter-accumulation, one global write per row), "Why it works".
 *
 *  out[i, m] = sum over the edges e of destination row i, in edge order, of
 *              edge_w[e] * v for every CBSR entry (v, m) of source row
 *              col_idx[e]; binary32 products and sums, one rounding each, no
 *              FMA -- deterministic, and bit-identical to that sequential sum
 *              for rows of at most 512 edges. Longer rows are split into
 *              equal chunks (multiples of 32 edges), one per warp of a block,
 *              each summed in edge order, and the partial rows are combined
 *              in warp order: still deterministic, and within
 *              2 (deg + 1) 2^-24 sum|terms| of the sequential sum.
 *
 *  row_ptr      device, n_dst + 1 int64: CSR offsets over destination rows
 *  col_idx      device, E int32: source row of each edge (0 <= j < n_src)
 *  edge_w       device, E fp32, or NULL for weight 1
 *  sp_data_bf16 device, n_src x k bf16: CBSR values (e.g. from maxk_forward)
 *  sp_index     device, n_src x k int16: CBSR columns, distinct within a row
 *  M, k         feature width (1..8192) and kept per row (1..min(M, 256))
 *  out          device, n_dst x M fp32, written in full
 *  status       device uint32 or NULL: RTOPK_STATUS_BAD_EDGE / _BAD_INDEX
 */
int maxk_spgemm_forward(const int64_t* row_ptr, const int32_t* col_idx, const float* edge_w, int64_t n_dst,
                        int64_t n_src, const void* sp_data_bf16, const int16_t* sp_index, int32_t M, int32_t k,
                        float* out, uint32_t* status, cudaStream_t stream);

/*
 * maxk_sspmm_backward -- MaxK-GNN backward of the aggregation: the gradient of
 * each CBSR value, a product sampled only at the forward sp_index.
 * [MaxK] "Asymmetric passes, one mask" (the sp_index computed forward is
 * reused backward; output positions are known before the kernel starts).
 *
 *  d_sp_data[j, t] = sum over the edges e of source row j in the transposed
 *              graph (t_row_ptr / t_dst / t_edge_w, edges in the order given),
 *              of t_edge_w[e] * dout[t_dst[e], sp_index[j, t]]; binary32, one
 *              rounding per product and sum, no FMA.
 *
 *  t_row_ptr   device, n_src + 1 int64: CSR offsets of the transposed graph
 *  t_dst       device, E int32: destination row of each edge (0 <= i < n_dst)
 *  t_edge_w    device, E fp32, or NULL for weight 1
 *  dout        device, n_dst x M fp32: gradient of the aggregation output
 *  sp_index    device, n_src x k int16: the forward CBSR columns
 *  d_sp_data   device, n_src x k fp32, written in full
 *  status      device uint32 or NULL: RTOPK_STATUS_BAD_EDGE / _BAD_INDEX
 */
int maxk_sspmm_backward(const int64_t* t_row_ptr, const int32_t* t_dst, const float* t_edge_w, int64_t n_src,
                        int64_t n_dst, const float* dout, const int16_t* sp_index, int32_t M, int32_t k,
                        float* d_sp_data, uint32_t* status, cudaStream_t stream);

/*
 * maxk_sspmm_backward_scatter -- maxk_sspmm_backward with the MaxK backward
 * scatter fused in: the gradient of the MaxK input, written dense.
 * [MaxK] "Asymmetric passes, one mask" (the backward SSpMM and the MaxK
 * backward share the forward sp_index; only kept features carry gradient).
 *
 *  grad[j, sp_index[j, t]] = bf16(d_sp_data[j, t]) with d_sp_data[j, t]
 *              exactly as maxk_sspmm_backward defines it, rounded to the
 *              nearest bf16 (ties to even); +0.0 at every other column. This
 *              equals maxk_sspmm_backward, a round-to-nearest conversion to
 *              bf16 and maxk_backward_scatter run in sequence, without the
 *              n_src x k intermediate in HBM.
 *
 *  grad_bf16   device, n_src x M bf16, written in full
 *  other arguments as for maxk_sspmm_backward
 * Indices repeated within a row leave which of their values lands unspecified.
 */
int maxk_sspmm_backward_scatter(const int64_t* t_row_ptr, const int32_t* t_dst, const float* t_edge_w,
                                int64_t n_src, int64_t n_dst, const float* dout, const int16_t* sp_index,
                                int32_t M, int32_t k, void* grad_bf16, uint32_t* status, cudaStream_t stream);

/*
 * rtopk_status_read -- read a device status word after the work that sets it.
 * Waits for `stream`, copies the word to the host and returns RTOPK_EDEVICE if
 * any RTOPK_STATUS_* bit is set, else RTOPK_OK (RTOPK_ECUDA if the copy or the
 * wait fails). The pages define no error reporting; this is the host side of
 * the status words the entry points above fill.
 *
 *  status  the word passed as `status` to the earlier calls (device or pinned host memory)
 *  bits    host uint32 or NULL: receives the word
 * Blocks the calling thread until `stream` has drained; allocates nothing.
 */
int rtopk_status_read(const uint32_t* status, uint32_t* bits, cudaStream_t stream);

/* Human-readable text for an rtopk_status code (static storage, never NULL). */
const char* rtopk_strerror(int code);

/* Library ABI version: major * 10000 + minor * 100 + patch. */
int rtopk_version(void);

#ifdef __cplusplus
}
#endif

#endif /* RTOPK_H_ */
