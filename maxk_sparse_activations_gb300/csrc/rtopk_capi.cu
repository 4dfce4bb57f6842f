// C ABI of librtopk.so: argument validation and dispatch (declared in rtopk.h).
#include <cmath>

#include "../../include/rtopk.h"
#include "launch.h"

namespace {

int check_select(const void* in, int64_t N, int32_t M, int32_t k, float eps, const void* vals,
                 const void* idx, int32_t max_m = RTOPK_MAX_M) {
  if (N < 0 || M < 1 || M > max_m) return RTOPK_EINVAL_SHAPE;
  if (k < 1 || k > M) return RTOPK_EINVAL_K;
  if (!(eps >= 0.0f)) return RTOPK_EINVAL_ARG;
  if (N > 0 && (in == nullptr || vals == nullptr || idx == nullptr)) return RTOPK_EINVAL_PTR;
  return RTOPK_OK;
}

int from_cuda(cudaError_t e) { return e == cudaSuccess ? RTOPK_OK : RTOPK_ECUDA; }

}  // namespace

extern "C" {

int rtopk_select_stats(const void* in, int64_t N, int32_t M, int32_t k, int32_t max_iter, float eps,
                       int32_t dtype, void* vals, int32_t* idx, int32_t* iters, uint32_t* status,
                       cudaStream_t stream) {
  if (dtype != RTOPK_F32 && dtype != RTOPK_BF16) return RTOPK_EINVAL_DTYPE;
  const int rc = check_select(in, N, M, k, eps, vals, idx, RTOPK_SELECT_MAX_M);
  if (rc != RTOPK_OK || N == 0) return rc;
  rtopk::SelectArgs a{in, N, M, k, max_iter, eps, vals, idx, iters, status};
  if (dtype == RTOPK_F32) return from_cuda(rtopk::launch_select_f32(a, stream));
  return from_cuda(rtopk::launch_select_bf16(a, /*idx16=*/false, stream));
}

int rtopk_select(const void* in, int64_t N, int32_t M, int32_t k, int32_t max_iter, float eps,
                 int32_t dtype, void* vals, int32_t* idx, cudaStream_t stream) {
  return rtopk_select_stats(in, N, M, k, max_iter, eps, dtype, vals, idx, nullptr, nullptr, stream);
}

int rtopk_select_bucketed(const void* in, int64_t N, int32_t M, int32_t k, int32_t buckets, int32_t max_iter,
                          float eps, int32_t dtype, void* vals, int32_t* idx, cudaStream_t stream) {
  if (dtype != RTOPK_F32 && dtype != RTOPK_BF16) return RTOPK_EINVAL_DTYPE;
  if (N < 0 || M < 1 || M > RTOPK_MAX_M) return RTOPK_EINVAL_SHAPE;
  if (k < 1 || k > M) return RTOPK_EINVAL_K;
  if (buckets < 1 || M % buckets != 0 || k % buckets != 0) return RTOPK_EINVAL_ARG;
  const int rc = check_select(in, N, M, k, eps, vals, idx);
  if (rc != RTOPK_OK || N == 0) return rc;
  rtopk::SelectArgs a{in, N, M, k, max_iter, eps, vals, idx, nullptr, nullptr};
  return from_cuda(rtopk::launch_select_bucketed(a, dtype == RTOPK_BF16, buckets, stream));
}

int maxk_forward(const void* in_bf16, int64_t N, int32_t M, int32_t k, int32_t max_iter, float eps,
                 void* vals_bf16, int16_t* idx, cudaStream_t stream) {
  const int rc = check_select(in_bf16, N, M, k, eps, vals_bf16, idx);
  if (rc != RTOPK_OK || N == 0) return rc;
  rtopk::SelectArgs a{in_bf16, N, M, k, max_iter, eps, vals_bf16, idx, nullptr, nullptr};
  return from_cuda(rtopk::launch_select_bf16(a, /*idx16=*/true, stream));
}

int maxk_backward_scatter(const void* dy_bf16, const int16_t* idx, int64_t N, int32_t M, int32_t k,
                          void* grad_bf16, uint32_t* status, cudaStream_t stream) {
  if (N < 0 || M < 1 || M > RTOPK_MAX_M) return RTOPK_EINVAL_SHAPE;
  if (k < 1 || k > M) return RTOPK_EINVAL_K;
  if (N > 0 && (dy_bf16 == nullptr || idx == nullptr || grad_bf16 == nullptr)) return RTOPK_EINVAL_PTR;
  if (N == 0) return RTOPK_OK;
  return from_cuda(rtopk::launch_maxk_backward(static_cast<const uint16_t*>(dy_bf16), idx, N, M, k,
                                               static_cast<uint16_t*>(grad_bf16), status, stream));
}

int maxk_spgemm_forward(const int64_t* row_ptr, const int32_t* col_idx, const float* edge_w, int64_t n_dst,
                        int64_t n_src, const void* sp_data_bf16, const int16_t* sp_index, int32_t M, int32_t k,
                        float* out, uint32_t* status, cudaStream_t stream) {
  if (n_dst < 0 || n_src < 0 || M < 1 || M > RTOPK_MAX_M) return RTOPK_EINVAL_SHAPE;
  if (k < 1 || k > M || k > RTOPK_GNN_MAX_K) return RTOPK_EINVAL_K;
  if (n_dst > 0 && (row_ptr == nullptr || out == nullptr || (n_src > 0 && (col_idx == nullptr ||
                    sp_data_bf16 == nullptr || sp_index == nullptr))))
    return RTOPK_EINVAL_PTR;
  if (n_dst == 0) return RTOPK_OK;
  return from_cuda(rtopk::launch_spgemm_fwd(row_ptr, col_idx, edge_w, n_dst, n_src,
                                            static_cast<const uint16_t*>(sp_data_bf16), sp_index, M, k, out,
                                            status, stream));
}

int maxk_sspmm_backward(const int64_t* t_row_ptr, const int32_t* t_dst, const float* t_edge_w, int64_t n_src,
                        int64_t n_dst, const float* dout, const int16_t* sp_index, int32_t M, int32_t k,
                        float* d_sp_data, uint32_t* status, cudaStream_t stream) {
  if (n_dst < 0 || n_src < 0 || M < 1 || M > RTOPK_MAX_M) return RTOPK_EINVAL_SHAPE;
  if (k < 1 || k > M || k > RTOPK_GNN_MAX_K) return RTOPK_EINVAL_K;
  if (n_src > 0 && (t_row_ptr == nullptr || sp_index == nullptr || d_sp_data == nullptr ||
                    (n_dst > 0 && (t_dst == nullptr || dout == nullptr))))
    return RTOPK_EINVAL_PTR;
  if (n_src == 0) return RTOPK_OK;
  return from_cuda(rtopk::launch_sspmm_bwd(t_row_ptr, t_dst, t_edge_w, n_src, n_dst, dout, sp_index, M, k,
                                           d_sp_data, nullptr, status, stream));
}

int maxk_sspmm_backward_scatter(const int64_t* t_row_ptr, const int32_t* t_dst, const float* t_edge_w,
                                int64_t n_src, int64_t n_dst, const float* dout, const int16_t* sp_index,
                                int32_t M, int32_t k, void* grad_bf16, uint32_t* status, cudaStream_t stream) {
  if (n_dst < 0 || n_src < 0 || M < 1 || M > RTOPK_MAX_M) return RTOPK_EINVAL_SHAPE;
  if (k < 1 || k > M || k > RTOPK_GNN_MAX_K) return RTOPK_EINVAL_K;
  if (n_src > 0 && (t_row_ptr == nullptr || sp_index == nullptr || grad_bf16 == nullptr ||
                    (n_dst > 0 && (t_dst == nullptr || dout == nullptr))))
    return RTOPK_EINVAL_PTR;
  if (n_src == 0) return RTOPK_OK;
  return from_cuda(rtopk::launch_sspmm_bwd(t_row_ptr, t_dst, t_edge_w, n_src, n_dst, dout, sp_index, M, k,
                                           nullptr, static_cast<uint16_t*>(grad_bf16), status, stream));
}

int rtopk_status_read(const uint32_t* status, uint32_t* bits, cudaStream_t stream) {
  if (status == nullptr) return RTOPK_EINVAL_PTR;
  uint32_t word = 0;
  if (cudaMemcpyAsync(&word, status, sizeof(word), cudaMemcpyDefault, stream) != cudaSuccess) return RTOPK_ECUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return RTOPK_ECUDA;
  if (bits != nullptr) *bits = word;
  return word == 0u ? RTOPK_OK : RTOPK_EDEVICE;
}

const char* rtopk_strerror(int code) {
  switch (code) {
    case RTOPK_OK: return "ok";
    case RTOPK_EINVAL_SHAPE:
      return "invalid shape: need N >= 0 and 1 <= M <= 65536 (rtopk_select) or 8192 (other entry points)";
    case RTOPK_EINVAL_K: return "invalid k: need 1 <= k <= M";
    case RTOPK_EINVAL_PTR: return "a required device pointer is NULL";
    case RTOPK_EINVAL_DTYPE: return "unknown dtype: use RTOPK_F32 or RTOPK_BF16";
    case RTOPK_ECUDA: return "a CUDA runtime call or kernel launch failed";
    case RTOPK_EDEVICE: return "the device status word reports invalid rows, a safety cap or bad indices";
    case RTOPK_EINVAL_ARG: return "invalid argument: need eps >= 0, and buckets dividing both M and k";
    default: return "unknown rtopk status code";
  }
}

int rtopk_version(void) { return 100; }

}  // extern "C"
