// Internal interface between the C ABI layer and the kernel translation units.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace rtopk {

struct SelectArgs {
  const void* in;
  int64_t N;
  int M;
  int k;
  int max_iter;
  float eps;
  void* vals;
  void* idx;
  int* iters;       // nullable
  uint32_t* status; // nullable
};

// fp32 input, int32 indices.
cudaError_t launch_select_f32(const SelectArgs& a, cudaStream_t s);
// bf16 input; int16 indices when idx16, else int32.
cudaError_t launch_select_bf16(const SelectArgs& a, bool idx16, cudaStream_t s);
// Bucketed approximate top-k: B buckets per row, k / B kept per bucket (int32 indices).
cudaError_t launch_select_bucketed(const SelectArgs& a, int dtype_bf16, int buckets, cudaStream_t s);
// MaxK backward scatter (bf16 values, int16 indices).
cudaError_t launch_maxk_backward(const uint16_t* dy, const int16_t* idx, int64_t N, int M, int k,
                                 uint16_t* grad, uint32_t* status, cudaStream_t s);

// MaxK-GNN aggregation over CBSR (forward SpGEMM, backward sampled product).
cudaError_t launch_spgemm_fwd(const int64_t* row_ptr, const int32_t* col, const float* w, int64_t n_dst,
                              int64_t n_src, const uint16_t* sp_data, const int16_t* sp_index, int M, int k,
                              float* out, uint32_t* status, cudaStream_t s);
// grad != nullptr: the MaxK scatter is fused in and grad (n_src x M bf16) is
// written instead of d_sp.
cudaError_t launch_sspmm_bwd(const int64_t* t_ptr, const int32_t* t_row, const float* t_w, int64_t n_src,
                             int64_t n_dst, const float* dout, const int16_t* sp_index, int M, int k,
                             float* d_sp, uint16_t* grad, uint32_t* status, cudaStream_t s);

// Persistent-grid size for `kernel` launched with `threads` threads per block:
// SM count x resident blocks per SM (cached per device and kernel), capped at
// the number of blocks the work needs.
int persistent_blocks(const void* kernel, int threads, size_t smem, int64_t blocks_needed);
// The same for a kernel launched in clusters of `cluster` CTAs: the number of
// clusters that can be resident at once, capped at the clusters the work needs
// (0 if none fits).
int persistent_clusters(const void* kernel, int threads, int cluster, int64_t clusters_needed);

}  // namespace rtopk
