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
// MaxK backward scatter (bf16 values, int16 indices).
cudaError_t launch_maxk_backward(const uint16_t* dy, const int16_t* idx, int64_t N, int M, int k,
                                 uint16_t* grad, uint32_t* status, cudaStream_t s);

// Persistent-grid size for `kernel` launched with `threads` threads per block:
// SM count x resident blocks per SM (cached per device and kernel), capped at
// the number of blocks the work needs.
int persistent_blocks(const void* kernel, int threads, size_t smem, int64_t blocks_needed);

}  // namespace rtopk
