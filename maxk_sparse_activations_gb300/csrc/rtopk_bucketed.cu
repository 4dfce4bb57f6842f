// Bucketed approximate row-wise top-k, sm_103a.
//
// Source: "Approximate Top-k for Increased Parallelism" (abstract): relax
// exactness by splitting the vector into buckets and computing many smaller
// top-k selections independently.
//
// A row of M elements is split into B contiguous buckets of M / B; each bucket
// keeps its own top-(k / B) under the same selection as rtopk_select (exact by
// default, or early-stopped). Viewed as (N * B) rows of M / B elements, the
// matrix and the CBSR output already have the layout of that smaller problem,
// so the selection kernels run unchanged; one pass then turns bucket-local
// column indices into row indices (+ bucket * M / B). Buckets are in column
// order and each bucket's indices ascend, so every output row ascends.
#include <cstdint>

#include "launch.h"

namespace rtopk {
namespace {

__global__ void __launch_bounds__(256)
bucket_index_offset_kernel(int32_t* __restrict__ idx, int64_t total, int kb, int buckets, int mb) {
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  for (int64_t p = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; p < total; p += stride) {
    const int64_t bucket_row = p / kb;  // row of the (N * B) x (M / B) problem
    idx[p] += int32_t(bucket_row % buckets) * mb;
  }
}

}  // namespace

cudaError_t launch_select_bucketed(const SelectArgs& a, int dtype_bf16, int buckets, cudaStream_t s) {
  SelectArgs b = a;
  b.N = a.N * buckets;
  b.M = a.M / buckets;
  b.k = a.k / buckets;
  cudaError_t e = dtype_bf16 ? launch_select_bf16(b, /*idx16=*/false, s) : launch_select_f32(b, s);
  if (e != cudaSuccess || buckets == 1) return e;
  const int64_t total = a.N * int64_t(a.k);
  const int blocks = persistent_blocks(reinterpret_cast<const void*>(bucket_index_offset_kernel), 256, 0,
                                       (total + 255) / 256);
  if (blocks <= 0) return cudaErrorInvalidConfiguration;
  bucket_index_offset_kernel<<<blocks, 256, 0, s>>>(static_cast<int32_t*>(a.idx), total, b.k, buckets, b.M);
  return cudaGetLastError();
}

}  // namespace rtopk
