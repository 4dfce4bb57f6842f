// Bucketed approximate row-wise top-k, sm_103a.
//
// Source: "Approximate Top-k for Increased Parallelism" (abstract): relax
// exactness by splitting the vector into buckets and computing many smaller
// top-k selections independently.
//
// A row of M elements is split into B contiguous buckets of M / B; each bucket
// keeps its own top-(k / B) under the same selection as rtopk_select (exact by
// default, or early-stopped).
//  * Exact mode on full rows of 128..512 (B = 2, 4, 8): the lean kernel with
//    the row's B buckets on B lane groups of one warp, searched side by side
//    (rtopk_lean.cuh, process_row_bucketed); indices come out as row columns.
//    When each bucket keeps one or two elements (k / B <= 2, B = 2 .. 32)
//    there is no search: per-lane best elements merged by shuffles
//    (process_row_bucket_small).
//  * Otherwise: viewed as (N * B) rows of M / B elements, the matrix and the
//    CBSR output already have the layout of the smaller problem, so the
//    selection kernels run unchanged; one pass then turns bucket-local column
//    indices into row indices (+ bucket * M / B). Buckets are in column order
//    and each bucket's indices ascend, so every output row ascends.
#include <cstdint>

#include "rtopk_lean.cuh"
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

template <typename T, int NE, int B, bool SMALLB = false>
cudaError_t launch_lean_bucketed(const SelectArgs& a, cudaStream_t s) {
  auto kern = lean::rtopk_lean_kernel<T, NE, int32_t, B, false, SMALLB>;
  const int blocks = persistent_blocks(reinterpret_cast<const void*>(kern), 256, 0, (a.N + 7) / 8);
  if (blocks <= 0) return cudaErrorInvalidConfiguration;
  kern<<<blocks, 256, 0, s>>>(static_cast<const T*>(a.in), a.N, a.k, static_cast<T*>(a.vals),
                              static_cast<int32_t*>(a.idx), a.status);
  return cudaGetLastError();
}

// small (k / B <= 2): each bucket keeps its best one or two elements without
// a search; otherwise B in {2, 4, 8}: the buckets' searches side by side.
template <typename T, int NE>
cudaError_t launch_lean_b(const SelectArgs& a, int buckets, bool small, cudaStream_t s) {
  if (small) {
    switch (buckets) {
      case 2: return launch_lean_bucketed<T, NE, 2, true>(a, s);
      case 4: return launch_lean_bucketed<T, NE, 4, true>(a, s);
      case 8: return launch_lean_bucketed<T, NE, 8, true>(a, s);
      case 16: return launch_lean_bucketed<T, NE, 16, true>(a, s);
      default: return launch_lean_bucketed<T, NE, 32, true>(a, s);
    }
  }
  switch (buckets) {
    case 2: return launch_lean_bucketed<T, NE, 2>(a, s);
    case 4: return launch_lean_bucketed<T, NE, 4>(a, s);
    default: return launch_lean_bucketed<T, NE, 8>(a, s);
  }
}

// Exact mode, rows of 32 * NE elements (NE the lean kernel's slice sizes),
// 16-byte aligned, and B in {2, 4, 8, 16, 32} with k / B <= 2, or B in
// {2, 4, 8}: returns true and launches.
bool try_lean_bucketed(const SelectArgs& a, bool bf16, int buckets, cudaStream_t s, cudaError_t& err) {
  const bool exact = a.max_iter < 0 && a.eps == 0.0f;
  if (!exact || a.iters != nullptr || a.k > lean::kListK) return false;
  const bool pow2 = buckets == 2 || buckets == 4 || buckets == 8 || buckets == 16 || buckets == 32;
  const bool small = pow2 && a.k / buckets <= 2;
  if (!small && buckets != 2 && buckets != 4 && buckets != 8) return false;
  if ((reinterpret_cast<uintptr_t>(a.in) & 15u) != 0) return false;
  if (bf16) {
    switch (a.M) {
      case 128: err = launch_lean_b<uint16_t, 4>(a, buckets, small, s); return true;
      case 256: err = launch_lean_b<uint16_t, 8>(a, buckets, small, s); return true;
      case 512: err = launch_lean_b<uint16_t, 16>(a, buckets, small, s); return true;
      default: return false;
    }
  }
  switch (a.M) {
    case 128: err = launch_lean_b<float, 4>(a, buckets, small, s); return true;
    case 256: err = launch_lean_b<float, 8>(a, buckets, small, s); return true;
    case 384: err = launch_lean_b<float, 12>(a, buckets, small, s); return true;
    case 512: err = launch_lean_b<float, 16>(a, buckets, small, s); return true;
    default: return false;
  }
}

}  // namespace

cudaError_t launch_select_bucketed(const SelectArgs& a, int dtype_bf16, int buckets, cudaStream_t s) {
  cudaError_t err = cudaSuccess;
  if (buckets > 1 && try_lean_bucketed(a, dtype_bf16 != 0, buckets, s, err)) return err;
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
