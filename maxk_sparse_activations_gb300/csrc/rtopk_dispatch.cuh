// Instantiation and launch of the row-wise top-k kernels for one element type.
#pragma once

#include "launch.h"
#include "rtopk_select.cuh"
#include "rtopk_warp.cuh"

namespace rtopk {

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// One warp per row (W = 1): exact-mode and general loops, full and padded rows.
template <typename T, int G, typename IdxT>
cudaError_t launch_warp(const SelectArgs& a, bool full, bool vec, cudaStream_t s) {
  constexpr int kThreads = 256;
  const bool exact = a.max_iter < 0 && a.eps == 0.0f;
  auto kern = full ? (exact ? rtopk_warp_kernel<T, G, true, true, IdxT> : rtopk_warp_kernel<T, G, true, false, IdxT>)
                   : (exact ? rtopk_warp_kernel<T, G, false, true, IdxT> : rtopk_warp_kernel<T, G, false, false, IdxT>);
  const int blocks = persistent_blocks(reinterpret_cast<const void*>(kern), kThreads, 0, (a.N + 7) / 8);
  if (blocks <= 0) return cudaErrorInvalidConfiguration;
  kern<<<blocks, kThreads, 0, s>>>(static_cast<const T*>(a.in), a.N, a.M, a.k, a.max_iter, a.eps, vec,
                                   static_cast<T*>(a.vals), static_cast<IdxT*>(a.idx), a.iters, a.status);
  return cudaGetLastError();
}

// One 256-thread block per row (W = 8) for rows longer than 1024 elements.
template <typename T, int G, typename IdxT>
cudaError_t launch_block(const SelectArgs& a, bool full, bool vec, cudaStream_t s) {
  constexpr int kThreads = 256;
  auto kern = full ? rtopk_select_kernel<T, G, 8, true, IdxT> : rtopk_select_kernel<T, G, 8, false, IdxT>;
  const int blocks = persistent_blocks(reinterpret_cast<const void*>(kern), kThreads, 0, a.N);
  if (blocks <= 0) return cudaErrorInvalidConfiguration;
  kern<<<blocks, kThreads, 0, s>>>(static_cast<const T*>(a.in), a.N, a.M, a.k, a.max_iter, a.eps, vec,
                                   static_cast<T*>(a.vals), static_cast<IdxT*>(a.idx), a.iters, a.status);
  return cudaGetLastError();
}

// Row-length dispatch for rows <= 1024 elements (one warp per row).
template <typename T, typename IdxT>
cudaError_t launch_short_rows(const SelectArgs& a, cudaStream_t s) {
  constexpr int V = ElemTraits<T>::V;
  constexpr int GS = 32 * V;
  const int M = a.M;
  const bool vec = (M % V == 0) && aligned16(a.in);
  const int need = (M + GS - 1) / GS;
  const int G = need <= 4 ? need : (need <= 6 ? 6 : 8);
  const bool full = vec && M == G * GS;
  switch (G) {
    case 1: return launch_warp<T, 1, IdxT>(a, full, vec, s);
    case 2: return launch_warp<T, 2, IdxT>(a, full, vec, s);
    case 3: return launch_warp<T, 3, IdxT>(a, full, vec, s);
    case 4: return launch_warp<T, 4, IdxT>(a, full, vec, s);
    case 6:
      if constexpr (GS * 6 <= 1024 + GS) return launch_warp<T, 6, IdxT>(a, full, vec, s);
      return cudaErrorInvalidValue;
    default:
      if constexpr (GS * 8 <= 1024) return launch_warp<T, 8, IdxT>(a, full, vec, s);
      return cudaErrorInvalidValue;
  }
}

// Row-length dispatch for 1024 < M <= 8192 (one block per row).
template <typename T, typename IdxT>
cudaError_t launch_long_rows(const SelectArgs& a, cudaStream_t s) {
  constexpr int V = ElemTraits<T>::V;
  constexpr int GS = 32 * V * 8;  // elements per group across the block
  const int M = a.M;
  const bool vec = (M % V == 0) && aligned16(a.in);
  const int need = (M + GS - 1) / GS;
  const int G = need <= 4 ? need : (need <= 6 ? 6 : 8);
  const bool full = vec && M == G * GS;
  switch (G) {
    case 1: return launch_block<T, 1, IdxT>(a, full, vec, s);
    case 2: return launch_block<T, 2, IdxT>(a, full, vec, s);
    case 3: return launch_block<T, 3, IdxT>(a, full, vec, s);
    case 4: return launch_block<T, 4, IdxT>(a, full, vec, s);
    case 6:
      if constexpr (GS * 4 < 8192) return launch_block<T, 6, IdxT>(a, full, vec, s);
      return cudaErrorInvalidValue;
    default:
      if constexpr (GS * 4 < 8192) return launch_block<T, 8, IdxT>(a, full, vec, s);
      return cudaErrorInvalidValue;
  }
}

}  // namespace rtopk
