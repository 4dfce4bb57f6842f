// Instantiation and launch of rtopk_select_kernel for one element type.
#pragma once

#include "launch.h"
#include "rtopk_select.cuh"

namespace rtopk {

template <typename T, int G, int W, typename IdxT>
cudaError_t launch_config(const SelectArgs& a, bool full, bool vec, cudaStream_t s) {
  static_assert(W == 1 || W == 8, "a team is one warp or the whole 256-thread block");
  constexpr int kThreads = 256;
  constexpr int kTeams = kThreads / (32 * W);
  auto kern = full ? rtopk_select_kernel<T, G, W, true, IdxT> : rtopk_select_kernel<T, G, W, false, IdxT>;
  const int blocks = persistent_blocks(reinterpret_cast<const void*>(kern), kThreads, 0,
                                       (a.N + kTeams - 1) / kTeams);
  if (blocks <= 0) return cudaErrorInvalidConfiguration;
  kern<<<blocks, kThreads, 0, s>>>(static_cast<const T*>(a.in), a.N, a.M, a.k, a.max_iter, a.eps, vec,
                                   static_cast<T*>(a.vals), static_cast<IdxT*>(a.idx), a.iters, a.status);
  return cudaGetLastError();
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace rtopk
