// Instantiation and launch of the row-wise top-k kernels for one element type.
#pragma once

#include "launch.h"
#include "rtopk_select.cuh"
#include "rtopk_block.cuh"
#include "rtopk_cluster.cuh"
#include "rtopk_lean.cuh"

namespace rtopk {

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

#ifndef RTOPK_LEAN_NE_MAX
#define RTOPK_LEAN_NE_MAX 32  // elements per lane of the largest rows the lean kernel takes
#endif

// Exact rows of 32 * NE elements without pass counts: the lean kernel
// (rtopk_lean.cuh).
template <typename T, int NE, typename IdxT>
cudaError_t launch_lean(const SelectArgs& a, cudaStream_t s) {
  constexpr int kThreads = 256;
  auto kern = lean::rtopk_lean_kernel<T, NE, IdxT>;
  if constexpr (lean::kGuessRows<T, NE>) {
    if (a.k > 32) kern = lean::rtopk_lean_kernel<T, NE, IdxT, 1, true>;
  }
  const int blocks = persistent_blocks(reinterpret_cast<const void*>(kern), kThreads, 0, (a.N + 7) / 8);
  if (blocks <= 0) return cudaErrorInvalidConfiguration;
  kern<<<blocks, kThreads, 0, s>>>(static_cast<const T*>(a.in), a.N, a.k, static_cast<T*>(a.vals),
                                   static_cast<IdxT*>(a.idx), a.status);
  return cudaGetLastError();
}

// Full rows of 32 * NE elements in replay mode: rtopk_lean_replay_kernel.
template <typename T, int NE, typename IdxT>
cudaError_t launch_lean_replay(const SelectArgs& a, cudaStream_t s) {
  constexpr int kThreads = 256;
  auto kern = lean::rtopk_lean_replay_kernel<T, NE, IdxT>;
  const int blocks = persistent_blocks(reinterpret_cast<const void*>(kern), kThreads, 0, (a.N + 7) / 8);
  if (blocks <= 0) return cudaErrorInvalidConfiguration;
  kern<<<blocks, kThreads, 0, s>>>(static_cast<const T*>(a.in), a.N, a.k, a.max_iter, a.eps,
                                   static_cast<T*>(a.vals), static_cast<IdxT*>(a.idx), a.iters, a.status);
  return cudaGetLastError();
}

// One warp per row (W = 1). L = compaction list entries per lane (0 = off).
// Measured on GB300 (2^18 N(0,1) rows): compaction costs more than it saves
// while a lane holds few elements (M = 256: 187 vs 160 us), and pays from 32
// elements per lane (M = 1024, k = 32: 358 vs 392 us with L = 4; M = 2048,
// k = 64: 849 vs 917 us with L = 8).
template <typename T, int G, typename IdxT>
cudaError_t launch_warp(const SelectArgs& a, bool full, bool vec, cudaStream_t s) {
  constexpr int kThreads = 256;
  constexpr int NE = G * ElemTraits<T>::V;
  const bool exact = a.max_iter < 0 && a.eps == 0.0f;
  if constexpr (NE <= RTOPK_LEAN_NE_MAX) {
    // exact mode without pass counts on full rows: the search counts on
    // packed 16-bit images of the row (rtopk_lean.cuh)
    if (exact && a.iters == nullptr && full && a.k <= lean::kListK) return launch_lean<T, NE, IdxT>(a, s);
    // early stop / eps on full rows: the replay on the same row ring (GB300,
    // 2^20 x 256 fp32, k = 32: max_iter = 2 494 -> 396 us, max_iter = 5 617 ->
    // 505 us). Exact mode with pass counts stays on the binary32 warp kernel,
    // whose exact-threshold exit is cheaper than the replay's general fill
    // (589 against 626 us).
    if (!exact && full && a.k <= lean::kListK) return launch_lean_replay<T, NE, IdxT>(a, s);
  }
  const int L = (NE >= 64 && a.k <= 128) ? 8 : ((NE >= 32 && a.k <= 64) ? 4 : 0);
  using K = void (*)(const T*, int64_t, int, int, int, float, bool, bool, T*, IdxT*, int*, uint32_t*);
  K kern;
  if (L == 4) {
    kern = exact ? rtopk_warp_kernel<T, G, true, (NE >= 32 ? 4 : 0), IdxT>
                 : rtopk_warp_kernel<T, G, false, (NE >= 32 ? 4 : 0), IdxT>;
  } else if (L == 8) {
    kern = exact ? rtopk_warp_kernel<T, G, true, (NE >= 64 ? 8 : 0), IdxT>
                 : rtopk_warp_kernel<T, G, false, (NE >= 64 ? 8 : 0), IdxT>;
  } else {
    kern = exact ? rtopk_warp_kernel<T, G, true, 0, IdxT> : rtopk_warp_kernel<T, G, false, 0, IdxT>;
  }
  const int blocks = persistent_blocks(reinterpret_cast<const void*>(kern), kThreads, 0, (a.N + 7) / 8);
  if (blocks <= 0) return cudaErrorInvalidConfiguration;
  kern<<<blocks, kThreads, 0, s>>>(static_cast<const T*>(a.in), a.N, a.M, a.k, a.max_iter, a.eps, full, vec,
                                   static_cast<T*>(a.vals), static_cast<IdxT*>(a.idx), a.iters, a.status);
  return cudaGetLastError();
}

// One 256-thread block per row for rows longer than kWarpMaxM elements. Once
// c(lo) fits the shared list, the search tail runs on the list: warp 0 alone
// for lists of <= 256 (k <= 128), all warps for lists of <= 2048 (k <= 1024).
template <typename T, int G, typename IdxT>
cudaError_t launch_block(const SelectArgs& a, bool full, bool vec, cudaStream_t s) {
  constexpr int kThreads = 256;
  const bool exact = a.max_iter < 0 && a.eps == 0.0f;
  const int LB = (a.k <= 128) ? 8 : (a.k <= 1024 ? 64 : 0);
  using K = void (*)(const T*, int64_t, int, int, int, float, bool, bool, T*, IdxT*, int*, uint32_t*);
  K kern;
  if (LB == 8) {
    kern = exact ? rtopk_block_kernel<T, G, true, 8, IdxT> : rtopk_block_kernel<T, G, false, 8, IdxT>;
  } else if (LB == 64) {
    kern = exact ? rtopk_block_kernel<T, G, true, 64, IdxT> : rtopk_block_kernel<T, G, false, 64, IdxT>;
  } else {
    kern = exact ? rtopk_block_kernel<T, G, true, 0, IdxT> : rtopk_block_kernel<T, G, false, 0, IdxT>;
  }
  const int blocks = persistent_blocks(reinterpret_cast<const void*>(kern), kThreads, 0, a.N);
  if (blocks <= 0) return cudaErrorInvalidConfiguration;
  kern<<<blocks, kThreads, 0, s>>>(static_cast<const T*>(a.in), a.N, a.M, a.k, a.max_iter, a.eps, full, vec,
                                   static_cast<T*>(a.vals), static_cast<IdxT*>(a.idx), a.iters, a.status);
  return cudaGetLastError();
}

// Row-length dispatch for rows <= kWarpMaxM elements (one warp per row).
#ifndef RTOPK_WARP_MAX_M
#define RTOPK_WARP_MAX_M 2048
#endif
constexpr int kWarpMaxM = RTOPK_WARP_MAX_M;
template <typename T, typename IdxT>
cudaError_t launch_short_rows(const SelectArgs& a, cudaStream_t s) {
  constexpr int V = ElemTraits<T>::V;
  constexpr int GS = 32 * V;
  const int M = a.M;
  const bool vec = (M % V == 0) && aligned16(a.in);
  if constexpr (sizeof(T) == 2) {
    // bf16 rows of 128 (4 per lane, 8 bytes): the lean kernel in exact mode,
    // its replay for early stop / eps
    const bool exact = a.max_iter < 0 && a.eps == 0.0f;
    if (M == 128 && vec && exact && a.iters == nullptr && a.k <= lean::kListK) return launch_lean<T, 4, IdxT>(a, s);
    if (M == 128 && vec && !exact && a.k <= lean::kListK) return launch_lean_replay<T, 4, IdxT>(a, s);
  }
  const int need = (M + GS - 1) / GS;
  const int G = need <= 4 ? need : (need <= 6 ? 6 : (need <= 8 ? 8 : (need <= 12 ? 12 : 16)));
  const bool full = vec && M == G * GS;
  switch (G) {
    case 1: return launch_warp<T, 1, IdxT>(a, full, vec, s);
    case 2: return launch_warp<T, 2, IdxT>(a, full, vec, s);
    case 3: return launch_warp<T, 3, IdxT>(a, full, vec, s);
    case 4: return launch_warp<T, 4, IdxT>(a, full, vec, s);
    case 6: return launch_warp<T, 6, IdxT>(a, full, vec, s);
    case 8: return launch_warp<T, 8, IdxT>(a, full, vec, s);
    case 12:
      if constexpr (GS * 12 <= kWarpMaxM) return launch_warp<T, 12, IdxT>(a, full, vec, s);
      return cudaErrorInvalidValue;
    default:
      if constexpr (GS * 16 <= kWarpMaxM) return launch_warp<T, 16, IdxT>(a, full, vec, s);
      return cudaErrorInvalidValue;
  }
}

// Row-length dispatch for kWarpMaxM < M <= 8192 (one block per row).
template <typename T, typename IdxT>
cudaError_t launch_long_rows(const SelectArgs& a, cudaStream_t s) {
  constexpr int V = ElemTraits<T>::V;
  constexpr int GS = 32 * V * kBlockWarps;  // elements per group across the block
  const int M = a.M;
  const bool vec = (M % V == 0) && aligned16(a.in);
  const int need = (M + GS - 1) / GS;
  const int G = need <= 4 ? need : (need <= 6 ? 6 : 8);
  const bool full = vec && M == G * GS;
  switch (G) {
    case 1:
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

// Rows of 8193..65536 elements: one cluster of C CTAs per row, NE elements per
// lane (8 warps x 32 lanes x NE per CTA). The kernel is bound by the latency of
// its exchange rounds, so what counts is how many rows are in flight: measured
// on GB300 (fp32, k = 256), rows of 16384 run best as 2 CTAs x 32 elements at 3
// CTAs per SM (929 us for 2^14 rows), rows of 32768 / 65536 as 2 / 4 CTAs x 64
// elements (843 / 912 us for 2^13 / 2^12 rows; 1020 / 1250 us with 32 elements).
template <typename T, int C, int NE, typename IdxT>
cudaError_t launch_cluster_c(const SelectArgs& a, cudaStream_t s) {
  constexpr int V = ElemTraits<T>::V;
  constexpr int G = NE / V;
  constexpr int kRow = C * kBlockWarps * 32 * NE;
  const bool vec = (a.M % V == 0) && aligned16(a.in);
  const bool full = vec && a.M == kRow;
  const bool exact = a.max_iter < 0 && a.eps == 0.0f;
  using K = void (*)(const T*, int64_t, int, int, int, float, bool, bool, T*, IdxT*, int*, uint32_t*);
  K kern = exact ? rtopk_cluster_kernel<T, G, true, C, IdxT> : rtopk_cluster_kernel<T, G, false, C, IdxT>;
  const int clusters = persistent_clusters(reinterpret_cast<const void*>(kern), 256, C, a.N);
  if (clusters <= 0) return cudaErrorInvalidConfiguration;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = unsigned(C);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(unsigned(clusters * C));
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<const T*>(a.in), a.N, a.M, a.k, a.max_iter, a.eps, full, vec,
                            static_cast<T*>(a.vals), static_cast<IdxT*>(a.idx), a.iters, a.status);
}

template <typename T, typename IdxT>
cudaError_t launch_cluster_rows(const SelectArgs& a, cudaStream_t s) {
  if (a.M <= 2 * 8192) return launch_cluster_c<T, 2, 32, IdxT>(a, s);
  if (a.M <= 2 * 16384) return launch_cluster_c<T, 2, 64, IdxT>(a, s);
  if (a.M <= 4 * 16384) return launch_cluster_c<T, 4, 64, IdxT>(a, s);
  return cudaErrorInvalidValue;
}

}  // namespace rtopk
