// MaxK backward scatter, sm_103a.
//
// Source: "MaxK-GNN: Extremely Fast GPU Kernel Design for Accelerating Graph
// Neural Networks Training", "How MaxK-GNN works" / "Asymmetric passes, one
// mask" and "Why it works": only the k kept features of a row carry gradient,
// at the positions (sp_index) recorded by the forward pass.
//
// The dense gradient is pure data movement bound by HBM writes: N x k x 4
// bytes in (bf16 values + int16 indices), N x M x 2 bytes out. A block takes
// a tile of consecutive rows, builds the tile in shared memory (zero, then
// scatter the k values of each row), and streams the tile out with 16-byte
// stores. Consecutive rows are contiguous in HBM, so a tile is one contiguous
// span and the output is written exactly once, with no separate zero-fill.
#include <cstdint>

#include "launch.h"

namespace rtopk {
namespace {

constexpr int kThreads = 256;
constexpr int kTileElems = 8192;  // 16 KB of bf16 per block
constexpr uint32_t kStatusBadIndex = 0x8u;

__device__ __forceinline__ void st_stream_u4(uint16_t* p, uint4 v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

__global__ void __launch_bounds__(kThreads)
maxk_backward_kernel(const uint16_t* __restrict__ dy, const int16_t* __restrict__ idx, int64_t N,
                     int M, int k, int rows_per_tile, bool vec, uint16_t* __restrict__ grad,
                     uint32_t* __restrict__ status) {
  __shared__ __align__(16) uint16_t tile[kTileElems];
  uint32_t st = 0;
  const int64_t ntiles = (N + rows_per_tile - 1) / rows_per_tile;
  for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x) {
    const int64_t r0 = t * rows_per_tile;
    const int64_t left = N - r0;
    const int rows = left < rows_per_tile ? int(left) : rows_per_tile;
    const int elems = rows * M;
    // zero the tile
    uint4* t4 = reinterpret_cast<uint4*>(tile);
    for (int i = threadIdx.x; i < (elems + 7) / 8; i += kThreads) t4[i] = make_uint4(0, 0, 0, 0);
    __syncthreads();
    // scatter the kept values of the tile's rows
    const int64_t e0 = r0 * int64_t(k);
    for (int i = threadIdx.x; i < rows * k; i += kThreads) {
      const int c = idx[e0 + i];
      if (c >= 0 && c < M) {
        tile[(i / k) * M + c] = dy[e0 + i];
      } else {
        st |= kStatusBadIndex;
      }
    }
    __syncthreads();
    // stream the tile out: one contiguous span of `elems` bf16
    uint16_t* out = grad + r0 * int64_t(M);
    if (vec) {
      for (int i = threadIdx.x; i < elems / 8; i += kThreads) st_stream_u4(out + 8 * i, t4[i]);
    } else {
      for (int i = threadIdx.x; i < elems; i += kThreads) out[i] = tile[i];
    }
    __syncthreads();
  }
  if (status != nullptr && st != 0u) atomicOr(status, st);
}

}  // namespace

cudaError_t launch_maxk_backward(const uint16_t* dy, const int16_t* idx, int64_t N, int M, int k,
                                 uint16_t* grad, uint32_t* status, cudaStream_t s) {
  const int rows_per_tile = kTileElems / M;  // M <= 8192, so at least one row
  // 16-byte stores need every tile span to start 16-byte aligned: M % 8 == 0
  const bool vec = (M % 8 == 0) && ((reinterpret_cast<uintptr_t>(grad) & 15u) == 0);
  const int64_t ntiles = (N + rows_per_tile - 1) / rows_per_tile;
  const int blocks = persistent_blocks(reinterpret_cast<const void*>(maxk_backward_kernel), kThreads,
                                       0, ntiles);
  if (blocks <= 0) return cudaErrorInvalidConfiguration;
  maxk_backward_kernel<<<blocks, kThreads, 0, s>>>(dy, idx, N, M, k, rows_per_tile, vec, grad, status);
  return cudaGetLastError();
}

}  // namespace rtopk
