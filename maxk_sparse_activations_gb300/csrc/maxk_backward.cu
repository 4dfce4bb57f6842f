// MaxK backward scatter, sm_103a.
//
// Source: "MaxK-GNN: Extremely Fast GPU Kernel Design for Accelerating Graph
// Neural Networks Training", "How MaxK-GNN works" / "Asymmetric passes, one
// mask" and "Why it works": only the k kept features of a row carry gradient,
// at the positions (sp_index) recorded by the forward pass.
//
// The dense gradient is pure data movement bound by HBM writes: N x k x 4
// bytes in (bf16 values + int16 indices), N x M x 2 bytes out, every output
// byte written exactly once (no separate zero-fill).
//
// Rows of at most 2048 elements with k <= 256 (the MaxK layer's shapes): one
// warp per group of R consecutive rows (R * M <= 2048, R * k <= 256, R <= 8),
// persistent over groups. The group's gradient block lives in the warp's own
// shared buffer: every lane zeroes 16-byte chunks, writes the values of its
// (index, value) pairs, and every lane streams 16-byte chunks out. Only
// __syncwarp orders the three steps, and the next group's pairs are already
// in registers (loaded before the current group is written), so a warp waits
// on neither a block barrier nor a dependent load.
// Other shapes: a block builds a tile of consecutive rows in shared memory
// (zero, scatter, barrier, stream out).
#include <cstdint>

#include "launch.h"

namespace rtopk {
namespace {

constexpr int kThreads = 256;
constexpr int kTileElems = 8192;  // 16 KB of bf16 per block (tile kernel)
constexpr int kWarpMaxM = 2048;   // warp kernel: groups of at most 2048 elements (4 KB)
constexpr int kWarpMaxK = 256;    // warp kernel: at most 256 pairs per group (8 per lane)
constexpr uint32_t kStatusBadIndex = 0x8u;

__device__ __forceinline__ void st_stream_u4(uint16_t* p, uint4 v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}
__device__ __forceinline__ int16_t ld_stream_s16(const int16_t* p) {
  short v;
  asm volatile("ld.global.nc.L1::no_allocate.s16 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ uint16_t ld_stream_u16(const uint16_t* p) {
  unsigned short v;
  asm volatile("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}

// One warp per group of R consecutive rows (M % 8 == 0, R * M <= 2048,
// R * k <= 256, grad 16-byte aligned), persistent over groups. The group's
// R * k (index, value) pairs are one contiguous block of both arrays: lane l
// takes entries [8 l, 8 l + 8) with one 16-byte load per array when k % 8 == 0
// (VEC), else entries l, l + 32, ... with 2-byte loads. The next group's pairs
// are loaded before the current group is written.
template <bool VEC>
__global__ void __launch_bounds__(kThreads)
maxk_backward_warp_kernel(const uint16_t* __restrict__ dy, const int16_t* __restrict__ idx, int64_t N, int M,
                          int k, int R, uint16_t* __restrict__ grad, uint32_t* __restrict__ status) {
  extern __shared__ __align__(16) uint16_t groupbuf_all[];
  constexpr int EP = 8;  // pairs per lane and group
  const int lane = threadIdx.x & 31;
  const int wib = threadIdx.x >> 5;
  const int GE = R * M;     // elements of a group's gradient block
  uint16_t* buf = groupbuf_all + wib * GE;
  uint4* buf4 = reinterpret_cast<uint4*>(buf);
  const int chunks = GE >> 3;  // 16-byte chunks per group
  const int64_t ngroups = (N + R - 1) / R;
  const int64_t nw = int64_t(gridDim.x) * (kThreads / 32);
  uint32_t st = 0;
  int64_t g = int64_t(blockIdx.x) * (kThreads / 32) + wib;
  int16_t c[EP];
  uint16_t v[EP];
  int ne = 0;  // valid entries of the fetched group
  // entry e of group gg: row gg * R + e / k, pair e % k
  auto fetch = [&](int64_t gg) {
    const int64_t rows = gg < ngroups ? (N - gg * R < R ? N - gg * R : R) : 0;
    ne = int(rows) * k;
    const int64_t e0 = gg * int64_t(R) * k;
    if (VEC) {
      if (lane * EP < ne) {  // k % 8 == 0: whole 16-byte chunks
        const uint4 ci = *reinterpret_cast<const uint4*>(idx + e0 + lane * EP);
        const uint4 vi = *reinterpret_cast<const uint4*>(dy + e0 + lane * EP);
        const uint32_t cw[4] = {ci.x, ci.y, ci.z, ci.w}, vw[4] = {vi.x, vi.y, vi.z, vi.w};
#pragma unroll
        for (int q = 0; q < EP; ++q) {
          c[q] = int16_t((q & 1) ? (cw[q / 2] >> 16) : (cw[q / 2] & 0xffffu));
          v[q] = uint16_t((q & 1) ? (vw[q / 2] >> 16) : (vw[q / 2] & 0xffffu));
        }
      }
    } else {
#pragma unroll
      for (int q = 0; q < EP; ++q) {
        const int e = lane + 32 * q;
        if (e < ne) {
          c[q] = ld_stream_s16(idx + e0 + e);
          v[q] = ld_stream_u16(dy + e0 + e);
        }
      }
    }
  };
  // VEC: k % 8 == 0, so a lane's 8 entries [8 l, 8 l + 8) lie in one row of
  // every group; its offset in the group block is fixed
  const int vrow_off = VEC ? ((lane * EP) / k) * M : 0;
  fetch(g);
  for (; g < ngroups; g += nw) {
    int16_t cc[EP];
    uint16_t vv[EP];
#pragma unroll
    for (int q = 0; q < EP; ++q) {
      cc[q] = c[q];
      vv[q] = v[q];
    }
    const int nec = ne;
    fetch(g + nw);  // the next group's pairs, in flight while this group is written
    for (int i = lane; i < chunks; i += 32) buf4[i] = make_uint4(0, 0, 0, 0);
    __syncwarp();
#pragma unroll
    for (int q = 0; q < EP; ++q) {
      const int e = VEC ? lane * EP + q : lane + 32 * q;
      if (e < nec) {
        const int off = VEC ? vrow_off : (e / k) * M;
        if (cc[q] >= 0 && cc[q] < M) {
          buf[off + cc[q]] = vv[q];
        } else {
          st |= kStatusBadIndex;
        }
      }
    }
    __syncwarp();
    const int64_t rows = N - g * R < R ? N - g * R : R;
    const int nch = int(rows) * (M >> 3);
    uint16_t* out = grad + g * int64_t(R) * M;
    for (int i = lane; i < nch; i += 32) st_stream_u4(out + 8 * i, buf4[i]);
    __syncwarp();
  }
  if (status != nullptr && st != 0u) atomicOr(status, st);
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
  // 16-byte stores need every row (or tile span) to start 16-byte aligned: M % 8 == 0
  const bool vec = (M % 8 == 0) && ((reinterpret_cast<uintptr_t>(grad) & 15u) == 0);
  if (vec && M <= kWarpMaxM && k <= kWarpMaxK) {
    // rows per warp iteration: a group block of at most 4 KB and 256 pairs
    int R = kWarpMaxM / M;
    if (R > kWarpMaxK / k) R = kWarpMaxK / k;
    if (R > 8) R = 8;
    const size_t smem = size_t(kThreads / 32) * size_t(R) * size_t(M) * 2;
    const int64_t ngroups = (N + R - 1) / R;
    // 16-byte pair loads need every group block to start 16-byte aligned
    const bool vpairs = (k % 8 == 0) && ((reinterpret_cast<uintptr_t>(idx) | reinterpret_cast<uintptr_t>(dy)) & 15u) == 0;
    auto launch = [&](auto kern) -> cudaError_t {
      const int blocks = persistent_blocks(reinterpret_cast<const void*>(kern), kThreads, smem, (ngroups + 7) / 8);
      if (blocks <= 0) return cudaErrorInvalidConfiguration;
      kern<<<blocks, kThreads, smem, s>>>(dy, idx, N, M, k, R, grad, status);
      return cudaGetLastError();
    };
    return vpairs ? launch(maxk_backward_warp_kernel<true>) : launch(maxk_backward_warp_kernel<false>);
  }
  const int rows_per_tile = kTileElems / M;  // M <= 8192, so at least one row
  const int64_t ntiles = (N + rows_per_tile - 1) / rows_per_tile;
  const int blocks = persistent_blocks(reinterpret_cast<const void*>(maxk_backward_kernel), kThreads,
                                       0, ntiles);
  if (blocks <= 0) return cudaErrorInvalidConfiguration;
  maxk_backward_kernel<<<blocks, kThreads, 0, s>>>(dy, idx, N, M, k, rows_per_tile, vec, grad, status);
  return cudaGetLastError();
}

}  // namespace rtopk
