// MaxK-GNN feature aggregation over CBSR, forward and backward, sm_103a.
//
// Source: "MaxK-GNN: Extremely Fast GPU Kernel Design for Accelerating Graph
// Neural Networks Training", "How MaxK-GNN works" (forward: row-wise-product
// SpGEMM over the compressed rows with shared-memory accumulation and one
// global write per row; backward: a sampled product whose output positions are
// the forward sp_index) and "Why it works" (each neighbour read shrinks from M
// to k values; scatter-accumulation stays on chip).
//
// Forward  out[i, m] = sum over the edges e of destination row i, in edge
//          order, of w_e * v for the CBSR entries (v, m) of source row col[e].
// Backward d_sp[j, t] = sum over the edges e of source row j (transposed
//          graph), in order, of w_e * dout[dst_e, sp_index[j, t]].
//
// Both kernels add in edge order with one rounding per product and per sum
// (__fmul_rn / __fadd_rn), so results are deterministic and bit-identical to
// the sequential binary32 definition -- except forward rows with more than
// 512 edges, which are summed in chunks (deterministic, within the binary32
// bound of the sequential sum). Forward: one warp per destination row
// with an M-float accumulator in shared memory; a source row's k indices are
// distinct, so the lanes of one edge never touch the same column and a
// __syncwarp between edges orders the updates. Edge lists are read 32 at a
// time (coalesced) and the CBSR rows of U edges are loaded before they are
// applied, so U gathers are in flight per warp. Rows with more than 512 edges
// (the heavy tail of power-law graphs) go to a second kernel that spreads
// each such row over the warps of one block. Backward: one warp per source
// row, lane t owns entry t, and the gathers of U edges are issued together.
#include <cstdint>

#include <cuda_bf16.h>

#include "launch.h"

namespace rtopk {
namespace {

constexpr uint32_t kStatusBadIndex = 0x8u;
constexpr uint32_t kStatusBadEdge = 0x10u;
constexpr int kThreads = 256;
#ifndef RTOPK_SPMM_U
#define RTOPK_SPMM_U 4  // k != 32 and the backward
#endif
#ifndef RTOPK_SPMM_HEAVY_WARPS
#define RTOPK_SPMM_HEAVY_WARPS 8
#endif
constexpr int kU = RTOPK_SPMM_U;  // edges whose rows are in flight together
// the same for the k == 32 loop (GB300, 2^17-node power-law graph: 576 /
// 497 / 582 us at 4 / 8 / 16)
constexpr int kU32 = 8;
constexpr int kHeavyThreads = 32 * RTOPK_SPMM_HEAVY_WARPS;  // warps sharing one heavy row
// Rows with more edges than this are split over the warps of one block.
constexpr int64_t kHeavyEdges = 512;

__device__ __forceinline__ float bf16f(uint16_t b) { return __uint_as_float(uint32_t(b) << 16); }

// Adds the edges [e0, e1) of one destination row into the warp's shared
// accumulator, in edge order (binary32, one rounding per product and sum).
template <int KS>
__device__ __forceinline__ void accumulate_edges(float* __restrict__ acc, const int32_t* __restrict__ col,
                                                 const float* __restrict__ w, int64_t e0, int64_t e1,
                                                 int64_t n_src, const uint16_t* __restrict__ sp_data,
                                                 const int16_t* __restrict__ sp_index, int M, int k, int lane,
                                                 uint32_t& st) {
  for (int64_t c0 = e0; c0 < e1; c0 += 32) {
    const int nc = (e1 - c0 < 32) ? int(e1 - c0) : 32;
    const int32_t cj = (lane < nc) ? col[c0 + lane] : 0;
    const float cw = (lane < nc) ? (w != nullptr ? w[c0 + lane] : 1.0f) : 0.0f;
    for (int u = 0; u < nc; u += kU) {
      float v[kU][KS];
      int c[kU][KS];
      float we[kU];
      bool okj[kU];
#pragma unroll
      for (int q = 0; q < kU; ++q) {
        const int64_t j = __shfl_sync(0xffffffffu, cj, (u + q) & 31);
        we[q] = __shfl_sync(0xffffffffu, cw, (u + q) & 31);
        okj[q] = (u + q < nc) && j >= 0 && j < n_src;
        if (u + q < nc && !okj[q]) st |= kStatusBadEdge;
#pragma unroll
        for (int s = 0; s < KS; ++s) {
          const int t = s * 32 + lane;
          if (okj[q] && t < k) {
            v[q][s] = bf16f(sp_data[j * k + t]);
            c[q][s] = sp_index[j * k + t];
          } else {
            v[q][s] = 0.0f;
            c[q][s] = -1;
          }
        }
      }
#pragma unroll
      for (int q = 0; q < kU; ++q) {
#pragma unroll
        for (int s = 0; s < KS; ++s) {
          const int t = s * 32 + lane;
          if (okj[q] && t < k) {
            const int m = c[q][s];
            if (m >= 0 && m < M) {
              acc[m] = __fadd_rn(acc[m], __fmul_rn(we[q], v[q][s]));
            } else {
              st |= kStatusBadIndex;
            }
          }
        }
        __syncwarp();
      }
    }
  }
}

// k == 32 (one CBSR entry per lane, the MaxK layer's shape): the same sums in
// the same order with no per-lane branch. A batch of 32 edges is validated
// once (a ballot of bad source rows; an edge is skipped with a warp-uniform
// test), the entries of U edges are loaded unconditionally (a skipped edge
// reads row 0, which exists because n_src > 0 is checked first), offsets are
// 32-bit when n_src * k fits, and a column index outside [0, M) is added into
// the accumulator's spare slot M instead of branching (and flagged). A full
// batch of valid edges (nearly all) runs without per-edge tests. GB300,
// 2^17-node power-law graph (8.05 M edges), M = 256: the forward (with the
// heavy rows) 1208 -> 497 us; 55 -> 30 warp-instructions per light edge, after
// which L1 / shared-memory throughput binds (77% of peak).
__device__ __forceinline__ void accumulate_edges_k32(float* __restrict__ acc, const int32_t* __restrict__ col,
                                                     const float* __restrict__ w, int64_t e0, int64_t e1,
                                                     int64_t n_src, const uint16_t* __restrict__ sp_data,
                                                     const int16_t* __restrict__ sp_index, int M, int lane,
                                                     uint32_t& st) {
  if (n_src <= 0) {
    if (e1 > e0) st |= kStatusBadEdge;
    return;
  }
  const bool off32 = n_src * 32 <= int64_t(0x7fffffff);
  bool bad_index = false;
  for (int64_t c0 = e0; c0 < e1; c0 += 32) {
    const int nc = (e1 - c0 < 32) ? int(e1 - c0) : 32;
    const int32_t cj = (lane < nc) ? col[c0 + lane] : 0;
    const float cw = (lane < nc) ? (w != nullptr ? w[c0 + lane] : 1.0f) : 0.0f;
    const bool bad_lane = lane < nc && !(cj >= 0 && cj < n_src);
    const unsigned bad = __ballot_sync(0xffffffffu, bad_lane);
    if (bad != 0u) st |= kStatusBadEdge;
    const int32_t cjs = bad_lane ? 0 : cj;  // a row that exists
    if (nc == 32 && bad == 0u) {
      // a full batch of valid edges (almost every batch): no per-edge tests
#pragma unroll 1
      for (int u = 0; u < 32; u += kU32) {
        uint16_t dv[kU32];
        int16_t di[kU32];
        float we[kU32];
#pragma unroll
        for (int q = 0; q < kU32; ++q) {
          const int32_t j = __shfl_sync(0xffffffffu, cjs, u + q);
          we[q] = __shfl_sync(0xffffffffu, cw, u + q);
          if (off32) {
            const uint32_t o = uint32_t(j) * 32u + uint32_t(lane);
            dv[q] = sp_data[o];
            di[q] = sp_index[o];
          } else {
            const int64_t o = int64_t(j) * 32 + lane;
            dv[q] = sp_data[o];
            di[q] = sp_index[o];
          }
        }
#pragma unroll
        for (int q = 0; q < kU32; ++q) {
          const uint32_t m = uint32_t(int32_t(di[q]));
          const bool in = m < uint32_t(M);
          bad_index |= !in;
          const uint32_t slot = in ? m : uint32_t(M);
          acc[slot] = __fadd_rn(acc[slot], __fmul_rn(we[q], bf16f(dv[q])));
          __syncwarp();
        }
      }
      continue;
    }
    for (int u = 0; u < nc; u += kU32) {
      uint16_t dv[kU32];
      int16_t di[kU32];
      float we[kU32];
#pragma unroll
      for (int q = 0; q < kU32; ++q) {
        const int32_t j = __shfl_sync(0xffffffffu, cjs, (u + q) & 31);
        we[q] = __shfl_sync(0xffffffffu, cw, (u + q) & 31);
        if (off32) {
          const uint32_t o = uint32_t(j) * 32u + uint32_t(lane);
          dv[q] = sp_data[o];
          di[q] = sp_index[o];
        } else {
          const int64_t o = int64_t(j) * 32 + lane;
          dv[q] = sp_data[o];
          di[q] = sp_index[o];
        }
      }
#pragma unroll
      for (int q = 0; q < kU32; ++q) {
        if (u + q < nc && !((bad >> ((u + q) & 31)) & 1u)) {  // warp-uniform
          const uint32_t m = uint32_t(int32_t(di[q]));
          const bool in = m < uint32_t(M);
          bad_index |= !in;
          const uint32_t slot = in ? m : uint32_t(M);
          acc[slot] = __fadd_rn(acc[slot], __fmul_rn(we[q], bf16f(dv[q])));
          __syncwarp();
        }
      }
    }
  }
  if (bad_index) st |= kStatusBadIndex;
}

__device__ __forceinline__ void zero_row(float* __restrict__ acc, int M, int lane, bool vec) {
  if (vec) {
    for (int m = lane * 4; m < M; m += 128) *reinterpret_cast<float4*>(acc + m) = make_float4(0.f, 0.f, 0.f, 0.f);
  } else {
    for (int m = lane; m < M; m += 32) acc[m] = 0.0f;
  }
}

// Destination rows with at most `heavy` edges: one warp per row, edges in
// order, rows round-robin over the warps (contiguous row ranges with equal
// edge counts per warp measured no faster on a power-law graph).
template <int KS>
__global__ void __launch_bounds__(kThreads)
spgemm_fwd_kernel(const int64_t* __restrict__ row_ptr, const int32_t* __restrict__ col,
                  const float* __restrict__ w, int64_t n_dst, int64_t n_src, const uint16_t* __restrict__ sp_data,
                  const int16_t* __restrict__ sp_index, int M, int k, int64_t heavy, bool vec,
                  float* __restrict__ out, uint32_t* __restrict__ status) {
  extern __shared__ __align__(16) float acc_all[];
  const int lane = threadIdx.x & 31;
  const int wib = threadIdx.x >> 5;
  const int wpb = blockDim.x >> 5;
  float* acc = acc_all + size_t(wib) * (M + 4);  // M columns + a spare slot, 16-byte aligned
  const int64_t nw = int64_t(gridDim.x) * wpb;
  uint32_t st = 0;
  for (int64_t i = int64_t(blockIdx.x) * wpb + wib; i < n_dst; i += nw) {
    const int64_t e0 = row_ptr[i], e1 = row_ptr[i + 1];
    if (e1 - e0 > heavy) continue;  // left to spgemm_heavy_kernel
    zero_row(acc, M, lane, vec);
    __syncwarp();
    if (KS == 1 && k == 32) {
      accumulate_edges_k32(acc, col, w, e0, e1, n_src, sp_data, sp_index, M, lane, st);
    } else {
      accumulate_edges<KS>(acc, col, w, e0, e1, n_src, sp_data, sp_index, M, k, lane, st);
    }
    float* o = out + i * int64_t(M);
    if (vec) {
      for (int m = lane * 4; m < M; m += 128) __stcs(reinterpret_cast<float4*>(o + m), *reinterpret_cast<const float4*>(acc + m));
    } else {
      for (int m = lane; m < M; m += 32) __stcs(o + m, acc[m]);
    }
    __syncwarp();
  }
  if (status != nullptr && st != 0u) atomicOr(status, st);
}

// Destination rows with more than `heavy` edges: one block (up to
// kHeavyThreads / 32 warps) per row. The row's edges are cut into W equal
// chunks (multiples of 32 edges); warp q adds chunk q, in edge order, into its
// own accumulator, and the W partial rows are then summed in warp order
// (fixed 512-edge chunks left most warps of a 600-edge row waiting at the
// barrier). Deterministic, but the terms of such a row are not added in plain
// edge order (the bound on the difference is in the C ABI header).
template <int KS>
__global__ void __launch_bounds__(kHeavyThreads)
spgemm_heavy_kernel(const int64_t* __restrict__ row_ptr, const int32_t* __restrict__ col,
                    const float* __restrict__ w, int64_t n_dst, int64_t n_src,
                    const uint16_t* __restrict__ sp_data, const int16_t* __restrict__ sp_index, int M, int k,
                    int64_t heavy, bool vec, float* __restrict__ out, uint32_t* __restrict__ status) {
  extern __shared__ __align__(16) float acc_all[];
  const int lane = threadIdx.x & 31;
  const int wib = threadIdx.x >> 5;
  const int wpb = blockDim.x >> 5;
  float* acc = acc_all + size_t(wib) * (M + 4);  // M columns + a spare slot, 16-byte aligned
  uint32_t st = 0;
  // every warp reads the same 32 row lengths, so the ballot is block-uniform
  for (int64_t i0 = int64_t(blockIdx.x) * 32; i0 < n_dst; i0 += int64_t(gridDim.x) * 32) {
    const int64_t il = i0 + lane;
    const bool is_heavy = il < n_dst && (row_ptr[il + 1] - row_ptr[il]) > heavy;
    unsigned todo = __ballot_sync(0xffffffffu, is_heavy);
    while (todo != 0u) {
    const int64_t i = i0 + (__ffs(todo) - 1);
    todo &= todo - 1u;
    const int64_t e0 = row_ptr[i], e1 = row_ptr[i + 1];
    zero_row(acc, M, lane, vec);
    __syncwarp();
    // the row's edges in wpb equal chunks (multiples of 32 edges): warp q adds
    // chunk q in edge order
    int64_t chunk = (e1 - e0 + wpb - 1) / wpb;
    chunk = (chunk + 31) & ~int64_t(31);
    const int64_t c0 = e0 + int64_t(wib) * chunk;
    const int64_t c1 = (e1 - c0 < chunk) ? e1 : c0 + chunk;
    if (c0 < c1) {
      if (KS == 1 && k == 32) {
        accumulate_edges_k32(acc, col, w, c0, c1, n_src, sp_data, sp_index, M, lane, st);
      } else {
        accumulate_edges<KS>(acc, col, w, c0, c1, n_src, sp_data, sp_index, M, k, lane, st);
      }
    }
    __syncthreads();
    float* o = out + i * int64_t(M);
    for (int m = threadIdx.x; m < M; m += blockDim.x) {
      float sum = acc_all[m];
      for (int q = 1; q < wpb; ++q) sum = __fadd_rn(sum, acc_all[size_t(q) * (M + 4) + m]);
      __stcs(o + m, sum);
    }
    __syncthreads();
    }
  }
  if (status != nullptr && st != 0u) atomicOr(status, st);
}

__device__ __forceinline__ void st_stream_u4(uint16_t* p, uint4 v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

// SCATTER = false: writes d_sp (n_src x k fp32). SCATTER = true: the MaxK
// backward scatter fused in -- writes the dense gradient row of the MaxK input
// instead, bf16(d_sp[j, t]) (round to nearest even) at column sp_index[j, t]
// and +0 elsewhere: each warp zeroes its shared slice of `row_stride` bf16,
// scatters its k values, and streams the row out (16-byte stores when `vec`).
template <int KS, bool SCATTER>
__global__ void __launch_bounds__(kThreads)
sspmm_bwd_kernel(const int64_t* __restrict__ t_ptr, const int32_t* __restrict__ t_row,
                 const float* __restrict__ t_w, int64_t n_src, int64_t n_dst, const float* __restrict__ dout,
                 const int16_t* __restrict__ sp_index, int M, int k, float* __restrict__ d_sp,
                 int row_stride, bool vec, uint16_t* __restrict__ grad, uint32_t* __restrict__ status) {
  extern __shared__ __align__(16) uint16_t grad_rows[];
  const int lane = threadIdx.x & 31;
  const int wib = threadIdx.x >> 5;
  const int wpb = blockDim.x >> 5;
  const int64_t nw = int64_t(gridDim.x) * wpb;
  uint32_t st = 0;
  for (int64_t j = int64_t(blockIdx.x) * wpb + wib; j < n_src; j += nw) {
    int c[KS];
    float acc[KS];
#pragma unroll
    for (int s = 0; s < KS; ++s) {
      const int t = s * 32 + lane;
      c[s] = (t < k) ? sp_index[j * k + t] : 0;
      if (t < k && (c[s] < 0 || c[s] >= M)) { st |= kStatusBadIndex; c[s] = -1; }
      acc[s] = 0.0f;
    }
    const int64_t e0 = t_ptr[j], e1 = t_ptr[j + 1];
    for (int64_t c0 = e0; c0 < e1; c0 += 32) {
      const int nc = (e1 - c0 < 32) ? int(e1 - c0) : 32;
      const int32_t ci = (lane < nc) ? t_row[c0 + lane] : 0;
      const float cw = (lane < nc) ? (t_w != nullptr ? t_w[c0 + lane] : 1.0f) : 0.0f;
      for (int u = 0; u < nc; u += kU) {
        float g[kU][KS], we[kU];
        bool oki[kU];
#pragma unroll
        for (int q = 0; q < kU; ++q) {
          const int64_t i = __shfl_sync(0xffffffffu, ci, (u + q) & 31);
          we[q] = __shfl_sync(0xffffffffu, cw, (u + q) & 31);
          oki[q] = (u + q < nc) && i >= 0 && i < n_dst;
          if (u + q < nc && !oki[q]) st |= kStatusBadEdge;
#pragma unroll
          for (int s = 0; s < KS; ++s) {
            const int t = s * 32 + lane;
            g[q][s] = (oki[q] && t < k && c[s] >= 0) ? __ldg(dout + i * int64_t(M) + c[s]) : 0.0f;
          }
        }
#pragma unroll
        for (int q = 0; q < kU; ++q)
#pragma unroll
          for (int s = 0; s < KS; ++s)
            if (oki[q]) acc[s] = __fadd_rn(acc[s], __fmul_rn(we[q], g[q][s]));
      }
    }
    if (!SCATTER) {
#pragma unroll
      for (int s = 0; s < KS; ++s) {
        const int t = s * 32 + lane;
        if (t < k) d_sp[j * k + t] = acc[s];
      }
    } else {
      uint16_t* srow = grad_rows + size_t(wib) * row_stride;
      uint4* s4 = reinterpret_cast<uint4*>(srow);
      for (int i = lane; i < row_stride / 8; i += 32) s4[i] = make_uint4(0u, 0u, 0u, 0u);
      __syncwarp();
#pragma unroll
      for (int s = 0; s < KS; ++s) {
        const int t = s * 32 + lane;
        if (t < k && c[s] >= 0) srow[c[s]] = __bfloat16_as_ushort(__float2bfloat16_rn(acc[s]));
      }
      __syncwarp();
      uint16_t* o = grad + j * int64_t(M);
      if (vec) {
        for (int i = lane; i < M / 8; i += 32) st_stream_u4(o + 8 * i, s4[i]);
      } else {
        for (int i = lane; i < M; i += 32) o[i] = srow[i];
      }
      __syncwarp();
    }
  }
  if (status != nullptr && st != 0u) atomicOr(status, st);
}

template <typename Kern>
cudaError_t launch_rows(Kern kern, int64_t rows, size_t smem_per_warp, cudaStream_t s, int& threads, int& blocks) {
  // warps per block limited by the shared accumulator (48 KB without opt-in)
  int wpb = kThreads / 32;
  if (smem_per_warp > 0) {
    const int fit = int((48 * 1024) / smem_per_warp);
    wpb = fit < wpb ? (fit < 1 ? 1 : fit) : wpb;
  }
  threads = wpb * 32;
  blocks = persistent_blocks(reinterpret_cast<const void*>(kern), threads, smem_per_warp * wpb,
                             (rows + wpb - 1) / wpb);
  return blocks > 0 ? cudaSuccess : cudaErrorInvalidConfiguration;
}

// Heavy rows: as many warps per block as the 48 KB of shared accumulators allow
// (up to kHeavyThreads / 32), one block per group of 32 rows.
template <typename Kern>
cudaError_t launch_heavy(Kern kern, int64_t rows, size_t smem_per_warp, int& threads, int& blocks) {
  int wpb = int((48 * 1024) / smem_per_warp);
  wpb = wpb > kHeavyThreads / 32 ? kHeavyThreads / 32 : (wpb < 1 ? 1 : wpb);
  threads = wpb * 32;
  // one block per 32-row group: a block meets only its group's heavy rows, so
  // the heavy rows of the graph spread over the SMs instead of queueing in a
  // persistent block; blocks of groups without one exit at once (2^17-node
  // power-law graph, 1118 rows > 512 edges: the forward 1207 -> 923 us)
  blocks = rows > 0x7fffffff ? 0x7fffffff : int(rows);
  (void)kern;
  return blocks > 0 ? cudaSuccess : cudaErrorInvalidConfiguration;
}

}  // namespace

cudaError_t launch_spgemm_fwd(const int64_t* row_ptr, const int32_t* col, const float* w, int64_t n_dst,
                              int64_t n_src, const uint16_t* sp_data, const int16_t* sp_index, int M, int k,
                              float* out, uint32_t* status, cudaStream_t s) {
  const int ks = (k + 31) / 32;
  const size_t smem_warp = size_t(M + 4) * sizeof(float);  // M columns + a spare slot, 16-byte aligned
  // 16-byte accumulator and output rows need M % 4 == 0 and an aligned output
  const bool vec = (M % 4 == 0) && ((reinterpret_cast<uintptr_t>(out) & 15u) == 0);
  int threads = 0, blocks = 0;
#define RTOPK_FWD(KS)                                                                                     \
  {                                                                                                       \
    cudaError_t e = launch_rows(spgemm_fwd_kernel<KS>, n_dst, smem_warp, s, threads, blocks);             \
    if (e != cudaSuccess) return e;                                                                       \
    spgemm_fwd_kernel<KS><<<blocks, threads, smem_warp * (threads / 32), s>>>(                            \
        row_ptr, col, w, n_dst, n_src, sp_data, sp_index, M, k, kHeavyEdges, vec, out, status);           \
    e = cudaGetLastError();                                                                               \
    if (e != cudaSuccess) return e;                                                                       \
    e = launch_heavy(spgemm_heavy_kernel<KS>, (n_dst + 31) / 32, smem_warp, threads, blocks);                         \
    if (e != cudaSuccess) return e;                                                                       \
    spgemm_heavy_kernel<KS><<<blocks, threads, smem_warp * (threads / 32), s>>>(                          \
        row_ptr, col, w, n_dst, n_src, sp_data, sp_index, M, k, kHeavyEdges, vec, out, status);           \
    return cudaGetLastError();                                                                            \
  }
  if (ks <= 1) RTOPK_FWD(1)
  if (ks <= 2) RTOPK_FWD(2)
  if (ks <= 4) RTOPK_FWD(4)
  RTOPK_FWD(8)
#undef RTOPK_FWD
}

cudaError_t launch_sspmm_bwd(const int64_t* t_ptr, const int32_t* t_row, const float* t_w, int64_t n_src,
                             int64_t n_dst, const float* dout, const int16_t* sp_index, int M, int k,
                             float* d_sp, uint16_t* grad, uint32_t* status, cudaStream_t s) {
  const int ks = (k + 31) / 32;
  int threads = 0, blocks = 0;
  // the fused scatter builds each row in a shared slice of M rounded up to 8 bf16
  const int row_stride = (M + 7) / 8 * 8;
  const size_t smem_warp = grad != nullptr ? size_t(row_stride) * 2 : 0;
  const bool vec = (M % 8 == 0) && ((reinterpret_cast<uintptr_t>(grad) & 15u) == 0);
#define RTOPK_BWD(KS, SC)                                                                                 \
  {                                                                                                       \
    cudaError_t e = launch_rows(sspmm_bwd_kernel<KS, SC>, n_src, smem_warp, s, threads, blocks);          \
    if (e != cudaSuccess) return e;                                                                       \
    sspmm_bwd_kernel<KS, SC><<<blocks, threads, smem_warp * (threads / 32), s>>>(                         \
        t_ptr, t_row, t_w, n_src, n_dst, dout, sp_index, M, k, d_sp, row_stride, vec, grad, status);      \
    return cudaGetLastError();                                                                            \
  }
  if (grad != nullptr) {
    if (ks <= 1) RTOPK_BWD(1, true)
    if (ks <= 2) RTOPK_BWD(2, true)
    if (ks <= 4) RTOPK_BWD(4, true)
    RTOPK_BWD(8, true)
  }
  if (ks <= 1) RTOPK_BWD(1, false)
  if (ks <= 2) RTOPK_BWD(2, false)
  if (ks <= 4) RTOPK_BWD(4, false)
  RTOPK_BWD(8, false)
#undef RTOPK_BWD
}

}  // namespace rtopk
