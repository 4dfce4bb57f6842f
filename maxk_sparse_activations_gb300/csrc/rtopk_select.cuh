// Row-wise top-k by per-row threshold bisection (RTop-K), sm_103a.
//
// Source: "RTop-K: Ultra-Fast Row-Wise Top-K Selection for Neural Network
// Acceleration on GPUs" (summary page), "Approach": a binary search over each
// row's value range finds a threshold that selects k elements, warp primitives
// count the elements above a candidate threshold, an optional cap on the number
// of passes stops early, and a second pass from the lower bound fills the
// borderline ties. Output layout: "MaxK-GNN: Extremely Fast GPU Kernel Design
// for Accelerating Graph Neural Networks Training", "How MaxK-GNN works" / "The
// idea" (exactly k survivors per row: dense N x k values + N x k indices).
//
// Mapping. A "team" of W warps owns one row at a time; the grid is persistent
// and teams stride over rows. Each lane holds V consecutive elements (16 bytes
// of input) of each of G groups; a group is 32 * V consecutive elements, so a
// warp covers G * 32 * V elements and a team covers W times that. Element j of
// the row sits in warp w, group g, lane l, slot e with
//     j = (w * G + g) * 32 * V + l * V + e.
// The row lives in registers for the whole search: it is read from HBM once
// (16-byte streaming loads), and every pass of the bisection re-reads
// registers only. W = 1 serves rows up to 1024 elements; W = 8 (one row per
// 256-thread block, counts combined through shared memory) serves longer rows.
//
// Arithmetic matches the replay of the method exactly: the midpoint is
// __fmul_rn(__fadd_rn(lo, hi), 0.5f), the precision test is
// __fsub_rn(hi, lo) > eps, comparisons are IEEE (-0 == +0, subnormals kept:
// the library is built without fast-math and without flush-to-zero), and
// counts are exact integers, so every pass takes the same branch as the
// scalar definition and the kept set is bit-identical.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "rtopk_device.cuh"

namespace rtopk {

// Passes after which a search is abandoned and flagged. A valid row (finite,
// |x| <= 1e38) needs fewer than 300: each pass halves a range of at most 2e38
// and the search ends once no binary32 value lies strictly inside it.
constexpr int kSafetyCap = 512;
constexpr uint32_t kStatusNonFinite = 0x1u;
constexpr uint32_t kStatusRange = 0x2u;
constexpr uint32_t kStatusSafetyCap = 0x4u;

template <typename T>
struct ElemTraits;
template <>
struct ElemTraits<float> {
  static constexpr int V = 4;  // 4 x fp32 = 16 bytes per lane per group
};
template <>
struct ElemTraits<uint16_t> {
  static constexpr int V = 8;  // 8 x bf16 = 16 bytes per lane per group
};

// Raw bits of a kept value for the output array (bit copy of the input).
__device__ __forceinline__ float out_value(float x, float*) { return x; }
__device__ __forceinline__ uint16_t out_value(float x, uint16_t*) {
  return static_cast<uint16_t>(__float_as_uint(x) >> 16);  // exact: x was widened from bf16
}

// ---------------------------------------------------------------------------
// Row load into registers. FULL: the row is exactly G * 32 * V * W elements
// and 16-byte aligned. Otherwise slots past M hold -inf, which no threshold
// counts and no bound admits; `vec` says 16-byte loads are legal slot by slot.
// ---------------------------------------------------------------------------
template <int G, int W, bool FULL>
__device__ __forceinline__ void load_row(const float* __restrict__ row, int M, int w, int lane,
                                         bool vec, float (&x)[G][4]) {
#pragma unroll
  for (int g = 0; g < G; ++g) {
    const int j0 = (w * G + g) * 128 + lane * 4;
    if (FULL) {
      float4 v = ld_stream_f4(row + j0);
      x[g][0] = v.x; x[g][1] = v.y; x[g][2] = v.z; x[g][3] = v.w;
    } else if (vec) {
      if (j0 < M) {  // M % 4 == 0: the 4 slots are all in or all out
        float4 v = ld_stream_f4(row + j0);
        x[g][0] = v.x; x[g][1] = v.y; x[g][2] = v.z; x[g][3] = v.w;
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) x[g][e] = neg_inf();
      }
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e) x[g][e] = (j0 + e < M) ? ld_stream_f1(row + j0 + e) : neg_inf();
    }
  }
}

template <int G, int W, bool FULL>
__device__ __forceinline__ void load_row(const uint16_t* __restrict__ row, int M, int w, int lane,
                                         bool vec, float (&x)[G][8]) {
#pragma unroll
  for (int g = 0; g < G; ++g) {
    const int j0 = (w * G + g) * 256 + lane * 8;
    if (FULL || (vec && j0 < M)) {
      uint4 u = ld_stream_u4(row + j0);
      const uint32_t wd[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        x[g][2 * q] = __uint_as_float(wd[q] << 16);              // element at the lower address
        x[g][2 * q + 1] = __uint_as_float(wd[q] & 0xffff0000u);  // element at the higher address
      }
    } else if (vec) {
#pragma unroll
      for (int e = 0; e < 8; ++e) x[g][e] = neg_inf();
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e)
        x[g][e] = (j0 + e < M) ? __uint_as_float(uint32_t(ld_stream_u1(row + j0 + e)) << 16)
                               : neg_inf();
    }
  }
}

// ---------------------------------------------------------------------------
// Team-wide reductions. W == 1: warp reductions only. W > 1: per-warp results
// meet in shared memory; `slot` alternates so one barrier per call suffices.
// ---------------------------------------------------------------------------
template <int W>
struct TeamShared {
  int cnt[2][W];
  int omax[W];
  int omin[W];
  int tot[W][2];
};
template <>
struct TeamShared<1> {};

template <int W>
__device__ __forceinline__ int team_sum(int v, int w, int lane, int& slot, TeamShared<W>& sh) {
  int s = (int)__reduce_add_sync(0xffffffffu, (unsigned)v);
  if constexpr (W == 1) {
    return s;
  } else {
    if (lane == 0) sh.cnt[slot][w] = s;
    __syncthreads();
    int t = 0;
#pragma unroll
    for (int i = 0; i < W; ++i) t += sh.cnt[slot][i];
    slot ^= 1;
    return t;
  }
}

template <int W>
__device__ __forceinline__ void team_minmax(int& omn, int& omx, int w, int lane, TeamShared<W>& sh) {
  omx = __reduce_max_sync(0xffffffffu, omx);
  omn = __reduce_min_sync(0xffffffffu, omn);
  if constexpr (W > 1) {
    if (lane == 0) { sh.omax[w] = omx; sh.omin[w] = omn; }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < W; ++i) { omx = max(omx, sh.omax[i]); omn = min(omn, sh.omin[i]); }
  }
}

template <int G, int V>
__device__ __forceinline__ int lane_count_ge(const float (&x)[G][V], float t) {
  int c = 0;
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int e = 0; e < V; ++e) c += (x[g][e] >= t) ? 1 : 0;
  return c;
}

// ---------------------------------------------------------------------------
// The kernel.
// ---------------------------------------------------------------------------
template <typename T, int G, int W, bool FULL, typename IdxT>
__global__ void __launch_bounds__(256)
rtopk_select_kernel(const T* __restrict__ in, int64_t N, int M, int k, int max_iter, float eps,
                    bool vec, T* __restrict__ vals, IdxT* __restrict__ idx,
                    int* __restrict__ iters, uint32_t* __restrict__ status) {
  constexpr int V = ElemTraits<T>::V;
  constexpr int GS = 32 * V;                // elements per group
  constexpr int FB = (GS <= 255) ? 8 : 16;  // bits per packed prefix-count field
  constexpr int FPW = 32 / FB;              // fields per 32-bit word
  constexpr int NF = 2 * G;                 // fields: (S count, B count) per group
  constexpr int NW = (NF + FPW - 1) / FPW;  // packed words
  constexpr unsigned FMASK = (1u << FB) - 1u;
  constexpr int TEAMS = 256 / (32 * W);     // teams per 256-thread block

  __shared__ TeamShared<W> sh;

  const int lane = threadIdx.x & 31;
  const int warp_in_block = threadIdx.x >> 5;
  const int w = warp_in_block % W;          // warp index inside the team
  const int64_t team = int64_t(blockIdx.x) * TEAMS + warp_in_block / W;
  const int64_t nteams = int64_t(gridDim.x) * TEAMS;
  int slot = 0;
  uint32_t st = 0;

  for (int64_t r = team; r < N; r += nteams) {
    const T* row = in + r * int64_t(M);
    float x[G][V];
    load_row<G, W, FULL>(row, M, w, lane, vec, x);

    // ---- value range [lo, hi] (NaN-propagating, pads excluded from the minimum)
    float mx = neg_inf(), mn = pos_inf();
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
      for (int e = 0; e < V; ++e) {
        mx = max_nan(mx, x[g][e]);
        if (FULL) {
          mn = min_nan(mn, x[g][e]);
        } else {
          const int j = (w * G + g) * GS + lane * V + e;
          mn = min_nan(mn, j < M ? x[g][e] : pos_inf());
        }
      }
    int omx = f2o(mx), omn = f2o(mn);
    team_minmax<W>(omn, omx, w, lane, sh);
    float lo = o2f(omn), hi = o2f(omx);
    if (!(lo >= -1e38f && hi <= 1e38f)) {
      st |= (isfinite(lo) && isfinite(hi)) ? kStatusRange : kStatusNonFinite;
    }

    // ---- ties at the maximum, then the bisection
    int c_hi = team_sum<W>(lane_count_ge<G, V>(x, hi), w, lane, slot, sh);
    int it = 0;
    if (c_hi >= k) {
      // threshold is the maximum: keep its k lowest-index ties via the fill rule
      lo = hi;
      hi = pos_inf();
      c_hi = 0;
    } else {
      while ((max_iter < 0 || it < max_iter) && __fsub_rn(hi, lo) > eps) {
        if (it >= kSafetyCap) { st |= kStatusSafetyCap; break; }
        const float mid = __fmul_rn(__fadd_rn(lo, hi), 0.5f);
        if (!(lo < mid && mid < hi)) break;  // no binary32 value strictly inside
        const int cnt = team_sum<W>(lane_count_ge<G, V>(x, mid), w, lane, slot, sh);
        ++it;
        if (cnt >= k) {
          lo = mid;
          if (cnt == k) break;
        } else {
          hi = mid;
          c_hi = cnt;
        }
      }
    }

    // ---- fill pass: S = {x >= hi} kept; B = {lo <= x < hi} fills `need` by index
    const int need = k - c_hi;
    unsigned pk[NW];
#pragma unroll
    for (int q = 0; q < NW; ++q) pk[q] = 0u;
#pragma unroll
    for (int g = 0; g < G; ++g) {
      unsigned cs = 0, cb = 0;
#pragma unroll
      for (int e = 0; e < V; ++e) {
        const bool s = x[g][e] >= hi;
        cs += s ? 1u : 0u;
        cb += (!s && x[g][e] >= lo) ? 1u : 0u;
      }
      pk[(2 * g) / FPW] += cs << (FB * ((2 * g) % FPW));
      pk[(2 * g + 1) / FPW] += cb << (FB * ((2 * g + 1) % FPW));
    }
    unsigned incl[NW], tot[NW];
#pragma unroll
    for (int q = 0; q < NW; ++q) {
      unsigned v = pk[q];
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const unsigned t = __shfl_up_sync(0xffffffffu, v, d);
        if (lane >= d) v += t;
      }
      incl[q] = v;
      tot[q] = __shfl_sync(0xffffffffu, v, 31);
    }
    int baseS = 0, baseB = 0;
    if constexpr (W > 1) {
      int ts = 0, tb = 0;
#pragma unroll
      for (int g = 0; g < G; ++g) {
        ts += int((tot[(2 * g) / FPW] >> (FB * ((2 * g) % FPW))) & FMASK);
        tb += int((tot[(2 * g + 1) / FPW] >> (FB * ((2 * g + 1) % FPW))) & FMASK);
      }
      if (lane == 0) { sh.tot[w][0] = ts; sh.tot[w][1] = tb; }
      __syncthreads();
      for (int i = 0; i < w; ++i) { baseS += sh.tot[i][0]; baseB += sh.tot[i][1]; }
    }
    const int64_t obase = r * int64_t(k);
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const int fs = 2 * g, fb = 2 * g + 1;
      int runS = baseS + int(((incl[fs / FPW] - pk[fs / FPW]) >> (FB * (fs % FPW))) & FMASK);
      int runB = baseB + int(((incl[fb / FPW] - pk[fb / FPW]) >> (FB * (fb % FPW))) & FMASK);
#pragma unroll
      for (int e = 0; e < V; ++e) {
        const float v = x[g][e];
        const bool s = v >= hi;
        const bool b = !s && v >= lo;
        if (s || (b && runB < need)) {
          const int pos = runS + min(runB, need);
          if (pos < k) {
            vals[obase + pos] = out_value(v, vals);
            idx[obase + pos] = IdxT((w * G + g) * GS + lane * V + e);
          }
        }
        runS += s ? 1 : 0;
        runB += b ? 1 : 0;
      }
      baseS += int((tot[fs / FPW] >> (FB * (fs % FPW))) & FMASK);
      baseB += int((tot[fb / FPW] >> (FB * (fb % FPW))) & FMASK);
    }
    if (iters != nullptr && w == 0 && lane == 0) iters[r] = it;
    if constexpr (W > 1) __syncthreads();  // shared slots are reused by the next row
  }
  if (status != nullptr && st != 0u && lane == 0) atomicOr(status, st);
}

}  // namespace rtopk
