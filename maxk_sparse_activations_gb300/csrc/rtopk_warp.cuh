// Row-wise top-k, one warp per row (rows up to 1024 elements), sm_103a.
//
// Source: "RTop-K: Ultra-Fast Row-Wise Top-K Selection for Neural Network
// Acceleration on GPUs" (summary page), "Approach" (binary search over each
// row's value range for a threshold that selects k, warp-level counting, early
// stop by capping passes, second pass filling borderline ties from the lower
// bound); output layout from "MaxK-GNN: Extremely Fast GPU Kernel Design for
// Accelerating Graph Neural Networks Training", "The idea" (CBSR: dense N x k
// values and indices).
//
// This is the instruction-lean variant of rtopk_select_kernel for W = 1. The
// search is issue-bound (about 8 passes over the row per N(0,1) row at
// M = 256), so everything around the passes is trimmed:
//  * the next row is loaded into a second register set while the current row
//    is searched (one row of HBM traffic always in flight per warp);
//  * the maximum-tie pass runs only when enough lanes hold the maximum for
//    c(max) >= k to be possible (a ballot bounds it), which for continuous
//    data is almost never;
//  * exact mode (max_iter < 0, eps == 0) compiles a loop with no cap or
//    precision test beyond the safety cap (the collapse test subsumes
//    hi - lo > 0);
//  * a pass counts x >= mid from the sign bit of x - mid (one subtract on the
//    FMA pipe and one shift-add per element);
//  * when the search ends on c(lo) == k (the usual exact-mode ending) the
//    fill keeps exactly {x >= lo}: one packed prefix scan of per-group counts;
//    other endings take the general S / borderline fill, whose per-slot step
//    is one straight-line predicated shared-memory store;
//  * kept (value, index) pairs are staged in shared memory and written out
//    with coalesced stores (k <= 256), else stored directly.
// Arithmetic and branch decisions are identical to rtopk_select_kernel.
#pragma once

#include "rtopk_select.cuh"

namespace rtopk {

constexpr int kStageK = 256;  // per-warp shared staging of the CBSR row (k <= 256)

template <typename T, int G>
__device__ __forceinline__ void load_row_w1(const T* __restrict__ in, int64_t r, int M, int lane,
                                            bool full, bool vec, float (&x)[G][ElemTraits<T>::V]) {
  const T* row = in + r * int64_t(M);
  if (full) {
    load_row<G, 1, true>(row, M, 0, lane, vec, x);
  } else {
    load_row<G, 1, false>(row, M, 0, lane, vec, x);
  }
}

// Prefix of per-lane packed counts across the warp: returns the exclusive
// prefix word and sets `tot` to the warp total word (fields never overflow).
__device__ __forceinline__ unsigned warp_excl_scan(unsigned v, int lane, unsigned& tot) {
  unsigned s = v;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const unsigned t = __shfl_up_sync(0xffffffffu, s, d);
    s += (lane >= d) ? t : 0u;
  }
  tot = __shfl_sync(0xffffffffu, s, 31);
  return s - v;
}

// One general fill slot, straight-line: S = v >= hi is kept; B = lo <= v < hi
// is kept while its rank among B (runB) is below `need`; position
// runS + min(runB, need), bounded by k. Advances runS / runB.
__device__ __forceinline__ void stage_general(float v, float lo, float hi, int need, int k, uint32_t sbase,
                                              int& runS, int& runB, int j) {
  asm volatile(
      "{\n\t.reg .pred ps, pb, pn, pk;\n\t.reg .s32 m, q;\n\t.reg .u32 a;\n\t"
      "setp.ge.f32 ps, %2, %4;\n\t"
      "setp.ge.and.f32 pb, %2, %3, !ps;\n\t"
      "setp.lt.and.s32 pn, %1, %5, pb;\n\t"
      "or.pred pk, ps, pn;\n\t"
      "min.s32 m, %1, %5;\n\t"
      "add.s32 q, %0, m;\n\t"
      "setp.lt.and.s32 pk, q, %6, pk;\n\t"
      "mad.lo.u32 a, q, 8, %7;\n\t"
      "@pk st.shared.v2.b32 [a], {%8, %9};\n\t"
      "@ps add.s32 %0, %0, 1;\n\t"
      "@pb add.s32 %1, %1, 1;\n\t}"
      : "+r"(runS), "+r"(runB)
      : "f"(v), "f"(lo), "f"(hi), "r"(need), "r"(k), "r"(sbase), "r"(__float_as_uint(v)), "r"(j)
      : "memory");
}

// Predicated global stores (rows whose k exceeds the shared staging area).
__device__ __forceinline__ void st_global_if(unsigned p, float* a, float v) {
  asm volatile("{\n\t.reg .pred q;\n\tsetp.ne.u32 q, %0, 0;\n\t@q st.global.b32 [%1], %2;\n\t}"
               ::"r"(p), "l"(a), "r"(__float_as_uint(v)) : "memory");
}
__device__ __forceinline__ void st_global_if(unsigned p, int32_t* a, int32_t v) {
  asm volatile("{\n\t.reg .pred q;\n\tsetp.ne.u32 q, %0, 0;\n\t@q st.global.b32 [%1], %2;\n\t}"
               ::"r"(p), "l"(a), "r"(v) : "memory");
}
__device__ __forceinline__ void st_global_if(unsigned p, uint16_t* a, uint16_t v) {
  asm volatile("{\n\t.reg .pred q;\n\tsetp.ne.u32 q, %0, 0;\n\t@q st.global.b16 [%1], %2;\n\t}"
               ::"r"(p), "l"(a), "h"(v) : "memory");
}
__device__ __forceinline__ void st_global_if(unsigned p, int16_t* a, int16_t v) {
  asm volatile("{\n\t.reg .pred q;\n\tsetp.ne.u32 q, %0, 0;\n\t@q st.global.b16 [%1], %2;\n\t}"
               ::"r"(p), "l"(a), "h"(v) : "memory");
}

template <typename T, int G, bool FULL, bool EXACT, typename IdxT>
__device__ __forceinline__ void process_row_w1(const float (&x)[G][ElemTraits<T>::V], int64_t r, int M,
                                               int k, int limit, bool cap_is_safety, float eps, int lane,
                                               float2* __restrict__ stage, T* __restrict__ vals,
                                               IdxT* __restrict__ idx, int* __restrict__ iters,
                                               uint32_t& st) {
  constexpr int V = ElemTraits<T>::V;
  constexpr int GS = 32 * V;
  constexpr int NE = G * V;
  constexpr int FB = (GS <= 255) ? 8 : 16;
  constexpr int FPW = 32 / FB;
  constexpr unsigned FMASK = (1u << FB) - 1u;

  // ---- value range (NaN-propagating; pads excluded from the minimum)
  float mx = neg_inf(), mn = pos_inf();
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int e = 0; e < V; ++e) {
      mx = max_nan(mx, x[g][e]);
      if (FULL) {
        mn = min_nan(mn, x[g][e]);
      } else {
        mn = min_nan(mn, (g * GS + lane * V + e < M) ? x[g][e] : pos_inf());
      }
    }
  const float hi0 = o2f(__reduce_max_sync(0xffffffffu, f2o(mx)));
  const float lo0 = o2f(__reduce_min_sync(0xffffffffu, f2o(mn)));
  float lo = lo0, hi = hi0;
  const bool ok = (lo >= -1e38f && hi <= 1e38f);
  if (!ok) st |= (isfinite(lo) && isfinite(hi)) ? kStatusRange : kStatusNonFinite;

  // ---- ties at the maximum: only possible if enough lanes hold the maximum
  bool max_tie = false;
  {
    const int lanes_at_max = __popc(__ballot_sync(0xffffffffu, mx == hi));
    if (lanes_at_max * NE >= k) {
      int c = 0;
#pragma unroll
      for (int g = 0; g < G; ++g)
#pragma unroll
        for (int e = 0; e < V; ++e) c += (x[g][e] >= hi) ? 1 : 0;
      max_tie = int(__reduce_add_sync(0xffffffffu, unsigned(c))) >= k;
    }
  }

  // ---- bisection. A pass counts x >= mid from the sign bit of x - mid
  // (finite |x|, |mid| <= 1e38, -inf pads); a zero threshold is taken as -0
  // so that x = -0 gives (-0) - (-0) = +0 and counts as >= (it equals +0).
  int it = 0;
  bool eq = false;
  if (max_tie) {
    lo = hi;           // keep the k lowest-index maxima through the fill rule:
    hi = pos_inf();    // S is empty and every maximum is borderline
  } else {
    for (;;) {
      if (EXACT) {
        if (it >= kSafetyCap) { st |= kStatusSafetyCap; break; }
      } else {
        if (it >= limit) {
          if (cap_is_safety) st |= kStatusSafetyCap;
          break;
        }
        if (!(__fsub_rn(hi, lo) > eps)) break;
      }
      const float mid = __fmul_rn(__fadd_rn(lo, hi), 0.5f);
      if (!(lo < mid && mid < hi)) break;
      const float t = (mid == 0.0f) ? -0.0f : mid;
      unsigned lt0 = 0, lt1 = 0;
#pragma unroll
      for (int g = 0; g < G; ++g)
#pragma unroll
        for (int e = 0; e < V; ++e) {
          const unsigned sb = __float_as_uint(__fsub_rn(x[g][e], t)) >> 31;
          if ((g * V + e) & 1) lt1 += sb; else lt0 += sb;
        }
      const int cnt = 32 * NE - int(__reduce_add_sync(0xffffffffu, lt0 + lt1));
      ++it;
      const bool ge = cnt >= k;
      lo = ge ? mid : lo;
      hi = ge ? hi : mid;
      if (cnt == k) { eq = true; break; }
    }
  }

  // ---- fill pass and CBSR store: S = {x >= hi} kept, B = {lo <= x < hi}
  // fills the remaining k - |S| in ascending index order (branch-free: every
  // slot issues one predicated store and advances its prefix counters)
  const int64_t obase = r * int64_t(k);
  const bool staged = (k <= kStageK);
  const uint32_t sbase = static_cast<uint32_t>(__cvta_generic_to_shared(stage));
  const int jl = lane * V;
  if (ok && eq && staged) {
    // the search ended on c(lo) == k: keep exactly {x >= lo}, in index order
    constexpr int NWF = (G + FPW - 1) / FPW;
    unsigned pkw[NWF];
#pragma unroll
    for (int q = 0; q < NWF; ++q) pkw[q] = 0u;
#pragma unroll
    for (int g = 0; g < G; ++g) {
      unsigned c = 0;
#pragma unroll
      for (int e = 0; e < V; ++e) c += (x[g][e] >= lo) ? 1u : 0u;
      pkw[g / FPW] += c << (FB * (g % FPW));
    }
    int base = 0;
#pragma unroll
    for (int q = 0; q < NWF; ++q) {
      unsigned tot;
      const unsigned ex = warp_excl_scan(pkw[q], lane, tot);
#pragma unroll
      for (int f = 0; f < FPW; ++f) {
        const int g = q * FPW + f;
        if (g < G) {
          int pos = base + int((ex >> (FB * f)) & FMASK);
#pragma unroll
          for (int e = 0; e < V; ++e) {
            if (x[g][e] >= lo) {
              stage[pos] = make_float2(x[g][e], __int_as_float(g * GS + jl + e));
              ++pos;
            }
          }
          base += int((tot >> (FB * f)) & FMASK);
        }
      }
    }
  } else
  {
    constexpr int NF = 2 * G;
    constexpr int NW = (NF + FPW - 1) / FPW;
    unsigned pkw[NW];
#pragma unroll
    for (int q = 0; q < NW; ++q) pkw[q] = 0u;
#pragma unroll
    for (int g = 0; g < G; ++g) {
      unsigned cs = 0, cb = 0;
#pragma unroll
      for (int e = 0; e < V; ++e) {
        cs += (x[g][e] >= hi) ? 1u : 0u;
        cb += (x[g][e] >= lo) ? 1u : 0u;  // S and B together; B = difference
      }
      pkw[(2 * g) / FPW] += cs << (FB * ((2 * g) % FPW));
      pkw[(2 * g + 1) / FPW] += (cb - cs) << (FB * ((2 * g + 1) % FPW));
    }
    unsigned ex[NW], tot[NW];
#pragma unroll
    for (int q = 0; q < NW; ++q) ex[q] = warp_excl_scan(pkw[q], lane, tot[q]);
    int sizeS = 0;
#pragma unroll
    for (int g = 0; g < G; ++g) sizeS += int((tot[(2 * g) / FPW] >> (FB * ((2 * g) % FPW))) & FMASK);
    const int need = max(k - sizeS, 0);  // sizeS < k for every valid row
    int baseS = 0, baseB = 0;
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const int fs = 2 * g, fb = 2 * g + 1;
      int runS = baseS + int((ex[fs / FPW] >> (FB * (fs % FPW))) & FMASK);
      int runB = baseB + int((ex[fb / FPW] >> (FB * (fb % FPW))) & FMASK);
#pragma unroll
      for (int e = 0; e < V; ++e) {
        const float v = x[g][e];
        const int j = g * GS + jl + e;
        if (staged) {
          stage_general(v, lo, hi, need, k, sbase, runS, runB, j);
        } else {
          const unsigned sf = (v >= hi) ? 1u : 0u;
          const unsigned bf = (v >= lo) ? 1u - sf : 0u;
          const int pos = runS + min(runB, need);
          const unsigned keep = (sf | (bf & unsigned(runB < need))) & unsigned(pos < k);
          st_global_if(keep, vals + obase + pos, out_value(v, vals));
          st_global_if(keep, idx + obase + pos, IdxT(j));
          runS += int(sf);
          runB += int(bf);
        }
      }
      baseS += int((tot[fs / FPW] >> (FB * (fs % FPW))) & FMASK);
      baseB += int((tot[fb / FPW] >> (FB * (fb % FPW))) & FMASK);
    }
  }
  if (staged) {
    __syncwarp();
    for (int p = lane; p < k; p += 32) {
      const float2 e = stage[p];
      vals[obase + p] = out_value(e.x, vals);
      idx[obase + p] = IdxT(__float_as_int(e.y));
    }
    __syncwarp();
  }
  if (iters != nullptr && lane == 0) iters[r] = it;
}

template <typename T, int G, bool FULL, bool EXACT, typename IdxT>
__global__ void __launch_bounds__(256)
rtopk_warp_kernel(const T* __restrict__ in, int64_t N, int M, int k, int max_iter, float eps, bool vec,
                  T* __restrict__ vals, IdxT* __restrict__ idx, int* __restrict__ iters,
                  uint32_t* __restrict__ status) {
  constexpr int V = ElemTraits<T>::V;
  __shared__ float2 stage_all[8][kStageK];
  const int lane = threadIdx.x & 31;
  const int wib = threadIdx.x >> 5;
  float2* stage = stage_all[wib];
  const int64_t nwarps = int64_t(gridDim.x) * 8;
  int64_t r = int64_t(blockIdx.x) * 8 + wib;
  const bool cap_is_safety = (max_iter < 0 || max_iter > kSafetyCap);
  const int limit = cap_is_safety ? kSafetyCap : max_iter;
  uint32_t st = 0;

  float xa[G][V], xb[G][V];
  if (r < N) load_row_w1<T, G>(in, r, M, lane, FULL, vec, xa);
  while (r < N) {
    int64_t rn = r + nwarps;
    if (rn < N) load_row_w1<T, G>(in, rn, M, lane, FULL, vec, xb);
    process_row_w1<T, G, FULL, EXACT, IdxT>(xa, r, M, k, limit, cap_is_safety, eps, lane, stage, vals, idx, iters, st);
    r = rn;
    if (r >= N) break;
    rn = r + nwarps;
    if (rn < N) load_row_w1<T, G>(in, rn, M, lane, FULL, vec, xa);
    process_row_w1<T, G, FULL, EXACT, IdxT>(xb, r, M, k, limit, cap_is_safety, eps, lane, stage, vals, idx, iters, st);
    r = rn;
  }
  if (status != nullptr && st != 0u && lane == 0) atomicOr(status, st);
}

}  // namespace rtopk
