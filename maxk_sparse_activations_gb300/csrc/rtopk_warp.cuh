// Row-wise top-k, one warp per row (rows up to 2048 elements), sm_103a.
//
// Source: "RTop-K: Ultra-Fast Row-Wise Top-K Selection for Neural Network
// Acceleration on GPUs" (summary page), "Approach" (binary search over each
// row's value range for a threshold that selects k, warp-level counting, early
// stop by capping passes, second pass filling borderline ties from the lower
// bound); output layout from "MaxK-GNN: Extremely Fast GPU Kernel Design for
// Accelerating Graph Neural Networks Training", "The idea" (CBSR: dense N x k
// values and indices).
//
// The search is issue-bound (about 8 passes over the row per N(0,1) row at
// M = 256), so the kernel is built around instruction count:
//  * the row lives in registers (lane l holds 16 bytes of each 32*V-element
//    group), one row per warp, no second register set: occupancy hides the
//    load latency better than a register prefetch;
//  * a pass counts x >= mid from the sign bit of x - mid (one subtract on the
//    FMA pipe and one shift-add per element);
//  * the maximum-tie pass runs only when enough lanes hold the maximum for
//    c(max) >= k to be possible (a ballot bounds it);
//  * exact mode (max_iter < 0, eps == 0) compiles a loop without the cap and
//    precision tests (the collapse test subsumes hi - lo > 0);
//  * compaction (L > 0): once c(lo) <= 32 L, the elements >= lo -- a superset
//    of every later candidate -- are written in index order to a per-warp
//    list, and the remaining passes count L list entries per lane instead of
//    the whole row; the CBSR row then comes straight from the list through
//    warp ballots. Counts, passes and results are unchanged: c(mid) over the
//    list equals c(mid) over the row for every mid > lo;
//  * when the search ends on c(lo) == k the kept set is exactly {x >= lo}: one
//    packed prefix scan of per-group counts places it; other endings take the
//    general S / borderline fill;
//  * kept (value, index) pairs are staged in shared memory and written out
//    with coalesced stores (k <= 256), else stored directly.
// Arithmetic and branch decisions are identical to the scalar definition of
// the method (and to rtopk_select_kernel).
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

// Count of this lane's x < t over the registers, t = mid with +0 taken as -0.
template <int G, int V>
__device__ __forceinline__ unsigned lane_count_lt(const float (&x)[G][V], float mid) {
  const float t = (mid == 0.0f) ? -0.0f : mid;
  unsigned lt0 = 0, lt1 = 0;
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int e = 0; e < V; ++e) {
      const unsigned sb = __float_as_uint(__fsub_rn(x[g][e], t)) >> 31;
      if ((g * V + e) & 1) lt1 += sb; else lt0 += sb;
    }
  return lt0 + lt1;
}

// A lower end for an exact search. The TEAM_LANES lanes that share a row are
// split into the largest number of equal lane groups that is still >= k
// (groups never span warps); each group holds an element >= its group
// maximum, so at least k elements of the row are >= the smallest group
// maximum: c(that value) >= k, a valid lower end whenever k <= TEAM_LANES.
// `mx` is the lane's maximum (-inf for a lane of pads, which leaves the bound
// at -inf). Returns this warp's smallest group maximum as an ordered integer.
template <int TEAM_LANES>
__device__ __forceinline__ int group_max_floor(float mx, int k) {
  int groups = TEAM_LANES;
  for (int d = 1; d < 32 && (groups >> 1) >= k; d <<= 1) {
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, d));
    groups >>= 1;
  }
  return __reduce_min_sync(0xffffffffu, f2o(mx));
}

// Counts of this lane's x below three thresholds in one sweep (same rule as
// lane_count_lt for each).
template <int G, int V>
__device__ __forceinline__ void lane_count_lt3(const float (&x)[G][V], float m1, float m2, float m3,
                                               unsigned& c1, unsigned& c2, unsigned& c3) {
  const float t1 = (m1 == 0.0f) ? -0.0f : m1;
  const float t2 = (m2 == 0.0f) ? -0.0f : m2;
  const float t3 = (m3 == 0.0f) ? -0.0f : m3;
  c1 = 0u; c2 = 0u; c3 = 0u;
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int e = 0; e < V; ++e) {
      c1 += __float_as_uint(__fsub_rn(x[g][e], t1)) >> 31;
      c2 += __float_as_uint(__fsub_rn(x[g][e], t2)) >> 31;
      c3 += __float_as_uint(__fsub_rn(x[g][e], t3)) >> 31;
    }
}

// True when [lo, hi) holds at most one bf16 value (lo <= hi finite). For bf16
// data every count c(t) only changes at bf16 values, so from then on further
// passes move lo and hi without changing S = {x >= hi} or B = {lo <= x < hi}:
// the kept set is final. (It cannot hold none: c(lo) >= k > c(hi).)
__device__ __forceinline__ bool bf16_single_value(float lo, float hi) {
  // l = smallest bf16 >= lo (round toward +inf)
  const uint32_t bl = __float_as_uint(lo);
  uint32_t l = bl;
  if (bl & 0xffffu) l = (bl & 0x80000000u) ? (bl & 0xffff0000u) : ((bl & 0xffff0000u) + 0x10000u);
  // u = largest bf16 < hi
  const uint32_t bh = __float_as_uint(hi);
  uint32_t u;
  if (bh & 0xffffu) {
    u = (bh & 0x80000000u) ? ((bh & 0xffff0000u) + 0x10000u) : (bh & 0xffff0000u);
  } else if ((bh & 0x7fffffffu) == 0u) {
    u = 0x80010000u;  // hi = +-0: the largest bf16 below it is -(smallest subnormal)
  } else {
    u = (bh & 0x80000000u) ? (bh + 0x10000u) : (bh - 0x10000u);
  }
  return __uint_as_float(u) <= __uint_as_float(l);
}

// Bisection passes from the current (lo, hi); `count_lt_team(mid)` returns the
// number of the team's elements below mid (identical in every thread), so a
// pass count is total - count_lt_team(mid). Returns true when a pass found
// c(mid) == k. With L > 0 it also stops (returning false, comp = true) right
// after a pass that moved lo to a value with k < c(lo) <= 32 L. With
// BF16STOP and `bf16_stop` set (bf16 data, pass counts not reported) it stops
// once the kept set is final (bf16_single_value): same result, fewer passes.
template <bool EXACT, int L, typename CountLtTeam, bool BF16STOP = false>
__device__ __forceinline__ bool search_passes(CountLtTeam count_lt_team, int total, int k, int limit,
                                              bool cap_is_safety,
                                              float eps, float& lo, float& hi, int& it, int& c_lo, bool& comp,
                                              uint32_t& st, bool bf16_stop = false) {
  for (;;) {
    if (EXACT) {
      if (it >= kSafetyCap) { st |= kStatusSafetyCap; return false; }
    } else {
      if (it >= limit) {
        if (cap_is_safety) st |= kStatusSafetyCap;
        return false;
      }
      if (!(__fsub_rn(hi, lo) > eps)) return false;
    }
    const float mid = __fmul_rn(__fadd_rn(lo, hi), 0.5f);
    if (!(lo < mid && mid < hi)) return false;
    const int cnt = total - int(count_lt_team(mid));
    ++it;
    const bool ge = cnt >= k;
    lo = ge ? mid : lo;
    hi = ge ? hi : mid;
    c_lo = ge ? cnt : c_lo;
    if (cnt == k) return true;
    if (L > 0 && ge && cnt <= 32 * L) { comp = true; return false; }
    // cheap necessary condition first: one bf16 value in [lo, hi) needs
    // hi - lo < 2 bf16 ulps <= max(|lo|, |hi|) * 2^-6 (+ the subnormal spacing)
    if (BF16STOP && bf16_stop &&
        __fsub_rn(hi, lo) <= fmaxf(fabsf(lo), fabsf(hi)) * 0.015625f + 1e-38f && bf16_single_value(lo, hi))
      return false;
  }
}

// Writes the elements x >= lo of the row, in ascending index order, as
// (value, index) pairs to stage[0 .. c(lo)).
template <int G, int V>
__device__ __forceinline__ void compact_ge(const float (&x)[G][V], float lo, int lane, float2* __restrict__ stage) {
  constexpr int GS = 32 * V;
  constexpr int FB = (GS <= 255) ? 8 : 16;
  constexpr int FPW = 32 / FB;
  constexpr unsigned FMASK = (1u << FB) - 1u;
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
  const int jl = lane * V;
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
}

// Finishes a row from its compacted list: the n (<= 32 L) elements >= lo in
// ascending index order, as (value, index) pairs in shared memory. Runs the
// remaining passes over the list (each lane holds entries lane + 32 s) and
// writes the CBSR row: S = {v >= hi} kept, B = {lo <= v < hi} fills the rest
// by index -- entry order is index order, so warp ballots give the ranks.
template <bool EXACT, int L, typename T, typename IdxT>
__device__ __forceinline__ void finish_from_list(const float2* __restrict__ list, int n, float lo, float hi,
                                                 int& it, int k, int limit, bool cap_is_safety, float eps,
                                                 int lane, T* __restrict__ vals, IdxT* __restrict__ idx,
                                                 int64_t obase, uint32_t& st) {
  float lv[L][1];
  int lj[L];
#pragma unroll
  for (int s = 0; s < L; ++s) {
    const int e = s * 32 + lane;
    const float2 p = (e < n) ? list[e] : make_float2(neg_inf(), 0.0f);
    lv[s][0] = p.x;
    lj[s] = __float_as_int(p.y);
  }
  int c_lo = n;
  bool dummy = false;
  search_passes<EXACT, 0>([&](float mid) { return __reduce_add_sync(0xffffffffu, lane_count_lt<L, 1>(lv, mid)); }, 32 * L, k, limit,
                          cap_is_safety, eps, lo, hi, it, c_lo, dummy, st);
  const unsigned lt_mask = (1u << lane) - 1u;
  unsigned bS[L], bB[L];
  int sizeS = 0;
#pragma unroll
  for (int s = 0; s < L; ++s) {
    const bool sf = lv[s][0] >= hi;
    const bool af = lv[s][0] >= lo;
    bS[s] = __ballot_sync(0xffffffffu, sf);
    bB[s] = __ballot_sync(0xffffffffu, af && !sf);
    sizeS += __popc(bS[s]);
  }
  const int need = max(k - sizeS, 0);
  int runS = 0, runB = 0;
#pragma unroll
  for (int s = 0; s < L; ++s) {
    const int rS = runS + __popc(bS[s] & lt_mask);
    const int rB = runB + __popc(bB[s] & lt_mask);
    const bool sf = (bS[s] >> lane) & 1u;
    const bool bf = (bB[s] >> lane) & 1u;
    const int pos = rS + min(rB, need);
    if ((sf || (bf && rB < need)) && pos < k) {
      vals[obase + pos] = out_value(lv[s][0], vals);
      idx[obase + pos] = IdxT(lj[s]);
    }
    runS += __popc(bS[s]);
    runB += __popc(bB[s]);
  }
}

// Fill pass and CBSR store of one row from the final bracket [lo, hi). With
// `exact_end` (the search ended on c(lo) == k) the kept set is exactly
// {x >= lo}; otherwise S = {x >= hi} is kept and B = {lo <= x < hi} fills the
// remaining k - |S| in ascending index order. Rows with k <= kStageK are
// staged in shared memory and written out coalesced.
template <typename T, int G, typename IdxT>
__device__ __forceinline__ void fill_store_w1(const float (&x)[G][ElemTraits<T>::V], float lo, float hi,
                                              bool exact_end, int k, int lane, float2* __restrict__ stage,
                                              T* __restrict__ vals, IdxT* __restrict__ idx, int64_t obase) {
  constexpr int V = ElemTraits<T>::V;
  constexpr int GS = 32 * V;
  constexpr int FB = (GS <= 255) ? 8 : 16;
  constexpr int FPW = 32 / FB;
  constexpr unsigned FMASK = (1u << FB) - 1u;
  const bool staged = (k <= kStageK);
  if (exact_end && staged) {
    // the search ended on c(lo) == k: keep exactly {x >= lo}, in index order
    compact_ge<G, V>(x, lo, lane, stage);
  } else {
    // general: S = {x >= hi} kept, B = {lo <= x < hi} fills the remaining
    // k - |S| in ascending index order
    const uint32_t sbase = static_cast<uint32_t>(__cvta_generic_to_shared(stage));
    const int jl = lane * V;
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
}

template <typename T, int G, bool EXACT, int L, typename IdxT>
__device__ __forceinline__ void process_row_w1(const float (&x)[G][ElemTraits<T>::V], bool full, int64_t r,
                                               int M, int k, int limit, bool cap_is_safety, float eps, int lane,
                                               float2* __restrict__ stage, T* __restrict__ vals,
                                               IdxT* __restrict__ idx, int* __restrict__ iters, uint32_t& st) {
  constexpr int V = ElemTraits<T>::V;
  constexpr int GS = 32 * V;
  constexpr int NE = G * V;

  // ---- value range (NaN-propagating; pads excluded from the minimum)
  float mx = neg_inf(), mn = pos_inf();
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int e = 0; e < V; ++e) {
      mx = max_nan(mx, x[g][e]);
      mn = min_nan(mn, (full || g * GS + lane * V + e < M) ? x[g][e] : pos_inf());
    }
  float hi = o2f(__reduce_max_sync(0xffffffffu, f2o(mx)));
  float lo = o2f(__reduce_min_sync(0xffffffffu, f2o(mn)));
  const bool ok = (lo >= -1e38f && hi <= 1e38f);
  if (!ok) st |= (isfinite(lo) && isfinite(hi)) ? kStatusRange : kStatusNonFinite;

  // ---- ties at the maximum: only possible if enough lanes hold the maximum
  bool max_tie = false;
  if (__popc(__ballot_sync(0xffffffffu, mx == hi)) * NE >= k) {
    int c = 0;
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
      for (int e = 0; e < V; ++e) c += (x[g][e] >= hi) ? 1 : 0;
    max_tie = int(__reduce_add_sync(0xffffffffu, unsigned(c))) >= k;
  }

  int it = 0;
  bool eq = false, comp = false;
  int c_lo = M;
  if (max_tie) {
    lo = hi;           // keep the k lowest-index maxima through the fill rule:
    hi = pos_inf();    // S is empty and every maximum is borderline
  } else {
    auto count_row = [&](float mid) { return __reduce_add_sync(0xffffffffu, lane_count_lt<G, V>(x, mid)); };
    eq = search_passes<EXACT, L, decltype(count_row), (V == 8)>(count_row, 32 * NE, k, limit, cap_is_safety,
                                                                 eps, lo, hi, it, c_lo, comp, st, iters == nullptr);
  }
  comp = comp && ok;

  const int64_t obase = r * int64_t(k);
  if (L > 0 && comp) {
    // ---- compacted phase: list of the c(lo) <= 32 L elements >= lo
    compact_ge<G, V>(x, lo, lane, stage);
    __syncwarp();
    finish_from_list<EXACT, (L > 0 ? L : 1), T, IdxT>(stage, c_lo, lo, hi, it, k, limit, cap_is_safety, eps,
                                                     lane, vals, idx, obase, st);
    __syncwarp();
    if (iters != nullptr && lane == 0) iters[r] = it;
    return;
  }

  fill_store_w1<T, G, IdxT>(x, lo, hi, ok && eq, k, lane, stage, vals, idx, obase);
  if (iters != nullptr && lane == 0) iters[r] = it;
}

// Minimum resident blocks per SM for a row of NE elements per lane.
template <int NE>
struct WarpOcc {
  static constexpr int value = NE <= 8 ? 5 : (NE <= 16 ? 3 : (NE <= 32 ? 2 : 1));
};

template <typename T, int G, bool EXACT, int L, typename IdxT>
__global__ void __launch_bounds__(256, WarpOcc<G * ElemTraits<T>::V>::value)
rtopk_warp_kernel(const T* __restrict__ in, int64_t N, int M, int k, int max_iter, float eps, bool full,
                  bool vec, T* __restrict__ vals, IdxT* __restrict__ idx, int* __restrict__ iters,
                  uint32_t* __restrict__ status) {
  constexpr int V = ElemTraits<T>::V;
  __shared__ float2 stage_all[8][kStageK];
  const int lane = threadIdx.x & 31;
  const int wib = threadIdx.x >> 5;
  float2* stage = stage_all[wib];
  const int64_t nwarps = int64_t(gridDim.x) * 8;
  const bool cap_is_safety = (max_iter < 0 || max_iter > kSafetyCap);
  const int limit = cap_is_safety ? kSafetyCap : max_iter;
  uint32_t st = 0;
  for (int64_t r = int64_t(blockIdx.x) * 8 + wib; r < N; r += nwarps) {
    float x[G][V];
    load_row_w1<T, G>(in, r, M, lane, full, vec, x);
    process_row_w1<T, G, EXACT, L, IdxT>(x, full, r, M, k, limit, cap_is_safety, eps, lane, stage, vals, idx,
                                         iters, st);
  }
  if (status != nullptr && st != 0u && lane == 0) atomicOr(status, st);
}

}  // namespace rtopk
