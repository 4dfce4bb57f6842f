// Row-wise top-k, one 256-thread block per row (rows of 2049..8192 elements), sm_103a.
//
// Source: "RTop-K: Ultra-Fast Row-Wise Top-K Selection for Neural Network
// Acceleration on GPUs" (summary page), "Approach" and "Limitations" (rows
// up to 8192 elements); CBSR output from "MaxK-GNN: Extremely Fast GPU Kernel
// Design for Accelerating Graph Neural Networks Training", "The idea".
//
// Eight warps share a row; warp w holds the contiguous slice
// [w * G * 32V, (w + 1) * G * 32V) in registers with the same per-lane layout
// as the warp kernel. A pass sums the eight warp counts through shared
// memory (double-buffered slots: one barrier per pass). With LB > 0, once
// k < c(lo) <= 32 LB the block writes its elements >= lo, in index order, to a
// shared list, and the rest of the search counts list entries only:
//  * LB = 8 (list <= 256, k <= 128): warp 0 alone finishes the search and the
//    CBSR row from the list (finish_from_list): no barriers in the tail;
//  * LB = 64 (list <= 2048, k <= 1024): all eight warps keep going, each lane
//    holding 8 list entries instead of its 4 G row elements, and the CBSR row
//    is written from the list through warp ballots and per-warp prefixes.
// For bf16 rows whose pass counts are not requested the search stops once
// the kept set is final (bf16_single_value). Arithmetic and branch decisions
// are those of the warp kernel.
#pragma once

#include "rtopk_warp.cuh"

namespace rtopk {

constexpr int kBlockWarps = 8;
constexpr int kBlockList = 2048;  // compaction list capacity (8 warps x 8 entries per lane)

struct BlockShared {
  unsigned cnt[2][kBlockWarps];
  int omax[kBlockWarps];
  int omin[kBlockWarps];
  int ofl[kBlockWarps];
  int tot[kBlockWarps][2];
  float2 list[kBlockList];
};

// Writes this block's elements x >= lo, in ascending index order, to sh.list
// (the caller guarantees at most kBlockList of them). Ends with a barrier.
template <int G, int V>
__device__ __forceinline__ void block_compact_ge(const float (&x)[G][V], float lo, int w, int lane,
                                                 BlockShared& sh) {
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
  unsigned ex[NWF], tot[NWF];
  int wtot = 0;
#pragma unroll
  for (int q = 0; q < NWF; ++q) {
    ex[q] = warp_excl_scan(pkw[q], lane, tot[q]);
#pragma unroll
    for (int f = 0; f < FPW; ++f)
      if (q * FPW + f < G) wtot += int((tot[q] >> (FB * f)) & FMASK);
  }
  if (lane == 0) sh.tot[w][0] = wtot;
  __syncthreads();
  int base = 0;
  for (int i = 0; i < w; ++i) base += sh.tot[i][0];
  const int j0 = w * G * GS + lane * V;
#pragma unroll
  for (int q = 0; q < NWF; ++q) {
#pragma unroll
    for (int f = 0; f < FPW; ++f) {
      const int g = q * FPW + f;
      if (g < G) {
        int pos = base + int((ex[q] >> (FB * f)) & FMASK);
#pragma unroll
        for (int e = 0; e < V; ++e) {
          if (x[g][e] >= lo) {
            if (pos < kBlockList) sh.list[pos] = make_float2(x[g][e], __int_as_float(j0 + g * GS + e));
            ++pos;
          }
        }
        base += int((tot[q] >> (FB * f)) & FMASK);
      }
    }
  }
  __syncthreads();
}

// LB = 64: the eight warps finish the search over the shared list of the
// n <= 2048 elements >= lo (entry e at warp e / 256, slot (e / 32) % 8,
// lane e % 32 -- entry order is index order) and write the CBSR row.
template <bool EXACT, bool BF16STOP, typename T, typename IdxT, typename BlockSum>
__device__ __forceinline__ void block_finish_from_list(BlockShared& sh, BlockSum block_sum, int n, float lo,
                                                       float hi, int& it, int k, int limit, bool cap_is_safety,
                                                       float eps, int w, int lane, T* __restrict__ vals,
                                                       IdxT* __restrict__ idx, int64_t obase, uint32_t& st,
                                                       bool bf16_stop) {
  constexpr int S = 8;
  float lv[S][1];
  int lj[S];
#pragma unroll
  for (int s = 0; s < S; ++s) {
    const int e = w * 256 + s * 32 + lane;
    const float2 p = (e < n) ? sh.list[e] : make_float2(neg_inf(), 0.0f);
    lv[s][0] = p.x;
    lj[s] = __float_as_int(p.y);
  }
  int c_lo = n;
  bool dummy = false;
  auto count_list = [&](float mid) { return block_sum(lane_count_lt<S, 1>(lv, mid)); };
  search_passes<EXACT, 0, decltype(count_list), BF16STOP>(count_list, kBlockWarps * 32 * S, k, limit,
                                                          cap_is_safety, eps, lo, hi, it, c_lo, dummy, st,
                                                          bf16_stop);
  const unsigned lt_mask = (1u << lane) - 1u;
  unsigned bS[S], bB[S];
  int tS = 0, tB = 0;
#pragma unroll
  for (int s = 0; s < S; ++s) {
    const bool sf = lv[s][0] >= hi;
    const bool af = lv[s][0] >= lo;
    bS[s] = __ballot_sync(0xffffffffu, sf);
    bB[s] = __ballot_sync(0xffffffffu, af && !sf);
    tS += __popc(bS[s]);
    tB += __popc(bB[s]);
  }
  if (lane == 0) { sh.tot[w][0] = tS; sh.tot[w][1] = tB; }
  __syncthreads();
  int runS = 0, runB = 0, sizeS = 0;
#pragma unroll
  for (int i = 0; i < kBlockWarps; ++i) {
    sizeS += sh.tot[i][0];
    if (i < w) { runS += sh.tot[i][0]; runB += sh.tot[i][1]; }
  }
  const int need = max(k - sizeS, 0);
#pragma unroll
  for (int s = 0; s < S; ++s) {
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

// Resident blocks per SM: at M = 8192 a thread holds 32 elements and one block
// per SM leaves too few warps to hide the per-pass barrier and reduction
// latency, so at least two (<= 128 registers a thread); rows of <= 16 elements
// a thread keep three.
template <int NE>
struct BlockOcc {
  static constexpr int value = NE <= 16 ? 3 : 2;
};

template <typename T, int G, bool EXACT, int LB, typename IdxT>
__global__ void __launch_bounds__(256, BlockOcc<G * ElemTraits<T>::V>::value)
rtopk_block_kernel(const T* __restrict__ in, int64_t N, int M, int k, int max_iter, float eps, bool full,
                   bool vec, T* __restrict__ vals, IdxT* __restrict__ idx, int* __restrict__ iters,
                   uint32_t* __restrict__ status) {
  constexpr int W = kBlockWarps;
  constexpr int V = ElemTraits<T>::V;
  constexpr int GS = 32 * V;
  constexpr int NE = G * V;
  constexpr int FB = (GS <= 255) ? 8 : 16;
  constexpr int FPW = 32 / FB;
  constexpr int NF = 2 * G;
  constexpr int NW = (NF + FPW - 1) / FPW;
  constexpr unsigned FMASK = (1u << FB) - 1u;
  static_assert(LB == 0 || LB == 8 || LB == 64, "list modes");
  static_assert(32 * LB <= kBlockList, "list capacity");

  __shared__ BlockShared sh;
  const int lane = threadIdx.x & 31;
  const int w = threadIdx.x >> 5;
  const bool cap_is_safety = (max_iter < 0 || max_iter > kSafetyCap);
  const int limit = cap_is_safety ? kSafetyCap : max_iter;
  int slot = 0;
  uint32_t st = 0;

  // sum over the block of a per-lane count (identical result in every thread)
  auto block_sum = [&](unsigned v) -> unsigned {
    const unsigned s = __reduce_add_sync(0xffffffffu, v);
    if (lane == 0) sh.cnt[slot][w] = s;
    __syncthreads();
    unsigned t = 0;
#pragma unroll
    for (int i = 0; i < W; ++i) t += sh.cnt[slot][i];
    slot ^= 1;
    return t;
  };

  for (int64_t r = blockIdx.x; r < N; r += gridDim.x) {
    const T* row = in + r * int64_t(M);
    float x[G][V];
    if (full) {
      load_row<G, W, true>(row, M, w, lane, vec, x);
    } else {
      load_row<G, W, false>(row, M, w, lane, vec, x);
    }

    // ---- value range [lo, hi] (NaN-propagating, pads excluded from the minimum)
    float mx = neg_inf(), mn = pos_inf();
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
      for (int e = 0; e < V; ++e) {
        mx = max_nan(mx, x[g][e]);
        mn = min_nan(mn, (full || (w * G + g) * GS + lane * V + e < M) ? x[g][e] : pos_inf());
      }
    // an exact search whose pass count is not reported may start from the
    // group-maximum lower end (the exact top-k set does not depend on it)
    const bool floor_lo = EXACT && iters == nullptr && k <= W * 32;
    int omx = __reduce_max_sync(0xffffffffu, f2o(mx));
    int omn = __reduce_min_sync(0xffffffffu, f2o(mn));
    int ofl = floor_lo ? group_max_floor<W * 32>(mx, k) : omn;
    if (lane == 0) { sh.omax[w] = omx; sh.omin[w] = omn; sh.ofl[w] = ofl; }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < W; ++i) {
      omx = max(omx, sh.omax[i]);
      omn = min(omn, sh.omin[i]);
      ofl = min(ofl, sh.ofl[i]);
    }
    float lo = o2f(omn), hi = o2f(omx);
    const bool ok = (lo >= -1e38f && hi <= 1e38f);
    if (!ok) st |= (isfinite(lo) && isfinite(hi)) ? kStatusRange : kStatusNonFinite;

    // ---- ties at the maximum
    unsigned cmax = 0;
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
      for (int e = 0; e < V; ++e) cmax += (x[g][e] >= hi) ? 1u : 0u;
    const bool max_tie = int(block_sum(cmax)) >= k;

    // ---- bisection over the block
    int it = 0;
    bool eq = false, comp = false;
    int c_lo = M;
    if (max_tie) {
      lo = hi;
      hi = pos_inf();
    } else {
      if (floor_lo && ok) lo = fmaxf(lo, o2f(ofl));
      auto count_row = [&](float mid) { return block_sum(lane_count_lt<G, V>(x, mid)); };
      eq = search_passes<EXACT, LB, decltype(count_row), (V == 8)>(count_row, W * 32 * NE, k, limit,
                                                                   cap_is_safety, eps, lo, hi, it, c_lo, comp,
                                                                   st, iters == nullptr);
    }
    comp = comp && ok;
    const int64_t obase = r * int64_t(k);

    if (LB == 8 && comp) {
      // ---- warp 0 finishes from the compacted list of the c(lo) elements >= lo
      block_compact_ge<G, V>(x, lo, w, lane, sh);
      if (w == 0) {
        finish_from_list<EXACT, 8, T, IdxT>(sh.list, c_lo, lo, hi, it, k, limit, cap_is_safety, eps, lane,
                                            vals, idx, obase, st);
        if (iters != nullptr && lane == 0) iters[r] = it;
      }
      __syncthreads();
      continue;
    }
    if (LB == 64 && comp) {
      // ---- the block finishes from the compacted list (8 entries per lane)
      block_compact_ge<G, V>(x, lo, w, lane, sh);
      block_finish_from_list<EXACT, (V == 8), T, IdxT>(sh, block_sum, c_lo, lo, hi, it, k, limit,
                                                       cap_is_safety, eps, w, lane, vals, idx, obase, st,
                                                       iters == nullptr);
      if (iters != nullptr && w == 0 && lane == 0) iters[r] = it;
      __syncthreads();
      continue;
    }
    if (ok && eq && k <= kBlockList) {
      // ---- the search ended on c(lo) == k: the list is the CBSR row
      block_compact_ge<G, V>(x, lo, w, lane, sh);
      for (int p = threadIdx.x; p < k; p += 256) {
        const float2 e = sh.list[p];
        vals[obase + p] = out_value(e.x, vals);
        idx[obase + p] = IdxT(__float_as_int(e.y));
      }
    } else {
      // ---- general fill: S = {x >= hi} kept; B = {lo <= x < hi} fills by index
      unsigned pk[NW];
#pragma unroll
      for (int q = 0; q < NW; ++q) pk[q] = 0u;
#pragma unroll
      for (int g = 0; g < G; ++g) {
        unsigned cs = 0, ca = 0;
#pragma unroll
        for (int e = 0; e < V; ++e) {
          cs += (x[g][e] >= hi) ? 1u : 0u;
          ca += (x[g][e] >= lo) ? 1u : 0u;
        }
        pk[(2 * g) / FPW] += cs << (FB * ((2 * g) % FPW));
        pk[(2 * g + 1) / FPW] += (ca - cs) << (FB * ((2 * g + 1) % FPW));
      }
      unsigned ex[NW], tot[NW];
#pragma unroll
      for (int q = 0; q < NW; ++q) ex[q] = warp_excl_scan(pk[q], lane, tot[q]);
      int ts = 0, tb = 0;
#pragma unroll
      for (int g = 0; g < G; ++g) {
        ts += int((tot[(2 * g) / FPW] >> (FB * ((2 * g) % FPW))) & FMASK);
        tb += int((tot[(2 * g + 1) / FPW] >> (FB * ((2 * g + 1) % FPW))) & FMASK);
      }
      if (lane == 0) { sh.tot[w][0] = ts; sh.tot[w][1] = tb; }
      __syncthreads();
      int baseS = 0, baseB = 0, sizeS = 0;
#pragma unroll
      for (int i = 0; i < W; ++i) {
        sizeS += sh.tot[i][0];
        if (i < w) { baseS += sh.tot[i][0]; baseB += sh.tot[i][1]; }
      }
      const int need = max(k - sizeS, 0);
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const int fs = 2 * g, fb = 2 * g + 1;
        int runS = baseS + int((ex[fs / FPW] >> (FB * (fs % FPW))) & FMASK);
        int runB = baseB + int((ex[fb / FPW] >> (FB * (fb % FPW))) & FMASK);
#pragma unroll
        for (int e = 0; e < V; ++e) {
          const float v = x[g][e];
          const bool s = v >= hi;
          const bool b = !s && v >= lo;
          const int pos = runS + min(runB, need);
          if ((s || (b && runB < need)) && pos < k) {
            vals[obase + pos] = out_value(v, vals);
            idx[obase + pos] = IdxT((w * G + g) * GS + lane * V + e);
          }
          runS += s ? 1 : 0;
          runB += b ? 1 : 0;
        }
        baseS += int((tot[fs / FPW] >> (FB * (fs % FPW))) & FMASK);
        baseB += int((tot[fb / FPW] >> (FB * (fb % FPW))) & FMASK);
      }
    }
    if (iters != nullptr && w == 0 && lane == 0) iters[r] = it;
    __syncthreads();  // shared slots and the list are reused by the next row
  }
  if (status != nullptr && st != 0u && lane == 0) atomicOr(status, st);
}

}  // namespace rtopk
