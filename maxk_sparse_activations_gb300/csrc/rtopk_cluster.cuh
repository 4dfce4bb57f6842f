// Row-wise top-k for rows longer than one block can hold: one thread-block
// cluster per row (rows of 8193..65536 elements), sm_103a.
//
// Source: "RTop-K: Ultra-Fast Row-Wise Top-K Selection for Neural Network
// Acceleration on GPUs" (summary page), "Approach" (per-row binary search over
// the value range, early stop, borderline ties filled from the lower bound)
// and "Limitations" (the method stops at 8192 elements per row; this kernel
// extends the same search past that limit); CBSR output from "MaxK-GNN:
// Extremely Fast GPU Kernel Design for Accelerating Graph Neural Networks
// Training", "The idea".
//
// C CTAs (C = 2, 4, 8) of 8 warps share one row. CTA q, warp w holds, in
// registers, the slice of team warp t = 8 q + w with the block kernel's lane
// layout (j = (t * G + g) * 32 V + l * V + e), so the row is read from HBM
// once. Every exchange between the CTAs is one "round": each warp reduces its
// value(s) with redux.sync, lanes 0..C-1 store them into the same slot of every
// CTA's shared memory (distributed shared memory, st.shared::cluster), then
// the whole cluster passes one hardware barrier (barrier.cluster, release /
// acquire) and every thread reduces the 8 C slots locally. Slots alternate
// between two buffers from round to round, so a buffer is rewritten only after
// a later barrier that every reader of its previous contents has passed.
// A pass of the search is one round; the range, the maximum-tie count and the
// general fill's two counts are one round each. All CTAs see the same sums and
// therefore take the same branches; no thread ever spins.
//
// Per row the arithmetic and branch decisions are those of the scalar
// definition: same midpoints, counts, pass numbers and kept set.
#pragma once

#include "rtopk_block.cuh"


namespace rtopk {

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_index() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_count() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}
// Every thread of every CTA of the cluster arrives and waits: shared-memory
// writes before the barrier (local or remote) are visible after it.
__device__ __forceinline__ void cluster_barrier() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Store v at the same shared-memory offset as `local` in CTA `rank` of the cluster.
__device__ __forceinline__ void st_cluster_u32(const void* local, uint32_t rank, uint32_t v) {
  const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(local));
  asm volatile("{\n\t.reg .u32 ra;\n\tmapa.shared::cluster.u32 ra, %0, %1;\n\tst.shared::cluster.u32 [ra], %2;\n\t}"
               ::"r"(a), "r"(rank), "r"(v) : "memory");
}

constexpr int kClusterMax = 8;
constexpr int kTeamWarpsMax = kBlockWarps * kClusterMax;  // 64 warps share a row at most

struct ClusterShared {
  uint32_t slot[2][3][kTeamWarpsMax];  // [buffer][value][team warp]
};

// One exchange round: lanes 0..C-1 of every warp publish up to three per-warp
// values into slot[buf][*][team warp] of every CTA, then the cluster barrier.
template <int C, int NV>
__device__ __forceinline__ void cluster_round(ClusterShared& sh, int buf, int t, int lane, uint32_t v0,
                                              uint32_t v1 = 0u, uint32_t v2 = 0u) {
  if (lane < C) {
    st_cluster_u32(&sh.slot[buf][0][t], uint32_t(lane), v0);
    if (NV > 1) st_cluster_u32(&sh.slot[buf][1][t], uint32_t(lane), v1);
    if (NV > 2) st_cluster_u32(&sh.slot[buf][2][t], uint32_t(lane), v2);
  }
  cluster_barrier();
}
// Sum of value `which` over the team warps [0, upto) (identical in every thread).
template <int C>
__device__ __forceinline__ uint32_t team_sum(const ClusterShared& sh, int buf, int which, int lane, int upto) {
  uint32_t a = (lane < upto) ? sh.slot[buf][which][lane] : 0u;
  if (8 * C > 32) a += (lane + 32 < upto) ? sh.slot[buf][which][lane + 32] : 0u;
  return __reduce_add_sync(0xffffffffu, a);
}
template <int C>
__device__ __forceinline__ int team_max(const ClusterShared& sh, int buf, int which, int lane) {
  int a = int(sh.slot[buf][which][lane & (8 * C - 1)]);
  if (8 * C > 32) a = max(a, int(sh.slot[buf][which][lane + 32]));
  return __reduce_max_sync(0xffffffffu, a);
}
template <int C>
__device__ __forceinline__ int team_min(const ClusterShared& sh, int buf, int which, int lane) {
  int a = int(sh.slot[buf][which][lane & (8 * C - 1)]);
  if (8 * C > 32) a = min(a, int(sh.slot[buf][which][lane + 32]));
  return __reduce_min_sync(0xffffffffu, a);
}

// C CTAs of 256 threads per row, G groups of V elements per lane (the row is
// at most C * 8 * G * 32 * V elements; shorter rows are padded with -inf).
// Resident CTAs per SM: 3 at 32 elements per lane (80 registers), 2 at 64.
// Measured on GB300 (fp32, k = 256): a third CTA per SM is 15% faster at 32
// elements per lane; a register prefetch of the next row (which rules the third
// CTA out) gained only 4%.
template <int NE>
struct ClusterOcc {
  static constexpr int value = NE <= 32 ? 3 : 2;
};
template <typename T, int G, bool EXACT, int C, typename IdxT>
__global__ void __launch_bounds__(256, ClusterOcc<G * ElemTraits<T>::V>::value)
rtopk_cluster_kernel(const T* __restrict__ in, int64_t N, int M, int k, int max_iter, float eps, bool full,
                     bool vec, T* __restrict__ vals, IdxT* __restrict__ idx, int* __restrict__ iters,
                     uint32_t* __restrict__ status) {
  constexpr int V = ElemTraits<T>::V;
  constexpr int W = kBlockWarps;
  constexpr int NE = G * V;
  constexpr int GS = 32 * V;
  constexpr int FB = (GS <= 255) ? 8 : 16;
  constexpr int FPW = 32 / FB;
  constexpr unsigned FMASK = (1u << FB) - 1u;
  constexpr int NW = (2 * G + FPW - 1) / FPW;
  static_assert(C == 2 || C == 4 || C == 8, "portable cluster sizes");
  __shared__ ClusterShared sh;
  const int lane = threadIdx.x & 31;
  const int w = threadIdx.x >> 5;
  const int q = int(cluster_rank());
  const int t = q * W + w;  // team warp: its slice starts at element t * G * GS
  const int TW = C * W;     // team warps
  const bool cap_is_safety = (max_iter < 0 || max_iter > kSafetyCap);
  const int limit = cap_is_safety ? kSafetyCap : max_iter;
  // every thread holds an element >= its own maximum, so the smallest thread
  // maximum is a valid lower end whenever k <= the number of threads
  const bool floor_lo = EXACT && iters == nullptr && k <= 32 * TW;
  const bool bf16_stop = (V == 8) && iters == nullptr;
  uint32_t st = 0;
  int buf = 0;
  cluster_barrier();  // every CTA of the cluster is running before the first remote store

  auto load = [&](int64_t rr, float (&dst)[G][V]) {
    const T* row = in + rr * int64_t(M);
    if (full) {
      load_row<G, W, true>(row, M, t, lane, vec, dst);
    } else {
      load_row<G, W, false>(row, M, t, lane, vec, dst);
    }
  };
  float x[G][V];
  float tprev = __int_as_float(0x7fc00000);  // the cluster's previous threshold (guessed probes)
  for (int64_t r = cluster_index(); r < N; r += cluster_count()) {
    load(r, x);

    // ---- round: value range and the lower end candidate
    float mx = neg_inf(), mn = pos_inf();
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
      for (int e = 0; e < V; ++e) {
        mx = max_nan(mx, x[g][e]);
        mn = min_nan(mn, (full || (t * G + g) * GS + lane * V + e < M) ? x[g][e] : pos_inf());
      }
    cluster_round<C, 3>(sh, buf, t, lane, uint32_t(__reduce_max_sync(0xffffffffu, f2o(mx))),
                        uint32_t(__reduce_min_sync(0xffffffffu, f2o(mn))),
                        uint32_t(__reduce_min_sync(0xffffffffu, f2o(mx))));
    float hi = o2f(team_max<C>(sh, buf, 0, lane));
    float lo = o2f(team_min<C>(sh, buf, 1, lane));
    const float floor_v = o2f(team_min<C>(sh, buf, 2, lane));
    buf ^= 1;
    const bool ok = (lo >= -1e38f && hi <= 1e38f);
    if (!ok) st |= (isfinite(lo) && isfinite(hi)) ? kStatusRange : kStatusNonFinite;

    // ---- round: ties at the maximum
    unsigned cmax = 0;
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
      for (int e = 0; e < V; ++e) cmax += (x[g][e] >= hi) ? 1u : 0u;
    cluster_round<C, 1>(sh, buf, t, lane, __reduce_add_sync(0xffffffffu, cmax));
    const bool max_tie = int(team_sum<C>(sh, buf, 0, lane, TW)) >= k;
    buf ^= 1;

    // ---- bisection: one round per pass
    int it = 0;
    bool eq = false;
    int last = buf;
    int lastw = 0;  // which of the last round's counts the last pass used
    if (max_tie) {
      lo = hi;           // keep the k lowest-index maxima through the fill rule:
      hi = pos_inf();    // S is empty and every maximum is borderline
    } else {
      if (floor_lo && ok) lo = fmaxf(lo, floor_v);
      // Each round settles up to two passes: it counts at the midpoint m1 and
      // at both midpoints the second pass can take, mid(lo, m1) and mid(m1, hi)
      // (the same binary32 values the second pass computes), so the passes,
      // their order and every stop test are exactly those of plain bisection.
      auto stop_before_pass = [&]() -> bool {
        if (EXACT) {
          if (it >= kSafetyCap) { st |= kStatusSafetyCap; return true; }
          return false;
        }
        if (it >= limit) {
          if (cap_is_safety) st |= kStatusSafetyCap;
          return true;
        }
        return !(__fsub_rn(hi, lo) > eps);
      };
      // one pass with count cnt at mid; true when the search is over
      auto take_pass = [&](float mid, int cnt) -> bool {
        ++it;
        const bool ge = cnt >= k;
        lo = ge ? mid : lo;
        hi = ge ? hi : mid;
        if (cnt == k) { eq = true; return true; }
        // one bf16 value left in [lo, hi): the kept set is final
        return V == 8 && bf16_stop && __fsub_rn(hi, lo) <= fmaxf(fabsf(lo), fabsf(hi)) * 0.015625f + 1e-38f &&
               bf16_single_value(lo, hi);
      };
      // Exact mode without pass counts: the round's middle probe is a guess --
      // the cluster's previous threshold in the first round, then the point
      // where the count, interpolated linearly between the bracket ends'
      // counts, crosses k + 1/2 -- and the outer probes the midpoints of the
      // two sub-brackets, so a poor guess still halves the bracket. Any count
      // of exactly k ends the search with the exact fill; the set is the same
      // whatever probes are taken. fp32 rows only: GB300, fp32 N(0,1), k = 64
      // / 256 / 1024: M = 16384 863 / 926 / 1070 -> 826 / 843 / 928 us, M =
      // 65536 850 / 910 / 978 -> 833 / 853 / 844 us; bf16 rows (ties at the
      // k-th value end on the single-value test anyway) were 1-3% slower.
      if (EXACT && iters == nullptr && V == 4) {
        int c_lo = M, c_hi = int(team_sum<C>(sh, buf ^ 1, 0, lane, TW));  // C(hi) from the max-tie round
        bool first = true;
        for (;;) {
          if (it >= kSafetyCap) {
            st |= kStatusSafetyCap;
            break;
          }
          const float mid = __fmul_rn(__fadd_rn(lo, hi), 0.5f);
          if (!(lo < mid && mid < hi)) break;  // no binary32 value strictly inside
          float g = first ? tprev
                          : fmaf(hi - lo, (float(c_lo - k) - 0.5f) / float(c_lo - c_hi), lo);
          first = false;
          const float m1 = (lo < g && g < hi) ? g : mid;
          const float mL = __fmul_rn(__fadd_rn(lo, m1), 0.5f);
          const float mR = __fmul_rn(__fadd_rn(m1, hi), 0.5f);
          unsigned l1, lL, lR;
          lane_count_lt3<G, V>(x, m1, mL, mR, l1, lL, lR);
          cluster_round<C, 3>(sh, buf, t, lane, unsigned(32 * NE) - __reduce_add_sync(0xffffffffu, l1),
                              unsigned(32 * NE) - __reduce_add_sync(0xffffffffu, lL),
                              unsigned(32 * NE) - __reduce_add_sync(0xffffffffu, lR));
          const int c1 = int(team_sum<C>(sh, buf, 0, lane, TW));
          const int cL = int(team_sum<C>(sh, buf, 1, lane, TW));
          const int cR = int(team_sum<C>(sh, buf, 2, lane, TW));
          last = buf;
          buf ^= 1;
          ++it;
          // counts are non-increasing in the threshold: mL <= m1 <= mR
          if (cL == k || c1 == k || cR == k) {
            lastw = cL == k ? 1 : (c1 == k ? 0 : 2);
            lo = cL == k ? mL : (c1 == k ? m1 : mR);
            eq = true;
            break;
          }
          if (cR > k) {
            lo = mR; c_lo = cR;
          } else if (c1 > k) {
            lo = m1; c_lo = c1; hi = mR; c_hi = cR;
          } else if (cL > k) {
            lo = mL; c_lo = cL; hi = m1; c_hi = c1;
          } else {
            hi = mL; c_hi = cL;
          }
          // one bf16 value left in [lo, hi): the kept set is final
          if (V == 8 && __fsub_rn(hi, lo) <= fmaxf(fabsf(lo), fabsf(hi)) * 0.015625f + 1e-38f &&
              bf16_single_value(lo, hi))
            break;
        }
        if (eq) tprev = lo;
      }
      for (;;) {
        if (EXACT && iters == nullptr && V == 4) break;  // searched above
        if (stop_before_pass()) break;
        const float m1 = __fmul_rn(__fadd_rn(lo, hi), 0.5f);
        if (!(lo < m1 && m1 < hi)) break;
        const float mL = __fmul_rn(__fadd_rn(lo, m1), 0.5f);
        const float mR = __fmul_rn(__fadd_rn(m1, hi), 0.5f);
        unsigned l1, lL, lR;
        lane_count_lt3<G, V>(x, m1, mL, mR, l1, lL, lR);
        cluster_round<C, 3>(sh, buf, t, lane, unsigned(32 * NE) - __reduce_add_sync(0xffffffffu, l1),
                            unsigned(32 * NE) - __reduce_add_sync(0xffffffffu, lL),
                            unsigned(32 * NE) - __reduce_add_sync(0xffffffffu, lR));
        const int c1 = int(team_sum<C>(sh, buf, 0, lane, TW));
        const int cL = int(team_sum<C>(sh, buf, 1, lane, TW));
        const int cR = int(team_sum<C>(sh, buf, 2, lane, TW));
        last = buf;
        buf ^= 1;
        lastw = 0;
        if (take_pass(m1, c1)) break;
        if (stop_before_pass()) break;
        const bool right = c1 >= k;  // pass 1 moved lo up to m1
        const float m2 = __fmul_rn(__fadd_rn(lo, hi), 0.5f);  // == (right ? mR : mL)
        if (!(lo < m2 && m2 < hi)) break;
        lastw = right ? 2 : 1;
        if (take_pass(m2, right ? cR : cL)) break;
      }
    }

    // ---- fill: positions from team prefixes, stores straight to the CBSR row
    const int64_t obase = r * int64_t(k);
    int preS, preB, need;
    if (ok && eq) {
      // the last pass counted x >= lo for every warp: S = {x >= lo}, B empty
      preS = int(team_sum<C>(sh, last, lastw, lane, t));
      preB = 0;
      need = 0;
      hi = lo;
    } else {
      unsigned cs = 0, cb = 0;
#pragma unroll
      for (int g = 0; g < G; ++g)
#pragma unroll
        for (int e = 0; e < V; ++e) {
          cs += (x[g][e] >= hi) ? 1u : 0u;
          cb += (x[g][e] >= lo && !(x[g][e] >= hi)) ? 1u : 0u;
        }
      cluster_round<C, 2>(sh, buf, t, lane, __reduce_add_sync(0xffffffffu, cs),
                          __reduce_add_sync(0xffffffffu, cb));
      const int sizeS = int(team_sum<C>(sh, buf, 0, lane, TW));
      preS = int(team_sum<C>(sh, buf, 0, lane, t));
      preB = int(team_sum<C>(sh, buf, 1, lane, t));
      buf ^= 1;
      need = max(k - sizeS, 0);
    }
    unsigned pkw[NW];
#pragma unroll
    for (int u = 0; u < NW; ++u) pkw[u] = 0u;
#pragma unroll
    for (int g = 0; g < G; ++g) {
      unsigned cs = 0, cb = 0;
#pragma unroll
      for (int e = 0; e < V; ++e) {
        cs += (x[g][e] >= hi) ? 1u : 0u;
        cb += (x[g][e] >= lo && !(x[g][e] >= hi)) ? 1u : 0u;
      }
      pkw[(2 * g) / FPW] += cs << (FB * ((2 * g) % FPW));
      pkw[(2 * g + 1) / FPW] += cb << (FB * ((2 * g + 1) % FPW));
    }
    unsigned ex[NW], tot[NW];
#pragma unroll
    for (int u = 0; u < NW; ++u) ex[u] = warp_excl_scan(pkw[u], lane, tot[u]);
    int baseS = preS, baseB = preB;
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const int fs = 2 * g, fb = 2 * g + 1;
      int runS = baseS + int((ex[fs / FPW] >> (FB * (fs % FPW))) & FMASK);
      int runB = baseB + int((ex[fb / FPW] >> (FB * (fb % FPW))) & FMASK);
#pragma unroll
      for (int e = 0; e < V; ++e) {
        const float v = x[g][e];
        const unsigned sf = (v >= hi) ? 1u : 0u;
        const unsigned bf = (v >= lo && !(v >= hi)) ? 1u : 0u;
        const int pos = runS + min(runB, need);
        const unsigned keep = (sf | (bf & unsigned(runB < need))) & unsigned(pos < k);
        st_global_if(keep, vals + obase + pos, out_value(v, vals));
        st_global_if(keep, idx + obase + pos, IdxT((t * G + g) * GS + lane * V + e));
        runS += int(sf);
        runB += int(bf);
      }
      baseS += int((tot[fs / FPW] >> (FB * (fs % FPW))) & FMASK);
      baseB += int((tot[fb / FPW] >> (FB * (fb % FPW))) & FMASK);
    }
    if (iters != nullptr && t == 0 && lane == 0) iters[r] = it;
  }
  cluster_barrier();  // no CTA leaves while a peer could still address its shared memory
  st = __reduce_or_sync(0xffffffffu, st);
  if (status != nullptr && st != 0u && lane == 0) atomicOr(status, st);
}

}  // namespace rtopk
