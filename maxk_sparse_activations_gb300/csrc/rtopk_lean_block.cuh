// Exact row-wise top-k on rows of 2048, 4096 and 8192 elements, one team of
// 2, 4 or 8 warps per row, the threshold search counted on packed 16-bit
// images of the row, sm_103a.
//
// Source: "RTop-K: Ultra-Fast Row-Wise Top-K Selection for Neural Network
// Acceleration on GPUs" (summary page), "Approach" (binary search over the
// row's value range for a threshold that selects k; ties filled by the
// lowest index) and "Limitations" (rows up to 8192); CBSR output from
// "MaxK-GNN: Extremely Fast GPU Kernel Design for Accelerating Graph Neural
// Networks Training", "The idea".
//
// The multi-warp version of rtopk_lean.cuh, for exact mode when per-row pass
// counts are not requested. A row belongs to a team of TW warps (TT = 32 * TW
// threads; a block of 256 threads holds 8 / TW teams): thread t of the team
// holds elements [t * NE, (t + 1) * NE) (NE = M / TT, 32 for rows of 2048 and
// 4096 on 2 and 4 warps, 32 for rows of 8192 on 8), rows stream through the
// team's 2-stage cp.async ring in shared memory (the same stage layout as the
// warp kernel's lane slices, swizzled for 4- and 8-chunk slices), and a pass
// counts the sign bits of h - t on the 16-bit images exactly as the warp
// kernel does. The per-pass count is the team sum of the warps' redux.sync
// results, exchanged through two alternating sets of shared slots (a set is
// rewritten two exchanges later, after a barrier that every reader of it has
// passed): one named barrier (bar.sync id, TT) per pass. Every decision that
// guards a barrier derives from team-wide sums, so all threads of a team take
// the same branches. The kept indices go to the team's shared list (k <= 1024)
// through a team prefix scan of thread counts, and all team threads write the
// CBSR row. Fewer warps per row means fewer warps waiting at each barrier and
// more rows in flight per SM (GB300, 2^16 fp32 rows of 2048, k = 64: 8 warps
// per row 374 us, 2 warps 191 us).
#pragma once

#include "rtopk_lean.cuh"

namespace rtopk {
namespace lean {

constexpr int kBlockListK = 1024;  // largest k of the block kernel



// Shared exchange area of one team (the TW warps of a row): two alternating
// slot sets.
struct BlockXchg {
  int isum[2][8];
  float fmax[2][8];
  float fmin[2][8];
  float fmin2[2][8];
  int scan[2][8];
};

// Barrier of one team: named barrier `id` (1..8) over its TW * 32 threads.
template <int TW>
__device__ __forceinline__ void team_sync(int id) {
  if constexpr (TW == 8) {
    __syncthreads();
  } else {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "n"(TW * 32) : "memory");
  }
}

// Team-wide sum of v (every thread of the team calls it).
template <int TW>
__device__ __forceinline__ int block_sum(int v, BlockXchg& x, int& par, int lane, int wib, int bid) {
  const int w = int(warp_sum(uint32_t(v)));
  if (lane == 0) x.isum[par][wib] = w;
  team_sync<TW>(bid);
  int r = 0;
#pragma unroll
  for (int i = 0; i < TW; ++i) r += x.isum[par][i];
  par ^= 1;
  return r;
}

// Team-wide NaN-propagating max of a, min of b and min of c in one exchange.
template <int TW>
__device__ __forceinline__ void block_max_min_min(float& a, float& b, float& c, BlockXchg& x, int& par, int lane,
                                                  int wib, int bid) {
  const float wa = warp_max_nan(a), wb = warp_min_nan(b), wc = warp_min_nan(c);
  if (lane == 0) {
    x.fmax[par][wib] = wa;
    x.fmin[par][wib] = wb;
    x.fmin2[par][wib] = wc;
  }
  team_sync<TW>(bid);
  float ra = x.fmax[par][0], rb = x.fmin[par][0], rc = x.fmin2[par][0];
#pragma unroll
  for (int i = 1; i < TW; ++i) {
    ra = max_nan(ra, x.fmax[par][i]);
    rb = min_nan(rb, x.fmin[par][i]);
    rc = min_nan(rc, x.fmin2[par][i]);
  }
  par ^= 1;
  a = ra;
  b = rb;
  c = rc;
}

// Exclusive team prefix of v; `tot` receives the team total.
template <int TW>
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, uint32_t& tot, BlockXchg& x, int& par, int lane,
                                                    int wib, int bid) {
  uint32_t incl = v;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1)
    asm("{\n\t.reg .pred p;\n\t.reg .u32 t;\n\t"
        "shfl.sync.up.b32 t|p, %0, %1, 0, -1;\n\t"
        "@p add.u32 %0, %0, t;\n\t}"
        : "+r"(incl) : "r"(d));
  if (lane == 31) x.scan[par][wib] = int(incl);
  team_sync<TW>(bid);
  uint32_t before = 0, all = 0;
#pragma unroll
  for (int i = 0; i < TW; ++i) {
    const uint32_t s = uint32_t(x.scan[par][i]);
    before += (i < wib) ? s : 0u;
    all += s;
  }
  par ^= 1;
  tot = all;
  return before + incl - v;
}

// Thread t's RW words of a staged row (4- / 8-chunk slices swizzled as in the
// warp kernel's stage layout, with the thread index in place of the lane).
template <int RW>
__device__ __forceinline__ void thread_words(const uint32_t* __restrict__ srow, int t, uint32_t (&w)[RW]) {
  static_assert(RW % 4 == 0, "whole 16-byte chunks per thread");
#pragma unroll
  for (int c = 0; c < RW / 4; ++c) {
    const uint4 q = *reinterpret_cast<const uint4*>(srow + StageLayout<RW>::chunk_pos(t, c) * 4);
    w[4 * c] = q.x; w[4 * c + 1] = q.y; w[4 * c + 2] = q.z; w[4 * c + 3] = q.w;
  }
}

// Asynchronous copy of one row (TT * RW words, TT threads) into a stage:
// thread t copies chunks t, t + TT, ... (coalesced) to their stage positions.
template <int RW, int TT>
__device__ __forceinline__ void issue_row_block(uint32_t stage, const uint32_t* __restrict__ src_t, int t,
                                                bool valid) {
  using SL = StageLayout<RW>;
#pragma unroll
  for (int i = 0; i < RW / 4; ++i) {
    const int g = t + TT * i;
    const uint32_t dst = stage + uint32_t(SL::chunk_pos(g / SL::CPL, g % SL::CPL)) * 16u;
    if (valid)
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src_t + i * TT * 4) : "memory");
  }
  asm volatile("cp.async.commit_group;" ::: "memory");
}

// The CBSR row from the list (all TT threads of the team; a barrier precedes it).
template <typename T, int RW, int TT, typename IdxT>
__device__ __forceinline__ void copy_out_block(const uint32_t* __restrict__ list, const uint32_t* __restrict__ srow,
                                               int k, int t, T* __restrict__ vrow, IdxT* __restrict__ irow) {
  using SL = StageLayout<RW>;
  for (int p = t; p < k; p += TT) {
    const uint32_t j = list[p];
    T v;
    if constexpr (sizeof(T) == 4) {
      v = __uint_as_float(srow[SL::word_of_f32(int(j))]);
    } else {
      v = reinterpret_cast<const uint16_t*>(srow)[SL::half_of_bf16(int(j))];
    }
    vrow[p] = v;
    irow[p] = IdxT(j);
  }
}

// General fill for a binary32 bracket [lo, hi) with c(lo) >= k > c(hi), over
// the block: keep every x >= hi, then the first k - c(hi) of lo <= x < hi in
// index order.
template <int NE, int TW>
__device__ __forceinline__ void stage_general_block(const float (&x)[NE], float lo, float hi, int k, int t,
                                                    uint32_t* __restrict__ list, BlockXchg& xc, int& par, int lane,
                                                    int wib, int bid) {
  uint32_t sc = 0, bc = 0;
#pragma unroll
  for (int e = 0; e < NE; ++e) {
    const bool s = x[e] >= hi;
    sc += s ? 1u : 0u;
    bc += (!s && x[e] >= lo) ? 1u : 0u;
  }
  uint32_t tot;
  const uint32_t ex = block_excl_scan<TW>(sc | (bc << 16), tot, xc, par, lane, wib, bid);
  const int need = k - int(tot & 0xffffu);
  int bpos = int(ex >> 16);
  int pos = int(ex & 0xffffu) + min(bpos, need);
#pragma unroll
  for (int e = 0; e < NE; ++e) {
    const bool s = x[e] >= hi;
    const bool b = !s && x[e] >= lo;
    if (s || (b && bpos < need)) {
      list[pos] = uint32_t(t * NE + e);
      ++pos;
    }
    bpos += b ? 1 : 0;
  }
}

template <typename T, int NE, int TW, typename IdxT>
__device__ __forceinline__ void process_row_block(const uint32_t* __restrict__ srow, int k, int t, int lane, int wib,
                                                  int bid, uint32_t* __restrict__ list, BlockXchg& xc, int& par,
                                                  float& tprev, float& rho, T* __restrict__ vrow,
                                                  IdxT* __restrict__ irow, uint32_t& st) {
  constexpr int TT = TW * 32;  // threads of the team
  using P = Packed16<T>;
  using I = Img<T>;
  constexpr int RW = Lane<T, NE>::RW;
  constexpr int W = Lane<T, NE>::W;
  uint32_t raw[RW];
  thread_words<RW>(srow, t, raw);

  // ---- image, range and precondition (one exchange)
  uint32_t h[W];
  float hi32, lo_row, lo_max;
  if constexpr (sizeof(T) == 4) {
    float x[NE];
    widen<T, NE>(raw, x);
#pragma unroll
    for (int w = 0; w < W; ++w) h[w] = P::pack(x[2 * w + 1], x[2 * w]);
    float a = fabsf(x[0]);
    int i = 1;
#pragma unroll
    for (; i + 1 < NE; i += 2) a = max3_nan(a, fabsf(x[i]), fabsf(x[i + 1]));
    if (i < NE) a = max_nan(a, fabsf(x[i]));
    hi32 = a;
    lo_row = -a;
    lo_max = lane_max<NE>(x);
  } else {
#pragma unroll
    for (int w = 0; w < W; ++w) h[w] = raw[w];
    uint32_t m = h[0], n = h[0];
#pragma unroll
    for (int w = 1; w < W; ++w) {
      m = I::max2(m, h[w]);
      n = I::min2(n, h[w]);
    }
    hi32 = __uint_as_float(I::max2(m, __byte_perm(m, 0, 0x1032)) & 0xffff0000u);
    lo_row = __uint_as_float(I::min2(n, __byte_perm(n, 0, 0x1032)) & 0xffff0000u);
    lo_max = hi32;
  }
  block_max_min_min<TW>(hi32, lo_row, lo_max, xc, par, lane, wib, bid);
  // fp32: hi32 = max |x|, lo_row = -max |x|; bf16: the row maximum and minimum
  if (!(hi32 <= 1e38f && lo_row >= -1e38f)) {
    float x[NE];
    uint32_t w2[RW];
    thread_words<RW>(srow, t, w2);
    widen<T, NE>(w2, x);
    bool nonfinite = false, range = false;
#pragma unroll
    for (int e = 0; e < NE; ++e) {
      const float a = fabsf(x[e]);
      nonfinite |= !(a <= 3.402823466e38f);
      range |= (a > 1e38f && a <= 3.402823466e38f);
    }
    // flags of all threads: counts of threads with each flag, in two fields
    const int bad = block_sum<TW>((nonfinite ? 1 : 0) + (range ? 0x10000 : 0), xc, par, lane, wib, bid);
    if (bad & 0xffff) st |= kStatusNonFinite;
    if (bad >> 16) st |= kStatusRange;
    for (int p = t; p < k; p += TT) list[p] = uint32_t(p);
    team_sync<TW>(bid);
    copy_out_block<T, RW, TT, IdxT>(list, srow, k, t, vrow, irow);
    return;
  }
  // lower end: each of the TT threads holds an element >= its maximum
  const float lo_src = (k <= TT) ? lo_max : lo_row;

  // ---- coarse bisection on 16-bit images (sign-bit counts, negated bracket)
#pragma unroll
  for (int w = 0; w < W; ++w) h[w] = P::add(h[w], 0u);  // no image is -0
  uint32_t lo2 = P::splat(lo_src);
  uint32_t hi2 = sizeof(T) == 4 ? P::splat(hi32) + 0x00010001u : next_up16(P::splat(hi32));
  if constexpr (sizeof(T) == 4) {
    if (hi2 == 0x7c007c00u) {
      // max |x| saturates the binary16 image (|x| >= 65488): a bracket up to
      // +inf would collapse at its first midpoint. Count the images at +65504
      // and -65504 and take the extremes of the others (one exchange each),
      // then start from a bracket that still has C(lo) >= k > C(hi):
      //   C(65504) >= k: [65504, +inf), the binary32 finish over those;
      //   else hi = the 16-bit value above the largest other image (or 65504),
      //   and for k > TT lo = the smallest other image when at least k images
      //   lie above -65504 (else -65504, where C = M).
      int sat = 0;
      float mxn = neg_inf(), mnn = pos_inf();
#pragma unroll
      for (int w = 0; w < W; ++w) {
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const float hv = half ? P::high_f32(h[w]) : P::low_f32(h[w]);
          const bool ps = hv == 65504.0f, ns = hv == -65504.0f;
          sat += (ps ? 1 : 0) + (ns ? 0x10000 : 0);
          mxn = (ps || ns) ? mxn : fmaxf(mxn, hv);
          mnn = (ps || ns) ? mnn : fminf(mnn, hv);
        }
      }
      const int both = block_sum<TW>(sat, xc, par, lane, wib, bid);
      float unused = pos_inf();
      block_max_min_min<TW>(mxn, mnn, unused, xc, par, lane, wib, bid);
      const int npos = both & 0xffff, nneg = both >> 16;
      if (npos >= k) {
        lo2 = 0x7bff7bffu;
      } else {
        hi2 = mxn == neg_inf() ? 0x7bff7bffu : next_up16(P::splat(mxn));
        if (k > TT) lo2 = (TT * NE - nneg >= k && mnn != pos_inf()) ? P::splat(mnn) : 0xfbfffbffu;
      }
    }
  }
  uint32_t nlo2 = lo2 ^ 0x80008000u, nhi2 = hi2 ^ 0x80008000u;
  const int kneg = k - TT * NE;  // C >= k  iff  -(negatives) >= k - M
  // Probes: the team's previous threshold first, then Newton steps
  // t + (C(t) - k - 1/2) / rho with the density rho (elements per unit value
  // near the threshold) estimated on earlier rows; a probe that is not
  // strictly inside the bracket (as a 16-bit value) is replaced by the
  // midpoint. Exact mode selects one set whatever thresholds are visited, so
  // the guesses change the pass count only (CPU emulation, 2^11 .. 2^13
  // columns, k = 64 .. 1024: 8-12.5 passes -> 4-5; GB300, 2^16 fp32 rows:
  // M = 2048 k = 256 227 -> 182 us, M = 4096 k = 1024 496 -> 400 us, M = 8192
  // k = 64 797 -> 717 us; bf16 rows, which often end tied, gain up to 18%
  // at k = 1024 and lose 4% at M = 2048, k = 64). At most kGuesses probes
  // of a row are guesses, so a poor density estimate (steps of one 16-bit
  // value) costs at most that many extra passes. tprev, rho and
  // every quantity below derive from team-wide sums, so all threads of the
  // team take the same branches.
  float lo_f = P::low_f32(lo2), hi_f = P::low_f32(hi2);
  const float inv_rho = rho > 0.0f ? 1.0f / rho : 0.0f;
  float t_last = tprev, t_first = 0.0f;
  int c_last = 0, c_first = 0;  // C - k at the last / first probe
  bool first = true;
  constexpr int kGuesses = 8;
  for (int pass = 0;; ++pass) {
    // guess: the previous row's threshold (NaN when none), then Newton
    const float tg = first ? tprev : fmaf(float(c_last) - 0.5f, inv_rho, t_last);
    const uint32_t ng2 = P::splat(-tg);  // negated image of the guess
    const float gv = -P::low_f32(ng2);
    uint32_t nm2;
    if (pass < kGuesses && lo_f < gv && gv < hi_f) {
      nm2 = ng2;
    } else {
      nm2 = P::midpoint(nlo2, nhi2);
      if (nm2 == nlo2 || nm2 == nhi2) break;  // no 16-bit value strictly inside
    }
    int acc = 0;
#pragma unroll
    for (int w = 0; w + 1 < W; w += 2) acc = sum_bytes(half_signs(P::add(h[w], nm2), P::add(h[w + 1], nm2)), acc);
    const int tot = block_sum<TW>(acc, xc, par, lane, wib, bid);
    const float mv = -P::low_f32(nm2);  // the probe's value
    if (tot == kneg) {
      // C(mid) == k: {h >= mid} is the top-k; this thread keeps NE + acc.
      // The differences are formed again here rather than kept through the
      // team barrier (16 fewer live registers across every pass).
      uint32_t d[W];
#pragma unroll
      for (int w = 0; w < W; ++w) d[w] = P::add(h[w], nm2);
      if (!first && c_first != 0 && t_first != mv) {
        const float est = fabsf(float(c_first)) / fabsf(t_first - mv);
        rho = rho > 0.0f ? 0.8f * rho + 0.2f * est : est;
      }
      tprev = mv;
      uint32_t all;
      const uint32_t ex = block_excl_scan<TW>(uint32_t(NE + acc), all, xc, par, lane, wib, bid);
      int pos = int(ex);
#pragma unroll
      for (int w = 0; w < W; ++w) {
        if ((d[w] & 0x8000u) == 0u) list[pos++] = uint32_t(t * NE + 2 * w);
        if (int(d[w]) >= 0) list[pos++] = uint32_t(t * NE + 2 * w + 1);
      }
      team_sync<TW>(bid);
      copy_out_block<T, RW, TT, IdxT>(list, srow, k, t, vrow, irow);
      return;
    }
    const bool ge = tot >= kneg;
    nlo2 = ge ? nm2 : nlo2;
    nhi2 = ge ? nhi2 : nm2;
    lo_f = ge ? mv : lo_f;
    hi_f = ge ? hi_f : mv;
    c_last = tot - kneg;
    t_last = mv;
    if (first) {
      c_first = c_last;
      t_first = mv;
      first = false;
    }
  }
  tprev = lo_f;  // collapsed: the threshold lies in [lo, hi)

  // ---- collapsed: the rest of the top-k lies in the bucket {lo <= h < hi}
  float x[NE];
  {
    uint32_t w2[RW];
    thread_words<RW>(srow, t, w2);
    widen<T, NE>(w2, x);
  }
  const float lo = P::low_f32(nlo2 ^ 0x80008000u), hi = P::low_f32(nhi2 ^ 0x80008000u);
  if (sizeof(T) == 2 && next_up_bf16(lo) == hi) {
    stage_general_block<NE, TW>(x, lo, hi, k, t, list, xc, par, lane, wib, bid);
  } else {
    float bmin = pos_inf(), bmax = neg_inf();
#pragma unroll
    for (int w = 0; w < W; ++w) {
      const float hl = P::low_f32(h[w]), hh = P::high_f32(h[w]);
      const bool il = hl >= lo && !(hl >= hi);
      const bool ih = hh >= lo && !(hh >= hi);
      bmin = fminf(bmin, il ? x[2 * w] : pos_inf());
      bmax = fmaxf(bmax, il ? x[2 * w] : neg_inf());
      bmin = fminf(bmin, ih ? x[2 * w + 1] : pos_inf());
      bmax = fmaxf(bmax, ih ? x[2 * w + 1] : neg_inf());
    }
    float dummy = pos_inf();
    block_max_min_min<TW>(bmax, bmin, dummy, xc, par, lane, wib, bid);
    // exact binary32 search on order-preserving keys (as the warp kernel's
    // finish: at most 32 passes for any range, e.g. up to 1e30 outliers)
    int olo = f2o(bmin), ohi = f2o(next_up_f32(bmax));
    for (int it = 0;; ++it) {
      const uint32_t gap = uint32_t(ohi) - uint32_t(olo);
      if (gap < 2u) break;
      if (it >= kSafetyCap) {
        st |= kStatusSafetyCap;
        break;
      }
      const int om = olo + int(gap >> 1);
      const float mid = o2f(om);
      int c = 0;
#pragma unroll
      for (int e = 0; e < NE; ++e) c += (x[e] >= mid) ? 1 : 0;
      const int cnt = block_sum<TW>(c, xc, par, lane, wib, bid);
      if (cnt >= k) olo = om;
      else ohi = om;
      if (cnt == k) break;
    }
    const float flo = o2f(olo), fhi = o2f(ohi);
    stage_general_block<NE, TW>(x, flo, fhi, k, t, list, xc, par, lane, wib, bid);
  }
  team_sync<TW>(bid);
  copy_out_block<T, RW, TT, IdxT>(list, srow, k, t, vrow, irow);
}

// A row of M = TW * 32 * NE elements on a team of TW warps; a block of 256
// threads holds 8 / TW teams (rows in flight), each with its own two stages,
// list and exchange slots. Resident blocks per SM (registers; at most about
// 70 KB of shared memory per block): 5 at 8 elements per thread, 3 at 16, 2 at
// 32 (up to 128 registers, no spills; GB300, 2^16 rows: M = 2048 fp32 k = 64
// 268 -> 191 us against 3 blocks, M = 8192 fp32 k = 256 1184 -> 955 us; at 3
// blocks the 80-register build spills 110-180 bytes, M = 4096 k = 256 387 ->
// 564 us).
template <typename T, int NE, int TW>
struct LeanBlockCfg {
  static constexpr int RW = Lane<T, NE>::RW;
  static constexpr int kTeams = 8 / TW;
  static constexpr int kBlocks = NE <= 8 ? 5 : (NE < 32 ? 3 : 2);
  static constexpr size_t kTeamWords = size_t(2) * TW * 32 * RW + kBlockListK + sizeof(BlockXchg) / 4;
  static constexpr size_t kSmem = kTeams * kTeamWords * 4;
};

// Full rows of TW * 32 * NE elements, exact mode, k <= kBlockListK, 16-byte
// aligned. One team of TW warps per row, persistent over rows, two rows in
// flight per team.
template <typename T, int NE, int TW, typename IdxT>
__global__ void __launch_bounds__(256, LeanBlockCfg<T, NE, TW>::kBlocks)
rtopk_lean_block_kernel(const T* __restrict__ in, int64_t N, int k, T* __restrict__ vals, IdxT* __restrict__ idx,
                        uint32_t* __restrict__ status) {
  using Cfg = LeanBlockCfg<T, NE, TW>;
  constexpr int RW = Lane<T, NE>::RW;
  constexpr int TT = TW * 32;
  constexpr int kRowWords = TT * RW;
  extern __shared__ __align__(16) uint32_t lb_smem[];
  const int team = threadIdx.x / TT;
  const int t = threadIdx.x % TT;  // thread index within the team
  const int lane = t & 31, wib = t >> 5;
  const int bid = team + 1;  // named barrier of the team
  uint32_t* base = lb_smem + size_t(team) * Cfg::kTeamWords;
  uint32_t* ring = base;                     // 2 stages of kRowWords
  uint32_t* list = base + 2 * kRowWords;     // kBlockListK entries
  BlockXchg& xc = *reinterpret_cast<BlockXchg*>(list + kBlockListK);
  const int64_t r0 = int64_t(blockIdx.x) * Cfg::kTeams + team;
  const int64_t nt = int64_t(gridDim.x) * Cfg::kTeams;
  const int nrows = r0 < N ? int((N - 1 - r0) / nt) + 1 : 0;
  const uint32_t ring_base = static_cast<uint32_t>(__cvta_generic_to_shared(ring));
  const uint32_t* src = reinterpret_cast<const uint32_t*>(in) + r0 * kRowWords + t * 4;
  const int64_t src_step = nt * kRowWords;
  int par = 0;
  uint32_t st = 0;
  float tprev = __int_as_float(0x7fc00000), rho = 0.0f;  // search guesses carried across the team's rows
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    issue_row_block<RW, TT>(ring_base + uint32_t(q * kRowWords * 4), src, t, q < nrows);
    src += src_step;
  }
  T* vrow = vals + r0 * int64_t(k);
  IdxT* irow = idx + r0 * int64_t(k);
  const int64_t out_step = nt * int64_t(k);
  int q = 0;
  for (int i = 0; i < nrows; ++i) {
    asm volatile("cp.async.wait_group 1;" ::: "memory");
    team_sync<TW>(bid);  // every team thread's copies of this row are visible
    process_row_block<T, NE, TW, IdxT>(ring + q * kRowWords, k, t, lane, wib, bid, list, xc, par, tprev, rho, vrow,
                                       irow, st);
    team_sync<TW>(bid);  // every team thread is done with this stage and the list
    issue_row_block<RW, TT>(ring_base + uint32_t(q * kRowWords * 4), src, t, i + 2 < nrows);
    src += src_step;
    vrow += out_step;
    irow += out_step;
    q ^= 1;
  }
  asm volatile("cp.async.wait_group 0;" ::: "memory");
  if (status != nullptr && st != 0u && t == 0) atomicOr(status, st);
}

}  // namespace lean
}  // namespace rtopk
