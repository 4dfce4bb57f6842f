// Exact row-wise top-k, one warp per row, with the threshold search counted on
// packed 16-bit images of the row (two elements per instruction), sm_103a.
//
// Source: "RTop-K: Ultra-Fast Row-Wise Top-K Selection for Neural Network
// Acceleration on GPUs" (summary page), "Approach" (binary search over the
// row's value range for a threshold that selects k; ties at the threshold
// filled by the lowest index); CBSR output from "MaxK-GNN: Extremely Fast GPU
// Kernel Design for Accelerating Graph Neural Networks Training", "The idea".
//
// Used for exact mode (max_iter < 0, eps == 0) when per-row pass counts are
// not requested. The result there is one set -- the k largest values, ties at
// the k-th value broken by the lowest index -- whatever thresholds the
// bisection visits, so the search may run on any order-preserving image of the
// row. Here the image h(x) is 16 bits wide:
//  * bf16 rows: the data themselves (h(x) = x, counts exact);
//  * fp32 rows: binary16 rounded to nearest, saturated at +-65504. Rounding is
//    monotone (x <= y implies h(x) <= h(y)), so for any 16-bit threshold t the
//    set {h(x) >= t} is an upper set of the row in value order.
// One pass counts C(t) = #{h(x) >= t} with one packed compare (set.ge.*x2,
// 1.0 or 0.0 per half) and one packed add per two elements, instead of two
// instructions per element on binary32. The coarse bisection keeps
// C(lo) >= k > C(hi) on 16-bit values lo < hi:
//  * C(mid) == k: {h(x) >= mid} has exactly k members and is an upper set, so
//    it is the exact top-k (two equal values have equal images: no tie at the
//    k-th value can straddle it). Stored straight from the packed compares.
//  * no 16-bit value strictly inside (lo, hi): A = {h(x) >= hi} (|A| < k) is
//    kept, everything below lo is dropped, and the rest of the top-k lies in
//    the bucket B = {lo <= h(x) < hi}, all of whose values are below A's and
//    above the dropped ones. The binary32 search then finishes from
//    [min B, next binary32 above max B], a valid bracket (c(min B) >= k,
//    c(above max B) = |A| < k), and the general fill writes the row. For bf16
//    rows lo and hi are adjacent, B holds one value, and the fill runs at once.
// Rows whose values are not all finite with |x| <= 1e38 take the binary32
// kernel's path (status bits, bounded search).
//
// Counting detail: the per-lane accumulator starts at 1024.0 (binary16) or
// 128.0 (bf16) in both halves, where the spacing is 1, so adding 1.0 per kept
// element is exact and the field bits read (magic + count). One integer
// multiply-add folds the two halves into bits 16..31 and removes the offsets,
// and one redux.sync sums the lanes.
#pragma once

#include "rtopk_warp.cuh"

namespace rtopk {

template <typename T>
struct Packed16;

// fp32 rows: binary16 image
template <>
struct Packed16<float> {
  static constexpr uint32_t kHalf2 = 0x38003800u;  // 0.5 in both halves
  // (lo + hi) / 2 with one rounding: lo * 0.5 + (hi * 0.5); lies in [lo, hi]
  static __device__ __forceinline__ uint32_t midpoint(uint32_t lo2, uint32_t hi2) {
    uint32_t t, d;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(t) : "r"(hi2), "r"(kHalf2));
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(lo2), "r"(kHalf2), "r"(t));
    return d;
  }
  // lo < m < hi, on one half (both halves of each operand are equal)
  static __device__ __forceinline__ bool strictly_inside(uint32_t lo2, uint32_t m2, uint32_t hi2) {
    uint32_t r;
    asm("{\n\t.reg .pred a, b, c, d;\n\t"
        "setp.gt.f16x2 a|b, %1, %2;\n\t"
        "setp.lt.and.f16x2 c|d, %1, %3, a;\n\t"
        "selp.u32 %0, 1, 0, c;\n\t}"
        : "=r"(r) : "r"(m2), "r"(lo2), "r"(hi2));
    return r != 0u;
  }
  static constexpr uint32_t kMagic2 = 0x64006400u;  // 1024.0 in both halves
  static constexpr uint32_t kFold = 0xc8006400u;     // (2 * 0x6400 << 16) + 0x6400
  static constexpr uint32_t kInf2 = 0x7c007c00u;     // +inf in both halves
  // both halves = round-to-nearest binary16 of v, saturated at +-65504
  static __device__ __forceinline__ uint32_t splat(float v) {
    uint32_t d;
    asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %1;" : "=r"(d) : "f"(v));
    return d;
  }
  // the pair (hi element, lo element) -> one word (lo element in bits 0..15)
  static __device__ __forceinline__ uint32_t pack(float hi_elem, float lo_elem) {
    uint32_t d;
    asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi_elem), "f"(lo_elem));
    return d;
  }
  static __device__ __forceinline__ float low_f32(uint32_t w) {
    float f;
    asm("{\n\t.reg .b16 l, u;\n\tmov.b32 {l, u}, %1;\n\tcvt.f32.f16 %0, l;\n\t}" : "=f"(f) : "r"(w));
    return f;
  }
  static __device__ __forceinline__ float high_f32(uint32_t w) {
    float f;
    asm("{\n\t.reg .b16 l, u;\n\tmov.b32 {l, u}, %1;\n\tcvt.f32.f16 %0, u;\n\t}" : "=f"(f) : "r"(w));
    return f;
  }
  static __device__ __forceinline__ uint32_t set_ge(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("set.ge.f16x2.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
  }
  static __device__ __forceinline__ uint32_t add(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("add.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
  }
};

// bf16 rows: the data themselves
template <>
struct Packed16<uint16_t> {
  static constexpr uint32_t kHalf2 = 0x3f003f00u;  // 0.5 in both halves
  // (lo + hi) / 2 with one rounding: lo * 0.5 + (hi * 0.5); lies in [lo, hi]
  static __device__ __forceinline__ uint32_t midpoint(uint32_t lo2, uint32_t hi2) {
    uint32_t t, d;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(t) : "r"(hi2), "r"(kHalf2));
    asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(lo2), "r"(kHalf2), "r"(t));
    return d;
  }
  // lo < m < hi, on one half (both halves of each operand are equal)
  static __device__ __forceinline__ bool strictly_inside(uint32_t lo2, uint32_t m2, uint32_t hi2) {
    uint32_t r;
    asm("{\n\t.reg .pred a, b, c, d;\n\t"
        "setp.gt.bf16x2 a|b, %1, %2;\n\t"
        "setp.lt.and.bf16x2 c|d, %1, %3, a;\n\t"
        "selp.u32 %0, 1, 0, c;\n\t}"
        : "=r"(r) : "r"(m2), "r"(lo2), "r"(hi2));
    return r != 0u;
  }
  static constexpr uint32_t kMagic2 = 0x43004300u;  // 128.0 in both halves
  static constexpr uint32_t kFold = 0x86004300u;     // (2 * 0x4300 << 16) + 0x4300
  static constexpr uint32_t kInf2 = 0x7f807f80u;
  static __device__ __forceinline__ uint32_t splat(float v) {
    uint32_t d;
    asm("cvt.rn.bf16x2.f32 %0, %1, %1;" : "=r"(d) : "f"(v));
    return d;
  }
  static __device__ __forceinline__ uint32_t pack(float hi_elem, float lo_elem) {
    return (__float_as_uint(hi_elem) & 0xffff0000u) | (__float_as_uint(lo_elem) >> 16);  // exact: bf16 data
  }
  static __device__ __forceinline__ float low_f32(uint32_t w) { return __uint_as_float(w << 16); }
  static __device__ __forceinline__ float high_f32(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
  static __device__ __forceinline__ uint32_t set_ge(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("set.ge.bf16x2.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
  }
  static __device__ __forceinline__ uint32_t add(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("add.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
  }
};

// Number of this lane's packed elements with h >= t in words [w0, w0 + n),
// shifted into bits 16..31 (low bits hold junk below 2^16).
template <typename P, int NW>
__device__ __forceinline__ uint32_t packed_count_hi16(const uint32_t (&h)[NW], int w0, int n, uint32_t t2) {
  uint32_t acc = P::add(P::kMagic2, P::set_ge(h[w0], t2));
#pragma unroll
  for (int q = 1; q < n; ++q) acc = P::add(acc, P::set_ge(h[w0 + q], t2));
  return acc * 0x10001u - P::kFold;  // (c_hi + c_lo) << 16 | c_lo
}

// Smallest binary32 above v (v finite).
__device__ __forceinline__ float next_up_f32(float v) {
  const int b = __float_as_int(v);
  if ((b & 0x7fffffff) == 0) return __int_as_float(1);
  return __int_as_float(b >= 0 ? b + 1 : b - 1);
}

// Smallest bf16 above v (v a finite bf16 value widened to binary32).
__device__ __forceinline__ float next_up_bf16(float v) {
  const uint32_t b = __float_as_uint(v);
  if ((b & 0x7fffffffu) == 0u) return __uint_as_float(0x10000u);
  return __uint_as_float((b & 0x80000000u) ? b - 0x10000u : b + 0x10000u);
}

// Stages one kept element when `flag` is set: its value bits at word `pos` of
// the warp's staging area and its index 256 words further on, then advances
// pos. HALF selects the flag's half-word (0: bits 0..15, 1: bits 16..31).
template <int HALF>
__device__ __forceinline__ void stage_split_if(uint32_t flag, int& pos, uint32_t sbase, uint32_t v, int j) {
  if (HALF == 0) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t.reg .u32 a, t;\n\t"
        "and.b32 t, %1, 65535;\n\t"
        "setp.ne.u32 p, t, 0;\n\t"
        "mad.lo.u32 a, %0, 4, %2;\n\t"
        "@p st.shared.b32 [a], %3;\n\t"
        "@p st.shared.b32 [a+1024], %4;\n\t"
        "@p add.s32 %0, %0, 1;\n\t}"
        : "+r"(pos) : "r"(flag), "r"(sbase), "r"(v), "r"(j) : "memory");
  } else {
    asm volatile(
        "{\n\t.reg .pred p;\n\t.reg .u32 a;\n\t"
        "setp.ge.u32 p, %1, 65536;\n\t"
        "mad.lo.u32 a, %0, 4, %2;\n\t"
        "@p st.shared.b32 [a], %3;\n\t"
        "@p st.shared.b32 [a+1024], %4;\n\t"
        "@p add.s32 %0, %0, 1;\n\t}"
        : "+r"(pos) : "r"(flag), "r"(sbase), "r"(v), "r"(j) : "memory");
  }
}

// Exclusive warp prefix of packed per-lane counts (as warp_excl_scan), each
// step a shfl.up whose in-range predicate guards the add. Used by the bf16
// instances: GB300, 2^20 x 256 bf16, k = 32: 411.6 against 429.2 us; the fp32
// instance measured faster with warp_excl_scan (397.3 against 405.3 us).
__device__ __forceinline__ unsigned warp_excl_scan_pred(unsigned v, unsigned& tot) {
  unsigned s = v;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1)
    asm("{\n\t.reg .pred p;\n\t.reg .u32 t;\n\t"
        "shfl.sync.up.b32 t|p, %0, %1, 0, -1;\n\t"
        "@p add.u32 %0, %0, t;\n\t}"
        : "+r"(s) : "r"(d));
  tot = __shfl_sync(0xffffffffu, s, 31);
  return s - v;
}

// Packed compares of one pass: s[w] = (h[w] >= t2) per half (1.0 or 0.0), and
// cum[g] = magic + the 1.0s of groups 0..g, accumulated in the 16-bit format.
template <typename P, int G, int WG>
__device__ __forceinline__ void packed_pass(const uint32_t (&h)[G * WG], uint32_t t2, uint32_t (&s)[G * WG],
                                            uint32_t (&cum)[G]) {
  uint32_t acc = P::kMagic2;
#pragma unroll
  for (int g = 0; g < G; ++g) {
#pragma unroll
    for (int q = 0; q < WG; ++q) {
      s[g * WG + q] = P::set_ge(h[g * WG + q], t2);
      acc = P::add(acc, s[g * WG + q]);
    }
    cum[g] = acc;
  }
}

// Lane count held in a packed accumulator (both halves, offsets removed).
template <typename P>
__device__ __forceinline__ uint32_t packed_lane_count(uint32_t acc) {
  return (acc * 0x10001u - P::kFold) >> 16;
}

// Writes the elements of the pass whose compares are s[] / cum[] (exactly k of
// them pass: an upper set of the row) in ascending index order: value bits to
// words [0, k) of the staging area, indices to words [256, 256 + k). The
// per-lane counts and the stored flags come from the same packed compares, so
// the positions fill exactly [0, k).
template <typename T, int G>
__device__ __forceinline__ void compact_packed(const float (&x)[G][ElemTraits<T>::V],
                                               const uint32_t (&s)[G * ElemTraits<T>::V / 2],
                                               const uint32_t (&cum)[G], int lane, float2* __restrict__ stage) {
  using P = Packed16<T>;
  constexpr int V = ElemTraits<T>::V;
  constexpr int WG = V / 2;  // words per group
  constexpr int GS = 32 * V;
  constexpr int FB = (GS <= 255) ? 8 : 16;
  constexpr int FPW = 32 / FB;
  constexpr unsigned FMASK = (1u << FB) - 1u;
  constexpr int NWF = (G + FPW - 1) / FPW;
  unsigned pkw[NWF];
#pragma unroll
  for (int q = 0; q < NWF; ++q) pkw[q] = 0u;
  unsigned prev = 0u;
#pragma unroll
  for (int g = 0; g < G; ++g) {
    const unsigned upto = packed_lane_count<P>(cum[g]);
    pkw[g / FPW] += (upto - prev) << (FB * (g % FPW));
    prev = upto;
  }
  const int jl = lane * V;
  const uint32_t sbase = static_cast<uint32_t>(__cvta_generic_to_shared(stage));
  int base = 0;
#pragma unroll
  for (int q = 0; q < NWF; ++q) {
    unsigned tot;
    const unsigned ex = (sizeof(T) == 2) ? warp_excl_scan_pred(pkw[q], tot) : warp_excl_scan(pkw[q], lane, tot);
#pragma unroll
    for (int f = 0; f < FPW; ++f) {
      const int g = q * FPW + f;
      if (g < G) {
        int pos = base + int((ex >> (FB * f)) & FMASK);
#pragma unroll
        for (int w = 0; w < WG; ++w) {
          stage_split_if<0>(s[g * WG + w], pos, sbase, __float_as_uint(x[g][2 * w]), g * GS + jl + 2 * w);
          stage_split_if<1>(s[g * WG + w], pos, sbase, __float_as_uint(x[g][2 * w + 1]), g * GS + jl + 2 * w + 1);
        }
        base += int((tot >> (FB * f)) & FMASK);
      }
    }
  }
}

template <typename T, int G, typename IdxT>
__device__ __forceinline__ void process_row_packed(const float (&x)[G][ElemTraits<T>::V], int64_t r, int M, int k,
                                                   int lane, float2* __restrict__ stage, T* __restrict__ vals,
                                                   IdxT* __restrict__ idx, uint32_t& st) {
  using P = Packed16<T>;
  constexpr int V = ElemTraits<T>::V;
  constexpr int NE = G * V;
  constexpr int NW = NE / 2;
  constexpr unsigned FULL = 0xffffffffu;

  // ---- value range (binary32, NaN-propagating) and the precondition. For
  // k <= 32 the search starts from the smallest lane maximum, so the row
  // minimum is not needed: the precondition is checked on max |x| instead.
  float mx = neg_inf();
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int e = 0; e < V; ++e) mx = max_nan(mx, x[g][e]);
  const float hi32 = o2f(__reduce_max_sync(FULL, f2o(mx)));
  float lo_src;
  bool valid;
  if (k <= 32) {
    float amax = 0.0f;
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
      for (int e = 0; e < V; ++e) amax = max_nan(amax, fabsf(x[g][e]));
    valid = __all_sync(FULL, amax <= 1e38f);
    // each of the 32 lanes holds an element >= its maximum: C(lane-max minimum) >= 32 >= k
    lo_src = o2f(__reduce_min_sync(FULL, f2o(mx)));
  } else {
    float mn = pos_inf();
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
      for (int e = 0; e < V; ++e) mn = min_nan(mn, x[g][e]);
    lo_src = o2f(__reduce_min_sync(FULL, f2o(mn)));
    valid = lo_src >= -1e38f && hi32 <= 1e38f;
  }
  if (!valid) {
    // invalid row: the binary32 path flags it and keeps every write in the row
    process_row_w1<T, G, true, 0, IdxT>(x, true, r, M, k, kSafetyCap, true, 0.0f, lane, stage, vals, idx,
                                        nullptr, st);
    return;
  }

  // ---- packed image: word w of group g holds elements 2w (bits 0..15) and 2w + 1
  uint32_t h[NW];
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int w = 0; w < V / 2; ++w) h[g * (V / 2) + w] = P::pack(x[g][2 * w + 1], x[g][2 * w]);
  auto count = [&](uint32_t t2) { return int(__reduce_add_sync(FULL, packed_count_hi16<P, NW>(h, 0, NW, t2)) >> 16); };

  // ---- coarse bracket: hi = image of the maximum; lo = image of lo_src (the
  // minimum, or for k <= 32 the smallest lane maximum)
  const uint32_t hi2 = P::splat(hi32);
  const float hi_img = P::low_f32(hi2);

  float b_lo, b_hi;  // coarse bucket [b_lo, b_hi) that the binary32 search finishes
  // ties at the top image: only possible when enough lanes' maxima share it
  if (__popc(__ballot_sync(FULL, P::low_f32(P::splat(mx)) >= hi_img)) * NE >= k && count(hi2) >= k) {
    b_lo = hi_img;
    b_hi = pos_inf();
  } else {
    // coarse bisection on the packed bracket (both halves of lo2 / hi2 equal)
    uint32_t lo2 = P::splat(lo_src), hi2_ = hi2;
    const uint32_t k0 = uint32_t(k) << 16, k1 = uint32_t(k + 1) << 16;  // C(t) >= k, >= k + 1 on the redux word
    const int64_t obase = r * int64_t(k);
    // C(t) == k: {h >= t} is the row's top-k; written from the pass's compares
    auto finish = [&](const uint32_t (&sp)[NW], const uint32_t (&cum)[G]) {
      compact_packed<T, G>(x, sp, cum, lane, stage);
      __syncwarp();
      const float* sv = reinterpret_cast<const float*>(stage);
      const int* si = reinterpret_cast<const int*>(stage) + kStageK;
      if (k <= 32) {  // one entry per lane, no loop (397.3 against 420.6 us at fp32 k = 32)
        if (lane < k) {
          vals[obase + lane] = out_value(sv[lane], vals);
          idx[obase + lane] = IdxT(si[lane]);
        }
      } else {
        for (int p = lane; p < k; p += 32) {
          vals[obase + p] = out_value(sv[p], vals);
          idx[obase + p] = IdxT(si[p]);
        }
      }
      __syncwarp();
    };
    // Two passes per iteration; only the first tests for collapse. The midpoint
    // always lies in [lo, hi], so once no 16-bit value is strictly inside, the
    // second pass counts at lo (C > k: lo unchanged) or at hi (C < k: hi
    // unchanged) and the next iteration's test ends the search. Each pass
    // keeps its own compares and writes the row from them where it ends.
    for (;;) {
      uint32_t m2 = P::midpoint(lo2, hi2_);
      if (!P::strictly_inside(lo2, m2, hi2_)) break;  // no 16-bit value strictly inside
      uint32_t sa[NW], ca[G];
      packed_pass<P, G, V / 2>(h, m2, sa, ca);
      uint32_t tot = __reduce_add_sync(FULL, ca[G - 1] * 0x10001u - P::kFold);
      bool ge = tot >= k0;
      if (ge && tot < k1) { finish(sa, ca); return; }
      lo2 = ge ? m2 : lo2;
      hi2_ = ge ? hi2_ : m2;
      m2 = P::midpoint(lo2, hi2_);
      uint32_t sb[NW], cb[G];
      packed_pass<P, G, V / 2>(h, m2, sb, cb);
      tot = __reduce_add_sync(FULL, cb[G - 1] * 0x10001u - P::kFold);
      ge = tot >= k0;
      if (ge && tot < k1) { finish(sb, cb); return; }
      lo2 = ge ? m2 : lo2;
      hi2_ = ge ? hi2_ : m2;
    }
    const float lo = P::low_f32(lo2), hi = P::low_f32(hi2_);
    if (sizeof(T) == 2 && next_up_bf16(lo) == hi) {
      // bf16 rows: B = {x == lo}, all tied; keep x >= hi and fill from B by index
      fill_store_w1<T, G, IdxT>(x, lo, hi, false, k, lane, stage, vals, idx, obase);
      return;
    }
    b_lo = lo;
    b_hi = hi;
  }

  // ---- binary32 search inside the bucket B = {b_lo <= h(x) < b_hi}
  float bmin = pos_inf(), bmax = neg_inf();
#pragma unroll
  for (int w = 0; w < NW; ++w) {
    const float hl = P::low_f32(h[w]), hh = P::high_f32(h[w]);
    const float xl = x[w / (V / 2)][2 * (w % (V / 2))], xh = x[w / (V / 2)][2 * (w % (V / 2)) + 1];
    const bool il = hl >= b_lo && !(hl >= b_hi);
    const bool ih = hh >= b_lo && !(hh >= b_hi);
    bmin = fminf(bmin, il ? xl : pos_inf());
    bmax = fmaxf(bmax, il ? xl : neg_inf());
    bmin = fminf(bmin, ih ? xh : pos_inf());
    bmax = fmaxf(bmax, ih ? xh : neg_inf());
  }
  float flo = o2f(__reduce_min_sync(FULL, f2o(bmin)));
  float fhi = next_up_f32(o2f(__reduce_max_sync(FULL, f2o(bmax))));
  int it = 0, c_lo = M;
  bool comp = false;
  auto count_row = [&](float mid) { return __reduce_add_sync(FULL, lane_count_lt<G, V>(x, mid)); };
  const bool eq32 = search_passes<true, 0>(count_row, 32 * NE, k, kSafetyCap, true, 0.0f, flo, fhi, it, c_lo,
                                           comp, st);
  fill_store_w1<T, G, IdxT>(x, flo, fhi, eq32, k, lane, stage, vals, idx, r * int64_t(k));
}

// fp32 rows (1 KB at M = 256) load the warp's next row into registers while
// the current one is searched; bf16 rows (half the bytes) measured faster
// without it (GB300, 2^20 x 256, k = 32, 4 blocks per SM: fp32 445 vs 469 us,
// bf16 519 vs 487 us).
#ifndef RTOPK_PACKED_PREFETCH_F32
#define RTOPK_PACKED_PREFETCH_F32 1
#endif
template <typename T>
struct PackedPrefetch {
  static constexpr bool value = sizeof(T) == 4 && RTOPK_PACKED_PREFETCH_F32;
};

// Minimum resident blocks per SM of the packed kernel. With the prefetch, 4
// blocks of 256 (64 registers) measured faster than 5 (48 registers, a small
// spill): 435.5 against 440.3 us at 2^20 x 256 fp32, k = 32.
#ifndef RTOPK_PACKED_MIN_BLOCKS
#define RTOPK_PACKED_MIN_BLOCKS 5
#endif
#ifndef RTOPK_PACKED_PREFETCH_MIN_BLOCKS
#define RTOPK_PACKED_PREFETCH_MIN_BLOCKS 4
#endif
template <typename T, int NE>
struct PackedOcc {
  static constexpr int value =
      NE <= 8 ? (PackedPrefetch<T>::value ? RTOPK_PACKED_PREFETCH_MIN_BLOCKS : RTOPK_PACKED_MIN_BLOCKS) : 3;
};

// Rows of exactly G * 32 * V elements, 16-byte aligned, exact mode, k <= kStageK.
template <typename T, int G, typename IdxT>
__global__ void __launch_bounds__(256, PackedOcc<T, G * ElemTraits<T>::V>::value)
rtopk_warp_packed_kernel(const T* __restrict__ in, int64_t N, int M, int k, T* __restrict__ vals,
                         IdxT* __restrict__ idx, uint32_t* __restrict__ status) {
  constexpr int V = ElemTraits<T>::V;
  __shared__ float2 stage_all[8][kStageK];
  const int lane = threadIdx.x & 31;
  const int wib = threadIdx.x >> 5;
  float2* stage = stage_all[wib];
  const int64_t nwarps = int64_t(gridDim.x) * 8;
  uint32_t st = 0;
  if constexpr (PackedPrefetch<T>::value) {
    float xn[G][V];
    int64_t r = int64_t(blockIdx.x) * 8 + wib;
    if (r < N) load_row<G, 1, true>(in + r * int64_t(M), M, 0, lane, true, xn);
    for (; r < N; r += nwarps) {
      float x[G][V];
#pragma unroll
      for (int g = 0; g < G; ++g)
#pragma unroll
        for (int e = 0; e < V; ++e) x[g][e] = xn[g][e];
      if (r + nwarps < N) load_row<G, 1, true>(in + (r + nwarps) * int64_t(M), M, 0, lane, true, xn);
      process_row_packed<T, G, IdxT>(x, r, M, k, lane, stage, vals, idx, st);
    }
  } else {
    for (int64_t r = int64_t(blockIdx.x) * 8 + wib; r < N; r += nwarps) {
      float x[G][V];
      load_row<G, 1, true>(in + r * int64_t(M), M, 0, lane, true, x);
      process_row_packed<T, G, IdxT>(x, r, M, k, lane, stage, vals, idx, st);
    }
  }
  if (status != nullptr && st != 0u && lane == 0) atomicOr(status, st);
}

}  // namespace rtopk
