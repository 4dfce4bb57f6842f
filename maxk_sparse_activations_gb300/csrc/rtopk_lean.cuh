// Exact row-wise top-k on rows of 128..1024 elements, one warp per row, each
// lane holding a contiguous slice of the row, the threshold search counted on
// packed 16-bit images of the row, sm_103a.
//
// Source: "RTop-K: Ultra-Fast Row-Wise Top-K Selection for Neural Network
// Acceleration on GPUs" (summary page), "Approach" (binary search over the
// row's value range for a threshold that selects k; ties at the threshold
// filled by the lowest index); CBSR output from "MaxK-GNN: Extremely Fast GPU
// Kernel Design for Accelerating Graph Neural Networks Training", "The idea".
//
// Used for exact mode (max_iter < 0, eps == 0) when per-row pass counts are
// not requested. The result there is one set -- the k largest values, ties at
// the k-th value broken by the lowest index -- whatever thresholds the search
// visits, so it may run on any order-preserving image h of the row: binary16
// (nearest, saturated at +-65504) for fp32 rows, the data themselves for bf16
// rows. Over 16-bit thresholds lo < hi with C(lo) >= k > C(hi),
// C(t) = #{h(x) >= t}:
//  * C(mid) == k: {h >= mid} is an upper set of the row with k members, the
//    exact top-k (equal values share an image, so no tie is split);
//  * no 16-bit value strictly inside (lo, hi): {h >= hi} (< k members) is kept
//    and the rest of the top-k lies in the bucket {lo <= h < hi}; a binary32
//    search over the row finishes from [min of the bucket, next binary32 above
//    its max] (a valid bracket), and the general fill writes the row. bf16
//    rows whose bracket ends on two adjacent bf16 values go to the fill at once.
//
// Design (the search, not the bytes, bounds the kernel: measured on GB300 at
// 2^20 x 256 fp32, k = 32, the same kernel without the search runs at 0.94 of
// the HBM copy bandwidth, with it at 0.61; the search passes load the
// half-rate ALU and FMA-heavy pipes about equally, so the compares run as
// fp16 subtractions and the counting as byte sums):
//  * lane l holds elements [l * NE, (l + 1) * NE), so the kept elements of a
//    lane are consecutive in index order and one warp prefix scan of lane
//    counts places them;
//  * rows stream through a ring of shared-memory stages per warp (cp.async,
//    coalesced 16-byte chunks, kStages rows in flight); a lane reads its slice
//    from the stage, and the stage is also the source of the CBSR values;
//  * range and precondition: NaN-propagating three-input max of |x| per lane
//    and redux.sync on binary32 (fp32 rows); packed bf16x2 max / min (bf16);
//  * the search bracket starts at [image of the smallest lane maximum (k <=
//    32: each lane holds an element at least that large, so C >= 32 >= k) or
//    of a row lower bound, next 16-bit value above the image of the upper
//    bound (C = 0)]: no test for ties at the maximum is needed;
//  * a pass forms h - t for two elements per packed add (FMA pipe), gathers
//    the sign bits of four halves into sign-replicated bytes with one prmt and
//    adds them with dp4a (the lane's negatives); one redux.sync sums the lanes;
//  * the finish stages only the kept indices (one predicated shared store per
//    element); the first k lanes gather values and indices and write the CBSR
//    row with coalesced stores.
// Rows whose values are not all finite with |x| <= 1e38 set their status bits
// and write the row's first k elements (output unspecified, writes in-row).
#pragma once

#include "rtopk_image16.cuh"
#include "rtopk_select.cuh"

namespace rtopk {
namespace lean {

constexpr int kListK = 256;  // per-warp list of kept indices (k <= 256)

#ifndef RTOPK_LEAN_SWZ
#define RTOPK_LEAN_SWZ 1
#endif

// ---- small device wrappers -------------------------------------------------
__device__ __forceinline__ float max3_nan(float a, float b, float c) {
  float r;
  asm("max.NaN.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}
__device__ __forceinline__ float min3_nan(float a, float b, float c) {
  float r;
  asm("min.NaN.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}
__device__ __forceinline__ float warp_max_nan(float v) {
  float r;
  asm volatile("redux.sync.max.NaN.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
  return r;
}
__device__ __forceinline__ float warp_min_nan(float v) {
  float r;
  asm volatile("redux.sync.min.NaN.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
  return r;
}
__device__ __forceinline__ uint32_t warp_sum(uint32_t v) { return __reduce_add_sync(0xffffffffu, v); }
// The sign bits of the four 16-bit halves of a and b, each replicated over a
// byte (0xff for a negative half): prmt with the sign-replicate selector bit.
__device__ __forceinline__ uint32_t half_signs(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, 0xFDB9;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
// c + the four bytes of a as signed integers (each 0 or -1 here)
__device__ __forceinline__ int sum_bytes(uint32_t a, int c) {
  int d;
  asm("dp4a.s32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(0x01010101), "r"(c));
  return d;
}

// c + minus the number of set sign bits of the binary32 words a and b: prmt
// copies their sign bits into bytes 0 and 1 as 0xff / 0x00 (bytes 2 and 3
// get weight 0 in the dp4a).
__device__ __forceinline__ int sum_sign_pair(uint32_t a, uint32_t b, int c) {
  uint32_t p;
  asm("prmt.b32 %0, %1, %2, 0x00FB;" : "=r"(p) : "r"(a), "r"(b));
  int d;
  asm("dp4a.s32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(p), "r"(0x00000101), "r"(c));
  return d;
}

// Number of a lane's values x >= t, for canonical values (no -0) and finite
// t: d = x - t has its sign bit clear iff x >= t (x == t gives +0, and a
// nonzero difference of binary32 values never rounds to zero), so a pass is
// subtractions on the FMA pipe and one prmt + one dp4a per two values instead
// of a compare and an add per value.
template <int NE>
__device__ __forceinline__ uint32_t lane_count_ge(const float (&x)[NE], float t) {
  int acc = 0;
#pragma unroll
  for (int e = 0; e + 1 < NE; e += 2)
    acc = sum_sign_pair(__float_as_uint(__fsub_rn(x[e], t)), __float_as_uint(__fsub_rn(x[e + 1], t)), acc);
  if constexpr ((NE & 1) != 0) acc -= int(__float_as_uint(__fsub_rn(x[NE - 1], t)) >> 31);
  return uint32_t(NE + acc);
}

// NaN-propagating maximum of a lane's values.
template <int NE>
__device__ __forceinline__ float lane_max(const float (&x)[NE]) {
  float m = x[0];
  int i = 1;
#pragma unroll
  for (; i + 1 < NE; i += 2) m = max3_nan(m, x[i], x[i + 1]);
  if (i < NE) m = max_nan(m, x[i]);
  return m;
}
// ---- 16-bit image traits ----------------------------------------------------
template <typename T>
struct Img;
template <>
struct Img<float> {
  static __device__ __forceinline__ uint32_t max2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.NaN.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
  }
  static __device__ __forceinline__ uint32_t min2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("min.NaN.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
  }
};
template <>
struct Img<uint16_t> {
  static __device__ __forceinline__ uint32_t max2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
  }
  static __device__ __forceinline__ uint32_t min2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("min.NaN.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
  }
};

// Next 16-bit value above the (splat) image word w, in both halves: +-0 ->
// smallest positive subnormal, positive -> +1 ulp, negative -> toward zero.
// The image of a valid fp32 maximum is at most 65504, whose successor is
// +inf; the search then collapses at once and the binary32 finish takes the
// whole bucket.
__device__ __forceinline__ uint32_t next_up16(uint32_t w) {
  const uint32_t b = w & 0xffffu;
  const uint32_t nb = (b & 0x7fffu) == 0u ? 1u : ((b & 0x8000u) ? b - 1u : b + 1u);
  return nb | (nb << 16);
}

// ---- loads and lane layout ---------------------------------------------------
// RW 32-bit words of input per lane: NE for fp32, NE / 2 for bf16.
template <typename T, int NE>
struct Lane {
  static constexpr int RW = sizeof(T) == 4 ? NE : NE / 2;
  static constexpr int W = NE / 2;  // packed image words
};

// Layout of a row in its shared stage, in 16-byte chunks. Lane L's slice is
// chunks [L * CPL, (L + 1) * CPL). When CPL is 4 or 8 the eight lanes of a
// shared-memory phase would read the same banks (slices 64 or 128 bytes
// apart: 4- / 8-way conflicts), so chunk c of lane L is stored at
// L * CPL + (c ^ s(L)), s(L) the lane bits the stride folds onto one bank
// group: every lane's chunk c then sits in its own bank group (GB300, 2^18
// rows of 1024 fp32: 385 -> 233 us at k = 16). Other slices keep the row in
// element order (a 2-chunk swizzle measured slower: its 2-way conflicts cost
// less than the address arithmetic).
template <int RW>
struct StageLayout {
  static constexpr int CPL = RW >= 4 ? RW / 4 : 1;  // 16-byte chunks per lane
  static constexpr int SH = CPL == 4 ? 1 : 0;
  static constexpr bool SWZ = RTOPK_LEAN_SWZ && (CPL == 4 || CPL == 8);
  static __device__ __forceinline__ int chunk_pos(int L, int c) {
    if constexpr (SWZ) {
      return L * CPL + (c ^ ((L >> SH) & (CPL - 1)));
    } else {
      return L * CPL + c;
    }
  }
  // word offset in the stage of element j (4-byte elements: 4 per chunk)
  static __device__ __forceinline__ int word_of_f32(int j) {
    if constexpr (SWZ) {
      const int g = j >> 2;
      return chunk_pos(g / CPL, g % CPL) * 4 + (j & 3);
    } else {
      return j;
    }
  }
  // 16-bit offset in the stage of element j (2-byte elements: 8 per chunk)
  static __device__ __forceinline__ int half_of_bf16(int j) {
    if constexpr (SWZ) {
      const int g = j >> 3;
      return chunk_pos(g / CPL, g % CPL) * 8 + (j & 7);
    } else {
      return j;
    }
  }
};

// Asynchronous copy of one row (32 * RW words) into a shared stage: lane l
// copies the 16-byte chunks l, l + 32, ... of the row (coalesced) to their
// stage positions. One commit group per row.
template <int RW>
__device__ __forceinline__ void issue_row(uint32_t stage, const uint32_t* __restrict__ src_lane, int lane,
                                          bool valid) {
  using SL = StageLayout<RW>;
  constexpr int CH = 8 * RW;  // 16-byte chunks per row
#pragma unroll
  for (int i = 0; i < (CH + 31) / 32; ++i) {
    const int g = lane + 32 * i;
    const uint32_t dst = SL::SWZ ? stage + uint32_t(SL::chunk_pos(g / SL::CPL, g % SL::CPL)) * 16u
                                 : stage + uint32_t(lane * 16 + i * 512);
    if (valid && (CH % 32 == 0 || g < CH))
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src_lane + i * 128) : "memory");
  }
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int PENDING>
__device__ __forceinline__ void wait_rows() {
  asm volatile("cp.async.wait_group %0;" ::"n"(PENDING) : "memory");
}

// The lane's RW consecutive words (elements [lane * NE, (lane + 1) * NE)) of a
// staged row.
template <int RW>
__device__ __forceinline__ void lane_words(const uint32_t* __restrict__ srow, int lane, uint32_t (&w)[RW]) {
  if constexpr (RW % 4 == 0) {
#pragma unroll
    for (int c = 0; c < RW / 4; ++c) {
      const uint4 q = *reinterpret_cast<const uint4*>(srow + StageLayout<RW>::chunk_pos(lane, c) * 4);
      w[4 * c] = q.x; w[4 * c + 1] = q.y; w[4 * c + 2] = q.z; w[4 * c + 3] = q.w;
    }
  } else {
    static_assert(RW == 2, "8-byte lane slices");
    const uint2 q = *reinterpret_cast<const uint2*>(srow + lane * RW);
    w[0] = q.x; w[1] = q.y;
  }
}

// Binary32 values of the lane's elements from its raw words.
template <typename T, int NE>
__device__ __forceinline__ void widen(const uint32_t (&w)[Lane<T, NE>::RW], float (&x)[NE]) {
#pragma unroll
  for (int e = 0; e < NE; ++e) {
    if constexpr (sizeof(T) == 4) {
      x[e] = __uint_as_float(w[e]);
    } else {  // element 2q in the low half of word q (lower address)
      x[e] = (e & 1) ? __uint_as_float(w[e / 2] & 0xffff0000u) : __uint_as_float(w[e / 2] << 16);
    }
  }
}

// The lane's values again, from the shared copy of the row (rare paths: the
// row's registers are not kept alive through the search for them).
template <typename T, int NE>
__device__ __forceinline__ void reload(const uint32_t* __restrict__ srow, int lane, float (&x)[NE]) {
  uint32_t w[Lane<T, NE>::RW];
  lane_words<Lane<T, NE>::RW>(srow, lane, w);
  widen<T, NE>(w, x);
}

// ---- finishes ---------------------------------------------------------------
// Kept indices of the exact ending C(t) == k, from that pass's compares s[]:
// this lane's kept elements go to list positions [ex, ex + count) in index
// order; one predicated shared store per element.
// SIGN: s[w] holds h - t per half (kept when the sign bit is clear) instead
// of the 1.0 / 0.0 compare results.
template <int W, bool SIGN = false>
__device__ __forceinline__ void stage_exact(const uint32_t (&s)[W], uint32_t c, int lane, uint32_t list_addr) {
  uint32_t incl = c;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1)
    asm("{\n\t.reg .pred p;\n\t.reg .u32 t;\n\t"
        "shfl.sync.up.b32 t|p, %0, %1, 0, -1;\n\t"
        "@p add.u32 %0, %0, t;\n\t}"
        : "+r"(incl) : "r"(d));
  uint32_t a = list_addr + (incl - c) * 4u;
  const uint32_t j0 = uint32_t(lane) * uint32_t(2 * W);
#pragma unroll
  for (int w = 0; w < W; ++w) {
    if constexpr (SIGN) {
      asm volatile(
          "{\n\t.reg .pred p;\n\t.reg .u32 t;\n\t"
          "and.b32 t, %1, 32768;\n\t"
          "setp.eq.u32 p, t, 0;\n\t"
          "@p st.shared.u32 [%0], %2;\n\t"
          "@p add.u32 %0, %0, 4;\n\t}"
          : "+r"(a) : "r"(s[w]), "r"(j0 + 2u * w) : "memory");
      asm volatile(
          "{\n\t.reg .pred p;\n\t"
          "setp.ge.s32 p, %1, 0;\n\t"
          "@p st.shared.u32 [%0], %2;\n\t"
          "@p add.u32 %0, %0, 4;\n\t}"
          : "+r"(a) : "r"(s[w]), "r"(j0 + 2u * w + 1u) : "memory");
    } else {
      asm volatile(
          "{\n\t.reg .pred p;\n\t.reg .u32 t;\n\t"
          "and.b32 t, %1, 65535;\n\t"
          "setp.ne.u32 p, t, 0;\n\t"
          "@p st.shared.u32 [%0], %2;\n\t"
          "@p add.u32 %0, %0, 4;\n\t}"
          : "+r"(a) : "r"(s[w]), "r"(j0 + 2u * w) : "memory");
      asm volatile(
          "{\n\t.reg .pred p;\n\t"
          "setp.ge.u32 p, %1, 65536;\n\t"
          "@p st.shared.u32 [%0], %2;\n\t"
          "@p add.u32 %0, %0, 4;\n\t}"
          : "+r"(a) : "r"(s[w]), "r"(j0 + 2u * w + 1u) : "memory");
    }
  }
}

// General fill for a binary32 bracket [lo, hi) with c(lo) >= k > c(hi): keep
// every x >= hi, then the first k - c(hi) of lo <= x < hi in index order, at
// list positions [base, base + k). Lanes with `active` false hold none of the
// elements concerned (a bucket of lanes selects on its own).
template <int NE>
__device__ __forceinline__ void stage_general(const float (&x)[NE], float lo, float hi, int k, int lane,
                                              uint32_t* __restrict__ list, bool active = true, int base = 0) {
  uint32_t sc = 0, bc = 0;
#pragma unroll
  for (int e = 0; e < NE; ++e) {
    const bool s = active && x[e] >= hi;
    sc += s ? 1u : 0u;
    bc += (active && !s && x[e] >= lo) ? 1u : 0u;
  }
  uint32_t incl = sc | (bc << 16);
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const uint32_t t = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= d) incl += t;
  }
  const uint32_t tot = __shfl_sync(0xffffffffu, incl, 31);
  const uint32_t ex = incl - (sc | (bc << 16));
  const int need = k - int(tot & 0xffffu);
  int bpos = int(ex >> 16);
  int pos = base + int(ex & 0xffffu) + min(bpos, need);
#pragma unroll
  for (int e = 0; e < NE; ++e) {
    const bool s = active && x[e] >= hi;
    const bool b = active && !s && x[e] >= lo;
    if (s || (b && bpos < need)) {
      list[pos] = uint32_t(lane * NE + e);
      ++pos;
    }
    bpos += b ? 1 : 0;
  }
}

// CBSR row from the staged list: value bits gathered from the staged row,
// indices as listed (ascending). vrow / irow point at the row's k outputs.
template <typename T, int RW, typename IdxT>
__device__ __forceinline__ void copy_out(const uint32_t* __restrict__ list, const uint32_t* __restrict__ srow,
                                         int k, int lane, T* __restrict__ vrow, IdxT* __restrict__ irow) {
  using SL = StageLayout<RW>;
  __syncwarp();
  auto one = [&](int p) {
    const uint32_t j = list[p];
    T v;
    if constexpr (sizeof(T) == 4) {
      v = __uint_as_float(srow[SL::word_of_f32(int(j))]);
    } else {
      v = reinterpret_cast<const uint16_t*>(srow)[SL::half_of_bf16(int(j))];
    }
    vrow[p] = v;
    irow[p] = IdxT(j);
  };
  if (k <= 32) {
    if (lane < k) one(lane);
  } else {
    for (int p = lane; p < k; p += 32) one(p);
  }
  __syncwarp();
}

// Exact binary32 search from a valid bracket [lo, hi] (c(lo) >= k > c(hi)),
// then the general fill. Used inside the last 16-bit bucket (and for the
// rare bf16 bracket that ends on two non-adjacent values). The bracket is
// bisected on order-preserving integer keys of binary32 (f2o), not on value
// midpoints: exact mode selects one set whatever thresholds are visited, and
// a key bisection ends within 32 passes for any range, where a value
// bisection from a small value up to a 1e30 outlier (whose 16-bit image
// saturates, so the 16-bit bracket collapses at once) takes 100+ passes.
// The count at a key is the count at its value, so -0 and +0 count alike;
// a final bracket [-0, +0) cannot occur (c(-0) == c(+0)).
template <int NE>
__device__ __forceinline__ void finish_binary32(const float (&x)[NE], float lo, float hi, int k, int lane,
                                                uint32_t* __restrict__ list, uint32_t& st, bool active = true,
                                                int base = 0) {
  int olo = f2o(lo), ohi = f2o(hi);
  for (int it = 0;; ++it) {
    const uint32_t gap = uint32_t(ohi) - uint32_t(olo);
    if (gap < 2u) break;  // adjacent keys: nothing strictly inside
    if (it >= kSafetyCap) {
      st |= kStatusSafetyCap;
      break;
    }
    const int om = olo + int(gap >> 1);
    const float mid = o2f(om);
    uint32_t c = 0;
#pragma unroll
    for (int e = 0; e < NE; ++e) c += (active && x[e] >= mid) ? 1u : 0u;
    const int cnt = int(warp_sum(c));
    if (cnt >= k) olo = om;
    else ohi = om;
    if (cnt == k) break;
  }
  stage_general<NE>(x, o2f(olo), o2f(ohi), k, lane, list, active, base);
}

// ---- one row ------------------------------------------------------------------
template <typename T, int NE, typename IdxT, bool GUESS>
__device__ __forceinline__ void process_row(const uint32_t* __restrict__ srow, int k, int lane,
                                            uint32_t* __restrict__ list, T* __restrict__ vrow,
                                            IdxT* __restrict__ irow, uint32_t& st, float& tprev, float& rho) {
  using P = Packed16<T>;
  using I = Img<T>;
  constexpr int RW = Lane<T, NE>::RW;
  constexpr int W = Lane<T, NE>::W;
  constexpr unsigned FULL = 0xffffffffu;
  uint32_t raw[RW];
  lane_words<RW>(srow, lane, raw);

  // ---- image, range and precondition. hi32 bounds every |x| (fp32) or x
  // (bf16) from above; lo_src is a value with at least k elements >= it.
  uint32_t h[W];
  float hi32, lo_src;
  bool valid;
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
    hi32 = warp_max_nan(a);  // NaN if any element is NaN
    valid = hi32 <= 1e38f;
    // k <= 32: each of the 32 lanes holds an element >= its maximum
    lo_src = (k <= 32) ? warp_min_nan(lane_max<NE>(x)) : -hi32;
  } else {
#pragma unroll
    for (int w = 0; w < W; ++w) h[w] = raw[w];
    uint32_t m = h[0], n = h[0];
#pragma unroll
    for (int w = 1; w < W; ++w) {
      m = I::max2(m, h[w]);
      n = I::min2(n, h[w]);
    }
    m = I::max2(m, __byte_perm(m, 0, 0x1032));  // both halves: the lane maximum
    n = I::min2(n, __byte_perm(n, 0, 0x1032));
    const float mx = __uint_as_float(m & 0xffff0000u);
    hi32 = warp_max_nan(mx);
    const float lo_row = warp_min_nan(__uint_as_float(n & 0xffff0000u));
    valid = hi32 <= 1e38f && lo_row >= -1e38f;
    lo_src = (k <= 32) ? warp_min_nan(mx) : lo_row;
  }
  if (!valid) {
    // invalid row: report which precondition fails, write the first k elements
    float x[NE];
    reload<T, NE>(srow, lane, x);
    bool nonfinite = false, range = false;
#pragma unroll
    for (int e = 0; e < NE; ++e) {
      const float a = fabsf(x[e]);
      nonfinite |= !(a <= 3.402823466e38f);
      range |= (a > 1e38f && a <= 3.402823466e38f);
    }
    if (__any_sync(FULL, nonfinite)) st |= kStatusNonFinite;
    if (__any_sync(FULL, range)) st |= kStatusRange;
    for (int p = lane; p < k; p += 32) list[p] = uint32_t(p);
    copy_out<T, Lane<T, NE>::RW, IdxT>(list, srow, k, lane, vrow, irow);
    return;
  }

  // ---- coarse bisection on 16-bit images: C(lo2) >= k > C(hi2) = 0
  uint32_t lo2 = P::splat(lo_src);
  // fp32: hi32 = max |x| >= 0, whose image is +0 or positive: the next 16-bit
  // value is one bit pattern up
  uint32_t hi2 = sizeof(T) == 4 ? P::splat(hi32) + 0x00010001u : next_up16(P::splat(hi32));
  const uint32_t list_addr = static_cast<uint32_t>(__cvta_generic_to_shared(list));
  // A pass forms d = h - t per half with packed adds of the negated
  // threshold (FMA pipe), gathers the halves' sign bits into sign-replicated
  // bytes (one prmt per two words) and adds the bytes with dp4a: C(t) = NE *
  // 32 minus the negatives. h >= t iff h - t has its sign bit clear, given no
  // image is -0 (the images are canonicalised by adding +0: -0 + 0 = +0) and a
  // zero threshold then gives +0 - 0 = +0. The bracket is kept negated
  // (nlo = -lo, nhi = -hi): the midpoint formula is odd-symmetric, so it
  // yields -mid exactly.
#pragma unroll
  for (int w = 0; w < W; ++w) h[w] = P::add(h[w], 0u);
  uint32_t nlo2 = lo2 ^ 0x80008000u, nhi2 = hi2 ^ 0x80008000u;
  const int kneg = k - 32 * NE;  // C >= k  iff  -(negatives) >= k - M
  auto pass = [&](uint32_t nm2, uint32_t (&s)[W], int& u) {
#pragma unroll
    for (int w = 0; w < W; ++w) s[w] = P::add(h[w], nm2);
    int acc = 0;
#pragma unroll
    for (int w = 0; w + 1 < W; w += 2) acc = sum_bytes(half_signs(s[w], s[w + 1]), acc);
    u = acc;  // -(this lane's negatives)
    return int(warp_sum(uint32_t(acc)));
  };
  // Two passes per collapse test: the midpoint always lies in the bracket (as a
  // value), so no 16-bit value strictly inside means it equals an end; after a
  // collapse the second pass counts at an end, leaves the bracket as it is,
  // and the next test ends the search (a midpoint of the other signed zero
  // than an end passes the test and costs one pass at the same value). Every
  // pass keeps its own differences and, on C == k, writes the row from them
  // where it ends (one exit per pass: a single shared exit measured slower).
  // Measured on GB300 (2^20 x 256 fp32, k = 32) and not kept: a test every 3
  // or 4 passes, 1.0 / 0.0 compares (set.ge, ALU pipe) summed with fp16 adds
  // (323.5 against 320.9 us; bf16 359.2 against 349.8), the same compares
  // summed with integer adds + dp2a (358), bracket updates as integer
  // multiply-adds, a bracket top from the warp maximum instead of max |x|, and
  // a row loop unrolled over the ring stages -- each 1-20% slower.
  // GUESS (the launcher's choice, kGuessRows): guessed probes, for rows where
  // a pass is large and the bracket starts wide (k > 32: from -max |x|): the
  // warp's previous threshold first, then Newton steps t + (C(t) - k - 1/2) /
  // rho with the density rho estimated on the warp's earlier rows, at most
  // kGuesses a row; a guess that is not strictly inside the bracket (as a
  // 16-bit value) is replaced by the midpoint. Exact mode selects one set
  // whatever thresholds are visited.
  if constexpr (GUESS) {
    float lo_f = P::low_f32(lo2), hi_f = P::low_f32(hi2);
    const float inv_rho = rho > 0.0f ? 1.0f / rho : 0.0f;
    float t_last = tprev, t_first = 0.0f;
    int c_last = 0, c_first = 0;  // C - k at the last / first probe
    constexpr int kGuesses = 8;
    for (int p = 0;; ++p) {
      const float tg = p == 0 ? tprev : fmaf(float(c_last) - 0.5f, inv_rho, t_last);
      const uint32_t ng2 = P::splat(-tg);  // negated image of the guess
      const float gv = -P::low_f32(ng2);
      uint32_t nm2;
      if (p < kGuesses && lo_f < gv && gv < hi_f) {
        nm2 = ng2;
      } else {
        nm2 = P::midpoint(nlo2, nhi2);
        if (nm2 == nlo2 || nm2 == nhi2) break;
      }
      uint32_t sd[W];
      int u;
      const int tot = pass(nm2, sd, u);
      const float mv = -P::low_f32(nm2);
      if (tot == kneg) {
        if (p > 0 && c_first != 0 && t_first != mv) {
          const float est = fabsf(float(c_first)) / fabsf(t_first - mv);
          rho = rho > 0.0f ? 0.8f * rho + 0.2f * est : est;
        }
        tprev = mv;
        stage_exact<W, true>(sd, uint32_t(NE + u), lane, list_addr);
        copy_out<T, Lane<T, NE>::RW, IdxT>(list, srow, k, lane, vrow, irow);
        return;
      }
      const bool ge = tot >= kneg;
      nlo2 = ge ? nm2 : nlo2;
      nhi2 = ge ? nhi2 : nm2;
      lo_f = ge ? mv : lo_f;
      hi_f = ge ? hi_f : mv;
      c_last = tot - kneg;
      t_last = mv;
      if (p == 0) {
        c_first = c_last;
        t_first = mv;
      }
    }
    tprev = lo_f;  // collapsed: the threshold lies in [lo, hi)
  } else {
    for (;;) {
      uint32_t nm2 = P::midpoint(nlo2, nhi2);
      if (nm2 == nlo2 || nm2 == nhi2) break;
  #pragma unroll
      for (int j = 0; j < 2; ++j) {
        if (j > 0) nm2 = P::midpoint(nlo2, nhi2);
        uint32_t s[W];
        int u;
        const int tot = pass(nm2, s, u);
        const bool ge = tot >= kneg;
        if (tot == kneg) {
          // C(mid) == k: {h >= mid} is the top-k
          stage_exact<W, true>(s, uint32_t(NE + u), lane, list_addr);
          copy_out<T, Lane<T, NE>::RW, IdxT>(list, srow, k, lane, vrow, irow);
          return;
        }
        nlo2 = ge ? nm2 : nlo2;
        nhi2 = ge ? nhi2 : nm2;
      }
    }
  }
  lo2 = nlo2 ^ 0x80008000u;
  hi2 = nhi2 ^ 0x80008000u;

  // ---- collapsed: the rest of the top-k lies in the bucket {lo <= h < hi}
  float x[NE];
  reload<T, NE>(srow, lane, x);
  const float lo = P::low_f32(lo2), hi = P::low_f32(hi2);
  if (sizeof(T) == 2 && next_up_bf16(lo) == hi) {
    // bf16: the bucket holds one value (every x in it equals lo)
    stage_general<NE>(x, lo, hi, k, lane, list);
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
    const float flo = o2f(__reduce_min_sync(FULL, f2o(bmin)));
    const float fhi = next_up_f32(o2f(__reduce_max_sync(FULL, f2o(bmax))));
    finish_binary32<NE>(x, flo, fhi, k, lane, list, st);
  }
  copy_out<T, Lane<T, NE>::RW, IdxT>(list, srow, k, lane, vrow, irow);
}

// ---- one row split into B buckets ------------------------------------------------
// "Approximate Top-k for Increased Parallelism" (abstract): each bucket of a
// row keeps its own top-(k / B) independently. With M = 32 * NE, bucket b is
// the columns of lanes [b * LB, (b + 1) * LB), LB = 32 / B, so the B searches
// run side by side in one warp: each lane holds its bucket's bracket, a pass
// compares every lane against its bucket's midpoint, and the bucket counts
// come from one redux.sync over fields of 32 / B bits (B <= 4; a bucket count
// is at most LB * NE < 2^(32 / B)) or an LB-lane butterfly (B >= 8). The
// loop runs until every bucket has found its threshold or collapsed. The
// buckets are in column order and each keeps exactly k / B, so the warp-wide
// placement of the kept elements is the bucketed CBSR row, indices already
// row columns. A bucket whose search ends on tied 16-bit images finishes with
// an exact binary32 search inside its last bracket, bucket by bucket.
template <int LB>
__device__ __forceinline__ float seg_max_nan(float v) {
#pragma unroll
  for (int d = LB / 2; d >= 1; d >>= 1) v = max_nan(v, __shfl_xor_sync(0xffffffffu, v, d));
  return v;
}
template <int LB>
__device__ __forceinline__ float seg_min_nan(float v) {
#pragma unroll
  for (int d = LB / 2; d >= 1; d >>= 1) v = min_nan(v, __shfl_xor_sync(0xffffffffu, v, d));
  return v;
}
// Sum of c over the lanes of bucket b (every lane of the warp calls it).
template <int B>
__device__ __forceinline__ uint32_t bucket_sum(uint32_t c, int b) {
  constexpr int LB = 32 / B;
  if constexpr (B <= 4) {
    constexpr int FW = 32 / B;
    const uint32_t tot = warp_sum(c << (FW * b));
    return FW == 32 ? tot : ((tot >> (FW * b)) & ((1u << (FW & 31)) - 1u));
  } else {
#pragma unroll
    for (int d = LB / 2; d >= 1; d >>= 1) c += __shfl_xor_sync(0xffffffffu, c, d);
    return c;
  }
}

template <typename T, int NE, int B, typename IdxT>
__device__ __forceinline__ void process_row_bucketed(const uint32_t* __restrict__ srow, int k, int lane,
                                                     uint32_t* __restrict__ list, T* __restrict__ vrow,
                                                     IdxT* __restrict__ irow, uint32_t& st) {
  using P = Packed16<T>;
  using I = Img<T>;
  constexpr int RW = Lane<T, NE>::RW;
  constexpr int W = Lane<T, NE>::W;
  constexpr int LB = 32 / B;
  constexpr unsigned FULL = 0xffffffffu;
  const int b = lane / LB;
  const int kb = k / B;
  uint32_t raw[RW];
  lane_words<RW>(srow, lane, raw);
  uint32_t h[W];
  float mx, mn;
  if constexpr (sizeof(T) == 4) {
    float x[NE];
    widen<T, NE>(raw, x);
#pragma unroll
    for (int w = 0; w < W; ++w) h[w] = P::pack(x[2 * w + 1], x[2 * w]);
    mx = lane_max<NE>(x);
    float m = x[0];
#pragma unroll
    for (int e = 1; e < NE; ++e) m = min_nan(m, x[e]);
    mn = m;
  } else {
#pragma unroll
    for (int w = 0; w < W; ++w) h[w] = raw[w];
    uint32_t m = h[0], n = h[0];
#pragma unroll
    for (int w = 1; w < W; ++w) {
      m = I::max2(m, h[w]);
      n = I::min2(n, h[w]);
    }
    mx = __uint_as_float(I::max2(m, __byte_perm(m, 0, 0x1032)) & 0xffff0000u);
    mn = __uint_as_float(I::min2(n, __byte_perm(n, 0, 0x1032)) & 0xffff0000u);
  }
  const float row_hi = warp_max_nan(mx), row_lo = warp_min_nan(mn);
  if (!(row_hi <= 1e38f && row_lo >= -1e38f)) {
    float x[NE];
    reload<T, NE>(srow, lane, x);
    bool nonfinite = false, range = false;
#pragma unroll
    for (int e = 0; e < NE; ++e) {
      const float a = fabsf(x[e]);
      nonfinite |= !(a <= 3.402823466e38f);
      range |= (a > 1e38f && a <= 3.402823466e38f);
    }
    if (__any_sync(FULL, nonfinite)) st |= kStatusNonFinite;
    if (__any_sync(FULL, range)) st |= kStatusRange;
    for (int p = lane; p < k; p += 32) list[p] = uint32_t(p);
    copy_out<T, Lane<T, NE>::RW, IdxT>(list, srow, k, lane, vrow, irow);
    return;
  }
  // bucket brackets: [image of the smallest lane maximum (kb <= LB) or of the
  // bucket minimum, next 16-bit value above the image of the bucket maximum]
  const float top = seg_max_nan<LB>(mx);
  const float lo_b = seg_min_nan<LB>(kb <= LB ? mx : mn);
  uint32_t lo2 = P::splat(lo_b);
  uint32_t hi2 = next_up16(P::splat(top));
  // Counting as in process_row: h - t per half with packed adds of the
  // negated threshold, the negative halves summed as bytes (images
  // canonicalised so that no image is -0); the brackets are kept negated.
#pragma unroll
  for (int w = 0; w < W; ++w) h[w] = P::add(h[w], 0u);
  uint32_t nlo2 = lo2 ^ 0x80008000u, nhi2 = hi2 ^ 0x80008000u;
  auto lane_count = [&](uint32_t nt2, uint32_t (&d)[W]) {
    int acc = 0;
#pragma unroll
    for (int w = 0; w < W; ++w) d[w] = P::add(h[w], nt2);
#pragma unroll
    for (int w = 0; w + 1 < W; w += 2) acc = sum_bytes(half_signs(d[w], d[w + 1]), acc);
    return uint32_t(NE + acc);
  };
  // Branch-free per bucket: once no 16-bit value lies strictly inside the
  // bracket (the midpoint equals an end), the pass counts at the lower end; if
  // C == k / B there the bucket's threshold is found (this catches a starting
  // lower end that already holds exactly k / B elements), else the bucket is
  // done unresolved (tied images at its k/B-th value). A finished bucket keeps
  // its bracket (lower end = its threshold when found).
  bool done = false, exact = false;
  for (;;) {
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const uint32_t nmid = P::midpoint(nlo2, nhi2);
      const bool coll = nmid == nlo2 || nmid == nhi2;
      const uint32_t nm2 = coll ? nlo2 : nmid;
      uint32_t d[W];
      const int cb = int(bucket_sum<B>(lane_count(nm2, d), b));
      const bool hit = cb == kb, ge = cb >= kb;
      nlo2 = (!done && ge) ? nm2 : nlo2;
      nhi2 = (!done && !ge) ? nm2 : nhi2;
      exact = exact || (!done && hit);
      done = done || hit || coll;
    }
    if (__all_sync(FULL, done)) break;
  }
  lo2 = nlo2 ^ 0x80008000u;
  hi2 = nhi2 ^ 0x80008000u;
  // Buckets with a threshold: their kept sets {h >= lo} placed in one pass.
  // An unresolved bucket reserves its k / B list positions (its first lane
  // counts k / B, its lanes store nothing: all differences negative) and is
  // finished below.
  uint32_t sw[W];
  const uint32_t cex = lane_count(nlo2, sw);
  if (!exact) {
#pragma unroll
    for (int w = 0; w < W; ++w) sw[w] = 0x80008000u;
  }
  const uint32_t cl = exact ? cex : ((lane % LB) == 0 ? uint32_t(kb) : 0u);
  stage_exact<W, true>(sw, cl, lane, static_cast<uint32_t>(__cvta_generic_to_shared(list)));
  const unsigned open = __ballot_sync(FULL, !exact);
  if (open != 0u) {
    // unresolved buckets (tied images at the k/B-th value): exact binary32
    // search inside the bucket's last 16-bit bracket {lo <= h < hi}, then the
    // general fill at the bucket's list positions
    __syncwarp();
    float x[NE];
    reload<T, NE>(srow, lane, x);
    const float lo = P::low_f32(lo2), hi = P::low_f32(hi2);
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
#pragma unroll 1
    for (int bs = 0; bs < B; ++bs) {
      if (!((open >> (bs * LB)) & 1u)) continue;  // warp-uniform
      const bool act = b == bs;
      const float flo = o2f(__reduce_min_sync(FULL, f2o(act ? bmin : pos_inf())));
      const float fhi = next_up_f32(o2f(__reduce_max_sync(FULL, f2o(act ? bmax : neg_inf()))));
      finish_binary32<NE>(x, flo, fhi, kb, lane, list, st, act, bs * kb);
    }
  }
  copy_out<T, Lane<T, NE>::RW, IdxT>(list, srow, k, lane, vrow, irow);
}

// ---- one row split into B buckets that keep one or two elements each --------
// Exact mode, k / B <= 2 (B = 2 .. 32 on a full row): no search. With
// S = 32 / B lanes per bucket, each lane keeps its best one or two elements in
// the definition's order (value descending, index ascending: only a strictly
// larger value replaces, so among equal values the earlier index stays), then
// log2(S) butterfly rounds merge the lanes' lists (a total order: indices are
// distinct), and the first lane of each bucket writes the bucket's entries in
// ascending index order straight to the CBSR row.
template <typename T, int NE, int B, typename IdxT>
__device__ __forceinline__ void process_row_bucket_small(const uint32_t* __restrict__ srow, int k, int lane,
                                                         uint32_t* __restrict__ list, T* __restrict__ vrow,
                                                         IdxT* __restrict__ irow, uint32_t& st) {
  constexpr unsigned FULL = 0xffffffffu;
  constexpr int S = 32 / B;  // lanes per bucket
  const int kb = k / B;      // 1 or 2
  float x[NE];
  reload<T, NE>(srow, lane, x);
  float a = fabsf(x[0]);
  int e = 1;
#pragma unroll
  for (; e + 1 < NE; e += 2) a = max3_nan(a, fabsf(x[e]), fabsf(x[e + 1]));
  if (e < NE) a = max_nan(a, fabsf(x[e]));
  if (!(warp_max_nan(a) <= 1e38f)) {
    // invalid row: report which precondition fails, write the first k elements
    bool nonfinite = false, range = false;
#pragma unroll
    for (int q = 0; q < NE; ++q) {
      const float b = fabsf(x[q]);
      nonfinite |= !(b <= 3.402823466e38f);
      range |= (b > 1e38f && b <= 3.402823466e38f);
    }
    if (__any_sync(FULL, nonfinite)) st |= kStatusNonFinite;
    if (__any_sync(FULL, range)) st |= kStatusRange;
    for (int p = lane; p < k; p += 32) list[p] = uint32_t(p);
    copy_out<T, Lane<T, NE>::RW, IdxT>(list, srow, k, lane, vrow, irow);
    return;
  }
  // the lane's best two, in the definition's order
  float v0 = x[0], v1 = neg_inf();
  int i0 = lane * NE, i1 = -1;
#pragma unroll
  for (int q = 1; q < NE; ++q) {
    const float xv = x[q];
    const int j = lane * NE + q;
    const bool g0 = xv > v0, g1 = xv > v1;
    v1 = g0 ? v0 : (g1 ? xv : v1);
    i1 = g0 ? i0 : (g1 ? j : i1);
    v0 = g0 ? xv : v0;
    i0 = g0 ? j : i0;
  }
  auto better = [](float av, int ai, float bv, int bi) { return av > bv || (av == bv && ai < bi); };
#pragma unroll
  for (int d = 1; d < S; d <<= 1) {
    const float pv0 = __shfl_xor_sync(FULL, v0, d);
    const int pi0 = __shfl_xor_sync(FULL, i0, d);
    const bool mine = better(v0, i0, pv0, pi0);  // this lane's first is the merged first
    if (kb == 2) {
      const float pv1 = __shfl_xor_sync(FULL, v1, d);
      const int pi1 = __shfl_xor_sync(FULL, i1, d);
      // second: the better of (my second, partner's first) or (my first, partner's second)
      const float av = mine ? v1 : v0, bv = mine ? pv0 : pv1;
      const int ai = mine ? i1 : i0, bi = mine ? pi0 : pi1;
      const bool ta = better(av, ai, bv, bi);
      v1 = ta ? av : bv;
      i1 = ta ? ai : bi;
    }
    v0 = mine ? v0 : pv0;
    i0 = mine ? i0 : pi0;
  }
  auto bits = [](float v) -> T {
    if constexpr (sizeof(T) == 4) {
      return v;
    } else {
      return T(__float_as_uint(v) >> 16);  // the bf16 pattern the value was widened from
    }
  };
  if ((lane & (S - 1)) == 0) {
    const int b = lane / S;
    if (kb == 1) {
      vrow[b] = bits(v0);
      irow[b] = IdxT(i0);
    } else {
      const bool o = i0 < i1;
      vrow[2 * b] = bits(o ? v0 : v1);
      irow[2 * b] = IdxT(o ? i0 : i1);
      vrow[2 * b + 1] = bits(o ? v1 : v0);
      irow[2 * b + 1] = IdxT(o ? i1 : i0);
    }
  }
  __syncwarp();
}

// The general fill of the replay (keep every x >= hi, then the first k - c(hi)
// of lo <= x < hi by index), for canonical values (no -0) and finite ends:
// the lane's classification as two bit masks from the sign bits of x - hi and
// x - lo (set: x below the end), lane counts by popc, one warp scan of both
// counts, and the lane's kept elements stored by walking its kept-bit mask.
// Used at 32 elements per lane with k <= 32 (GB300, rows of 1024, max_iter 2:
// fp32 k = 16 / 32 306 / 308 -> 277 / 285 us, bf16 304 / 310 -> 261 / 269 us;
// max_iter 5, k = 32: fp32 370 -> 315 us). Where a lane keeps many elements
// (k >= 64: rows of 512, k = 256: 195 -> 230 us) or holds fewer (rows of 512,
// k = 32: 160 -> 173 us; rows of 128: 271 -> 347 us) the divergent mask walk
// costs more than one predicated store per element.
template <int NE>
__device__ __forceinline__ void stage_general_masks(const float (&x)[NE], float lo, float hi, int k, int lane,
                                                    uint32_t* __restrict__ list) {
  static_assert(NE <= 32, "one mask word per lane");
  uint32_t lt_hi = 0u, lt_lo = 0u;  // bit e: x[e] < hi, x[e] < lo
#pragma unroll
  for (int e = 0; e < NE; ++e) {
    lt_hi |= (__float_as_uint(__fsub_rn(x[e], hi)) >> 31) << e;
    lt_lo |= (__float_as_uint(__fsub_rn(x[e], lo)) >> 31) << e;
  }
  constexpr uint32_t kAll = NE == 32 ? 0xffffffffu : ((1u << NE) - 1u);
  const uint32_t s_m = ~lt_hi & kAll;   // x >= hi: kept
  const uint32_t b_m = lt_hi & ~lt_lo;  // lo <= x < hi: the first need of them by index
  const uint32_t sc = uint32_t(__popc(s_m)), bc = uint32_t(__popc(b_m));
  uint32_t incl = sc | (bc << 16);
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const uint32_t t = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= d) incl += t;
  }
  const uint32_t tot = __shfl_sync(0xffffffffu, incl, 31);
  const uint32_t ex = incl - (sc | (bc << 16));
  const int need = k - int(tot & 0xffffu);
  const int bstart = int(ex >> 16);
  int r = need - bstart;  // this lane keeps its first r borderline elements
  r = r < 0 ? 0 : (r > int(bc) ? int(bc) : r);
  uint32_t kb = b_m;
  for (int d = int(bc) - r; d > 0; --d) kb ^= 0x80000000u >> __clz(kb);  // drop the highest
  uint32_t km = s_m | kb;
  uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(list)) +
               4u * (uint32_t(ex & 0xffffu) + uint32_t(bstart < need ? bstart : need));
  const uint32_t j0 = uint32_t(lane * NE);
  while (km != 0u) {
    const uint32_t e = uint32_t(__ffs(km) - 1);
    asm volatile("st.shared.u32 [%0], %1;" ::"r"(a), "r"(j0 + e) : "memory");
    a += 4u;
    km &= km - 1u;
  }
}

// ---- one row, replay of the value-space bisection ---------------------------
// Early stop (max_iter cap, eps) or exact mode with per-row pass counts: the
// RTop-K summary page, "Approach": bisection over the row's value range
// [min, max] with the binary32 midpoint (lo + hi) * 0.5, at most `limit`
// counting passes, stopping once hi - lo <= eps, once no binary32 value lies
// strictly inside, or at a threshold that keeps exactly k; then every x >= hi
// is kept and the rest of k comes from lo <= x < hi by ascending index (the
// general fill). When ties at the row maximum alone fill k, the k
// lowest-index maxima are kept after no pass. Every comparison, midpoint and
// difference is binary32 and rounded as written, so the pass count and the
// kept set are those of the plain sequential replay.
template <typename T, int NE, typename IdxT>
__device__ __forceinline__ void process_row_replay(const uint32_t* __restrict__ srow, int k, int limit,
                                                   bool cap_is_safety, float eps, int lane,
                                                   uint32_t* __restrict__ list, T* __restrict__ vrow,
                                                   IdxT* __restrict__ irow, int* __restrict__ it_out,
                                                   uint32_t& st) {
  constexpr unsigned FULL = 0xffffffffu;
  float x[NE];
  reload<T, NE>(srow, lane, x);
  float mx = x[0], mn = x[0];
  int e = 1;
#pragma unroll
  for (; e + 1 < NE; e += 2) {
    mx = max3_nan(mx, x[e], x[e + 1]);
    mn = min3_nan(mn, x[e], x[e + 1]);
  }
  if (e < NE) {
    mx = max_nan(mx, x[e]);
    mn = min_nan(mn, x[e]);
  }
  float hi = warp_max_nan(mx), lo = warp_min_nan(mn);
  int it = 0;
#pragma unroll
  for (int q = 0; q < NE; ++q) x[q] = __fadd_rn(x[q], 0.0f);  // -0 -> +0 (counts, not output bits)
  if (!(hi <= 1e38f && lo >= -1e38f)) {
    // invalid row: report which precondition fails, write the first k elements
    bool nonfinite = false, range = false;
#pragma unroll
    for (int q = 0; q < NE; ++q) {
      const float a = fabsf(x[q]);
      nonfinite |= !(a <= 3.402823466e38f);
      range |= (a > 1e38f && a <= 3.402823466e38f);
    }
    if (__any_sync(FULL, nonfinite)) st |= kStatusNonFinite;
    if (__any_sync(FULL, range)) st |= kStatusRange;
    for (int p = lane; p < k; p += 32) list[p] = uint32_t(p);
  } else {
    // ties at the maximum fill k only if k / NE lanes hold the maximum
    bool max_tie = false;
    if (__popc(__ballot_sync(FULL, mx == hi)) * NE >= k) max_tie = int(warp_sum(lane_count_ge<NE>(x, hi))) >= k;
    if (max_tie) {
      lo = hi;  // [max, next above max): the maxima, filled by lowest index
      hi = next_up_f32(hi);
    } else {
      // invariant: c(lo) >= k > c(hi)
      for (;;) {
        if (it >= limit) {
          if (cap_is_safety) st |= kStatusSafetyCap;
          break;
        }
        if (!(__fsub_rn(hi, lo) > eps)) break;
        const float mid = __fmul_rn(__fadd_rn(lo, hi), 0.5f);
        if (!(lo < mid && mid < hi)) break;
        const int cnt = int(warp_sum(lane_count_ge<NE>(x, mid)));
        ++it;
        if (cnt >= k) lo = mid;
        else hi = mid;
        if (cnt == k) break;
      }
    }
    bool masks = false;
    if constexpr (NE >= 32) masks = k <= 32;
    if (masks) {
      stage_general_masks<NE>(x, lo, hi, k, lane, list);
    } else {
      stage_general<NE>(x, lo, hi, k, lane, list);
    }
  }
  if (it_out != nullptr && lane == 0) *it_out = it;
  copy_out<T, Lane<T, NE>::RW, IdxT>(list, srow, k, lane, vrow, irow);
}

#ifndef RTOPK_LEAN_MIN_BLOCKS
#define RTOPK_LEAN_MIN_BLOCKS 5
#endif
// Rows in flight per warp (shared stages) and resident blocks of 256 per SM.
// Rows of 1024 fp32 (128 bytes per lane): 2 blocks (72 KB of stages each, 80+
// registers; at 3 blocks the kernel spills); measured on GB300 at 2^18 rows:
// 224-333 us at 2 blocks against 233-343 us at 3 (k = 16..256), bf16 rows of
// 1024 the other way round (234-367 against 250-392 us).
template <typename T, int NE>
struct LeanCfg {
  static constexpr int kStages = NE <= 8 ? 3 : 2;
  static constexpr int kBlocks =
      NE <= 8 ? RTOPK_LEAN_MIN_BLOCKS : ((NE >= 32 && sizeof(T) == 4) ? 2 : 3);
};

// Whether rows of 32 * NE elements take guessed probes (process_row, GUESS)
// when k > 32. Measured on GB300, 2^18 N(0,1) rows, k = 64..256: fp32 rows of
// 1024 4-8% faster (k = 256 327 -> 303 us), bf16 rows of 512 / 1024 2-15%
// faster; fp32 rows of 512 were not faster, and every k <= 32 (bracket from
// the smallest lane maximum) was slower with guesses.
template <typename T, int NE>
constexpr bool kGuessRows = NE >= 32 || (NE >= 16 && sizeof(T) == 2);

// Full rows of 32 * NE elements, exact mode, k <= kListK, 16-byte aligned
// (B > 1: B buckets per row, B dividing 32 and k). One warp per row,
// persistent over rows; each warp keeps kStages rows in flight through
// cp.async copies into its own shared stages.
// SMALLB (B > 1): the buckets keep one or two elements each
// (process_row_bucket_small) instead of searching side by side.
template <typename T, int NE, typename IdxT, int B = 1, bool GUESS = false, bool SMALLB = false>
__global__ void __launch_bounds__(256, LeanCfg<T, NE>::kBlocks)
rtopk_lean_kernel(const T* __restrict__ in, int64_t N, int k, T* __restrict__ vals, IdxT* __restrict__ idx,
                  uint32_t* __restrict__ status) {
  constexpr int RW = Lane<T, NE>::RW;
  constexpr int S = LeanCfg<T, NE>::kStages;
  constexpr int kRowWords = 32 * RW;
  __shared__ __align__(16) uint32_t ring_all[8][S][kRowWords];
  __shared__ uint32_t list_all[8][kListK];
  const int lane = threadIdx.x & 31;
  const int wib = threadIdx.x >> 5;
  uint32_t* list = list_all[wib];
  const int64_t nw = int64_t(gridDim.x) * 8;
  const int64_t r0 = int64_t(blockIdx.x) * 8 + wib;
  const int nrows = r0 < N ? int((N - 1 - r0) / nw) + 1 : 0;  // rows r0, r0 + nw, ... < N
  constexpr uint32_t kStageBytes = uint32_t(kRowWords) * 4u;
  const uint32_t ring_base = static_cast<uint32_t>(__cvta_generic_to_shared(ring_all[wib][0]));
  const uint32_t* src = reinterpret_cast<const uint32_t*>(in) + r0 * kRowWords + lane * 4;  // next row to issue
  const int64_t src_step = nw * kRowWords;
  uint32_t st = 0;
  float tprev = __int_as_float(0x7fc00000), rho = 0.0f;  // search guesses carried across the warp's rows
  // prologue: the warp's first S rows
#pragma unroll
  for (int q = 0; q < S; ++q) {
    issue_row<RW>(ring_base + uint32_t(q) * kStageBytes, src, lane, q < nrows);
    src += src_step;
  }
  T* vrow = vals + r0 * int64_t(k);
  IdxT* irow = idx + r0 * int64_t(k);
  const int64_t out_step = nw * int64_t(k);
  int q = 0;
  for (int i = 0; i < nrows; ++i) {
    wait_rows<S - 1>();  // this row's copy group is complete
    __syncwarp();
    if constexpr (B == 1) {
      process_row<T, NE, IdxT, GUESS>(ring_all[wib][q], k, lane, list, vrow, irow, st, tprev, rho);
    } else if constexpr (SMALLB) {
      process_row_bucket_small<T, NE, B, IdxT>(ring_all[wib][q], k, lane, list, vrow, irow, st);
    } else {
      process_row_bucketed<T, NE, B, IdxT>(ring_all[wib][q], k, lane, list, vrow, irow, st);
    }
    // process_row ends with __syncwarp: every lane is done with this stage
    issue_row<RW>(ring_base + uint32_t(q) * kStageBytes, src, lane, i + S < nrows);
    src += src_step;
    vrow += out_step;
    irow += out_step;
    q = (q + 1 == S) ? 0 : q + 1;
  }
  wait_rows<0>();
  if (status != nullptr && st != 0u && lane == 0) atomicOr(status, st);
}

// Full rows of 32 * NE elements, replay mode (process_row_replay: early stop,
// eps, or pass counts written to iters when it is not null), k <= kListK,
// 16-byte aligned; the same row ring as rtopk_lean_kernel.
template <typename T, int NE, typename IdxT>
__global__ void __launch_bounds__(256, LeanCfg<T, NE>::kBlocks)
rtopk_lean_replay_kernel(const T* __restrict__ in, int64_t N, int k, int max_iter, float eps, T* __restrict__ vals,
                         IdxT* __restrict__ idx, int* __restrict__ iters, uint32_t* __restrict__ status) {
  constexpr int RW = Lane<T, NE>::RW;
  constexpr int S = LeanCfg<T, NE>::kStages;
  constexpr int kRowWords = 32 * RW;
  __shared__ __align__(16) uint32_t ring_all[8][S][kRowWords];
  __shared__ uint32_t list_all[8][kListK];
  const int lane = threadIdx.x & 31;
  const int wib = threadIdx.x >> 5;
  uint32_t* list = list_all[wib];
  const int64_t nw = int64_t(gridDim.x) * 8;
  const int64_t r0 = int64_t(blockIdx.x) * 8 + wib;
  const int nrows = r0 < N ? int((N - 1 - r0) / nw) + 1 : 0;  // rows r0, r0 + nw, ... < N
  constexpr uint32_t kStageBytes = uint32_t(kRowWords) * 4u;
  const uint32_t ring_base = static_cast<uint32_t>(__cvta_generic_to_shared(ring_all[wib][0]));
  const uint32_t* src = reinterpret_cast<const uint32_t*>(in) + r0 * kRowWords + lane * 4;  // next row to issue
  const int64_t src_step = nw * kRowWords;
  const bool cap_is_safety = (max_iter < 0 || max_iter > kSafetyCap);
  const int limit = cap_is_safety ? kSafetyCap : max_iter;
  uint32_t st = 0;
#pragma unroll
  for (int q = 0; q < S; ++q) {
    issue_row<RW>(ring_base + uint32_t(q) * kStageBytes, src, lane, q < nrows);
    src += src_step;
  }
  T* vrow = vals + r0 * int64_t(k);
  IdxT* irow = idx + r0 * int64_t(k);
  int* itrow = iters != nullptr ? iters + r0 : nullptr;
  const int64_t out_step = nw * int64_t(k);
  int q = 0;
  for (int i = 0; i < nrows; ++i) {
    wait_rows<S - 1>();  // this row's copy group is complete
    __syncwarp();
    process_row_replay<T, NE, IdxT>(ring_all[wib][q], k, limit, cap_is_safety, eps, lane, list, vrow, irow, itrow,
                                    st);
    // copy_out ends with __syncwarp: every lane is done with this stage
    issue_row<RW>(ring_base + uint32_t(q) * kStageBytes, src, lane, i + S < nrows);
    src += src_step;
    vrow += out_step;
    irow += out_step;
    if (itrow != nullptr) itrow += nw;
    q = (q + 1 == S) ? 0 : q + 1;
  }
  wait_rows<0>();
  if (status != nullptr && st != 0u && lane == 0) atomicOr(status, st);
}

}  // namespace lean
}  // namespace rtopk
