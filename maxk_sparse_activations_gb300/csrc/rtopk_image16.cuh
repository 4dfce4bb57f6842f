// 16-bit images of a row for the packed threshold search, sm_103a: binary16
// (nearest, saturated at +-65504) of fp32 rows, the data themselves for bf16
// rows, two elements per 32-bit word (lower index in bits 0..15).
//
// Source: "RTop-K: Ultra-Fast Row-Wise Top-K Selection for Neural Network
// Acceleration on GPUs" (summary page), "Approach": the exact top-k is one set,
// whatever thresholds the bisection visits, so it may count on any
// order-preserving image of the row (x <= y implies h(x) <= h(y)).
//
// Operations: the bracket midpoint lo * 0.5 + (hi * 0.5) (one rounding, always
// in [lo, hi], odd-symmetric: the midpoint of the negated ends is the negated
// midpoint), packed adds, splats of a binary32 value, and the halves widened
// back to binary32.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

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
  static __device__ __forceinline__ uint32_t add(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("add.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
  }
};

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

}  // namespace rtopk
