// Shared definitions of the row-wise top-k kernels (RTop-K), sm_103a:
// element traits, the register layout of a row and its loads, status bits.
//
// Source: "RTop-K: Ultra-Fast Row-Wise Top-K Selection for Neural Network
// Acceleration on GPUs" (summary page), "Approach"; output layout from
// "MaxK-GNN: Extremely Fast GPU Kernel Design for Accelerating Graph Neural
// Networks Training", "How MaxK-GNN works" / "The idea".
//
// Layout. A "team" of W warps owns one row at a time (W = 1: rtopk_warp.cuh,
// W = 8: rtopk_block.cuh). Each lane holds V consecutive elements (16 bytes of
// input) of each of G groups; a group is 32 * V consecutive elements, so a
// warp covers G * 32 * V elements and a team covers W times that. Element j
// of the row sits in warp w, group g, lane l, slot e with
//     j = (w * G + g) * 32 * V + l * V + e.
// The row lives in registers for the whole search: it is read from HBM once.
//
// Arithmetic matches the scalar definition of the method exactly: the
// midpoint is __fmul_rn(__fadd_rn(lo, hi), 0.5f), the precision test is
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

}  // namespace rtopk
