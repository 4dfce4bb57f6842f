// Rows of 2048, 4096 and 8192 elements in exact mode without pass counts: one
// team of 2, 4 or 8 warps per row (rtopk_lean_block.cuh). Other rows and
// modes are not taken.
#include <cstdint>

#include "rtopk_lean_block.cuh"
#include "launch.h"

namespace rtopk {
namespace {

template <typename T, int NE, int TW, typename IdxT>
cudaError_t launch_lb(const SelectArgs& a, cudaStream_t s) {
  using Cfg = lean::LeanBlockCfg<T, NE, TW>;
  auto kern = lean::rtopk_lean_block_kernel<T, NE, TW, IdxT>;
  const size_t smem = Cfg::kSmem;
  cudaError_t e = cudaFuncSetAttribute(reinterpret_cast<const void*>(kern),
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  if (e != cudaSuccess) return e;
  const int blocks =
      persistent_blocks(reinterpret_cast<const void*>(kern), 256, smem, (a.N + Cfg::kTeams - 1) / Cfg::kTeams);
  if (blocks <= 0) return cudaErrorInvalidConfiguration;
  kern<<<blocks, 256, smem, s>>>(static_cast<const T*>(a.in), a.N, a.k, static_cast<T*>(a.vals),
                                 static_cast<IdxT*>(a.idx), a.status);
  return cudaGetLastError();
}

#ifndef RTOPK_LEAN_BLOCK
#define RTOPK_LEAN_BLOCK 1
#endif

bool takes(const SelectArgs& a) {
  return RTOPK_LEAN_BLOCK && a.max_iter < 0 && a.eps == 0.0f && a.iters == nullptr && a.k <= lean::kBlockListK &&
         (reinterpret_cast<uintptr_t>(a.in) & 15u) == 0 && (a.M == 2048 || a.M == 4096 || a.M == 8192);
}

// 32 elements per thread: 2, 4 and 8 warps per row (GB300, 2^16 fp32 rows of
// 2048, k = 64: 8 warps 374 us, 4 warps 234 us, 2 warps 191 us).
template <typename T, typename IdxT>
cudaError_t launch_by_m(const SelectArgs& a, cudaStream_t s) {
  switch (a.M) {
    case 2048: return launch_lb<T, 32, 2, IdxT>(a, s);
    case 4096: return launch_lb<T, 32, 4, IdxT>(a, s);
    default: return launch_lb<T, 32, 8, IdxT>(a, s);
  }
}

}  // namespace

bool launch_lean_block_f32(const SelectArgs& a, cudaStream_t s, cudaError_t& err) {
  if (!takes(a)) return false;
  err = launch_by_m<float, int32_t>(a, s);
  return true;
}

bool launch_lean_block_bf16(const SelectArgs& a, bool idx16, cudaStream_t s, cudaError_t& err) {
  if (!takes(a)) return false;
  err = idx16 ? launch_by_m<uint16_t, int16_t>(a, s) : launch_by_m<uint16_t, int32_t>(a, s);
  return true;
}

}  // namespace rtopk
