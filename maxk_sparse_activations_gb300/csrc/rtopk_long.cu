// Rows of 2049..8192 elements: one 256-thread block per row; 8193..65536: one
// CTA cluster per row; all dtypes; and the dtype / row-length dispatch behind
// launch.h (exact rows of 2048 / 4096 / 8192 without pass counts go to the
// 16-bit multi-warp kernel first).
#include "rtopk_dispatch.cuh"

namespace rtopk {

cudaError_t launch_select_f32_short(const SelectArgs& a, cudaStream_t s);
cudaError_t launch_select_bf16_short_i32(const SelectArgs& a, cudaStream_t s);
cudaError_t launch_select_bf16_short_i16(const SelectArgs& a, cudaStream_t s);
cudaError_t launch_select_f32_cluster(const SelectArgs& a, cudaStream_t s);
cudaError_t launch_select_bf16_cluster(const SelectArgs& a, cudaStream_t s);
// exact rows of 2048 / 4096 / 8192 without pass counts: true when launched
bool launch_lean_block_f32(const SelectArgs& a, cudaStream_t s, cudaError_t& err);
bool launch_lean_block_bf16(const SelectArgs& a, bool idx16, cudaStream_t s, cudaError_t& err);

cudaError_t launch_select_f32(const SelectArgs& a, cudaStream_t s) {
  cudaError_t err = cudaSuccess;
  if (launch_lean_block_f32(a, s, err)) return err;
  if (a.M <= kWarpMaxM) return launch_select_f32_short(a, s);
  if (a.M > 8192) return launch_select_f32_cluster(a, s);
  return launch_long_rows<float, int32_t>(a, s);
}

cudaError_t launch_select_bf16(const SelectArgs& a, bool idx16, cudaStream_t s) {
  cudaError_t err = cudaSuccess;
  if (launch_lean_block_bf16(a, idx16, s, err)) return err;
  if (a.M <= kWarpMaxM) return idx16 ? launch_select_bf16_short_i16(a, s) : launch_select_bf16_short_i32(a, s);
  if (a.M > 8192) return idx16 ? cudaErrorInvalidValue : launch_select_bf16_cluster(a, s);
  return idx16 ? launch_long_rows<uint16_t, int16_t>(a, s) : launch_long_rows<uint16_t, int32_t>(a, s);
}

}  // namespace rtopk
