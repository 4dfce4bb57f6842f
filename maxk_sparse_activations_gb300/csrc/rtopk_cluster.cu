// Rows of 8193..65536 elements (one CTA cluster per row), fp32 and bf16 with int32 indices.
#include "rtopk_dispatch.cuh"

namespace rtopk {

cudaError_t launch_select_f32_cluster(const SelectArgs& a, cudaStream_t s) {
  return launch_cluster_rows<float, int32_t>(a, s);
}

cudaError_t launch_select_bf16_cluster(const SelectArgs& a, cudaStream_t s) {
  return launch_cluster_rows<uint16_t, int32_t>(a, s);
}

}  // namespace rtopk
