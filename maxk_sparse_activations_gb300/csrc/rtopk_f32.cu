// fp32 rows of at most 1024 elements: one warp per row (int32 indices).
#include "rtopk_dispatch.cuh"

namespace rtopk {

cudaError_t launch_select_f32_short(const SelectArgs& a, cudaStream_t s) {
  return launch_short_rows<float, int32_t>(a, s);
}

}  // namespace rtopk
