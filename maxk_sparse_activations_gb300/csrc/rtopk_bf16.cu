// bf16 rows of at most 1024 elements with int32 indices (rtopk_select).
#include "rtopk_dispatch.cuh"

namespace rtopk {

cudaError_t launch_select_bf16_short_i32(const SelectArgs& a, cudaStream_t s) {
  return launch_short_rows<uint16_t, int32_t>(a, s);
}

}  // namespace rtopk
