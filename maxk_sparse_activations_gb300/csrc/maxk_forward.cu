// bf16 rows of at most 1024 elements with int16 indices (maxk_forward).
#include "rtopk_dispatch.cuh"

namespace rtopk {

cudaError_t launch_select_bf16_short_i16(const SelectArgs& a, cudaStream_t s) {
  return launch_short_rows<uint16_t, int16_t>(a, s);
}

}  // namespace rtopk
