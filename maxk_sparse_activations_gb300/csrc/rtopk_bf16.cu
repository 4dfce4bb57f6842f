// bf16 instances of the row-wise top-k kernel (int32 or int16 indices).
#include "rtopk_dispatch.cuh"

namespace rtopk {

template <typename IdxT>
static cudaError_t launch_bf16_idx(const SelectArgs& a, cudaStream_t s) {
  const int M = a.M;
  const bool vec = (M % 8 == 0) && aligned16(a.in);
  if (M <= 1024) {  // one warp per row, G groups of 256
    const int G = (M + 255) / 256;
    const bool full = vec && M == G * 256;
    switch (G) {
      case 1: return launch_config<uint16_t, 1, 1, IdxT>(a, full, vec, s);
      case 2: return launch_config<uint16_t, 2, 1, IdxT>(a, full, vec, s);
      case 3: return launch_config<uint16_t, 3, 1, IdxT>(a, full, vec, s);
      default: return launch_config<uint16_t, 4, 1, IdxT>(a, full, vec, s);
    }
  }
  const int G = (M + 2047) / 2048;  // one 256-thread block per row
  const bool full = vec && M == G * 2048;
  switch (G) {
    case 1: return launch_config<uint16_t, 1, 8, IdxT>(a, full, vec, s);
    case 2: return launch_config<uint16_t, 2, 8, IdxT>(a, full, vec, s);
    case 3: return launch_config<uint16_t, 3, 8, IdxT>(a, full, vec, s);
    default: return launch_config<uint16_t, 4, 8, IdxT>(a, full, vec, s);
  }
}

cudaError_t launch_select_bf16(const SelectArgs& a, bool idx16, cudaStream_t s) {
  return idx16 ? launch_bf16_idx<int16_t>(a, s) : launch_bf16_idx<int32_t>(a, s);
}

}  // namespace rtopk
