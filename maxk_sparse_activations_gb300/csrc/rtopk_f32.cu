// fp32 instances of the row-wise top-k kernel (int32 indices).
#include "rtopk_dispatch.cuh"

namespace rtopk {

cudaError_t launch_select_f32(const SelectArgs& a, cudaStream_t s) {
  const int M = a.M;
  const bool vec = (M % 4 == 0) && aligned16(a.in);
  if (M <= 1024) {  // one warp per row, G groups of 128
    const int need = (M + 127) / 128;
    const int G = need <= 4 ? need : (need <= 6 ? 6 : 8);
    const bool full = vec && M == G * 128;
    switch (G) {
      case 1: return launch_config<float, 1, 1, int32_t>(a, full, vec, s);
      case 2: return launch_config<float, 2, 1, int32_t>(a, full, vec, s);
      case 3: return launch_config<float, 3, 1, int32_t>(a, full, vec, s);
      case 4: return launch_config<float, 4, 1, int32_t>(a, full, vec, s);
      case 6: return launch_config<float, 6, 1, int32_t>(a, full, vec, s);
      default: return launch_config<float, 8, 1, int32_t>(a, full, vec, s);
    }
  }
  // one 256-thread block per row, G groups of 128 per warp
  const int need = (M + 1023) / 1024;
  const int G = need <= 4 ? need : (need <= 6 ? 6 : 8);
  const bool full = vec && M == G * 1024;
  switch (G) {
    case 2: return launch_config<float, 2, 8, int32_t>(a, full, vec, s);
    case 3: return launch_config<float, 3, 8, int32_t>(a, full, vec, s);
    case 4: return launch_config<float, 4, 8, int32_t>(a, full, vec, s);
    case 6: return launch_config<float, 6, 8, int32_t>(a, full, vec, s);
    default: return launch_config<float, 8, 8, int32_t>(a, full, vec, s);
  }
}

}  // namespace rtopk
