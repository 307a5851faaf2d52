// Scan-kernel instantiations: f32 I/O, head dim 32, every chunk length.
#include "kernels_inst.cuh"

namespace prism {
cudaError_t launch_k2_f32_32(int C, const K2Args& a, cudaStream_t s) {
  switch (C) {
    case 16: return launch_k2_t<float, 32, 16>(a, s);
    case 32: return launch_k2_t<float, 32, 32>(a, s);
    case 64: return launch_k2_t<float, 32, 64>(a, s);
  }
  return cudaErrorInvalidValue;
}
}  // namespace prism
