// Scan-kernel instantiations: bf16 I/O, head dim 128, every chunk length.
#include "kernels_inst.cuh"

namespace prism {
cudaError_t launch_k2_bf16_128(int C, const K2Args& a, cudaStream_t s) {
  switch (C) {
    case 16: return launch_k2_t<__nv_bfloat16, 128, 16>(a, s);
    case 32: return launch_k2_t<__nv_bfloat16, 128, 32>(a, s);
    case 64: return launch_k2_t<__nv_bfloat16, 128, 64>(a, s);
  }
  return cudaErrorInvalidValue;
}
}  // namespace prism
