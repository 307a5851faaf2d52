// Anchor/refinement-kernel instantiations for every I/O type and head dim.
#include "kernels_inst.cuh"

namespace prism {
cudaError_t launch_k1(int dtype, int D, const K1Args& a, cudaStream_t s) {
  if (dtype == 1) {
    switch (D) {
      case 16: return launch_k1_t<__nv_bfloat16, 16>(a, s);
      case 32: return launch_k1_t<__nv_bfloat16, 32>(a, s);
      case 64: return launch_k1_t<__nv_bfloat16, 64>(a, s);
      case 128: return launch_k1_t<__nv_bfloat16, 128>(a, s);
    }
  } else {
    switch (D) {
      case 16: return launch_k1_t<float, 16>(a, s);
      case 32: return launch_k1_t<float, 32>(a, s);
      case 64: return launch_k1_t<float, 64>(a, s);
    }
  }
  return cudaErrorInvalidValue;
}

size_t k1_smem_bytes(int dtype, int D) {
  if (dtype == 0 && D == 128) return 0;
  return dtype == 1 ? k1_bytes_t<__nv_bfloat16>(D) : k1_bytes_t<float>(D);
}
size_t k2_smem_bytes(int dtype, int D, int C) {
  if (dtype == 0 && D == 128) return 0;
  return dtype == 1 ? k2_bytes_t<__nv_bfloat16>(D, C) : k2_bytes_t<float>(D, C);
}
}  // namespace prism
