// fp32-path instantiations of the anchor/refinement kernel (SIMT fp32).
#include "kernels_inst.cuh"

namespace prism {
cudaError_t launch_k1(int dtype, int D, const K1Args& a, cudaStream_t s) {
  if (dtype == 0) {
    switch (D) {
      case 16: return launch_k1_t<float, 16>(a, s);
      case 32: return launch_k1_t<float, 32>(a, s);
      case 64: return launch_k1_t<float, 64>(a, s);
    }
  }
  return cudaErrorInvalidValue;
}

size_t k1_smem_bytes(int dtype, int D) { return dtype == 0 && D <= 64 ? k1_bytes_t<float>(D) : 0; }
size_t k2_smem_bytes(int dtype, int D, int C) { return dtype == 0 && D <= 64 ? k2_bytes_t<float>(D, C) : 0; }
}  // namespace prism
