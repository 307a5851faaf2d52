// bf16-path instantiations for head dim 32: prep and scan kernels (tcgen05).
#include "kernels_tc.cuh"

namespace prism {
cudaError_t launch_prep_32(int C, const PrepArgs& a, cudaStream_t s) {
  switch (C) {
    case 16: return launch_prep_t<32, 16>(a, s);
    case 32: return launch_prep_t<32, 32>(a, s);
    case 64: return launch_prep_t<32, 64>(a, s);
  }
  return cudaErrorInvalidValue;
}
cudaError_t launch_weights_32(const float* Wk, const float* Wp, int H, int L, unsigned char* blocks,
                              int* flag, cudaStream_t s) {
  prep_weights_kernel<32><<<H * L * 2 * WeightBlock<32>::kCtas, 256, 0, s>>>(Wk, Wp, H, L, blocks, flag);
  return cudaGetLastError();
}
size_t prep_smem_32(int C) {
  switch (C) {
    case 16: return PrepSmem<32, 16>::bytes;
    case 32: return PrepSmem<32, 32>::bytes;
    case 64: return PrepSmem<32, 64>::bytes;
  }
  return 0;
}
cudaError_t launch_scan_tc_32(int C, const ScanTcArgs& a, cudaStream_t s) {
  switch (C) {
    case 16: return launch_scan_tc_t<32, 16>(a, s);
    case 32: return launch_scan_tc_t<32, 32>(a, s);
    case 64: return launch_scan_tc_t<32, 64>(a, s);
  }
  return cudaErrorInvalidValue;
}
}  // namespace prism
