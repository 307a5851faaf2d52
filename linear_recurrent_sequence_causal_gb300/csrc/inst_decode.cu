// Single-token decode step: instantiations for both I/O dtypes and every head dim.
#include <cuda_runtime.h>

#include "decode.cuh"

namespace prism {
template <class T, int D>
cudaError_t launch_decode_t(const DecodeArgs& a, cudaStream_t s) {
  using S = DecodeSmem<D>;
  auto fn = decode_kernel<T, D>;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)S::bytes);
  if (e != cudaSuccess) return e;
  fn<<<a.B * a.H, kDecodeThreads, S::bytes, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_decode(int dtype, int D, const DecodeArgs& a, cudaStream_t s) {
  if (dtype == 0) {
    switch (D) {
      case 16: return launch_decode_t<float, 16>(a, s);
      case 32: return launch_decode_t<float, 32>(a, s);
      case 64: return launch_decode_t<float, 64>(a, s);
      case 128: return launch_decode_t<float, 128>(a, s);
    }
  } else {
    switch (D) {
      case 16: return launch_decode_t<__nv_bfloat16, 16>(a, s);
      case 32: return launch_decode_t<__nv_bfloat16, 32>(a, s);
      case 64: return launch_decode_t<__nv_bfloat16, 64>(a, s);
      case 128: return launch_decode_t<__nv_bfloat16, 128>(a, s);
    }
  }
  return cudaErrorInvalidValue;
}
}  // namespace prism
