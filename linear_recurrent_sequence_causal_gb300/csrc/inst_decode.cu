// Single-token decode step: instantiations for both I/O dtypes and every head dim, and
// the choice of the batch grouping and the weight-ring depth.
#include <cuda_runtime.h>

#include "decode.cuh"

namespace prism {
template <class T, int D, int BB>
cudaError_t launch_decode_t(DecodeArgs a, cudaStream_t s) {
  using G = DecodeGeom<D, BB>;
  int dev = 0, sms = 0, smem_sm = 0, smem_optin = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e != cudaSuccess) return e;
  const int ctas = (a.B + BB - 1) / BB * a.H * G::NCL;
  // as many weight slices in flight as fit while the grid still runs in one wave
  // (capped at the 2L slices of the step)
  const int per_sm = (ctas + sms - 1) / sms;
  long budget = (long)smem_sm / (per_sm < 1 ? 1 : per_sm) - 1024;
  if (budget > smem_optin) budget = smem_optin;
  const long fixed = (long)G::bytes(0, a.L, a.w);
  const long slice = (long)sizeof(float) * G::kSlice;
  // (the two slices of a refinement step are used together: at least 2)
  int nbuf = (int)((budget - fixed) / slice);
  if (nbuf > 2 * a.L) nbuf = 2 * a.L;
  if (nbuf < 2) nbuf = a.L > 0 ? 2 : 0;
  a.nbuf = nbuf;
  const size_t bytes = G::bytes(nbuf, a.L, a.w);
  if (bytes > (size_t)smem_optin) return cudaErrorInvalidValue;
  auto fn = decode_kernel<T, D, BB>;
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e != cudaSuccess) return e;
  fn<<<ctas, G::NT, bytes, s>>>(a);   // clusters of G::NCL CTAs
  return cudaGetLastError();
}

template <class T, int D>
cudaError_t launch_decode_d(const DecodeArgs& a, cudaStream_t s) {
  return a.B >= 2 ? launch_decode_t<T, D, 2>(a, s) : launch_decode_t<T, D, 1>(a, s);
}

cudaError_t launch_decode(int dtype, int D, const DecodeArgs& a, cudaStream_t s) {
  if (dtype == 0) {
    switch (D) {
      case 16: return launch_decode_d<float, 16>(a, s);
      case 32: return launch_decode_d<float, 32>(a, s);
      case 64: return launch_decode_d<float, 64>(a, s);
      case 128: return launch_decode_d<float, 128>(a, s);
    }
  } else {
    switch (D) {
      case 16: return launch_decode_d<__nv_bfloat16, 16>(a, s);
      case 32: return launch_decode_d<__nv_bfloat16, 32>(a, s);
      case 64: return launch_decode_d<__nv_bfloat16, 64>(a, s);
      case 128: return launch_decode_d<__nv_bfloat16, 128>(a, s);
    }
  }
  return cudaErrorInvalidValue;
}
}  // namespace prism
