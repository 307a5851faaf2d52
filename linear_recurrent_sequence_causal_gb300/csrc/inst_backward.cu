// Backward pass: launches of the five kernels for both I/O dtypes and every head dim.
#include <cuda_runtime.h>

#include "backward.cuh"

namespace prism {

template <class T, int D, int RS>
cudaError_t launch_state(const BwdArgs& a, cudaStream_t s) {
  using S = BwdBSmem<D, RS>;
  auto fn = bwd_state_kernel<T, D, RS>;
  const size_t bytes = S::bytes(a.L, (int)sizeof(T));
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e != cudaSuccess) return e;
  fn<<<dim3(a.H, a.B, RS), S::NT, bytes, s>>>(a);
  return cudaGetLastError();
}

template <class T, int D>
cudaError_t launch_backward_t(const BwdArgs& a, cudaStream_t s) {
  cudaError_t e;
  const int L = a.L;
  {
    auto fn = bwd_refine_fwd_kernel<T, D>;
    if ((e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)BwdASmem<D>::bytes)) != cudaSuccess)
      return e;
    fn<<<dim3((a.T + kBwdTT - 1) / kBwdTT, a.H, a.B), kBwdThreads, BwdASmem<D>::bytes, s>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  switch (a.rs) {
    case 1: e = launch_state<T, D, 1>(a, s); break;
    case 2: e = launch_state<T, D, 2>(a, s); break;
    case 4: e = (D >= 32) ? launch_state<T, D, (D >= 32 ? 4 : 2)>(a, s) : cudaErrorInvalidValue; break;
    default: e = cudaErrorInvalidValue;
  }
  if (e != cudaSuccess) return e;
  if (a.rs > 1) {
    const size_t total = (size_t)a.B * a.T * a.H * ((2 + L) * D + 2);
    const size_t blocks = (total + kBwdThreads - 1) / kBwdThreads;
    bwd_state_reduce_kernel<D><<<(unsigned)(blocks < 4864 ? blocks : 4864), kBwdThreads, 0, s>>>(a, a.rs);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  {
    auto fn = bwd_refine_kernel<T, D>;
    if ((e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)BwdCSmem<D>::bytes)) != cudaSuccess)
      return e;
    fn<<<dim3((a.T + kBwdTC - 1) / kBwdTC, a.H, a.B), kBwdThreads, BwdCSmem<D>::bytes, s>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (L > 0) {
    using WT = BwdWTile<D>;
    bwd_weight_kernel<D><<<dim3(WT::TILES, 2 * L, a.H * a.nsw), WT::NT, 0, s>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (a.nsw > 1) {
      const size_t total = (size_t)a.H * 2 * L * D * D;
      const size_t blocks = (total + kBwdThreads - 1) / kBwdThreads;
      bwd_weight_reduce_kernel<D><<<(unsigned)(blocks < 4864 ? blocks : 4864), kBwdThreads, 0, s>>>(a);
      if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
  }
  bwd_small_weight_kernel<T, D><<<dim3((D + 31) / 32, a.H, a.nss), kBwdThreads, 0, s>>>(a);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (a.nss > 1) {
    const size_t total = (size_t)a.H * (L + a.w) * D;
    const size_t blocks = (total + kBwdThreads - 1) / kBwdThreads;
    bwd_small_reduce_kernel<D><<<(unsigned)(blocks < 4864 ? blocks : 4864), kBwdThreads, 0, s>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  {
    const size_t total = (size_t)a.B * a.T * a.H * D;
    const size_t blocks = (total + kBwdThreads - 1) / kBwdThreads;
    bwd_conv_dv_kernel<D><<<(unsigned)(blocks < 4864 ? blocks : 4864), kBwdThreads, 0, s>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_backward(int dtype, int D, const BwdArgs& a, cudaStream_t s) {
  if (dtype == 0) {
    switch (D) {
      case 16: return launch_backward_t<float, 16>(a, s);
      case 32: return launch_backward_t<float, 32>(a, s);
      case 64: return launch_backward_t<float, 64>(a, s);
      case 128: return launch_backward_t<float, 128>(a, s);
    }
  } else {
    switch (D) {
      case 16: return launch_backward_t<__nv_bfloat16, 16>(a, s);
      case 32: return launch_backward_t<__nv_bfloat16, 32>(a, s);
      case 64: return launch_backward_t<__nv_bfloat16, 64>(a, s);
      case 128: return launch_backward_t<__nv_bfloat16, 128>(a, s);
    }
  }
  return cudaErrorInvalidValue;
}

}  // namespace prism
