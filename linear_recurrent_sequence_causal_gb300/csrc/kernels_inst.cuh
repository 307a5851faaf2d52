// Instantiation helpers: each translation unit that includes this header and
// defines PRISM_INST_DTYPE (0 = fp32, 1 = bf16) compiles the kernels of that
// type for every supported head dim and chunk length.  Splitting by type lets
// the build compile the two halves in parallel.
#pragma once

#include "kernels.h"

namespace prism {

template <class T, int D>
cudaError_t launch_k1_t(const K1Args& a, cudaStream_t s) {
  using S = K1Smem<T, D>;
  auto fn = anchor_refine_kernel<T, D>;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)S::bytes);
  if (e != cudaSuccess) return e;
  dim3 grid((a.T + S::TT - 1) / S::TT, a.H, a.B);
  fn<<<grid, kThreads, S::bytes, s>>>(a);
  return cudaGetLastError();
}

template <class T, int D, int C>
cudaError_t launch_k2_t(const K2Args& a, cudaStream_t s) {
  using S = K2Smem<T, D, C>;
  auto fn = chunk_scan_kernel<T, D, C>;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)S::bytes);
  if (e != cudaSuccess) return e;
  fn<<<a.B * a.H, kThreads, S::bytes, s>>>(a);
  return cudaGetLastError();
}

template <class T>
size_t k1_bytes_t(int D) {
  switch (D) {
    case 16: return K1Smem<T, 16>::bytes;
    case 32: return K1Smem<T, 32>::bytes;
    case 64: return K1Smem<T, 64>::bytes;
    case 128: return K1Smem<T, 128>::bytes;
  }
  return 0;
}

template <class T, int D>
size_t k2_bytes_td(int C) {
  switch (C) {
    case 16: return K2Smem<T, D, 16>::bytes;
    case 32: return K2Smem<T, D, 32>::bytes;
    case 64: return K2Smem<T, D, 64>::bytes;
  }
  return 0;
}

template <class T>
size_t k2_bytes_t(int D, int C) {
  switch (D) {
    case 16: return k2_bytes_td<T, 16>(C);
    case 32: return k2_bytes_td<T, 32>(C);
    case 64: return k2_bytes_td<T, 64>(C);
    case 128: return k2_bytes_td<T, 128>(C);
  }
  return 0;
}

}  // namespace prism
