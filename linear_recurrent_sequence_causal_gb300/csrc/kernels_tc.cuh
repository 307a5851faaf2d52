// Launch helpers for the bf16 I/O path (prep kernel on tcgen05, scan kernel).
#pragma once

#include <cuda_runtime.h>

#include "prep_tc.cuh"
#include "scan_affine.cuh"
#include "scan_tc.cuh"

namespace prism {

template <int D, int C>
cudaError_t launch_prep_t(const PrepArgs& a, cudaStream_t s) {
  using S = PrepSmem<D, C>;
  auto fn = prep_tc_kernel<D, C>;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)S::bytes);
  if (e != cudaSuccess) return e;
  dim3 grid((a.T + C - 1) / C, a.H, a.B);
  fn<<<grid, S::NTA, S::bytes, s>>>(a);
  return cudaGetLastError();
}

template <int D, int C, int BV>
cudaError_t launch_scan_t(const ScanArgs& a, cudaStream_t s) {
  using S = ScanSmem<D, C, BV>;
  auto fn = scan_affine_kernel<D, C, BV>;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)S::bytes);
  if (e != cudaSuccess) return e;
  fn<<<a.B * a.H * (D / BV), S::NW * 32, S::bytes, s>>>(a);
  return cudaGetLastError();
}

template <int C>
cudaError_t launch_scan_tc_t(const ScanTcArgs& a, cudaStream_t s) {
  using S = ScanTcSmem<C>;
  auto fn = scan_tc_kernel<C>;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)S::bytes);
  if (e != cudaSuccess) return e;
  fn<<<a.B * a.H * (S::D / S::BV), S::NT, S::bytes, s>>>(a);
  return cudaGetLastError();
}

}  // namespace prism
