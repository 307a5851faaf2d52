// Launch helpers for the bf16 I/O path (prep kernel on tcgen05, scan kernel).
#pragma once

#include <cuda_runtime.h>

#include "prep_tc.cuh"
#include "scan_tc.cuh"

namespace prism {

template <int D, int C>
cudaError_t launch_prep_t(const PrepArgs& a, cudaStream_t s) {
  using S = PrepSmem<D, C>;
  auto fn = prep_tc_kernel<D, C>;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)S::bytes);
  if (e != cudaSuccess) return e;
  // Persistent CTAs walk the chunks (the next chunk's tiles come in during a tail): as many
  // as are resident at once (one or two per SM), never more than there are chunks.  With
  // per-sequence lengths the chunks past a sequence's end are skipped, which a fixed
  // stride shares out unevenly: there each chunk gets its own CTA and the hardware
  // scheduler balances them.
  const long long chunks = (long long)a.B * a.H * ((a.T + C - 1) / C);
  long long grid = chunks;
  if (S::kPrefetch && !a.seq_lens) {
    int dev = 0, sms = 0;
    static int per_sm = 0;                     // CTAs resident per SM (asked once per process)
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if (per_sm == 0) {
      int n = 0;
      if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, S::NTA, S::bytes)) != cudaSuccess) return e;
      per_sm = n;
    }
    const long long resident = (long long)sms * (per_sm > 0 ? per_sm : 1);
    if (grid > resident) grid = resident;
  }
  fn<<<(unsigned)grid, S::NTA, S::bytes, s>>>(a);
  return cudaGetLastError();
}

// The scan: one chain per sequence (a.nseg <= 1), or the sequence split in three
// launches (affine maps, entering states, final pass; see scan_tc.cuh).
template <int D, int C>
cudaError_t launch_scan_tc_t(const ScanTcArgs& a, cudaStream_t s) {
  using S = ScanTcSmem<D, C>;
  auto fn = scan_tc_kernel<D, C>;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)S::bytes);
  if (e != cudaSuccess) return e;
  const int NSL = S::D / S::BV, BH = a.B * a.H;
  if (a.nseg <= 1) {
    ScanTcArgs p0 = a;
    p0.phase = 0;
    fn<<<BH * NSL, S::NT, S::bytes, s>>>(p0);
    return cudaGetLastError();
  }
  ScanTcArgs p1 = a;
  p1.phase = 1;
  fn<<<BH * NSL * (1 + 2 * (a.nseg - 1)), S::NT, S::bytes, s>>>(p1);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (a.nseg > 2) {
    auto fc = scan_seg_chain_kernel<S::D>;
    e = cudaFuncSetAttribute(fc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SegChainSmem<S::D>::bytes);
    if (e != cudaSuccess) return e;
    fc<<<BH * (S::D / kSegRows), 256, SegChainSmem<S::D>::bytes, s>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  ScanTcArgs p3 = a;
  p3.phase = 3;
  fn<<<BH * NSL * (a.nseg - 1), S::NT, S::bytes, s>>>(p3);
  return cudaGetLastError();
}

}  // namespace prism
