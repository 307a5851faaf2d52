// Host-side declarations of the kernel launchers (one per instantiation).
// Each launcher sets the dynamic shared-memory limit it needs and enqueues its
// kernel on `stream`.  They return the cudaError_t of the launch.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>

#include "anchor_refine.cuh"
#include "chunk_scan.cuh"

namespace prism {

// dtype: 0 = fp32, 1 = bf16
size_t k1_smem_bytes(int dtype, int D);
size_t k2_smem_bytes(int dtype, int D, int C);
cudaError_t launch_k1(int dtype, int D, const K1Args& a, cudaStream_t s);
cudaError_t launch_k2(int dtype, int D, int C, const K2Args& a, cudaStream_t s);

}  // namespace prism
