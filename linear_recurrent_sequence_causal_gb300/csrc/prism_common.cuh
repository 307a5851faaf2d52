// Shared device helpers for the PRISM kernels: element types, the warp-level
// tile product used by both kernels, and small numeric helpers.
//
// The tile product computes a warp's share of C[M x N] += A[M x K] * B[K x N]
// in 16 x 16 output tiles held in the register layout of the m16n8k16 MMA
// (thread (g = lane/4, c = lane%4) owns rows g, g+8 and columns 2c, 2c+1 of
// each 16 x 8 half).  bf16 operands go through ldmatrix + mma.sync; fp32
// operands use the same register layout with FMA (exact fp32 products, for
// the fp32 I/O workloads whose tolerance bf16 cannot meet).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include <type_traits>

namespace prism {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;

template <class T> struct Elem;
template <> struct Elem<float> {
  static __device__ __forceinline__ float to_f(float x) { return x; }
  static __device__ __forceinline__ float from_f(float x) { return x; }
  static constexpr int kPad = 4;       // row padding (elements) of shared tiles
};
template <> struct Elem<__nv_bfloat16> {
  static __device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
  static __device__ __forceinline__ __nv_bfloat16 from_f(float x) { return __float2bfloat16_rn(x); }
  static constexpr int kPad = 8;       // 16 bytes: ldmatrix rows land in distinct banks
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr));
}

__device__ __forceinline__ void mma_f16_16816(float (&d)[4], const uint32_t (&a)[4],
                                              uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4],
                                               uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Accumulator of one 16 x 16 output tile: acc[h][e], h = which 8-column half,
// e = 0..3 -> (row g + 8*(e/2), col 8h + 2c + (e%2)).
struct Acc16 {
  float v[2][4];
  __device__ __forceinline__ void zero() {
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int e = 0; e < 4; ++e) v[h][e] = 0.f;
  }
};

__device__ __forceinline__ int acc_row(int e) { return ((threadIdx.x & 31) >> 2) + 8 * (e >> 1); }
__device__ __forceinline__ int acc_col(int h, int e) {
  return 8 * h + 2 * (threadIdx.x & 3) + (e & 1);
}

// Operand views.  A is logically M x K, B is logically K x N.
//   A_T == false: A(m,k) = a[m*lda + k]   (row-major)
//   A_T == true : A(m,k) = a[k*lda + m]   (stored transposed)
//   B_NK == true : B(k,n) = b[n*ldb + k]  (stored N x K, "K-major")
//   B_NK == false: B(k,n) = b[k*ldb + n]  (stored K x N, row-major)
// Offsets m0, n0 are multiples of 16; K is a multiple of 16; all row strides
// are multiples of 8 elements and the bases 16-byte aligned.
template <bool A_T, bool B_NK, class H16>
__device__ __forceinline__ void tile_mma16(Acc16& acc, const H16* a, int lda, const H16* b, int ldb,
                                           int m0, int n0, int K) {
  const int lane = threadIdx.x & 31;
  const int j = lane >> 3;      // which 8x8 matrix this lane addresses
  const int r = lane & 7;       // which row of it
  for (int k0 = 0; k0 < K; k0 += 16) {
    uint32_t af[4], bf[4];
    if (!A_T) {
      // matrices: (m+0,k+0) (m+8,k+0) (m+0,k+8) (m+8,k+8)
      const H16* p = a + (size_t)(m0 + r + 8 * (j & 1)) * lda + k0 + 8 * (j >> 1);
      ldsm_x4(smem_u32(p), af);
    } else {
      // stored [k][m]; same four blocks, rows of the stored matrix are k
      const H16* p = a + (size_t)(k0 + r + 8 * (j >> 1)) * lda + m0 + 8 * (j & 1);
      ldsm_x4_t(smem_u32(p), af);
    }
    if (B_NK) {
      // matrices: (n+0,k+0) (n+0,k+8) (n+8,k+0) (n+8,k+8)
      const H16* p = b + (size_t)(n0 + r + 8 * (j >> 1)) * ldb + k0 + 8 * (j & 1);
      ldsm_x4(smem_u32(p), bf);
    } else {
      // stored [k][n]: matrices (k+0,n+0) (k+8,n+0) (k+0,n+8) (k+8,n+8)
      const H16* p = b + (size_t)(k0 + r + 8 * (j & 1)) * ldb + n0 + 8 * (j >> 1);
      ldsm_x4_t(smem_u32(p), bf);
    }
    if constexpr (sizeof(H16) == 2 && std::is_same<H16, __half>::value) {
      mma_f16_16816(acc.v[0], af, bf[0], bf[1]);
      mma_f16_16816(acc.v[1], af, bf[2], bf[3]);
    } else {
      mma_bf16_16816(acc.v[0], af, bf[0], bf[1]);
      mma_bf16_16816(acc.v[1], af, bf[2], bf[3]);
    }
  }
}

// Same product with operands addressed through functors: a(m0_row, k_col) and
// b(...) return the shared address of the 16-byte ldmatrix row the lane loads.
//   AMode 0: A row-major,  address of (row m, cols k..k+7)    -> ldmatrix
//   AMode 1: A transposed, address of (row k, cols m..m+7)    -> ldmatrix.trans
//   BMode 0: B stored N x K, address of (row n, cols k..k+7)  -> ldmatrix
//   BMode 1: B stored K x N, address of (row k, cols n..n+7)  -> ldmatrix.trans
template <int AMode, int BMode, class AF, class BF>
__device__ __forceinline__ void tile_mma_f16(Acc16& acc, AF a, BF b, int m0, int n0, int K) {
  const int lane = threadIdx.x & 31;
  const int j = lane >> 3, r = lane & 7;
  for (int k0 = 0; k0 < K; k0 += 16) {
    uint32_t af[4], bf[4];
    if (AMode == 0) ldsm_x4(a(m0 + r + 8 * (j & 1), k0 + 8 * (j >> 1)), af);
    else            ldsm_x4_t(a(k0 + r + 8 * (j >> 1), m0 + 8 * (j & 1)), af);
    if (BMode == 0) ldsm_x4(b(n0 + r + 8 * (j >> 1), k0 + 8 * (j & 1)), bf);
    else            ldsm_x4_t(b(k0 + r + 8 * (j & 1), n0 + 8 * (j >> 1)), bf);
    mma_f16_16816(acc.v[0], af, bf[0], bf[1]);
    mma_f16_16816(acc.v[1], af, bf[2], bf[3]);
  }
}

template <bool A_T, bool B_NK>
__device__ __forceinline__ void tile_mma(Acc16& acc, const __nv_bfloat16* a, int lda,
                                         const __nv_bfloat16* b, int ldb, int m0, int n0, int K) {
  tile_mma16<A_T, B_NK>(acc, a, lda, b, ldb, m0, n0, K);
}
template <bool A_T, bool B_NK>
__device__ __forceinline__ void tile_mma(Acc16& acc, const __half* a, int lda, const __half* b,
                                         int ldb, int m0, int n0, int K) {
  tile_mma16<A_T, B_NK>(acc, a, lda, b, ldb, m0, n0, K);
}

template <bool A_T, bool B_NK>
__device__ __forceinline__ void tile_mma(Acc16& acc, const float* a, int lda, const float* b,
                                         int ldb, int m0, int n0, int K) {
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  for (int k = 0; k < K; ++k) {
    float a0, a1;
    if (!A_T) { a0 = a[(size_t)(m0 + g) * lda + k]; a1 = a[(size_t)(m0 + g + 8) * lda + k]; }
    else      { a0 = a[(size_t)k * lda + m0 + g];   a1 = a[(size_t)k * lda + m0 + g + 8]; }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int n = n0 + 8 * h + 2 * c;
      float b0, b1;
      if (B_NK) { b0 = b[(size_t)n * ldb + k]; b1 = b[(size_t)(n + 1) * ldb + k]; }
      else      { b0 = b[(size_t)k * ldb + n]; b1 = b[(size_t)k * ldb + n + 1]; }
      acc.v[h][0] = fmaf(a0, b0, acc.v[h][0]);
      acc.v[h][1] = fmaf(a0, b1, acc.v[h][1]);
      acc.v[h][2] = fmaf(a1, b0, acc.v[h][2]);
      acc.v[h][3] = fmaf(a1, b1, acc.v[h][3]);
    }
  }
}

// Tiles of an M x N output, numbered row-major in 16 x 16 units, dealt
// round-robin to the NW warps: warp w owns tiles w, w + NW, ...
template <int M, int N, int NW = kWarps>
struct TileMap {
  static constexpr int kTM = M / 16, kTN = N / 16, kTiles = kTM * kTN;
  static constexpr int kPerWarp = (kTiles + NW - 1) / NW;
  static __device__ __forceinline__ bool valid(int i) {
    return (threadIdx.x >> 5) + i * NW < kTiles;
  }
  static __device__ __forceinline__ int m0(int i) {
    return (((threadIdx.x >> 5) + i * NW) / kTN) * 16;
  }
  static __device__ __forceinline__ int n0(int i) {
    return (((threadIdx.x >> 5) + i * NW) % kTN) * 16;
  }
};

__device__ __forceinline__ float gelu_erf(float x) {
  return 0.5f * x * (1.0f + erff(x * 0.70710678118654752f));
}
__device__ __forceinline__ float sigmoidf(float x) { return 1.0f / (1.0f + expf(-x)); }

}  // namespace prism
