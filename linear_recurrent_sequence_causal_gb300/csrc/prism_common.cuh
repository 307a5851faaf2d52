// Shared device helpers for the PRISM kernels: element types, the warp-level fp32
// tile product of the fp32 I/O path, and small numeric helpers.
//
// The tile product computes a warp's share of C[M x N] += A[M x K] * B[K x N] in
// 16 x 16 output tiles (thread (g = lane/4, c = lane%4) owns rows g, g+8 and columns
// 2c, 2c+1 of each 16 x 8 half) with exact fp32 FMA products, for the fp32 workloads
// whose tolerance 16-bit operands cannot meet.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>


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

// Bounds checks of the debug build (compiled with PRISM_DEBUG_BOUNDS): an access whose
// index falls outside its array is skipped and bit 2 of the word `bounds` records it
// (prism_debug_bounds reads the word).  In the normal build every check is the constant
// true, the word is never touched and the code is the same as without the checks.
#ifdef PRISM_DEBUG_BOUNDS
__device__ __forceinline__ bool in_bounds(bool ok, int* word) {
  if (!ok && word) atomicOr(word, 2);
  return ok;
}
#define PRISM_IN_BOUNDS(cond, word) ::prism::in_bounds((cond), (word))
#else
#define PRISM_IN_BOUNDS(cond, word) true
#endif
// [p, p + bytes) inside [base, base + extent)
__device__ __forceinline__ bool within(const void* p, size_t bytes, const void* base, size_t extent) {
  const char* a = static_cast<const char*>(p);
  const char* o = static_cast<const char*>(base);
  return a >= o && a + bytes <= o + extent;
}

// checked store / load: the access happens only when [ptr, ptr + sizeof(T)) lies inside
// [base, base + extent) (always, in the normal build)
template <class T>
__device__ __forceinline__ void put(T* ptr, const T& v, const void* base, size_t extent, int* word) {
  if (PRISM_IN_BOUNDS(within(ptr, sizeof(T), base, extent), word)) *ptr = v;
}
template <class T>
__device__ __forceinline__ T get(const T* ptr, const void* base, size_t extent, int* word) {
  return PRISM_IN_BOUNDS(within(ptr, sizeof(T), base, extent), word) ? *ptr : T();
}
// bytes of dynamic shared memory this launch has
__device__ __forceinline__ uint32_t dyn_smem_bytes() {
  uint32_t n;
  asm volatile("mov.u32 %0, %%dynamic_smem_size;\n" : "=r"(n));
  return n;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
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
// Offsets m0, n0 are multiples of 16.
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

__device__ __forceinline__ float rcp_approx(float z) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(z));
  return r;
}
// x Phi(x) with erf from Hastings' rational approximation (Abramowitz and Stegun,
// "Handbook of Mathematical Functions", 7.1.26: |error of erf(y)| <= 1.5e-7 for y >= 0, and
// erf is odd): with y = |x| / sqrt(2), t = 1 / (1 + 0.3275911 y) and
// h = (1 - erf(y)) / 2 = t (a1 + t (a2 + t (a3 + t (a4 + t a5)))) exp(-y^2) / 2,
// Phi(x) = 1 - h for x >= 0 and h for x < 0.  Within about 4e-7 max(|x|, 1) of the exact
// GELU with the approximate reciprocal and exponential (the erff form is within about the
// same of it in fp32); fewer instructions than erff, which matters in the tensor-core
// prepare kernel's refinement loop.
__device__ __forceinline__ float gelu_hastings(float x) {
  const float y = fabsf(x) * 0.70710678118654752f;
  const float t = rcp_approx(fmaf(0.3275911f, y, 1.0f));
  const float poly =
      t * fmaf(t, fmaf(t, fmaf(t, fmaf(t, 1.061405429f, -1.453152027f), 1.421413741f), -0.284496736f), 0.254829592f);
  const float h = 0.5f * poly * __expf(-y * y);
  return x * (x >= 0.f ? 1.0f - h : h);
}
__device__ __forceinline__ float sigmoidf(float x) { return 1.0f / (1.0f + expf(-x)); }

}  // namespace prism
