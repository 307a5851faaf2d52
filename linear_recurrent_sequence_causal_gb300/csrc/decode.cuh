// Single-token step of the PRISM mixer ("Technical Summary: PRISM", §2.1 and §2.2,
// read token by token): for each (b, h), from the carried state S (d_v x d_k, fp32)
// and the v rows of the w previous tokens,
//   u = sum_j c_j (.) v_{t-j},  r = v_t - u,
//   for l: k^(l) = normalize(W_k^(l) u), p^(l) = W_p^(l) u, beta^(l) = sigmoid(w_beta^(l) . u),
//          delta^(l) = GELU(p^(l) (.) r), r -= delta^(l)
//   S <- alpha (S - beta (S k) k^T) + beta v k^T + sum_l beta^(l) delta^(l) k^(l)^T,   o = S q,
// then the history moves by one token.  Everything is fp32 (one token is small:
// matrix-vector products on the CUDA cores), one CTA per (b, h).
#pragma once

#include "prism_common.cuh"

namespace prism {

struct DecodeArgs {
  int B, H, w, L;
  unsigned flags;
  const void* q;            // [B][H][D] one token (I/O dtype)
  const void* k;
  const void* v;
  const float* log_alpha;   // [B][H]
  const float* beta;        // [B][H]
  const float* conv_w;      // [H][w][D]
  const float* Wk;          // [H][L][D][D]
  const float* Wp;          // [H][L][D][D]
  const float* wbeta;       // [H][L][D]
  float* state;             // [B][H][D][D] in/out
  void* vhist;              // [B][H][w][D] in/out (I/O dtype), oldest first
  float* out;               // [B][H][D]
};

constexpr int kDecodeThreads = 256, kDecodeLmax = 8;

template <int D>
struct DecodeSmem {
  static constexpr int LDS = D + 1;                       // padded state rows
  static constexpr size_t oS = 0;                         // f32 [D][LDS]
  static constexpr size_t oVec = oS + sizeof(float) * D * LDS;   // v, k, q, u, r, p, Sk: 7 x D
  static constexpr size_t oKl = oVec + sizeof(float) * 7 * D;    // [Lmax][D] directions
  static constexpr size_t oDl = oKl + sizeof(float) * kDecodeLmax * D;   // [Lmax][D] beta^(l) delta^(l)
  static constexpr size_t oRed = oDl + sizeof(float) * kDecodeLmax * D;  // block-reduction scratch
  static constexpr size_t bytes = oRed + sizeof(float) * 64;
};

// Sum over the CTA of one value per thread (all threads call it).
__device__ __forceinline__ float block_sum(float x, float* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  __syncthreads();
  if (lane == 0) red[warp] = x;
  __syncthreads();
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < kDecodeThreads / 32; ++i) s += red[i];
  return s;
}

// y[a] = sum_c M[a][c] x[c] for a < D (M row-major D x D in global memory), one warp per
// row, lanes along the row (coalesced).
template <int D>
__device__ __forceinline__ void matvec_rows(const float* M, const float* x, float* y) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int a = warp; a < D; a += kDecodeThreads / 32) {
    float s = 0.f;
    for (int c = lane; c < D; c += 32) s = fmaf(M[(size_t)a * D + c], x[c], s);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (lane == 0) y[a] = s;
  }
}

template <class T, int D>
__global__ void __launch_bounds__(kDecodeThreads) decode_kernel(DecodeArgs p) {
  using S = DecodeSmem<D>;
  constexpr int LDS = S::LDS;
  extern __shared__ __align__(128) unsigned char smem[];
  float* sS = reinterpret_cast<float*>(smem + S::oS);
  float* sv = reinterpret_cast<float*>(smem + S::oVec);
  float* sk = sv + D;
  float* sq = sk + D;
  float* su = sq + D;
  float* sr = su + D;
  float* sp = sr + D;
  float* sSk = sp + D;
  float* skl = reinterpret_cast<float*>(smem + S::oKl);
  float* sdl = reinterpret_cast<float*>(smem + S::oDl);
  float* red = reinterpret_cast<float*>(smem + S::oRed);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int bh = blockIdx.x, h = bh % p.H;
  const int w = p.w, L = p.L;
  const T* q = static_cast<const T*>(p.q) + (size_t)bh * D;
  const T* k = static_cast<const T*>(p.k) + (size_t)bh * D;
  const T* v = static_cast<const T*>(p.v) + (size_t)bh * D;
  T* hist = static_cast<T*>(p.vhist) + (size_t)bh * w * D;
  float* st = p.state + (size_t)bh * D * D;
  const float alpha = expf(p.log_alpha[bh]), beta = p.beta[bh];

  for (int idx = tid; idx < D * D; idx += kDecodeThreads) sS[(idx / D) * LDS + idx % D] = st[idx];
  for (int c = tid; c < D; c += kDecodeThreads) {
    sv[c] = Elem<T>::to_f(v[c]);
    sk[c] = Elem<T>::to_f(k[c]);
    sq[c] = Elem<T>::to_f(q[c]);
    float u = 0.f;                                   // anchor from the history rows
    for (int j = 1; j <= w; ++j)
      u = fmaf(p.conv_w[((size_t)h * w + (j - 1)) * D + c], Elem<T>::to_f(hist[(size_t)(w - j) * D + c]), u);
    su[c] = u;
    sr[c] = sv[c] - u;
  }
  __syncthreads();

  const bool gelu = !(p.flags & 1u);
  for (int l = 0; l < L; ++l) {
    float* kl = skl + l * D;
    matvec_rows<D>(p.Wk + ((size_t)h * L + l) * D * D, su, kl);
    matvec_rows<D>(p.Wp + ((size_t)h * L + l) * D * D, su, sp);
    __syncthreads();
    float n2 = 0.f, z = 0.f;
    for (int c = tid; c < D; c += kDecodeThreads) {
      n2 = fmaf(kl[c], kl[c], n2);
      z = fmaf(p.wbeta[((size_t)h * L + l) * D + c], su[c], z);
    }
    const float inv = 1.0f / sqrtf(block_sum(n2, red) + 1e-6f);
    const float bl = sigmoidf(block_sum(z, red));
    for (int c = tid; c < D; c += kDecodeThreads) {
      kl[c] *= inv;
      const float x = sp[c] * sr[c];
      const float dl = gelu ? gelu_erf(x) : x;
      sr[c] -= dl;
      sdl[l * D + c] = bl * dl;
    }
    __syncthreads();
  }

  // S k, then S <- alpha (S - beta (S k) k^T) + beta v k^T + sum_l D^(l) k^(l)^T, then o = S q
  for (int i = warp; i < D; i += kDecodeThreads / 32) {
    float s = 0.f;
    for (int j = lane; j < D; j += 32) s = fmaf(sS[i * LDS + j], sk[j], s);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (lane == 0) sSk[i] = s;
  }
  __syncthreads();
  for (int idx = tid; idx < D * D; idx += kDecodeThreads) {
    const int i = idx / D, j = idx % D;
    float x = alpha * (sS[i * LDS + j] - beta * sSk[i] * sk[j]) + beta * sv[i] * sk[j];
    for (int l = 0; l < L; ++l) x = fmaf(sdl[l * D + i], skl[l * D + j], x);
    sS[i * LDS + j] = x;
    st[idx] = x;
  }
  __syncthreads();
  for (int i = warp; i < D; i += kDecodeThreads / 32) {
    float s = 0.f;
    for (int j = lane; j < D; j += 32) s = fmaf(sS[i * LDS + j], sq[j], s);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (lane == 0) p.out[(size_t)bh * D + i] = s;
  }
  // history: drop the oldest row, append v_t (all reads before any write)
  T keep[(kDecodeLmax * 128 + kDecodeThreads - 1) / kDecodeThreads];
  int n = 0;
  for (int idx = tid; idx < (w - 1) * D; idx += kDecodeThreads) keep[n++] = hist[idx + D];
  __syncthreads();
  n = 0;
  for (int idx = tid; idx < (w - 1) * D; idx += kDecodeThreads) hist[idx] = keep[n++];
  for (int c = tid; c < D; c += kDecodeThreads) hist[(size_t)(w - 1) * D + c] = v[c];
}

}  // namespace prism
