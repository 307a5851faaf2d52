// Single-token step of the PRISM mixer ("Technical Summary: PRISM", §2.1 and §2.2,
// read token by token): for each (b, h), from the carried state S (d_v x d_k, fp32)
// and the v rows of the w previous tokens,
//   u = sum_j c_j (.) v_{t-j},  r = v_t - u,
//   for l: k^(l) = normalize(W_k^(l) u), p^(l) = W_p^(l) u, beta^(l) = sigmoid(w_beta^(l) . u),
//          delta^(l) = GELU(p^(l) (.) r), r -= delta^(l)
//   S <- alpha (S - beta (S k) k^T) + beta v k^T + sum_l beta^(l) delta^(l) k^(l)^T,   o = S q,
// then the history moves by one token.  Everything is fp32 (one token is small:
// matrix-vector products on the CUDA cores), one CTA per (b, h); the 2L weight matrices
// stream through two shared-memory buffers (cp.async, the next one loading while the
// current one is used) and every product reads shared memory.
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
  static constexpr int LDW = D + 4;                       // weight rows (16-byte aligned)
  static constexpr size_t oS = 0;                         // f32 [D][LDS]
  static constexpr size_t oW = (sizeof(float) * D * LDS + 15) / 16 * 16;   // f32 [2][D][LDW]
  static constexpr size_t oVec = oW + sizeof(float) * 2 * D * LDW;         // v, k, q, u, r, p, Sk: 7 x D
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

// y[a] = sum_c M[a][c] x[c] for a < D (M in shared memory, rows `ld` floats apart): a warp
// takes four rows at a time (four independent reductions), lanes along the row.
template <int D>
__device__ __forceinline__ void matvec_smem(const float* M, int ld, const float* x, float* y) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  constexpr int NWp = kDecodeThreads / 32;
  for (int a0 = warp * 4; a0 < D; a0 += NWp * 4) {
    float s[4] = {0.f, 0.f, 0.f, 0.f};
    for (int c = lane; c < D; c += 32) {
      const float xc = x[c];
#pragma unroll
      for (int q = 0; q < 4; ++q) s[q] = fmaf(M[(a0 + q) * ld + c], xc, s[q]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
#pragma unroll
      for (int q = 0; q < 4; ++q) s[q] += __shfl_xor_sync(0xffffffffu, s[q], o);
    if (lane < 4) y[a0 + lane] = lane == 0 ? s[0] : lane == 1 ? s[1] : lane == 2 ? s[2] : s[3];
  }
}

// Weight matrix m (W_k^(l) for m = 2l, W_p^(l) for m = 2l + 1) into buffer m % 2.
template <int D>
__device__ __forceinline__ void decode_load_w(const DecodeArgs& p, int h, int m, float* sW) {
  const int l = m >> 1;
  const float* g = ((m & 1) ? p.Wp : p.Wk) + ((size_t)h * p.L + l) * D * D;
  float* dst = sW + (size_t)(m & 1) * D * DecodeSmem<D>::LDW;
  for (int i = threadIdx.x; i < D * D / 4; i += kDecodeThreads) {
    const int a = (i * 4) / D, c = (i * 4) % D;
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(smem_u32(dst + a * DecodeSmem<D>::LDW + c)),
                 "l"(g + (size_t)i * 4) : "memory");
  }
  asm volatile("cp.async.commit_group;\n" ::: "memory");
}

template <class T, int D>
__global__ void __launch_bounds__(kDecodeThreads) decode_kernel(DecodeArgs p) {
  using S = DecodeSmem<D>;
  constexpr int LDS = S::LDS;
  extern __shared__ __align__(128) unsigned char smem[];
  float* sS = reinterpret_cast<float*>(smem + S::oS);
  float* sW = reinterpret_cast<float*>(smem + S::oW);
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

  if (L > 0) decode_load_w<D>(p, h, 0, sW);          // W_k^(0) streams in meanwhile
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
#pragma unroll
    for (int which = 0; which < 2; ++which) {        // W_k^(l) then W_p^(l)
      const int m = 2 * l + which;
      if (m + 1 < 2 * L) {
        decode_load_w<D>(p, h, m + 1, sW);           // the next matrix into the other buffer
        asm volatile("cp.async.wait_group 1;\n" ::: "memory");
      } else {
        asm volatile("cp.async.wait_group 0;\n" ::: "memory");
      }
      __syncthreads();
      matvec_smem<D>(sW + (size_t)(m & 1) * D * S::LDW, S::LDW, su, which ? sp : kl);
      __syncthreads();                               // buffer m % 2 free for matrix m + 2
    }
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
  matvec_smem<D>(sS, LDS, sk, sSk);
  __syncthreads();
  for (int idx = tid; idx < D * D; idx += kDecodeThreads) {
    const int i = idx / D, j = idx % D;
    float x = alpha * (sS[i * LDS + j] - beta * sSk[i] * sk[j]) + beta * sv[i] * sk[j];
    for (int l = 0; l < L; ++l) x = fmaf(sdl[l * D + i], skl[l * D + j], x);
    sS[i * LDS + j] = x;
    st[idx] = x;
  }
  __syncthreads();
  matvec_smem<D>(sS, LDS, sq, p.out + (size_t)bh * D);
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
