// Kernel K1: ShortConv anchor + L-step refinement ("Technical Summary: PRISM",
// §2.2 stages 1 and 2).  Fully parallel over tokens: one CTA takes TT tokens
// of one (b, h) sequence.
//
// Per token t (row i of the tile):
//   u = sum_{j=1..w} c_j (.) v_{t-j}           (zero before t = 0)
//   r = v_t - u
//   for l: [khat | p] = u [W_k^(l)^T | W_p^(l)^T]     (one tile product)
//          k^(l) = khat / sqrt(|khat|^2 + 1e-6)
//          delta = GELU(p (.) r);  r -= delta
//          D^(l) = sigmoid(w_beta^(l) . u) * delta
// Outputs Kl[b,t,h,l,:] = k^(l) and Dl[b,t,h,l,:] = D^(l) in the I/O type;
// zeros at padded tokens (len_b <= t < T).
#pragma once

#include "prism_common.cuh"

namespace prism {

template <class T, int D>
struct K1Smem {
  static constexpr int TT = 64;                         // tokens per CTA
  static constexpr int WMAX = 8;                        // max conv width
  static constexpr int LDT = D + Elem<T>::kPad;         // row stride of T tiles
  static constexpr int LDX = 2 * D + 4;                 // fp32 product dump
  // Offsets in bytes.
  static constexpr size_t oU = 0;                                        // T [TT][LDT]
  static constexpr size_t oW = oU + sizeof(T) * TT * LDT;                // T [2D][LDT]
  static constexpr size_t oR = oW + sizeof(T) * 2 * D * LDT;             // f32 [TT][D]
  static constexpr size_t oX = oR + sizeof(float) * TT * D;              // f32 [TT][LDX]
  static constexpr size_t oVw = oX;                                      // f32 [TT+WMAX][D] (aliases X)
  static constexpr size_t oBeta = oX + sizeof(float) *
      ((TT * LDX) > ((TT + WMAX) * D) ? (TT * LDX) : ((TT + WMAX) * D));   // f32 [TT][8]
  static constexpr size_t oInv = oBeta + sizeof(float) * TT * 8;         // f32 [TT]
  static constexpr size_t bytes = oInv + sizeof(float) * TT;
};

struct K1Args {
  int B, T, H, w, L;
  unsigned flags;
  const void* v;
  const float* conv_w;
  const float* Wk;
  const float* Wp;
  const float* wbeta;
  const int* seq_lens;
  const void* vhist;     // [B][H][w][D] v of the w tokens before t = 0 (oldest first), or null
  void* Kl;
  void* Dl;
};

template <class T, int D>
__global__ void __launch_bounds__(kThreads, 1) anchor_refine_kernel(K1Args p) {
  using S = K1Smem<T, D>;
  constexpr int TT = S::TT, LDT = S::LDT, LDX = S::LDX;
  extern __shared__ __align__(128) unsigned char smem[];
  T* sU = reinterpret_cast<T*>(smem + S::oU);
  T* sW = reinterpret_cast<T*>(smem + S::oW);
  float* sR = reinterpret_cast<float*>(smem + S::oR);
  float* sX = reinterpret_cast<float*>(smem + S::oX);
  float* sVw = reinterpret_cast<float*>(smem + S::oVw);
  float* sBeta = reinterpret_cast<float*>(smem + S::oBeta);
  float* sInv = reinterpret_cast<float*>(smem + S::oInv);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int t0 = blockIdx.x * TT;
  const int h = blockIdx.y, b = blockIdx.z;
  const int H = p.H, T_ = p.T, w = p.w, L = p.L;
  const int len = p.seq_lens ? min(max(p.seq_lens[b], 0), T_) : T_;
  const T* v = static_cast<const T*>(p.v);

  // 1. v window: rows t0-w .. t0+TT-1 -> sVw[(i + w)][c] for token t0 + i.
  //    Tokens outside [0, len) read as 0 (padding is selected away, never used); tokens
  //    before t = 0 come from the history when one is given.
  for (int idx = tid; idx < (TT + w) * D; idx += kThreads) {
    const int rr = idx / D, c = idx % D;
    const int t = t0 - w + rr;
    float x = 0.f;
    if (t >= 0 && t < len) x = Elem<T>::to_f(v[(((size_t)b * T_ + t) * H + h) * D + c]);
    else if (t < 0 && p.vhist)                 // [B][H][w][D], or [B][w][H][D] (token-major flag)
      x = Elem<T>::to_f(static_cast<const T*>(p.vhist)[(p.flags & 2u) ? (((size_t)b * w + (w + t)) * H + h) * D + c
                                                                     : (((size_t)b * H + h) * w + (w + t)) * D + c]);
    sVw[rr * D + c] = x;
  }
  __syncthreads();

  // 2. anchor u (fp32 in sR for now, tile type in sU).
  for (int idx = tid; idx < TT * D; idx += kThreads) {
    const int i = idx / D, c = idx % D;
    float u = 0.f;
    for (int j = 1; j <= w; ++j)
      u = fmaf(p.conv_w[((size_t)h * w + (j - 1)) * D + c], sVw[(i + w - j) * D + c], u);
    sU[i * LDT + c] = Elem<T>::from_f(u);
    sR[i * D + c] = u;
  }
  __syncthreads();
  // confidence gates beta^(l) = sigmoid(w_beta^(l) . u) from the fp32 anchor.
  for (int il = warp; il < TT * L; il += kWarps) {
    const int i = il / L, l = il % L;
    const float* wb = p.wbeta + ((size_t)h * L + l) * D;
    float z = 0.f;
    for (int c = lane; c < D; c += 32) z = fmaf(wb[c], sR[i * D + c], z);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
    if (lane == 0) sBeta[i * 8 + l] = sigmoidf(z);
  }
  __syncthreads();
  // first residual r^(1) = v - u.
  for (int idx = tid; idx < TT * D; idx += kThreads) {
    const int i = idx / D, c = idx % D;
    sR[i * D + c] = sVw[(i + w) * D + c] - sR[i * D + c];
  }
  __syncthreads();

  using Map = TileMap<TT, 2 * D>;
  T* Kl = static_cast<T*>(p.Kl);
  T* Dl = static_cast<T*>(p.Dl);
  const bool gelu = !(p.flags & 1u);
  for (int l = 0; l < L; ++l) {
    // 3. stage [W_k^(l) ; W_p^(l)] (2D rows of length D) in the tile type.
    const float* wk = p.Wk + ((size_t)h * L + l) * D * D;
    const float* wp = p.Wp + ((size_t)h * L + l) * D * D;
    for (int idx = tid; idx < 2 * D * D; idx += kThreads) {
      const int n = idx / D, c = idx % D;
      const float x = n < D ? wk[(size_t)n * D + c] : wp[(size_t)(n - D) * D + c];
      sW[n * LDT + c] = Elem<T>::from_f(x);
    }
    __syncthreads();
    // 4. X = U W^T  (TT x 2D, K = D); B(k, n) = W[n][k] -> stored N x K.
#pragma unroll
    for (int i = 0; i < Map::kPerWarp; ++i) {
      if (!Map::valid(i)) continue;
      Acc16 acc;
      acc.zero();
      const int m0 = Map::m0(i), n0 = Map::n0(i);
      tile_mma<false, true>(acc, sU, LDT, sW, LDT, m0, n0, D);
#pragma unroll
      for (int hh = 0; hh < 2; ++hh)
#pragma unroll
        for (int e = 0; e < 4; ++e) sX[(m0 + acc_row(e)) * LDX + n0 + acc_col(hh, e)] = acc.v[hh][e];
    }
    __syncthreads();
    // 5. direction norms.
    for (int i = warp; i < TT; i += kWarps) {
      float s = 0.f;
      for (int a = lane; a < D; a += 32) { const float x = sX[i * LDX + a]; s = fmaf(x, x, s); }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
      if (lane == 0) sInv[i] = 1.0f / sqrtf(s + 1e-6f);
    }
    __syncthreads();
    // 6. residual step and outputs (one warp per token row, lanes over columns).
    for (int i = warp; i < TT; i += kWarps) {
      const int t = t0 + i;
      if (t >= T_) continue;
      const bool valid = t < len;
      const size_t base = ((((size_t)b * T_ + t) * H + h) * L + l) * D;
      const float inv = sInv[i], bl = sBeta[i * 8 + l];
      for (int a = lane; a < D; a += 32) {
        const float kd = valid ? sX[i * LDX + a] * inv : 0.f;
        Kl[base + a] = Elem<T>::from_f(kd);
        const float x = sX[i * LDX + D + a] * sR[i * D + a];
        const float dl = gelu ? gelu_erf(x) : x;
        sR[i * D + a] -= dl;
        Dl[base + a] = Elem<T>::from_f(valid ? bl * dl : 0.f);
      }
    }
    __syncthreads();
  }
}

}  // namespace prism
