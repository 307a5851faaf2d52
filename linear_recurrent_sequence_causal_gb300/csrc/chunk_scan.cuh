// Kernel K2: chunkwise scan of S_t = S_{t-1} A_t + B_t with readout o_t = S_t q_t
// ("Technical Summary: PRISM", §2.1 Write-Forget Decoupling, and §2.2: the write
// depends on the input only, so the recurrence admits a parallel/chunked scan).
//
// One CTA walks the chunks of one (b, h) sequence in order, holding the state S
// (d_v x d_k, fp32) in registers.  Per chunk of C tokens with entering state S0,
// g = inclusive cumsum of log alpha inside the chunk, gamma = exp(g),
// Gamma_ij = exp(g_i - g_j) (<= 1 for i >= j; never formed for i < j):
//   A   = strict_tril(diag(beta) (K K^T (.) Gamma))
//   T   = (I + A)^-1                                 (fp32 blocked substitution)
//   R   = sum_l strict_tril(K K_l^T (.) Gamma) D_l
//   W   = T diag(beta gamma) K,   X = diag(beta) (V - R)
//   E   = T X - W S0^T                               (delta-rule pseudo-values)
//   O   = diag(gamma) Q S0^T + tril(Q K^T (.) Gamma) E + sum_l tril(Q K_l^T (.) Gamma) D_l
//   S   = gamma_C S0 + E^T diag(gamma_C / gamma) K + sum_l D_l^T diag(gamma_C / gamma) K_l
// where K_l, D_l are the refinement directions k^(l) and write values
// beta^(l) delta^(l) produced by the anchor/refinement kernel.  The Gated
// DeltaNet write beta v k^T enters through E.
//
// Padding (t >= len_b) and the ragged tail are handled by selection: padded
// rows load as zeros with beta = 0 and log alpha = 0, which leaves the state
// untouched, and their outputs are written as zeros.
#pragma once

#include "prism_common.cuh"

namespace prism {

template <class T, int D, int C>
struct K2Smem {
  static constexpr int LDD = D + Elem<T>::kPad;   // row stride of C x D / D x D tiles
  static constexpr int LDC = C + Elem<T>::kPad;   // row stride of C x C tiles
  static constexpr int LDA = C + 1;               // fp32 solve buffers
  static constexpr size_t kRowTile = sizeof(T) * C * LDD;
  static constexpr size_t kSqTile = sizeof(T) * C * LDC;
  static constexpr size_t kSolve = sizeof(float) * C * LDA;
  static constexpr size_t kRegion1 = (2 * kRowTile > 2 * kSolve) ? 2 * kRowTile : 2 * kSolve;
  static constexpr size_t oQ = 0;
  static constexpr size_t oK = oQ + kRowTile;
  static constexpr size_t oV = oK + kRowTile;
  static constexpr size_t oR1 = oV + kRowTile;           // {Kl, Dl} or {A, T} (solve)
  static constexpr size_t oKl = oR1;
  static constexpr size_t oDl = oR1 + kRowTile;
  static constexpr size_t oSA = oR1;
  static constexpr size_t oST = oR1 + kSolve;
  static constexpr size_t oDt = oR1 + ((kRegion1 + 15) / 16) * 16;
  static constexpr size_t oS0 = oDt + kRowTile;
  static constexpr size_t oTb = oS0 + sizeof(T) * D * LDD;
  static constexpr size_t oP = oTb + kSqTile;
  static constexpr size_t oG = oP + kSqTile;
  static constexpr size_t oPl = oG + kSqTile;
  static constexpr size_t oX = oPl + kSqTile;
  static constexpr size_t oKb = oX + kRowTile;
  static constexpr size_t oY = oKb + kRowTile;                      // f32 [C/16-1][16][16]
  static constexpr size_t oGate = oY + sizeof(float) * 256 * (C / 16 > 1 ? C / 16 - 1 : 1);
  static constexpr size_t bytes = oGate + sizeof(float) * 4 * C + 16;
};

struct K2Args {
  int B, T, H, L;
  const void* q;
  const void* k;
  const void* v;
  const float* log_alpha;
  const float* beta;
  const void* Kl;
  const void* Dl;
  const int* seq_lens;
  void* out;
  float* final_state;
  const float* initial_state;   // [B][H][D][D] entering state, or null (zero)
};

// Load rows [0, n_valid) of a C x D tile from global rows spaced `stride`
// elements apart; rows >= n_valid are written as zeros (selected, never read).
template <class T, int D, int C>
__device__ __forceinline__ void load_tile(T* s, int lds, const T* g, size_t stride, int n_valid) {
  constexpr int V = 16 / sizeof(T), VPR = D / V;
  for (int idx = threadIdx.x; idx < C * VPR; idx += kThreads) {
    const int i = idx / VPR, c = (idx % VPR) * V;
    uint4 x = make_uint4(0u, 0u, 0u, 0u);
    if (i < n_valid) x = *reinterpret_cast<const uint4*>(g + (size_t)i * stride + c);
    *reinterpret_cast<uint4*>(s + (size_t)i * lds + c) = x;
  }
}

// Same, also writing a copy scaled per row by f[i].
template <class T, int D, int C>
__device__ __forceinline__ void load_tile_scaled(T* s, T* s2, int lds, const T* g, size_t stride,
                                                 int n_valid, const float* f) {
  constexpr int V = 16 / sizeof(T), VPR = D / V;
  for (int idx = threadIdx.x; idx < C * VPR; idx += kThreads) {
    const int i = idx / VPR, c = (idx % VPR) * V;
    union { uint4 u; T e[V]; } x, y;
    x.u = make_uint4(0u, 0u, 0u, 0u);
    if (i < n_valid) x.u = *reinterpret_cast<const uint4*>(g + (size_t)i * stride + c);
    const float fi = f[i];
#pragma unroll
    for (int e = 0; e < V; ++e) y.e[e] = Elem<T>::from_f(Elem<T>::to_f(x.e[e]) * fi);
    *reinterpret_cast<uint4*>(s + (size_t)i * lds + c) = x.u;
    *reinterpret_cast<uint4*>(s2 + (size_t)i * lds + c) = y.u;
  }
}

// T = (I + A)^-1 for the strictly lower triangular C x C matrix A in sA (fp32),
// by blocked forward substitution with 16 x 16 blocks:
//   T_ii = (I + A_ii)^-1                           (row-by-row, one warp per block)
//   T_ij = -T_ii sum_{k=j}^{i-1} A_ik T_kj,  i > j (block rows in order)
// Result in sT (fp32, full C x C with zeros above the diagonal).
template <int C>
__device__ __forceinline__ void solve_unit_lower(const float* sA, float* sT, float* sY) {
  constexpr int LDA = C + 1, NB = C / 16;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int idx = tid; idx < C * C; idx += kThreads) sT[(idx / C) * LDA + idx % C] = 0.f;
  __syncthreads();
  if (warp < NB && lane < 16) {
    const int o = warp * 16, jj = lane;
    for (int ii = 0; ii < 16; ++ii) {
      float s = (ii == jj) ? 1.f : 0.f;
      if (jj < ii) {
        for (int m = jj; m < ii; ++m) s -= sA[(o + ii) * LDA + o + m] * sT[(o + m) * LDA + o + jj];
      }
      sT[(o + ii) * LDA + o + jj] = s;
      __syncwarp(0x0000ffffu);
    }
  }
  __syncthreads();
  for (int bi = 1; bi < NB; ++bi) {
    // Y_j = sum_{k=j}^{bi-1} A_{bi,k} T_{k,j} for j < bi
    for (int idx = tid; idx < bi * 256; idx += kThreads) {
      const int bj = idx / 256, r = (idx % 256) / 16, c = idx % 16;
      float s = 0.f;
      for (int m = bj * 16; m < bi * 16; ++m) s += sA[(bi * 16 + r) * LDA + m] * sT[m * LDA + bj * 16 + c];
      sY[idx] = s;
    }
    __syncthreads();
    for (int idx = tid; idx < bi * 256; idx += kThreads) {
      const int bj = idx / 256, r = (idx % 256) / 16, c = idx % 16;
      float s = 0.f;
      for (int m = 0; m < 16; ++m) s += sT[(bi * 16 + r) * LDA + bi * 16 + m] * sY[bj * 256 + m * 16 + c];
      sT[(bi * 16 + r) * LDA + bj * 16 + c] = -s;
    }
    __syncthreads();
  }
}

template <class T, int D, int C>
__global__ void __launch_bounds__(kThreads, 1) chunk_scan_kernel(K2Args p) {
  using S = K2Smem<T, D, C>;
  constexpr int LDD = S::LDD, LDC = S::LDC, LDA = S::LDA;
  extern __shared__ __align__(128) unsigned char smem[];
  T* sQ = reinterpret_cast<T*>(smem + S::oQ);
  T* sK = reinterpret_cast<T*>(smem + S::oK);
  T* sV = reinterpret_cast<T*>(smem + S::oV);
  T* sKl = reinterpret_cast<T*>(smem + S::oKl);
  T* sDl = reinterpret_cast<T*>(smem + S::oDl);
  float* sA = reinterpret_cast<float*>(smem + S::oSA);
  float* sT = reinterpret_cast<float*>(smem + S::oST);
  T* sDt = reinterpret_cast<T*>(smem + S::oDt);
  T* sS0 = reinterpret_cast<T*>(smem + S::oS0);
  T* sTb = reinterpret_cast<T*>(smem + S::oTb);
  T* sP = reinterpret_cast<T*>(smem + S::oP);
  T* sG = reinterpret_cast<T*>(smem + S::oG);
  T* sPl = reinterpret_cast<T*>(smem + S::oPl);
  T* sX = reinterpret_cast<T*>(smem + S::oX);
  T* sKb = reinterpret_cast<T*>(smem + S::oKb);
  float* sY = reinterpret_cast<float*>(smem + S::oY);
  float* sg = reinterpret_cast<float*>(smem + S::oGate);   // g_i
  float* sgam = sg + C;                                     // gamma_i
  float* sbeta = sgam + C;                                  // beta_i
  float* sdec = sbeta + C;                                  // gamma_C / gamma_i

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int h = blockIdx.x % p.H, b = blockIdx.x / p.H;
  const int H = p.H, T_ = p.T, L = p.L;
  const int len = p.seq_lens ? min(max(p.seq_lens[b], 0), T_) : T_;
  const size_t row = (size_t)H * D;                  // stride between tokens in q/k/v/out
  const size_t rowl = (size_t)H * L * D;             // stride between tokens in Kl/Dl
  const T* q = static_cast<const T*>(p.q) + ((size_t)b * T_ * H + h) * D;
  const T* k = static_cast<const T*>(p.k) + ((size_t)b * T_ * H + h) * D;
  const T* v = static_cast<const T*>(p.v) + ((size_t)b * T_ * H + h) * D;
  T* out = static_cast<T*>(p.out) + ((size_t)b * T_ * H + h) * D;

  using MapCD = TileMap<C, D>;
  using MapDD = TileMap<D, D>;
  using MapCC = TileMap<C, C>;
  Acc16 accS[MapDD::kPerWarp];
#pragma unroll
  for (int i = 0; i < MapDD::kPerWarp; ++i) accS[i].zero();
  if (p.initial_state) {
    const float* s0 = p.initial_state + ((size_t)b * H + h) * D * D;
#pragma unroll
    for (int i = 0; i < MapDD::kPerWarp; ++i) {
      if (!MapDD::valid(i)) continue;
      const int m0 = MapDD::m0(i), n0 = MapDD::n0(i);
#pragma unroll
      for (int hh = 0; hh < 2; ++hh)
#pragma unroll
        for (int e = 0; e < 4; ++e) accS[i].v[hh][e] = s0[(m0 + acc_row(e)) * D + n0 + acc_col(hh, e)];
    }
  }

  for (int c0 = 0; c0 < len; c0 += C) {
    const int nv = min(C, len - c0);
    // ---- phase 0: chunk inputs, gates, entering state ----
    load_tile<T, D, C>(sQ, LDD, q + (size_t)c0 * row, row, nv);
    load_tile<T, D, C>(sK, LDD, k + (size_t)c0 * row, row, nv);
    load_tile<T, D, C>(sV, LDD, v + (size_t)c0 * row, row, nv);
#pragma unroll
    for (int i = 0; i < MapDD::kPerWarp; ++i) {
      if (!MapDD::valid(i)) continue;
      const int m0 = MapDD::m0(i), n0 = MapDD::n0(i);
#pragma unroll
      for (int hh = 0; hh < 2; ++hh)
#pragma unroll
        for (int e = 0; e < 4; ++e)
          sS0[(m0 + acc_row(e)) * LDD + n0 + acc_col(hh, e)] = Elem<T>::from_f(accS[i].v[hh][e]);
    }
    if (warp == 0) {
      // inclusive scan of log alpha over the chunk (two halves of 32)
      float run = 0.f;
      for (int half = 0; half < C; half += 32) {
        const int i = half + lane;
        const size_t gi = ((size_t)b * T_ + c0 + i) * H + h;
        float la = 0.f, be = 0.f;
        if (i < nv) { la = p.log_alpha[gi]; be = p.beta[gi]; }
        float x = (i < C) ? la : 0.f;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const float y = __shfl_up_sync(0xffffffffu, x, o);
          if (lane >= o) x += y;
        }
        x += run;
        run = __shfl_sync(0xffffffffu, x, 31);
        if (i < C) { sg[i] = x; sbeta[i] = be; }
      }
      __syncwarp();
      const float gC = sg[C - 1];
      for (int i = lane; i < C; i += 32) {
        sgam[i] = expf(sg[i]);
        sdec[i] = expf(gC - sg[i]);
      }
    }
    __syncthreads();
    const float gammaC = sgam[C - 1];
#pragma unroll
    for (int i = 0; i < MapDD::kPerWarp; ++i)
#pragma unroll
      for (int hh = 0; hh < 2; ++hh)
#pragma unroll
        for (int e = 0; e < 4; ++e) accS[i].v[hh][e] *= gammaC;

    // ---- phase 1: A = strict_tril(beta (K K^T)(.)Gamma), P = tril(Q K^T (.) Gamma), O = gamma (.) Q S0^T
#pragma unroll
    for (int mat = 0; mat < 2; ++mat) {
#pragma unroll
      for (int i = 0; i < MapCC::kPerWarp; ++i) {
        if (!MapCC::valid(i)) continue;
        const int m0 = MapCC::m0(i), n0 = MapCC::n0(i);
        if (n0 > m0 + 15) continue;                    // tile entirely above the diagonal
        Acc16 acc;
        acc.zero();
        tile_mma<false, true>(acc, mat == 0 ? sK : sQ, LDD, sK, LDD, m0, n0, D);
#pragma unroll
        for (int hh = 0; hh < 2; ++hh)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int ii = m0 + acc_row(e), jj = n0 + acc_col(hh, e);
            if (mat == 0) {
              sA[ii * LDA + jj] = (ii > jj) ? sbeta[ii] * expf(sg[ii] - sg[jj]) * acc.v[hh][e] : 0.f;
            } else {
              sP[ii * LDC + jj] = Elem<T>::from_f((ii >= jj) ? expf(sg[ii] - sg[jj]) * acc.v[hh][e] : 0.f);
            }
          }
      }
    }
    // zero the tiles skipped above the diagonal
    for (int idx = tid; idx < C * C; idx += kThreads) {
      const int ii = idx / C, jj = idx % C;
      if ((jj / 16) > (ii / 16)) { sA[ii * LDA + jj] = 0.f; sP[ii * LDC + jj] = Elem<T>::from_f(0.f); }
    }
    Acc16 accO[MapCD::kPerWarp];
#pragma unroll
    for (int i = 0; i < MapCD::kPerWarp; ++i) {
      accO[i].zero();
      if (!MapCD::valid(i)) continue;
      const int m0 = MapCD::m0(i), n0 = MapCD::n0(i);
      tile_mma<false, true>(accO[i], sQ, LDD, sS0, LDD, m0, n0, D);
#pragma unroll
      for (int hh = 0; hh < 2; ++hh)
#pragma unroll
        for (int e = 0; e < 4; ++e) accO[i].v[hh][e] *= sgam[m0 + acc_row(e)];
    }
    __syncthreads();

    // ---- phase 2: T = (I + A)^-1 ----
    solve_unit_lower<C>(sA, sT, sY);
    for (int idx = tid; idx < C * C; idx += kThreads) {
      const int ii = idx / C, jj = idx % C;
      sTb[ii * LDC + jj] = Elem<T>::from_f(sT[ii * LDA + jj]);
    }
    __syncthreads();

    // ---- phase 3: rank-L write terms ----
    Acc16 accR[MapCD::kPerWarp];
#pragma unroll
    for (int i = 0; i < MapCD::kPerWarp; ++i) accR[i].zero();
    for (int l = 0; l < L; ++l) {
      const T* kl = static_cast<const T*>(p.Kl) + (((size_t)b * T_ + c0) * H + h) * L * D + (size_t)l * D;
      const T* dl = static_cast<const T*>(p.Dl) + (((size_t)b * T_ + c0) * H + h) * L * D + (size_t)l * D;
      load_tile<T, D, C>(sKl, LDD, kl, rowl, nv);
      load_tile_scaled<T, D, C>(sDl, sDt, LDD, dl, rowl, nv, sdec);
      __syncthreads();
#pragma unroll
      for (int mat = 0; mat < 2; ++mat) {
#pragma unroll
        for (int i = 0; i < MapCC::kPerWarp; ++i) {
          if (!MapCC::valid(i)) continue;
          const int m0 = MapCC::m0(i), n0 = MapCC::n0(i);
          T* dst = mat == 0 ? sG : sPl;
          Acc16 acc;
          acc.zero();
          if (n0 <= m0 + 15) tile_mma<false, true>(acc, mat == 0 ? sK : sQ, LDD, sKl, LDD, m0, n0, D);
#pragma unroll
          for (int hh = 0; hh < 2; ++hh)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int ii = m0 + acc_row(e), jj = n0 + acc_col(hh, e);
              const bool keep = mat == 0 ? (ii > jj) : (ii >= jj);
              dst[ii * LDC + jj] = Elem<T>::from_f(keep ? expf(sg[ii] - sg[jj]) * acc.v[hh][e] : 0.f);
            }
        }
      }
      __syncthreads();
#pragma unroll
      for (int i = 0; i < MapCD::kPerWarp; ++i) {
        if (!MapCD::valid(i)) continue;
        const int m0 = MapCD::m0(i), n0 = MapCD::n0(i);
        tile_mma<false, false>(accR[i], sG, LDC, sDl, LDD, m0, n0, C);
        tile_mma<false, false>(accO[i], sPl, LDC, sDl, LDD, m0, n0, C);
      }
#pragma unroll
      for (int i = 0; i < MapDD::kPerWarp; ++i) {
        if (!MapDD::valid(i)) continue;
        tile_mma<true, false>(accS[i], sDt, LDD, sKl, LDD, MapDD::m0(i), MapDD::n0(i), C);
      }
      __syncthreads();
    }

    // ---- phase 4: X = diag(beta)(V - R), Kb = diag(beta gamma) K, K <- diag(gamma_C/gamma) K
#pragma unroll
    for (int i = 0; i < MapCD::kPerWarp; ++i) {
      if (!MapCD::valid(i)) continue;
      const int m0 = MapCD::m0(i), n0 = MapCD::n0(i);
#pragma unroll
      for (int hh = 0; hh < 2; ++hh)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int ii = m0 + acc_row(e), cc = n0 + acc_col(hh, e);
          const float x = sbeta[ii] * (Elem<T>::to_f(sV[ii * LDD + cc]) - accR[i].v[hh][e]);
          sX[ii * LDD + cc] = Elem<T>::from_f(x);
        }
    }
    for (int idx = tid; idx < C * D; idx += kThreads) {
      const int ii = idx / D, cc = idx % D;
      const float kv = Elem<T>::to_f(sK[ii * LDD + cc]);
      sKb[ii * LDD + cc] = Elem<T>::from_f(sbeta[ii] * sgam[ii] * kv);
      sK[ii * LDD + cc] = Elem<T>::from_f(sdec[ii] * kv);
    }
    __syncthreads();
    // W = T Kb  (kept in registers, stored negated over Kb)
    Acc16 accW[MapCD::kPerWarp];
#pragma unroll
    for (int i = 0; i < MapCD::kPerWarp; ++i) {
      accW[i].zero();
      if (!MapCD::valid(i)) continue;
      tile_mma<false, false>(accW[i], sTb, LDC, sKb, LDD, MapCD::m0(i), MapCD::n0(i), C);
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < MapCD::kPerWarp; ++i) {
      if (!MapCD::valid(i)) continue;
      const int m0 = MapCD::m0(i), n0 = MapCD::n0(i);
#pragma unroll
      for (int hh = 0; hh < 2; ++hh)
#pragma unroll
        for (int e = 0; e < 4; ++e)
          sKb[(m0 + acc_row(e)) * LDD + n0 + acc_col(hh, e)] = Elem<T>::from_f(-accW[i].v[hh][e]);
    }
    __syncthreads();
    // E = T X + (-W) S0^T
#pragma unroll
    for (int i = 0; i < MapCD::kPerWarp; ++i) {
      accW[i].zero();
      if (!MapCD::valid(i)) continue;
      const int m0 = MapCD::m0(i), n0 = MapCD::n0(i);
      tile_mma<false, false>(accW[i], sTb, LDC, sX, LDD, m0, n0, C);
      tile_mma<false, true>(accW[i], sKb, LDD, sS0, LDD, m0, n0, D);
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < MapCD::kPerWarp; ++i) {
      if (!MapCD::valid(i)) continue;
      const int m0 = MapCD::m0(i), n0 = MapCD::n0(i);
#pragma unroll
      for (int hh = 0; hh < 2; ++hh)
#pragma unroll
        for (int e = 0; e < 4; ++e)
          sX[(m0 + acc_row(e)) * LDD + n0 + acc_col(hh, e)] = Elem<T>::from_f(accW[i].v[hh][e]);
    }
    __syncthreads();

    // ---- phase 5: O += P E;  S += E^T diag(gamma_C/gamma) K;  write O ----
#pragma unroll
    for (int i = 0; i < MapCD::kPerWarp; ++i) {
      if (!MapCD::valid(i)) continue;
      const int m0 = MapCD::m0(i), n0 = MapCD::n0(i);
      tile_mma<false, false>(accO[i], sP, LDC, sX, LDD, m0, n0, C);
#pragma unroll
      for (int hh = 0; hh < 2; ++hh)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int ii = m0 + acc_row(2 * e), cc = n0 + acc_col(hh, 2 * e);
          if (ii < nv) {
            T* dst = out + (size_t)(c0 + ii) * row + cc;
            dst[0] = Elem<T>::from_f(accO[i].v[hh][2 * e]);
            dst[1] = Elem<T>::from_f(accO[i].v[hh][2 * e + 1]);
          }
        }
    }
#pragma unroll
    for (int i = 0; i < MapDD::kPerWarp; ++i) {
      if (!MapDD::valid(i)) continue;
      tile_mma<true, false>(accS[i], sX, LDD, sK, LDD, MapDD::m0(i), MapDD::n0(i), C);
    }
    __syncthreads();
  }

  // padded tokens: zero output
  for (size_t idx = tid; idx < (size_t)(T_ - len) * D; idx += kThreads) {
    const int t = len + (int)(idx / D), cc = (int)(idx % D);
    out[(size_t)t * row + cc] = Elem<T>::from_f(0.f);
  }
  if (p.final_state) {
    float* fs = p.final_state + ((size_t)b * H + h) * D * D;
#pragma unroll
    for (int i = 0; i < MapDD::kPerWarp; ++i) {
      if (!MapDD::valid(i)) continue;
      const int m0 = MapDD::m0(i), n0 = MapDD::n0(i);
#pragma unroll
      for (int hh = 0; hh < 2; ++hh)
#pragma unroll
        for (int e = 0; e < 4; ++e) fs[(m0 + acc_row(e)) * D + n0 + acc_col(hh, e)] = accS[i].v[hh][e];
    }
  }
}

}  // namespace prism
