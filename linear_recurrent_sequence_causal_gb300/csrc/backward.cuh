// Backward pass of the PRISM mixer ("Technical Summary: PRISM", §2.1 and §2.2, read as the
// forward kernels read them): the gradients of a scalar loss with respect to q, k, v,
// log_alpha, beta and the per-head parameters (conv taps, W_k, W_p, w_beta), given the
// loss's gradient with respect to the outputs (and, optionally, the final state).
//
// All arithmetic is fp32 on the CUDA cores; five kernels, in launch order:
//   A  bwd_refine_fwd   per tile of tokens: anchor u, the L refinement steps; keeps u,
//                       k^(l), D^(l) = beta^(l) delta^(l), p^(l), 1/|k_hat^(l)|, z^(l)
//   B  bwd_state        per (b, h): the state S_t forward (checkpoints every kBwdCK tokens),
//                       then backward block by block, recomputing the block's states from
//                       its checkpoint: dS_(t-1) = alpha (dS_t - beta (dS_t k) k^T) with
//                       dS_t += do_t q_t^T, and the per-token gradients of q, k, v (base
//                       write), beta, log_alpha, D^(l) and k^(l)
//   C  bwd_refine       per tile of tokens: the refinement chain backwards (GELU, the
//                       residual, the normalisation, the gate), du_t, dv_t (residual part)
//   D  bwd_weights      dW_k, dW_p (token-sum outer products), dw_beta, dconv_w
//   E  bwd_conv_dv      dv_t += sum_j c_j (.) du_(t+j)  (the anchor's taps, transposed)
#pragma once

#include <algorithm>

#include "prism_common.cuh"

namespace prism {

constexpr int kBwdTT = 32;        // tokens per tile, kernel A
constexpr int kBwdTC = 16;        // tokens per tile, kernel C
constexpr int kBwdCK = 16;        // tokens between state checkpoints, kernel B
constexpr int kBwdLmax = 8;
constexpr int kBwdThreads = 256;

// Rows-of-S slices per (b, h) in the state kernel: enough CTAs to fill the SMs twice over.
inline int bwd_pick_rs(long long BH, int D) {
  if (BH >= 152) return 1;
  if (BH >= 76) return 2;
  return D >= 32 ? 4 : 2;
}

// Token splits of the weight-gradient sums: each split sums its share of the tokens into a
// partial array, and a second kernel adds the partials in split order (deterministic).
inline int bwd_pick_nsw(long long ntok) { return (int)std::min<long long>(32, std::max<long long>(1, ntok / 2048)); }
inline int bwd_pick_nss(long long ntok) { return (int)std::min<long long>(64, std::max<long long>(1, ntok / 512)); }

struct BwdArgs {
  int B, T, H, L, w;
  int rs;                         // rows-of-S slices per (b, h) in the state kernel
  int nsw, nss;                   // token splits of dW_k / dW_p and of dw_beta / dconv
  unsigned flags;                 // bit 0: identity in place of GELU
  const void* q;                  // [B][T][H][D] (I/O dtype)
  const void* k;
  const void* v;
  const float* log_alpha;         // [B][T][H]
  const float* beta;
  const float* conv_w;            // [H][w][D]
  const float* Wk;                // [H][L][D][D]
  const float* Wp;
  const float* wbeta;             // [H][L][D]
  const float* d_out;             // [B][T][H][D]
  const float* d_fs;              // [B][H][D][D] or null
  const int* seq_lens;
  float* dq;                      // [B][T][H][D]
  float* dk;
  float* dv;
  float* dla;                     // [B][T][H]
  float* dbeta;
  float* dconv;                   // [H][w][D]
  float* dWk;                     // [H][L][D][D]
  float* dWp;
  float* dwb;                     // [H][L][D]
  // workspace (token-head n = (b T + t) H + h)
  float* U;                       // [n][D]
  float* KL;                      // [n][L][D]  k^(l)
  float* DL;                      // [n][L][D]  D^(l); then dp^(l) (kernel C)
  float* P;                       // [n][L][D]  p^(l)
  float* NRM;                     // [n][L]     1 / sqrt(|k_hat|^2 + eps)
  float* Z;                       // [n][L]     w_beta^(l) . u
  float* dDL;                     // [n][L][D]
  float* dKL;                     // [n][L][D]
  float* dKH;                     // [n][L][D]  gradient of k_hat^(l)
  float* dZ;                      // [n][L]
  float* dU;                      // [n][D]
  float* CK;                      // [B][H][RS][ceil(T/kBwdCK)][D/RS][D] states before each block
  float* SCR;                     // [B][H][RS][kBwdCK][D/RS][D] states of the block being reversed
  // per-slice partial column sums when the state kernel splits rows over RS CTAs
  float* PQ;                      // [RS][n][D]
  float* PK;                      // [RS][n][D]
  float* PKL;                     // [RS][n][L][D]
  float* PB;                      // [RS][n]
  float* PA;                      // [RS][n]
  float* PW;                      // [nsw][H][2L][D][D] partial dW_k, dW_p (nsw > 1)
  float* PSW;                     // [nss][H][L + w][D] partial dw_beta, dconv (nss > 1)
};

__device__ __forceinline__ int bwd_len(const BwdArgs& p, int b) {
  return p.seq_lens ? min(max(p.seq_lens[b], 0), p.T) : p.T;
}

__device__ __forceinline__ float gelu_grad(float x) {     // d/dx of x Phi(x)
  return 0.5f * (1.0f + erff(x * 0.70710678118654752f)) + x * 0.39894228040143268f * expf(-0.5f * x * x);
}

__device__ __forceinline__ void bwd_cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void bwd_cp_async4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void bwd_cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void bwd_cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory"); }
__device__ __forceinline__ void bwd_cp_async_wait_all() { asm volatile("cp.async.wait_all;\n" ::: "memory"); }

// ------------------------------------------------------------------------------------
// A: refinement forward for kBwdTT tokens of one (b, h)

template <int D>
struct BwdASmem {
  static constexpr size_t oW = 0;                                   // W [2][D][D] (swizzled pieces)
  static constexpr size_t oV = oW + 4u * 2 * D * D;                 // v rows t0-8 .. t0+TT-1
  static constexpr size_t oU = oV + 4u * (kBwdTT + 8) * D;          // u  [TT][D]
  static constexpr size_t oR = oU + 4u * kBwdTT * D;                // r  [TT][D]
  static constexpr size_t oK = oR + 4u * kBwdTT * D;                // k_hat [TT][D]
  static constexpr size_t oP = oK + 4u * kBwdTT * D;                // p [TT][D]
  static constexpr size_t oS = oP + 4u * kBwdTT * D;                // 1/|k_hat| [TT], beta^(l) [TT]
  static constexpr size_t bytes = oS + 4u * 2 * kBwdTT;
};

// W [D][D] (row-major, global) into shared memory asynchronously (one cp.async group):
// row a's 16-byte piece j lands at piece j ^ (a mod D/4) of the row, so threads reading
// one column (consecutive a) or one row (consecutive c) hit different banks.
template <int D>
__device__ __forceinline__ void bwd_load_w_async(float* sW, const float* W) {
  constexpr int NP = D / 4;
  for (int i = threadIdx.x; i < D * NP; i += blockDim.x) {
    const int a = i / NP, j = i % NP;
    bwd_cp_async16(sW + a * D + ((j ^ (a & (NP - 1))) << 2), W + (size_t)i * 4);
  }
  bwd_cp_async_commit();
}
template <int D>
__device__ __forceinline__ float bwd_w(const float* sW, int a, int c) {
  return sW[a * D + (((c >> 2) ^ (a & (D / 4 - 1))) << 2) + (c & 3)];
}

// Y[i][a] = sum_c W[a][c] X[i][a'=c] for the NTOK token rows of X (shared memory, rows
// 16-byte aligned).  Four columns at a time: one 16-byte piece of W's row a and one of
// each token row.
template <int D, int NTOK>
__device__ __forceinline__ void bwd_matvec(const float* sW, const float* X, float* Y) {
  constexpr int NG = kBwdThreads / D, TPG = NTOK / NG;
  const int a = threadIdx.x % D, g = threadIdx.x / D;
  float acc[TPG];
#pragma unroll
  for (int i = 0; i < TPG; ++i) acc[i] = 0.f;
#pragma unroll 1
  for (int c = 0; c < D; c += 4) {
    const float4 wv = *reinterpret_cast<const float4*>(sW + a * D + (((c >> 2) ^ (a & (D / 4 - 1))) << 2));
#pragma unroll
    for (int i = 0; i < TPG; ++i) {
      const float4 xv = *reinterpret_cast<const float4*>(X + (g * TPG + i) * D + c);
      acc[i] = fmaf(wv.x, xv.x, fmaf(wv.y, xv.y, fmaf(wv.z, xv.z, fmaf(wv.w, xv.w, acc[i]))));
    }
  }
#pragma unroll
  for (int i = 0; i < TPG; ++i) Y[(g * TPG + i) * D + a] = acc[i];
}

// Y[i][c] += sum_a W[a][c] X[i][a] (the transposed product), NTOK token rows.
template <int D, int NTOK>
__device__ __forceinline__ void bwd_matvec_t_add(const float* sW, const float* X, float* Y) {
  constexpr int NG = kBwdThreads / D, TPG = NTOK / NG;
  const int c = threadIdx.x % D, g = threadIdx.x / D;
  float acc[TPG];
#pragma unroll
  for (int i = 0; i < TPG; ++i) acc[i] = 0.f;
  for (int a = 0; a < D; ++a) {
    const float wv = bwd_w<D>(sW, a, c);
#pragma unroll
    for (int i = 0; i < TPG; ++i) acc[i] = fmaf(wv, X[(g * TPG + i) * D + a], acc[i]);
  }
#pragma unroll
  for (int i = 0; i < TPG; ++i) Y[(g * TPG + i) * D + c] += acc[i];
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}



template <class T, int D>
__global__ void __launch_bounds__(kBwdThreads) bwd_refine_fwd_kernel(BwdArgs p) {
  using S = BwdASmem<D>;
  extern __shared__ __align__(1024) unsigned char sm[];
  float* sW = reinterpret_cast<float*>(sm + S::oW);
  float* sV = reinterpret_cast<float*>(sm + S::oV);
  float* sU = reinterpret_cast<float*>(sm + S::oU);
  float* sR = reinterpret_cast<float*>(sm + S::oR);
  float* sK = reinterpret_cast<float*>(sm + S::oK);
  float* sP = reinterpret_cast<float*>(sm + S::oP);
  float* sInv = reinterpret_cast<float*>(sm + S::oS);
  float* sBl = sInv + kBwdTT;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int t0 = blockIdx.x * kBwdTT, h = blockIdx.y, b = blockIdx.z;
  const int H = p.H, T_ = p.T, L = p.L, w = p.w;
  const int len = bwd_len(p, b);
  const T* v = static_cast<const T*>(p.v);
  const bool gelu = !(p.flags & 1u);

  // the 2L weight matrices (W_k^(0), W_p^(0), W_k^(1), ...) stream through two buffers
  auto wmat = [&](int m) { return ((m & 1) ? p.Wp : p.Wk) + ((size_t)h * L + (m >> 1)) * D * D; };
  if (L > 0) bwd_load_w_async<D>(sW, wmat(0));
  for (int idx = tid; idx < (kBwdTT + 8) * D; idx += kBwdThreads) {
    const int t = t0 - 8 + idx / D;
    sV[idx] = (t >= 0 && t < len) ? Elem<T>::to_f(v[(((size_t)b * T_ + t) * H + h) * D + idx % D]) : 0.f;
  }
  __syncthreads();
  for (int idx = tid; idx < kBwdTT * D; idx += kBwdThreads) {
    const int i = idx / D, c = idx % D, t = t0 + i;
    float u = 0.f;
    for (int j = 1; j <= w; ++j) u = fmaf(p.conv_w[((size_t)h * w + (j - 1)) * D + c], sV[(i + 8 - j) * D + c], u);
    const bool valid = t < len;
    sU[idx] = valid ? u : 0.f;
    sR[idx] = valid ? sV[(i + 8) * D + c] - u : 0.f;
    if (t < T_) p.U[(((size_t)b * T_ + t) * H + h) * D + c] = valid ? u : 0.f;
  }
  __syncthreads();
  for (int l = 0; l < L; ++l) {
#pragma unroll
    for (int which = 0; which < 2; ++which) {
      const int m = 2 * l + which;
      if (m + 1 < 2 * L) {
        bwd_load_w_async<D>(sW + (size_t)((m + 1) & 1) * D * D, wmat(m + 1));
        bwd_cp_async_wait<1>();
      } else {
        bwd_cp_async_wait<0>();
      }
      __syncthreads();
      bwd_matvec<D, kBwdTT>(sW + (size_t)(m & 1) * D * D, sU, which ? sP : sK);
      __syncthreads();                               // buffer m % 2 free for matrix m + 2
    }
    for (int i = warp; i < kBwdTT; i += kBwdThreads / 32) {   // reads sK, sU (ready)
      float n2 = 0.f, z = 0.f;
      for (int a = lane; a < D; a += 32) {
        const float kk = sK[i * D + a];
        n2 = fmaf(kk, kk, n2);
        z = fmaf(p.wbeta[((size_t)h * L + l) * D + a], sU[i * D + a], z);
      }
      n2 = warp_sum(n2);
      z = warp_sum(z);
      const int t = t0 + i;
      const bool valid = t < len;
      const float inv = 1.0f / sqrtf(n2 + 1e-6f);
      if (lane == 0) {
        sInv[i] = inv;
        sBl[i] = sigmoidf(z);
        if (t < T_) {
          const size_t n = ((size_t)b * T_ + t) * H + h;
          p.NRM[n * L + l] = valid ? inv : 0.f;
          p.Z[n * L + l] = valid ? z : 0.f;
        }
      }
    }
    __syncthreads();
    for (int idx = tid; idx < kBwdTT * D; idx += kBwdThreads) {
      const int i = idx / D, a = idx % D, t = t0 + i;
      if (t >= T_) continue;
      const size_t o = ((((size_t)b * T_ + t) * H + h) * L + l) * D + a;
      if (t < len) {
        const float x = sP[idx] * sR[idx];
        const float dl = gelu ? gelu_erf(x) : x;
        sR[idx] -= dl;
        p.KL[o] = sK[idx] * sInv[i];
        p.DL[o] = sBl[i] * dl;
        p.P[o] = sP[idx];
      } else {
        p.KL[o] = 0.f;
        p.DL[o] = 0.f;
        p.P[o] = 0.f;
      }
    }
    __syncthreads();
  }
}

// ------------------------------------------------------------------------------------
// B: the state, forward with checkpoints and backward block by block (one CTA per (b, h),
// 4 D threads).  Row mapping: thread (r = tid / 4, cq = tid % 4) owns columns cq + 4 i of
// row r; column mapping: thread (c = tid % D, rq = tid / D) owns rows rq D/4 + i of column c.

// RS CTAs share a (b, h): each owns R = D / RS rows of S and dS (rows evolve independently)
// and writes its part of the column sums (dq, dk, dk^(l), dbeta, dlog_alpha) to per-slice
// partial arrays, which bwd_state_reduce adds in slice order (RS = 1 writes them directly).
template <int D, int RS>
struct BwdBSmem {
  static constexpr int R = D / RS;                                  // rows of S in this CTA
  static constexpr int LDS = D + 4;                                 // 16-byte rows, no bank conflicts
  static constexpr int NT = 4 * R, NW = NT / 32;
  static constexpr int NGRP = NT / D;                               // row groups of the column mapping
  static constexpr int RPG = R / NGRP;                              // rows per group (= D / 4)
  static constexpr int TOKF = (4 + 2 * kBwdLmax) * D + 2;           // floats of one token's vectors
  static constexpr size_t oDS = 0;                                  // dS [R][D+4]
  static constexpr size_t oS = oDS + 4u * R * LDS;                  // S  [R][D+4]
  static constexpr size_t oVec = oS + 4u * R * LDS;                 // k | v | do | q | k^(l) | D^(l) | la, beta
  static constexpr size_t oY = oVec + 4u * ((TOKF + 3) / 4 * 4);    // y [R]
  static constexpr size_t oZS = oY + 4u * R;                        // S_(t-1) k_t of the block [CK][R]
  static constexpr size_t oPart = oZS + 4u * kBwdCK * R;            // column partial sums [NGRP][3 + Lmax][D]
  static constexpr size_t oRed = oPart + 4u * NGRP * (3 + kBwdLmax) * D;   // scalar partials [NW][16]
  static constexpr size_t oRing = (oRed + 4u * NW * 16 + 15) / 16 * 16;     // raw token vectors [NSTAGE]
  static constexpr int NSTAGE = 4;                                  // tokens in flight
  // raw bytes of one token's vectors at L steps (k, v, q in the I/O type, do, k^(l), D^(l), gates)
  static __host__ __device__ constexpr size_t tok_bytes(int L, int esz) {
    return (size_t)3 * D * esz + 4u * D + 8u * L * D + 16;
  }
  static __host__ __device__ constexpr size_t bytes(int L, int esz) { return oRing + NSTAGE * tok_bytes(L, esz); }
  static_assert(NT >= D && NT % D == 0 && NT % 32 == 0, "row slice too small");
};


template <int D, int RS>
__device__ __forceinline__ void bwd_state_load_async(float* sS, const float* g) {
  using S = BwdBSmem<D, RS>;
  for (int idx = threadIdx.x; idx < S::R * D / 4; idx += S::NT) {
    const int r = (idx * 4) / D, c = (idx * 4) % D;
    bwd_cp_async16(sS + r * S::LDS + c, g + (size_t)idx * 4);
  }
  bwd_cp_async_commit();
}

template <class T, int D, int RS>
__global__ void __launch_bounds__(4 * (D / RS)) bwd_state_kernel(BwdArgs p) {
  using S = BwdBSmem<D, RS>;
  constexpr int R = S::R, LDS = S::LDS, NT = S::NT, NW = S::NW, CPT = D / 4;
  constexpr int RPG = S::RPG;
  constexpr int NSLOT = 3 + kBwdLmax;
  extern __shared__ __align__(1024) unsigned char sm[];
  float* sDS = reinterpret_cast<float*>(sm + S::oDS);
  float* sS = reinterpret_cast<float*>(sm + S::oS);
  float* svec = reinterpret_cast<float*>(sm + S::oVec);
  float* sy = reinterpret_cast<float*>(sm + S::oY);
  float* sZS = reinterpret_cast<float*>(sm + S::oZS);
  float* sPart = reinterpret_cast<float*>(sm + S::oPart);
  float* sRed = reinterpret_cast<float*>(sm + S::oRed);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int r = tid >> 2, cq = tid & 3;              // row mapping (local row r of the slice)
  const int cc = tid % D, rq = tid / D;              // column mapping (row group rq)
  const int h = blockIdx.x, b = blockIdx.y, slice = blockIdx.z;
  const int r0 = slice * R;                          // first row of S owned here
  const int H = p.H, T_ = p.T, L = p.L;
  const int len = bwd_len(p, b);
  const int NCK = (T_ + kBwdCK - 1) / kBwdCK;
  const size_t NTH = (size_t)p.B * T_ * H;
  const T* qg = static_cast<const T*>(p.q);
  const T* kg = static_cast<const T*>(p.k);
  const T* vg = static_cast<const T*>(p.v);
  float* ck = p.CK + (((size_t)b * H + h) * RS + slice) * NCK * R * D;
  float* scr = p.SCR + (((size_t)b * H + h) * RS + slice) * kBwdCK * R * D;
  // column-sum outputs: the final arrays (RS = 1) or this slice's partial arrays
  float* oq = RS > 1 ? p.PQ + slice * NTH * D : p.dq;
  float* ok_ = RS > 1 ? p.PK + slice * NTH * D : p.dk;
  float* okl = RS > 1 ? p.PKL + slice * NTH * L * D : p.dKL;
  float* ob = RS > 1 ? p.PB + slice * NTH : p.dbeta;
  float* oa = RS > 1 ? p.PA + slice * NTH : p.dla;
  float* sk = svec;
  float* sv = svec + D;
  float* sdo = svec + 2 * D;
  float* sq = svec + 3 * D;
  float* skl = svec + 4 * D;
  float* sdl = skl + L * D;
  const float* sgate = sdl + L * D;                  // log alpha, beta
  auto tok = [&](int t) { return ((size_t)b * T_ + t) * H + h; };

  // padding tokens: every per-token gradient is zero (this slice's rows and partials)
  for (int t = len; t < T_; ++t) {
    const size_t n = tok(t);
    for (int idx = tid; idx < D; idx += NT) {
      oq[n * D + idx] = 0.f;
      ok_[n * D + idx] = 0.f;
    }
    for (int idx = tid; idx < R; idx += NT) p.dv[n * D + r0 + idx] = 0.f;
    for (int idx = tid; idx < L * D; idx += NT) okl[n * L * D + idx] = 0.f;
    for (int idx = tid; idx < L * R; idx += NT) p.dDL[(n * L + idx / R) * D + r0 + idx % R] = 0.f;
    if (tid == 0) {
      oa[n] = 0.f;
      ob[n] = 0.f;
    }
  }
  if (len <= 0) return;

  // A token's vectors stream through a ring of NSTAGE raw buffers (cp.async, one group per
  // token, issued NSTAGE - 1 tokens ahead so the loads' latency overlaps the work) and are
  // converted to fp32 vectors in svec when the token's turn comes.
  constexpr int NSTAGE = S::NSTAGE;
  constexpr int ESZ = sizeof(T);
  const size_t TB = S::tok_bytes(L, ESZ);
  unsigned char* ring = sm + S::oRing;
  const int nk16 = D * ESZ / 16, nf16 = D / 4, nl16 = L * D / 4;   // 16-byte pieces per vector
  auto issue = [&](int t, bool valid) {          // token t into stage t % NSTAGE (empty if !valid)
    if (valid) {
      unsigned char* st = ring + (size_t)(t % NSTAGE) * TB;
      const size_t n = tok(t);
      const int total = 3 * nk16 + nf16 + 2 * nl16;
      for (int i = tid; i < total; i += NT) {
        int j = i;
        const void* src;
        if (j < nk16) src = kg + n * D + j * (16 / ESZ);
        else if ((j -= nk16) < nk16) src = vg + n * D + j * (16 / ESZ);
        else if ((j -= nk16) < nk16) src = qg + n * D + j * (16 / ESZ);
        else if ((j -= nk16) < nf16) src = p.d_out + n * D + j * 4;
        else if ((j -= nf16) < nl16) src = p.KL + n * L * D + j * 4;
        else src = p.DL + n * L * D + (j - nl16) * 4;
        bwd_cp_async16(st + (size_t)i * 16, src);
      }
      if (tid == 0) {
        bwd_cp_async4(st + TB - 16, p.log_alpha + n);
        bwd_cp_async4(st + TB - 12, p.beta + n);
      }
    }
    bwd_cp_async_commit();
  };
  auto convert = [&](int t) {                    // stage of token t -> svec (k | v | do | q | k^(l) | D^(l) | gates)
    const unsigned char* st = ring + (size_t)(t % NSTAGE) * TB;
    const T* rk = reinterpret_cast<const T*>(st);
    const T* rv = rk + D;
    const T* rqq = rv + D;
    const float* rf = reinterpret_cast<const float*>(st + 3 * D * ESZ);   // do | k^(l) | D^(l)
    for (int i = tid; i < D; i += NT) {
      sk[i] = Elem<T>::to_f(rk[i]);
      sv[i] = Elem<T>::to_f(rv[i]);
      sq[i] = Elem<T>::to_f(rqq[i]);
      sdo[i] = rf[i];
    }
    for (int i = tid; i < 2 * L * D; i += NT) skl[i] = rf[D + i];     // k^(l) then D^(l): contiguous
    if (tid < 2) svec[(4 + 2 * L) * D + tid] = reinterpret_cast<const float*>(st + TB - 16)[tid];
  };
  // z_r = S[r] . k (row mapping; every thread of the row gets it)
  auto row_dot_k = [&]() {
    float z0 = 0.f, z1 = 0.f, z2 = 0.f, z3 = 0.f;      // four independent chains
#pragma unroll
    for (int i = 0; i < CPT; i += 4) {
      z0 = fmaf(sS[r * LDS + cq + 4 * i], sk[cq + 4 * i], z0);
      if (i + 1 < CPT) z1 = fmaf(sS[r * LDS + cq + 4 * (i + 1)], sk[cq + 4 * (i + 1)], z1);
      if (i + 2 < CPT) z2 = fmaf(sS[r * LDS + cq + 4 * (i + 2)], sk[cq + 4 * (i + 2)], z2);
      if (i + 3 < CPT) z3 = fmaf(sS[r * LDS + cq + 4 * (i + 3)], sk[cq + 4 * (i + 3)], z3);
    }
    float z = (z0 + z1) + (z2 + z3);
    z += __shfl_xor_sync(0xffffffffu, z, 1);
    z += __shfl_xor_sync(0xffffffffu, z, 2);
    return z;
  };
  // S <- alpha (S - beta z k^T) + beta v k^T + sum_l D^(l) k^(l)^T on this thread's elements
  // (rows of S evolve independently: no barrier between tokens)
  // (the row's coefficients in registers: alpha, beta v - alpha beta z, D^(l)[r])
  auto row_update = [&](float z) {
    const float al = expf(sgate[0]), be = sgate[1];
    const int gr = r0 + r;
    const float a0 = be * sv[gr] - al * be * z;
    float al_[kBwdLmax];
#pragma unroll
    for (int l = 0; l < kBwdLmax; ++l) al_[l] = l < L ? sdl[l * D + gr] : 0.f;
#pragma unroll 4
    for (int i = 0; i < CPT; ++i) {
      const int c = cq + 4 * i;
      float x = fmaf(al, sS[r * LDS + c], a0 * sk[c]);
#pragma unroll
      for (int l = 0; l < kBwdLmax; ++l)
        if (l < L) x = fmaf(al_[l], skl[l * D + c], x);
      sS[r * LDS + c] = x;
    }
  };
  auto row_store = [&](float* g) {                   // this thread's elements of S to global
#pragma unroll 4
    for (int i = 0; i < CPT; ++i) g[r * D + cq + 4 * i] = sS[r * LDS + cq + 4 * i];
  };

  // ---- forward: checkpoints (the state before tokens 0, CK, 2 CK, ...) ----
  for (int idx = tid; idx < R * LDS; idx += NT) sS[idx] = 0.f;
  __syncthreads();
  row_store(ck);
  for (int j = 0; j < NSTAGE - 1; ++j) issue(j, j < len);
  for (int t = 0; t < len; ++t) {
    issue(t + NSTAGE - 1, t + NSTAGE - 1 < len);
    bwd_cp_async_wait<NSTAGE - 1>();
    __syncthreads();
    convert(t);
    __syncthreads();
    row_update(row_dot_k());
    if ((t + 1) % kBwdCK == 0 && t + 1 < len) row_store(ck + (size_t)((t + 1) / kBwdCK) * R * D);
  }

  // ---- backward ----
  for (int idx = tid; idx < R * LDS; idx += NT) {
    const int rr = idx / LDS, c = idx % LDS;
    sDS[idx] = (p.d_fs && c < D) ? p.d_fs[(((size_t)b * H + h) * D + r0 + rr) * D + c] : 0.f;
  }
  const int nblk = (len + kBwdCK - 1) / kBwdCK;
  for (int blk = nblk - 1; blk >= 0; --blk) {
    const int c0 = blk * kBwdCK, c1 = min(c0 + kBwdCK, len);
    __syncthreads();
    bwd_state_load_async<D, RS>(sS, ck + (size_t)blk * R * D);
    bwd_cp_async_wait_all();
    for (int j = 0; j < NSTAGE - 1; ++j) issue(c0 + j, c0 + j < c1);
    // recompute the block: z_t = S_(t-1) k_t, and the states after tokens c0 .. c1-2
    for (int t = c0; t < c1; ++t) {
      issue(t + NSTAGE - 1, t + NSTAGE - 1 < c1);
      bwd_cp_async_wait<NSTAGE - 1>();
      __syncthreads();
      convert(t);
      __syncthreads();
      const float z = row_dot_k();
      if (cq == 0) sZS[(t - c0) * R + r] = z;
      if (t < c1 - 1) {
        row_update(z);
        row_store(scr + (size_t)(t - c0) * R * D);
      }
    }
    // reverse through the block (tokens in decreasing order through the same ring)
    bwd_cp_async_wait<0>();
    __syncthreads();
    for (int j = 0; j < NSTAGE - 1; ++j) issue(c1 - 1 - j, c1 - 1 - j >= c0);
    for (int t = c1 - 1; t >= c0; --t) {
      __syncthreads();                                 // previous token done with the buffers
      bwd_state_load_async<D, RS>(sS, t > c0 ? scr + (size_t)(t - 1 - c0) * R * D : ck + (size_t)blk * R * D);
      issue(t - (NSTAGE - 1), t - (NSTAGE - 1) >= c0);
      bwd_cp_async_wait<2>();                          // token t's vectors (older groups) landed
      __syncthreads();
      convert(t);
      __syncthreads();
      const size_t n = tok(t);
      const float al = expf(sgate[0]), be = sgate[1];
      const float* zs = sZS + (t - c0) * R;
      // phase 1 (rows): dS += do q^T; y = dS k; y_l = dS k^(l)
      const int gr = r0 + r;
      const float dor = sdo[gr];
      float y = 0.f;
#pragma unroll 4
      for (int i = 0; i < CPT; ++i) {
        const int c = cq + 4 * i;
        const float ds = fmaf(dor, sq[c], sDS[r * LDS + c]);
        sDS[r * LDS + c] = ds;
        y = fmaf(ds, sk[c], y);
      }
      y += __shfl_xor_sync(0xffffffffu, y, 1);
      y += __shfl_xor_sync(0xffffffffu, y, 2);
      const bool own = cq == 0;
      for (int l = 0; l < L; ++l) {
        float yl = 0.f;
#pragma unroll 4
        for (int i = 0; i < CPT; ++i) yl = fmaf(sDS[r * LDS + cq + 4 * i], skl[l * D + cq + 4 * i], yl);
        yl += __shfl_xor_sync(0xffffffffu, yl, 1);
        yl += __shfl_xor_sync(0xffffffffu, yl, 2);
        if (own) p.dDL[(n * L + l) * D + gr] = yl;
        const float s = warp_sum(own ? sdl[l * D + gr] * dor : 0.f);   // D^(l) . do over these rows
        if (lane == 0) sRed[warp * 16 + 4 + l] = s;
      }
      {
        // per-row scalars summed over this slice's rows: v.y, z.y, z.do, v.do
        const float zr = zs[r], vr = sv[gr];
        const float s0 = warp_sum(own ? vr * y : 0.f);
        const float s1 = warp_sum(own ? zr * y : 0.f);
        const float s2 = warp_sum(own ? zr * dor : 0.f);
        const float s3 = warp_sum(own ? vr * dor : 0.f);
        if (lane == 0) {
          sRed[warp * 16 + 0] = s0;
          sRed[warp * 16 + 1] = s1;
          sRed[warp * 16 + 2] = s2;
          sRed[warp * 16 + 3] = s3;
        }
        if (own) {
          sy[r] = y;
          p.dv[n * D + gr] = be * y;
        }
      }
      bwd_cp_async_wait<1>();                          // S_(t-1) landed (only the newest prefetch may pend)
      __syncthreads();
      // phase 2 (columns, this slice's rows): dS^T D^(l); S_(t-1)^T y, S_(t-1)^T do,
      // dS^T (beta v - alpha beta z), <S_(t-1), dS>; then dS <- alpha (dS - beta y k^T)
      for (int l = 0; l < L; ++l) {
        float f = 0.f;
#pragma unroll 4
        for (int i = 0; i < RPG; ++i) {
          const int rr = rq * RPG + i;
          f = fmaf(sDS[rr * LDS + cc], sdl[l * D + r0 + rr], f);
        }
        sPart[(rq * NSLOT + 3 + l) * D + cc] = f;
      }
      {
        float bS = 0.f, e = 0.f, a = 0.f, fro = 0.f;
        const float kc = sk[cc];
#pragma unroll 4
        for (int i = 0; i < RPG; ++i) {
          const int rr = rq * RPG + i;
          const float s = sS[rr * LDS + cc], ds = sDS[rr * LDS + cc], yr = sy[rr];
          bS = fmaf(s, yr, bS);
          a = fmaf(s, sdo[r0 + rr], a);
          e = fmaf(ds, be * (sv[r0 + rr] - al * zs[rr]), e);
          fro = fmaf(s, ds, fro);
          sDS[rr * LDS + cc] = al * (ds - be * yr * kc);
        }
        sPart[(rq * NSLOT + 0) * D + cc] = bS;
        sPart[(rq * NSLOT + 1) * D + cc] = e;
        sPart[(rq * NSLOT + 2) * D + cc] = a;
        fro = warp_sum(fro);
        if (lane == 0) sRed[warp * 16 + 15] = fro;
      }
      __syncthreads();
      // phase 3: this slice's part of the per-token gradients
      if (tid < D) {
        const int c = tid;
        float t0s = 0.f, t1s = 0.f, t2s = 0.f, zd = 0.f, vd = 0.f;
#pragma unroll
        for (int q4 = 0; q4 < S::NGRP; ++q4) {
          t0s += sPart[(q4 * NSLOT + 0) * D + c];
          t1s += sPart[(q4 * NSLOT + 1) * D + c];
          t2s += sPart[(q4 * NSLOT + 2) * D + c];
        }
        for (int wv = 0; wv < NW; ++wv) {
          zd += sRed[wv * 16 + 2];
          vd += sRed[wv * 16 + 3];
        }
        ok_[n * D + c] = t1s - al * be * t0s;
        float dqc = al * (t2s - be * zd * sk[c]) + be * vd * sk[c];
        for (int l = 0; l < L; ++l) {
          float ddl = 0.f, tl = 0.f;
          for (int wv = 0; wv < NW; ++wv) ddl += sRed[wv * 16 + 4 + l];
#pragma unroll
          for (int q4 = 0; q4 < S::NGRP; ++q4) tl += sPart[(q4 * NSLOT + 3 + l) * D + c];
          dqc = fmaf(ddl, skl[l * D + c], dqc);
          okl[(n * L + l) * D + c] = tl;
        }
        oq[n * D + c] = dqc;
        if (c == 0) {
          float vy = 0.f, zy = 0.f, fr = 0.f;
          for (int wv = 0; wv < NW; ++wv) {
            vy += sRed[wv * 16 + 0];
            zy += sRed[wv * 16 + 1];
            fr += sRed[wv * 16 + 15];
          }
          ob[n] = vy - al * zy;
          oa[n] = al * (fr - be * zy);
        }
      }
    }
  }
  bwd_cp_async_wait<0>();
}

// Sum of the RS slices' partial column sums, in slice order.
template <int D>
__global__ void __launch_bounds__(kBwdThreads) bwd_state_reduce_kernel(BwdArgs p, int RS) {
  const size_t NTH = (size_t)p.B * p.T * p.H;
  const int L = p.L;
  const size_t per = (size_t)(2 + L) * D + 2;        // outputs per token-head
  for (size_t idx = (size_t)blockIdx.x * kBwdThreads + threadIdx.x; idx < NTH * per;
       idx += (size_t)gridDim.x * kBwdThreads) {
    const size_t n = idx / per;
    const int j = (int)(idx % per);
    float s = 0.f;
    if (j < D) {
      for (int r = 0; r < RS; ++r) s += p.PQ[(r * NTH + n) * D + j];
      p.dq[n * D + j] = s;
    } else if (j < 2 * D) {
      for (int r = 0; r < RS; ++r) s += p.PK[(r * NTH + n) * D + j - D];
      p.dk[n * D + j - D] = s;
    } else if (j < (2 + L) * D) {
      const int e = j - 2 * D;
      for (int r = 0; r < RS; ++r) s += p.PKL[(r * NTH + n) * L * D + e];
      p.dKL[n * L * D + e] = s;
    } else if (j == (2 + L) * D) {
      for (int r = 0; r < RS; ++r) s += p.PB[r * NTH + n];
      p.dbeta[n] = s;
    } else {
      for (int r = 0; r < RS; ++r) s += p.PA[r * NTH + n];
      p.dla[n] = s;
    }
  }
}

// ------------------------------------------------------------------------------------
// C: the refinement chain backwards for kBwdTC tokens of one (b, h)

template <int D>
struct BwdCSmem {
  static constexpr size_t oW = 0;                                       // W [2][D][D] (swizzled pieces)
  static constexpr size_t oR = oW + 4u * 2 * D * D;                     // r^(l) [Lmax][TC][D]
  static constexpr size_t oDR = oR + 4u * kBwdLmax * kBwdTC * D;        // dr [TC][D]
  static constexpr size_t oDU = oDR + 4u * kBwdTC * D;                  // du [TC][D]
  static constexpr size_t oG = oDU + 4u * kBwdTC * D;                   // d k_hat [TC][D]
  static constexpr size_t oH = oG + 4u * kBwdTC * D;                    // dp [TC][D]
  static constexpr size_t oZ = oH + 4u * kBwdTC * D;                    // dz [TC]
  static constexpr size_t bytes = oZ + 4u * kBwdTC;
};

template <class T, int D>
__global__ void __launch_bounds__(kBwdThreads) bwd_refine_kernel(BwdArgs p) {
  using S = BwdCSmem<D>;
  extern __shared__ __align__(1024) unsigned char sm[];
  float* sW = reinterpret_cast<float*>(sm + S::oW);
  float* sR = reinterpret_cast<float*>(sm + S::oR);
  float* sDR = reinterpret_cast<float*>(sm + S::oDR);
  float* sDU = reinterpret_cast<float*>(sm + S::oDU);
  float* sG = reinterpret_cast<float*>(sm + S::oG);
  float* sH = reinterpret_cast<float*>(sm + S::oH);
  float* sZ = reinterpret_cast<float*>(sm + S::oZ);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int t0 = blockIdx.x * kBwdTC, h = blockIdx.y, b = blockIdx.z;
  const int H = p.H, T_ = p.T, L = p.L;
  const int len = bwd_len(p, b);
  const T* vg = static_cast<const T*>(p.v);
  const bool gelu = !(p.flags & 1u);
  auto tok = [&](int t) { return ((size_t)b * T_ + t) * H + h; };

  // the weight matrices in the order they are used: W_k^(L-1), W_p^(L-1), W_k^(L-2), ...
  auto wmat = [&](int m) {
    const int l = L - 1 - (m >> 1);
    return ((m & 1) ? p.Wp : p.Wk) + ((size_t)h * L + l) * D * D;
  };
  if (L > 0) bwd_load_w_async<D>(sW, wmat(0));
  // forward recompute of the residual chain: r^(1) = v - u, r^(l+1) = r^(l) - delta^(l)
  for (int idx = tid; idx < kBwdTC * D; idx += kBwdThreads) {
    const int i = idx / D, c = idx % D, t = t0 + i;
    float rr = 0.f;
    if (t < len) {
      const size_t n = tok(t);
      rr = Elem<T>::to_f(vg[n * D + c]) - p.U[n * D + c];
      for (int l = 0; l < L; ++l) {
        sR[(l * kBwdTC + i) * D + c] = rr;
        const float x = p.P[(n * L + l) * D + c] * rr;
        rr -= gelu ? gelu_erf(x) : x;
      }
    } else {
      for (int l = 0; l < L; ++l) sR[(l * kBwdTC + i) * D + c] = 0.f;
    }
    sDR[idx] = 0.f;
    sDU[idx] = 0.f;
  }
  __syncthreads();
  for (int l = L - 1; l >= 0; --l) {
    // elementwise: dp, dr, and per token d beta^(l) (-> dz) and k^(l) . dk^(l) (-> d k_hat)
    for (int i = warp; i < kBwdTC; i += kBwdThreads / 32) {
      const int t = t0 + i;
      const bool valid = t < len;
      const size_t n = valid ? tok(t) : 0;
      const float bl = valid ? sigmoidf(p.Z[n * L + l]) : 0.f;
      const float inv = valid ? p.NRM[n * L + l] : 0.f;
      float sdb = 0.f, skd = 0.f;
      for (int a = lane; a < D; a += 32) {
        if (!valid) {
          sH[i * D + a] = 0.f;
          continue;
        }
        const float rr = sR[(l * kBwdTC + i) * D + a];
        const float pp = p.P[(n * L + l) * D + a];
        const float x = pp * rr;
        const float dl = gelu ? gelu_erf(x) : x;
        const float dD = p.dDL[(n * L + l) * D + a];
        const float ddel = bl * dD - sDR[i * D + a];
        const float dx = ddel * (gelu ? gelu_grad(x) : 1.0f);
        sH[i * D + a] = dx * rr;
        sDR[i * D + a] += dx * pp;
        sdb = fmaf(dl, dD, sdb);
        skd = fmaf(p.KL[(n * L + l) * D + a], p.dKL[(n * L + l) * D + a], skd);
      }
      sdb = warp_sum(sdb);
      skd = warp_sum(skd);
      const float dz = sdb * bl * (1.0f - bl);
      if (lane == 0) sZ[i] = valid ? dz : 0.f;
      for (int a = lane; a < D; a += 32) {
        const float g = valid ? (p.dKL[(n * L + l) * D + a] - p.KL[(n * L + l) * D + a] * skd) * inv : 0.f;
        sG[i * D + a] = g;
        if (t < T_) {
          const size_t o = (tok(t) * L + l) * D + a;
          p.dKH[o] = g;
          p.DL[o] = sH[i * D + a];          // dp^(l) (the forward's D^(l) is no longer needed)
        }
      }
      if (lane == 0 && t < T_) p.dZ[tok(t) * L + l] = valid ? dz : 0.f;
    }
    __syncthreads();
    // du += W_k^T d k_hat + W_p^T dp + dz w_beta
#pragma unroll
    for (int which = 0; which < 2; ++which) {
      const int m = 2 * (L - 1 - l) + which;
      if (m + 1 < 2 * L) {
        bwd_load_w_async<D>(sW + (size_t)((m + 1) & 1) * D * D, wmat(m + 1));
        bwd_cp_async_wait<1>();
      } else {
        bwd_cp_async_wait<0>();
      }
      __syncthreads();
      bwd_matvec_t_add<D, kBwdTC>(sW + (size_t)(m & 1) * D * D, which ? sH : sG, sDU);
      __syncthreads();                               // buffer m % 2 free for matrix m + 2
    }
    for (int idx = tid; idx < kBwdTC * D; idx += kBwdThreads)
      sDU[idx] = fmaf(sZ[idx / D], p.wbeta[((size_t)h * L + l) * D + idx % D], sDU[idx]);
    __syncthreads();
  }
  // r^(1) = v - u: dv += dr^(1), du -= dr^(1)
  for (int idx = tid; idx < kBwdTC * D; idx += kBwdThreads) {
    const int i = idx / D, c = idx % D, t = t0 + i;
    if (t >= T_) continue;
    const size_t n = tok(t);
    if (t < len) {
      p.dv[n * D + c] += sDR[idx];
      p.dU[n * D + c] = sDU[idx] - sDR[idx];
    } else {
      p.dU[n * D + c] = 0.f;
    }
  }
}

// ------------------------------------------------------------------------------------
// D: dW_k^(l), dW_p^(l): sums over the head's tokens of d k_hat u^T and dp u^T.  One CTA
// per (TILE x TILE output tile, step and matrix, head, token split); thread (ty, tx) of
// a (TILE/4)^2 grid keeps a 4 x 4 block of outputs in registers, and 32-token slabs of
// the two operands pass through shared memory.
template <int D>
struct BwdWTile {
  static constexpr int TILE = D < 64 ? D : 64, NT = (TILE / 4) * (TILE / 4), TILES = (D / TILE) * (D / TILE);
};
template <int D>
__global__ void __launch_bounds__(BwdWTile<D>::NT) bwd_weight_kernel(BwdArgs p) {
  constexpr int TILE = BwdWTile<D>::TILE, NT = BwdWTile<D>::NT;
  __shared__ __align__(16) float sA[32][TILE], sU[32][TILE];
  const int tid = threadIdx.x, ty = tid / (TILE / 4), tx = tid % (TILE / 4);
  const int tile = blockIdx.x, lw = blockIdx.y, which = lw % 2, l = lw / 2;
  const int h = blockIdx.z % p.H, split = blockIdx.z / p.H;
  const int a0 = (tile / (D / TILE)) * TILE, c0 = (tile % (D / TILE)) * TILE;
  const int H = p.H, L = p.L, NTOK = p.B * p.T;
  const int per = ((NTOK + p.nsw - 1) / p.nsw + 31) / 32 * 32;
  const int m_begin = split * per, m_end = min(NTOK, m_begin + per);
  const float* src = which == 0 ? p.dKH : p.DL;      // DL holds dp^(l) after kernel C
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
  for (int m0 = m_begin; m0 < m_end; m0 += 32) {
    for (int idx = tid; idx < 32 * (TILE / 4); idx += NT) {
      const int i = idx / (TILE / 4), j4 = (idx % (TILE / 4)) * 4, m = m0 + i;
      const size_t n = (size_t)m * H + h;
      const bool in = m < m_end;
      *reinterpret_cast<float4*>(&sA[i][j4]) =
          in ? *reinterpret_cast<const float4*>(src + (n * L + l) * D + a0 + j4) : make_float4(0.f, 0.f, 0.f, 0.f);
      *reinterpret_cast<float4*>(&sU[i][j4]) =
          in ? *reinterpret_cast<const float4*>(p.U + n * D + c0 + j4) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    __syncthreads();
#pragma unroll 4
    for (int i = 0; i < 32; ++i) {
      const float4 av = *reinterpret_cast<const float4*>(&sA[i][ty * 4]);
      const float4 uv = *reinterpret_cast<const float4*>(&sU[i][tx * 4]);
      const float a[4] = {av.x, av.y, av.z, av.w}, u[4] = {uv.x, uv.y, uv.z, uv.w};
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[r][c] = fmaf(a[r], u[c], acc[r][c]);
    }
    __syncthreads();
  }
  // one split: the sums themselves; else this split's partials, added by the reduce kernel
  float* dst = p.nsw == 1
                   ? (which == 0 ? p.dWk : p.dWp) + ((size_t)h * L + l) * D * D
                   : p.PW + (((size_t)split * H + h) * 2 * L + lw) * D * D;
#pragma unroll
  for (int r = 0; r < 4; ++r)
    *reinterpret_cast<float4*>(dst + (size_t)(a0 + ty * 4 + r) * D + c0 + tx * 4) =
        make_float4(acc[r][0], acc[r][1], acc[r][2], acc[r][3]);
}

// dW_k, dW_p = the nsw partials added in split order.
template <int D>
__global__ void __launch_bounds__(kBwdThreads) bwd_weight_reduce_kernel(BwdArgs p) {
  const size_t per = (size_t)p.H * 2 * p.L * D * D;
  for (size_t idx = (size_t)blockIdx.x * kBwdThreads + threadIdx.x; idx < per; idx += (size_t)gridDim.x * kBwdThreads) {
    float s = 0.f;
    for (int q = 0; q < p.nsw; ++q) s += p.PW[(size_t)q * per + idx];
    const size_t hl = idx / ((size_t)D * D), e = idx % ((size_t)D * D);
    const int h = (int)(hl / (2 * p.L)), lw = (int)(hl % (2 * p.L));
    (lw % 2 == 0 ? p.dWk : p.dWp)[((size_t)h * p.L + lw / 2) * D * D + e] = s;
  }
}

// dw_beta^(l)[c] = sum_tokens dz^(l) u[c];  dconv[j-1][c] = sum_tokens du_t[c] v_(t-j)[c].
// One CTA per (32 channels, head, token split); thread (channel, token lane) over every 8th
// token of the split's share of the flattened (b, t) axis.
template <class T, int D>
__global__ void __launch_bounds__(kBwdThreads) bwd_small_weight_kernel(BwdArgs p) {
  __shared__ float sRed[8][32][kBwdLmax + 8 + 1];
  const int tid = threadIdx.x, cl = tid % 32, tl = tid / 32;
  const int c = blockIdx.x * 32 + cl, h = blockIdx.y, split = blockIdx.z;
  const int H = p.H, T_ = p.T, L = p.L, w = p.w;
  const long long NTOK = (long long)p.B * T_;
  const long long per = (NTOK + p.nss - 1) / p.nss;
  const long long m_begin = split * per, m_end = m_begin + per < NTOK ? m_begin + per : NTOK;
  const T* vg = static_cast<const T*>(p.v);
  float acc[kBwdLmax + 8];
#pragma unroll
  for (int j = 0; j < kBwdLmax + 8; ++j) acc[j] = 0.f;
  for (long long m = m_begin + tl; m < m_end && c < D; m += 8) {
    const int b = (int)(m / T_), t = (int)(m % T_);
    if (t >= bwd_len(p, b)) continue;
    const size_t n = (size_t)m * H + h;
    const float uc = p.U[n * D + c], du = p.dU[n * D + c];
    // (fixed trip counts with predicates, so that acc stays in registers)
#pragma unroll
    for (int l = 0; l < kBwdLmax; ++l)
      if (l < L) acc[l] = fmaf(p.dZ[n * L + l], uc, acc[l]);
#pragma unroll
    for (int j = 1; j <= 8; ++j)
      if (j <= w && j <= t)
        acc[kBwdLmax + j - 1] = fmaf(du, Elem<T>::to_f(vg[(((size_t)b * T_ + t - j) * H + h) * D + c]), acc[kBwdLmax + j - 1]);
  }
#pragma unroll
  for (int j = 0; j < kBwdLmax + 8; ++j) sRed[tl][cl][j] = acc[j];
  __syncthreads();
  if (tl == 0 && c < D) {
    // one split: the sums themselves; else this split's partials [split][h][L + w][D]
    float* part = p.PSW + ((size_t)split * H + h) * (L + w) * D;
    for (int l = 0; l < L; ++l) {
      float s = 0.f;
      for (int q = 0; q < 8; ++q) s += sRed[q][cl][l];
      if (p.nss == 1) p.dwb[((size_t)h * L + l) * D + c] = s;
      else part[(size_t)l * D + c] = s;
    }
    for (int j = 1; j <= w; ++j) {
      float s = 0.f;
      for (int q = 0; q < 8; ++q) s += sRed[q][cl][kBwdLmax + j - 1];
      if (p.nss == 1) p.dconv[((size_t)h * w + j - 1) * D + c] = s;
      else part[(size_t)(L + j - 1) * D + c] = s;
    }
  }
}

// dw_beta, dconv = the nss partials added in split order.
template <int D>
__global__ void __launch_bounds__(kBwdThreads) bwd_small_reduce_kernel(BwdArgs p) {
  const int LW = p.L + p.w;
  const size_t per = (size_t)p.H * LW * D;
  for (size_t idx = (size_t)blockIdx.x * kBwdThreads + threadIdx.x; idx < per; idx += (size_t)gridDim.x * kBwdThreads) {
    float s = 0.f;
    for (int q = 0; q < p.nss; ++q) s += p.PSW[(size_t)q * per + idx];
    const int c = (int)(idx % D), j = (int)((idx / D) % LW), h = (int)(idx / ((size_t)D * LW));
    if (j < p.L) p.dwb[((size_t)h * p.L + j) * D + c] = s;
    else p.dconv[((size_t)h * p.w + j - p.L) * D + c] = s;
  }
}

// E: dv_t += sum_{j=1..w} c_j (.) du_(t+j) over tokens t + j inside the sequence.
template <int D>
__global__ void __launch_bounds__(kBwdThreads) bwd_conv_dv_kernel(BwdArgs p) {
  const size_t total = (size_t)p.B * p.T * p.H * D;
  for (size_t idx = (size_t)blockIdx.x * kBwdThreads + threadIdx.x; idx < total; idx += (size_t)gridDim.x * kBwdThreads) {
    const int c = idx % D;
    const size_t n = idx / D;
    const int h = n % p.H;
    const size_t bt = n / p.H;
    const int t = bt % p.T, b = bt / p.T;
    const int len = bwd_len(p, b);
    if (t >= len) continue;
    float s = 0.f;
    for (int j = 1; j <= p.w && t + j < len; ++j)
      s = fmaf(p.conv_w[((size_t)h * p.w + j - 1) * D + c], p.dU[(n + (size_t)j * p.H) * D + c], s);
    p.dv[idx] += s;
  }
}

}  // namespace prism
