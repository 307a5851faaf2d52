// Kernel A (bf16 I/O path): anchor + refinement + the chunk's rank-L write
// summaries, on tcgen05 tensor cores.  ("Technical Summary: PRISM", §2.2
// stages 1-2 and the injection B_t = sum_l beta^(l) delta^(l) k^(l)^T.)
//
// Everything here is state-independent, so it runs fully parallel: one CTA per
// (chunk, head, batch).  For the chunk's C tokens it computes the anchor u, the
// L refinement steps (directions K_l = k^(l), write values D_l = beta^(l) delta^(l))
// and reduces them at once to what the state scan needs:
//   R   = sum_l strict_tril(K K_l^T (.) Gamma) D_l      (C x d_v)  value-side correction
//   O_l = sum_l tril(Q K_l^T (.) Gamma) D_l             (C x d_v)  intra-chunk output
//   N_l = sum_l D_l^T diag(gamma_C / gamma) K_l          (d_v x d_k) state injection
// with Gamma_ts = exp(g_t - g_s), g the in-chunk cumulative sum of log alpha.
// The per-token factors never leave the SM.  The kernel then also does the
// state-independent part of the gated delta rule for the chunk (strictly lower
// A = beta (K K^T (.) Gamma), T = (I + A)^-1, P = tril(Q K^T (.) Gamma)) and
// writes the chunk's affine state map in factored form for the scan kernel:
//   E = U - W S0^T,  O = O_intra + Qt S0^T,  S1 = gamma_C S0 + E^T Kt + N
// with W = T diag(beta gamma) K, U = T diag(beta)(V - R), Kt = diag(gamma_C/gamma) K,
// Qt = diag(gamma) Q - P W, O_intra = P U + O_l, N = N_l.
//
// Precision: tensor-core operands are fp16 (q, k, v arrive as bf16 and convert
// exactly).  Values that carry large magnitudes are split x = hi + lo into two
// fp16 halves and multiplied in 2-3 passes (hi*hi + hi*lo + lo*hi), which keeps
// ~fp32 accuracy: the anchor u in the projections, k^(l), D_l, the scaled
// D_l, and the output-side scores Q K_l^T.  Accumulation is fp32 in TMEM.
//
// Operand orientation (all MMAs are M = 128, fp32 accumulators in TMEM):
//   projections  [k_hat ; p]^T = W u^T : A = W (features x d_v),  B = U (tokens x d_v)
//   scores       [G ; P]  = [K ; Q] K_l^T : A = [K ; Q] rows,   B = K_l (MN-major)
//   corrections  [R ; O_l] += [G ; P] D_l : A = [G ; P],          B = D_l^T rows
//   injection    N_l += Dt_l^T K_l         : A = Dt_l^T rows,     B = K_l rows
// so each epilogue thread owns one TMEM lane (a feature or a token row).
#pragma once

#include "chunk_scan.cuh"
#include "prism_common.cuh"
#include "tc_common.cuh"

namespace prism {

struct PrepArgs {
  int B, T, H, w, L;
  unsigned flags;
  const __nv_bfloat16* q;
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  const float* log_alpha;
  const float* beta;
  const float* conv_w;
  const float* wbeta;
  const unsigned char* wblocks;   // fp16 weight blocks laid out for the A operand
  const int* wflag;               // nonzero: weights need their lo halves
  const int* seq_lens;
  // Per-chunk outputs, chunk-major [B][H][NC][...].  Inside a chunk each array is
  // stored "piece-major": 16-byte column pieces, rows contiguous within a piece:
  // element (r, f) of an R-row array at ((f / V) * R + r) * V + f % V, V = 16 / elem
  // size.  A warp whose lanes hold consecutive rows then writes 512 contiguous bytes.
  __half* Wc;                     // [C][D]  W = T diag(beta gamma) K
  __half* Kt;                     // [C][D]  Kt = diag(gamma_C / gamma) K
  __half* Qth;                    // [C][D]  Qt = diag(gamma) Q - P W, hi half
  __half* Qtl;                    // [C][D]  lo half
  float* U;                       // [C][D]  U = T diag(beta) (V - R)
  float* Oi;                      // [C][D]  O_intra = P U + O_l
  float* Nl;                      // [D][D]  N = U^T Kt + N_l
  float* gC;                      // [1]     gamma_C
  int* status;                    // device error word (bounded waits)
};

// One weight block: 128 rows (features, zero beyond D) x D columns, fp16,
// K-major with SBO = 128 and LBO = 2048:  (row, c) at (c/8)*2048 + row*16 + (c%8)*2.
template <int D>
struct WeightBlock {
  static constexpr uint32_t bytes = 128u * D * 2u;
  // block index of (h, l, which = 0 W_k / 1 W_p, part = 0 hi / 1 lo)
  static __host__ __device__ size_t index(int h, int l, int L, int which, int part) {
    return (((size_t)h * L + l) * 2 + which) * 2 + part;
  }
};

// Converts W_k, W_p (fp32 [H][L][D][D]) into fp16 hi/lo blocks; sets *flag if
// any lo half is significant (|lo| > 2^-22 of its row norm), in which case the
// projections take a third pass with the lo halves.
template <int D>
__global__ void prep_weights_kernel(const float* Wk, const float* Wp, int H, int L,
                                    unsigned char* blocks, int* flag) {
  const int blk = blockIdx.x;              // (h*L + l)*2 + which
  const int which = blk & 1, hl = blk >> 1;
  const float* W = (which == 0 ? Wk : Wp) + (size_t)hl * D * D;
  unsigned char* hi = blocks + (size_t)(blk * 2 + 0) * WeightBlock<D>::bytes;
  unsigned char* lo = blocks + (size_t)(blk * 2 + 1) * WeightBlock<D>::bytes;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarp = blockDim.x >> 5;
  bool need = false;
  for (int row = warp; row < 128; row += nwarp) {
    float n2 = 0.f;
    if (row < D)
      for (int c = lane; c < D; c += 32) { const float x = W[(size_t)row * D + c]; n2 = fmaf(x, x, n2); }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) n2 += __shfl_xor_sync(0xffffffffu, n2, o);
    const float tol = sqrtf(n2) * 0x1p-22f;
    for (int c = lane; c < D; c += 32) {
      const float x = row < D ? W[(size_t)row * D + c] : 0.f;
      __half h, l;
      tc::split_f16(x, h, l);
      const uint32_t off = (c / 8) * 2048u + row * 16u + (c % 8) * 2u;
      *reinterpret_cast<__half*>(hi + off) = h;
      *reinterpret_cast<__half*>(lo + off) = l;
      need |= fabsf(__half2float(l)) > tol;
    }
  }
  if (__any_sync(0xffffffffu, need) && lane == 0) atomicOr(flag, 1);
}

// First-fit placement helper for the tail buffers: region 1 is [r1, r1_end),
// region 2 starts at r2 and may grow past the refinement loop's footprint.
struct Place {
  uint32_t o1, e1, o2;
  constexpr Place at(uint32_t size) const {
    return (((o1 + 127) / 128) * 128 + size <= e1)
               ? Place{((o1 + 127) / 128) * 128 + size, e1, o2}
               : Place{o1, e1, ((o2 + 127) / 128) * 128 + size};
  }
  constexpr uint32_t where(uint32_t size) const {
    return (((o1 + 127) / 128) * 128 + size <= e1) ? ((o1 + 127) / 128) * 128 : ((o2 + 127) / 128) * 128;
  }
};

template <int D, int C>
struct PrepSmem {
  static constexpr int NTH = C / 2;                      // tokens per column half
  static constexpr uint32_t kW = WeightBlock<D>::bytes;  // 128 x D
  static constexpr uint32_t kU = C * D * 2;              // tokens x D
  static constexpr uint32_t kKQ = 128 * D * 2;           // 128 rows x D
  static constexpr uint32_t kF = D * C * 2;              // features x tokens
  static constexpr uint32_t kF128 = 128 * C * 2;         // 128 rows x tokens
  static constexpr bool kWpInGP = kW <= 2 * kF128;       // W_p staged in the [G;P] buffers
  // small arrays first
  static constexpr uint32_t oG = 0;                      // f32 g[C]
  static constexpr uint32_t oDec = oG + 4 * C;           // f32 gamma_C/gamma [C]
  static constexpr uint32_t oBeta = oDec + 4 * C;        // f32 beta^(l) [C]
  static constexpr uint32_t oInv = oBeta + 4 * C;        // f32 1/|k_hat| [C]
  static constexpr uint32_t oBar = oInv + 4 * C;         // mbarriers: mma, W_k, W_p
  static constexpr uint32_t oSlot = oBar + 24;
  static constexpr uint32_t oTiles = ((oSlot + 8 + 127) / 128) * 128;
  // refinement-loop tiles
  static constexpr uint32_t oW = oTiles;
  static constexpr uint32_t oGP = oW + kW;               // hi, lo (2 * kF128)
  static constexpr uint32_t oWp = kWpInGP ? oGP : oGP + 2 * kF128;
  static constexpr uint32_t oU = oGP + 2 * kF128 + (kWpInGP ? 0 : kW);   // hi, lo
  static constexpr uint32_t oKQ = oU + 2 * kU;
  static constexpr uint32_t oKl = oKQ + kKQ;             // hi, lo
  static constexpr uint32_t oD = oKl + 2 * kF;           // hi, lo
  static constexpr uint32_t oDt = oD + 2 * kF;           // hi, lo (128 rows)
  static constexpr uint32_t loop_end = oDt + 2 * kF128;
  // tail buffers (after the loop), placed around the [K;Q] tile which stays live
  static constexpr uint32_t sKX = 4 * C * D, sSq = 4 * C * (C + 1), sY = 1024 * (C / 16), sB = 8 * C;
  static constexpr uint32_t sTB = 2 * C * C;               // f16 T as B operand (C x C)
  static constexpr Place p0{oW, oKQ, oKl};
  static constexpr uint32_t tKX = p0.where(sKX);         // f16 [Kb | X] MN-major, C x 2D
  static constexpr Place p1 = p0.at(sKX);
  static constexpr uint32_t tTP = p1.where(kF128);       // f16 [T ; PT] 128 x C  (also [I ; P])
  static constexpr Place p2 = p1.at(kF128);
  static constexpr uint32_t tA = p2.where(sSq);          // f32 [C][C+1]
  static constexpr Place p3 = p2.at(sSq);
  static constexpr uint32_t tP = p3.where(sSq);          // f32 [C][C+1]
  static constexpr Place p4 = p3.at(sSq);
  static constexpr uint32_t tT = p4.where(sSq);          // f32 [C][C+1]
  static constexpr Place p5 = p4.at(sSq);
  static constexpr uint32_t tY = p5.where(sY);           // f32 block-solve scratch
  static constexpr Place p6 = p5.at(sY);
  static constexpr uint32_t tB = p6.where(sB);           // f32 beta[C], gamma[C]
  static constexpr Place p7a = p6.at(sB);
  static constexpr uint32_t tTB = p7a.where(sTB);        // f16 T (B operand)
  static constexpr Place p7 = p7a.at(sTB);
  static constexpr uint32_t bytes = p7.o2 > loop_end ? p7.o2 : loop_end;
  static constexpr bool kExtraX = D > 2 * C;             // U/PU need their own TMEM columns
  // columns: k_hat | p | [R;O_l] | N_l | r, u (refinement loop) or U/PU (tail, when D > 2C)
  static constexpr uint32_t tmem_cols_needed = 2 * C + 2 * D + (kExtraX ? D : 2 * C);
  static constexpr uint32_t tmem_cols =
      tmem_cols_needed <= 32 ? 32 : tmem_cols_needed <= 64 ? 64 : tmem_cols_needed <= 128 ? 128
                                  : tmem_cols_needed <= 256 ? 256 : 512;
};

// T = (I + A)^-1 for the strictly lower triangular C x C matrix A (fp32, row
// stride C+1), by blocked forward substitution with 16 x 16 blocks:
//   diagonal blocks  T_ii = (I + A_ii)^-1 : one lane per column, the column kept
//                    in registers (row i needs only A's row i and rows < i of
//                    the lane's own column);
//   off-diagonal     T_ij = -T_ii sum_{k=j}^{i-1} A_ik T_kj, by diagonal level.
// Result in sT (fp32, zeros above the diagonal).  All 256 threads take part.
template <int C>
__device__ __forceinline__ void solve_tri(const float* sA, float* sT, float* sY) {
  constexpr int LD = C + 1, NB = C / 16;
  const int tid = threadIdx.x;
  for (int idx = tid; idx < C * C; idx += 256) {
    const int i = idx / C, j = idx % C;
    if (j / 16 != i / 16 && j > i) sT[i * LD + j] = 0.f;
  }
  if (tid < 16 * NB) {
    const int blk = tid / 16, j = tid % 16, o = blk * 16;
    float col[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      float s = (i == j) ? 1.f : 0.f;
#pragma unroll
      for (int m = 0; m < i; ++m) s -= (m >= j) ? sA[(o + i) * LD + o + m] * col[m] : 0.f;
      col[i] = (i >= j) ? s : 0.f;
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) sT[(o + i) * LD + o + j] = col[i];
  }
  __syncthreads();
  // Off-diagonal blocks by level (distance lev = i - j).  At one level every
  // block has the same inner length 16*lev, so a thread walks its (up to
  // NB-1) elements in lockstep: independent FMA chains instead of one long one.
  const int r = (tid & 255) / 16, cc = tid % 16;
  for (int lev = 1; lev < NB; ++lev) {
    const int nblk = NB - lev;                       // blocks (i = lev + e, j = e)
    if (tid < 256) {
      float acc[NB > 1 ? NB - 1 : 1];
#pragma unroll
      for (int e = 0; e < NB - 1; ++e) acc[e] = 0.f;
#pragma unroll 4
      for (int mo = 0; mo < 16 * lev; ++mo) {
#pragma unroll
        for (int e = 0; e < NB - 1; ++e)
          if (e < nblk) {
            const int bi = lev + e, bj = e;
            acc[e] = fmaf(sA[(bi * 16 + r) * LD + bj * 16 + mo], sT[(bj * 16 + mo) * LD + bj * 16 + cc], acc[e]);
          }
      }
#pragma unroll
      for (int e = 0; e < NB - 1; ++e)
        if (e < nblk) sY[e * 256 + r * 16 + cc] = acc[e];
    }
    __syncthreads();
    if (tid < 256) {
      float acc[NB > 1 ? NB - 1 : 1];
#pragma unroll
      for (int e = 0; e < NB - 1; ++e) acc[e] = 0.f;
#pragma unroll
      for (int m = 0; m < 16; ++m) {
#pragma unroll
        for (int e = 0; e < NB - 1; ++e)
          if (e < nblk) {
            const int bi = lev + e;
            acc[e] = fmaf(sT[(bi * 16 + r) * LD + bi * 16 + m], sY[e * 256 + m * 16 + cc], acc[e]);
          }
      }
#pragma unroll
      for (int e = 0; e < NB - 1; ++e)
        if (e < nblk) sT[((lev + e) * 16 + r) * LD + e * 16 + cc] = -acc[e];
    }
    __syncthreads();
  }
}

template <int D, int C>
__global__ void __launch_bounds__(256, 1) prep_tc_kernel(PrepArgs p) {
  using S = PrepSmem<D, C>;
  constexpr int NTH = S::NTH;
  extern __shared__ __align__(1024) unsigned char sm[];
  unsigned char* sW = sm + S::oW;
  unsigned char* sWp = sm + S::oWp;
  unsigned char* sGP = sm + S::oGP;
  unsigned char* sU = sm + S::oU;
  unsigned char* sKQ = sm + S::oKQ;
  unsigned char* sKl = sm + S::oKl;
  unsigned char* sD = sm + S::oD;
  unsigned char* sDt = sm + S::oDt;
  float* sg = reinterpret_cast<float*>(sm + S::oG);
  float* sdec = reinterpret_cast<float*>(sm + S::oDec);
  float* sbl = reinterpret_cast<float*>(sm + S::oBeta);
  float* sinv = reinterpret_cast<float*>(sm + S::oInv);
  uint64_t* bar_mma = reinterpret_cast<uint64_t*>(sm + S::oBar);
  uint64_t* bar_wk = bar_mma + 1;
  uint64_t* bar_wp = bar_mma + 2;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + S::oSlot);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int quarter = warp & 3, half = warp >> 2;
  const int row = quarter * 32 + lane;         // this thread's TMEM lane
  const int chunk = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int H = p.H, T_ = p.T, L = p.L, w = p.w;
  const int NC = (T_ + C - 1) / C;
  const int len = p.seq_lens ? min(max(p.seq_lens[b], 0), T_) : T_;
  const int t0 = chunk * C;
  const int nv = min(C, len - t0);
  if (nv <= 0) return;                         // chunk entirely padding: never read
  const bool need_lo = *p.wflag != 0;
  const unsigned char* wsrc = p.wblocks;
  auto wblock = [&](int l, int which, int part) {
    return wsrc + WeightBlock<D>::index(h, l, L, which, part) * S::kW;
  };

  // ---- setup: barriers, TMEM, first weights, gates, [K;Q] rows, v window ----
  if (tid == 0) {
    tc::bar_init(bar_mma, 1);
    tc::bar_init(bar_wk, 1);
    tc::bar_init(bar_wp, 1);
    tc::bar_fence_init();
    if (L > 0) {                               // W^(0) streams in while the anchor is built
      tc::bar_expect_tx(bar_wk, S::kW);
      tc::bulk_g2s(sW, wblock(0, 0, 0), S::kW, bar_wk);
      tc::bar_expect_tx(bar_wp, S::kW);
      tc::bulk_g2s(sWp, wblock(0, 1, 0), S::kW, bar_wp);
    }
  }
  if (warp == 0) tc::alloc(tslot, S::tmem_cols);
  if (warp == 1) {
    // inclusive scan of log alpha over the chunk
    float run = 0.f;
    for (int base = 0; base < C; base += 32) {
      const int i = base + lane;
      float x = 0.f;
      if (i < nv) x = p.log_alpha[((size_t)b * T_ + t0 + i) * H + h];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      x += run;
      run = __shfl_sync(0xffffffffu, x, 31);
      if (i < C) sg[i] = x;
    }
    __syncwarp();
    for (int i = lane; i < C; i += 32) sdec[i] = expf(sg[C - 1] - sg[i]);
  }
  // [K ; Q] rows as fp16: (row, a) at (a/8)*2048 + row*16 + (a%8)*2, and the v window,
  // rows t0-w .. t0+C-1 as bf16 [C + w][D] (zero outside [0, len)), in the D tiles.
  // All global loads are issued before any is used.
  __nv_bfloat16* vwin = reinterpret_cast<__nv_bfloat16*>(sD);
  {
    constexpr int NKQ = (128 * (D / 8) + 255) / 256;
    constexpr int NVW = ((C + 8) * (D / 8) + 255) / 256;
    uint4 kq[NKQ], vw[NVW];
#pragma unroll
    for (int i = 0; i < NKQ; ++i) {
      const int idx = tid + i * 256, r = idx % 128, a8 = idx / 128;
      const int t = r < C ? r : r - C;
      kq[i] = make_uint4(0u, 0u, 0u, 0u);
      if (idx < 128 * (D / 8) && r < 2 * C && t < nv)
        kq[i] = *reinterpret_cast<const uint4*>((r < C ? p.k : p.q) + (((size_t)b * T_ + t0 + t) * H + h) * D + a8 * 8);
    }
#pragma unroll
    for (int i = 0; i < NVW; ++i) {
      const int idx = tid + i * 256, rr = idx / (D / 8), c8 = idx % (D / 8);
      const int t = t0 - w + rr;
      vw[i] = make_uint4(0u, 0u, 0u, 0u);
      if (rr < C + w && t >= 0 && t < len)
        vw[i] = *reinterpret_cast<const uint4*>(p.v + (((size_t)b * T_ + t) * H + h) * D + c8 * 8);
    }
#pragma unroll
    for (int i = 0; i < NKQ; ++i) {
      const int idx = tid + i * 256, r = idx % 128, a8 = idx / 128;
      if (idx < 128 * (D / 8)) {
        const __nv_bfloat16* e = reinterpret_cast<const __nv_bfloat16*>(&kq[i]);
        __half hv[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) hv[j] = __float2half_rn(__bfloat162float(e[j]));
        *reinterpret_cast<uint4*>(sKQ + a8 * 2048u + r * 16u) = *reinterpret_cast<const uint4*>(hv);
      }
    }
#pragma unroll
    for (int i = 0; i < NVW; ++i) {
      const int idx = tid + i * 256, rr = idx / (D / 8), c8 = idx % (D / 8);
      if (rr < C + w) *reinterpret_cast<uint4*>(vwin + rr * D + c8 * 8) = vw[i];
    }
  }
  // rows D..127 of the scaled-write tiles stay zero (A operand of the injection)
  if constexpr (D < 128)
    for (int idx = tid; idx < (128 - D) * (C / 8) * 2; idx += 256) {
      const int part = idx / ((128 - D) * (C / 8));
      const int rem = idx % ((128 - D) * (C / 8));
      const int r = D + rem % (128 - D), s8 = rem / (128 - D);
      *reinterpret_cast<uint4*>(sDt + part * S::kF128 + s8 * 2048u + r * 16u) = make_uint4(0u, 0u, 0u, 0u);
    }
  tc::fence_before();
  __syncthreads();

  tc::fence_after();
  const uint32_t tmem = *tslot;
  const uint32_t t_proj = tmem, t_p = tmem + C, t_ro = tmem + 2 * C, t_n = tmem + 2 * C + D;
  const uint32_t t_r = tmem + 2 * C + 2 * D, t_u = t_r + C;   // residual r and anchor u
  const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;

  // ---- anchor u = sum_j c_j (.) v_{t-j} and residual r = v - u, kept in TMEM ----
  // thread (feature c = row, token half) owns tokens [half*NTH, half*NTH + NTH)
  const int c = row;
  const bool cvalid = c < D;
  {
    float taps[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) taps[j] = (cvalid && j < w) ? p.conv_w[((size_t)h * w + j) * D + c] : 0.f;
#pragma unroll 1
    for (int j8 = 0; j8 < NTH; j8 += 8) {
      float uu[8], rr[8];
      __half uh[8], ul[8];
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) {
        const int tl = half * NTH + j8 + jj;
        float u = 0.f, vt = 0.f;
        if (cvalid) {
#pragma unroll
          for (int j = 1; j <= 8; ++j)
            if (j <= w) u = fmaf(taps[j - 1], __bfloat162float(vwin[(tl + w - j) * D + c]), u);
          vt = __bfloat162float(vwin[(tl + w) * D + c]);
        }
        uu[jj] = u;
        rr[jj] = (tl < nv) ? vt - u : 0.f;
        tc::split_f16(u, uh[jj], ul[jj]);
        if (cvalid) {
          // U tile (B operand, N = tokens, K = features): (t, c) at (c/8)*(C*16) + t*16 + (c%8)*2
          const uint32_t off = (c / 8) * (C * 16u) + tl * 16u + (c % 8) * 2u;
          *reinterpret_cast<__half*>(sU + off) = uh[jj];
          *reinterpret_cast<__half*>(sU + S::kU + off) = ul[jj];
        }
      }
      tc::st8(t_u + lane_base + half * NTH + j8, uu);
      tc::st8(t_r + lane_base + half * NTH + j8, rr);
    }
  }
  tc::fence_smem_to_async();
  tc::fence_before();
  __syncthreads();
  tc::fence_after();

  uint32_t ph_mma = 0, ph_wk = 0, ph_wp = 0;
  bool ok = true;
  auto wait_mma = [&]() {
    ok &= tc::bar_wait(bar_mma, ph_mma & 1);
    ++ph_mma;
    tc::fence_after();
  };
  auto wait_bar = [&](uint64_t* bar, uint32_t& ph) {
    ok &= tc::bar_wait(bar, ph & 1);
    ++ph;
  };

  constexpr uint32_t idesc_proj = tc::idesc_f16(C, false, false);
  constexpr uint32_t idesc_gp = tc::idesc_f16(C, false, true);
  constexpr uint32_t idesc_dd = tc::idesc_f16(D, false, false);
  constexpr uint32_t S_s = (D / 8) * 128;      // token step of the feature x token tiles
  const bool gelu = !(p.flags & 1u);
  float* spart = reinterpret_cast<float*>(sGP);  // per-warp partial sums during [3]

  for (int l = 0; l < L; ++l) {
    // [1] W_p^(l) into the [G;P] buffers once the previous step's MMAs are done
    //     (W_k^(l) was requested as soon as the previous projection finished)
    if (l > 0) {
      wait_mma();
      if (tid == 0) {
        tc::bar_expect_tx(bar_wp, S::kW);
        tc::bulk_g2s(sWp, wblock(l, 1, 0), S::kW, bar_wp);
      }
    }
    wait_bar(bar_wk, ph_wk);
    wait_bar(bar_wp, ph_wp);
    // [2] projections: k_hat^T = W_k u^T, p^T = W_p u^T (u = hi + lo)
    if (tid == 0) {
      tc::fence_after();
      for (int pass = 0; pass < 2; ++pass)
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t bdesc = tc::desc(sU + pass * S::kU + kk * 2 * C * 16, C * 16, 128);
          const bool acc = pass > 0 || kk > 0;
          tc::mma(t_proj, tc::desc(sW + kk * 4096, 2048, 128), bdesc, idesc_proj, acc);
          tc::mma(t_p, tc::desc(sWp + kk * 4096, 2048, 128), bdesc, idesc_proj, acc);
        }
      tc::commit(bar_mma);
    }
    if (need_lo) {       // weights not exact in fp16: add W_lo u_hi
      wait_mma();
      if (tid == 0) {
        tc::bar_expect_tx(bar_wk, S::kW);
        tc::bulk_g2s(sW, wblock(l, 0, 1), S::kW, bar_wk);
        tc::bar_expect_tx(bar_wp, S::kW);
        tc::bulk_g2s(sWp, wblock(l, 1, 1), S::kW, bar_wp);
      }
      wait_bar(bar_wk, ph_wk);
      wait_bar(bar_wp, ph_wp);
      if (tid == 0) {
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t bdesc = tc::desc(sU + kk * 2 * C * 16, C * 16, 128);
          tc::mma(t_proj, tc::desc(sW + kk * 4096, 2048, 128), bdesc, idesc_proj, true);
          tc::mma(t_p, tc::desc(sWp + kk * 4096, 2048, 128), bdesc, idesc_proj, true);
        }
        tc::commit(bar_mma);
      }
    }
    wait_mma();
    // the projection has read W_k^(l): stream W_k^(l+1) in behind the epilogues
    if (tid == 0 && l + 1 < L) {
      tc::bar_expect_tx(bar_wk, S::kW);
      tc::bulk_g2s(sW, wblock(l + 1, 0, 0), S::kW, bar_wk);
    }
    // [3] epilogue.  Pass A: per token |k_hat|^2 and the gate logit w_beta . u,
    //     summed over this warp's 32 features (reduce-scatter over 8-token groups).
    {
      const float wb = cvalid ? p.wbeta[((size_t)h * L + l) * D + c] : 0.f;
#pragma unroll 1
      for (int j8 = 0; j8 < NTH; j8 += 8) {
        float kv[8], uv[8], rn[8], rz[8];
        tc::ld8(t_proj + lane_base + half * NTH + j8, kv);
        tc::ld8(t_u + lane_base + half * NTH + j8, uv);
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
          rn[jj] = cvalid ? kv[jj] * kv[jj] : 0.f;
          rz[jj] = wb * uv[jj];
        }
        int n = 8;
#pragma unroll
        for (int m = 16; m >= 1; m >>= 1) {
          if (n > 1) {
            const int hn = n / 2;
            const bool upper = lane & m;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              if (j < hn) {
                const float sn = upper ? rn[j] : rn[j + hn], kn = upper ? rn[j + hn] : rn[j];
                const float sz = upper ? rz[j] : rz[j + hn], kz = upper ? rz[j + hn] : rz[j];
                rn[j] = kn + __shfl_xor_sync(0xffffffffu, sn, m);
                rz[j] = kz + __shfl_xor_sync(0xffffffffu, sz, m);
              }
            }
            n = hn;
          } else {
            rn[0] += __shfl_xor_sync(0xffffffffu, rn[0], m);
            rz[0] += __shfl_xor_sync(0xffffffffu, rz[0], m);
          }
        }
        if ((lane & 3) == 0) {                  // lane holds token j8 + lane/4 of its half
          const int t = half * NTH + j8 + (lane >> 2);
          spart[quarter * C + t] = rn[0];
          spart[4 * C + quarter * C + t] = rz[0];
        }
      }
      __syncthreads();
      if (tid < C) {
        const float ss = spart[tid] + spart[C + tid] + spart[2 * C + tid] + spart[3 * C + tid];
        const float zz = spart[4 * C + tid] + spart[5 * C + tid] + spart[6 * C + tid] + spart[7 * C + tid];
        sinv[tid] = 1.0f / sqrtf(ss + 1e-6f);
        sbl[tid] = sigmoidf(zz);
      }
      __syncthreads();
      // Pass B: directions, residual step, factor tiles
#pragma unroll 1
      for (int j8 = 0; j8 < NTH; j8 += 8) {
        float kv[8], pv[8], rr[8];
        tc::ld8(t_proj + lane_base + half * NTH + j8, kv);
        tc::ld8(t_p + lane_base + half * NTH + j8, pv);
        tc::ld8(t_r + lane_base + half * NTH + j8, rr);
        __half kh[8], kl[8], dh[8], dlo[8], th[8], tl[8];
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
          const int t = half * NTH + j8 + jj;
          const bool valid = cvalid && t < nv;
          const float kd = valid ? kv[jj] * sinv[t] : 0.f;
          const float x = pv[jj] * rr[jj];
          const float dl = gelu ? gelu_erf(x) : x;
          rr[jj] -= dl;
          const float dval = valid ? sbl[t] * dl : 0.f;
          tc::split_f16(kd, kh[jj], kl[jj]);
          tc::split_f16(dval, dh[jj], dlo[jj]);
          tc::split_f16(dval * sdec[t], th[jj], tl[jj]);
        }
        tc::st8(t_r + lane_base + half * NTH + j8, rr);
        if (cvalid) {
          // feature x token tiles: (f, s) at (s/8)*S_s + f*16 + (s%8)*2  (f < D)
          const uint32_t off = ((half * NTH + j8) / 8) * S_s + c * 16u;
          *reinterpret_cast<uint4*>(sKl + off) = *reinterpret_cast<const uint4*>(kh);
          *reinterpret_cast<uint4*>(sKl + S::kF + off) = *reinterpret_cast<const uint4*>(kl);
          *reinterpret_cast<uint4*>(sD + off) = *reinterpret_cast<const uint4*>(dh);
          *reinterpret_cast<uint4*>(sD + S::kF + off) = *reinterpret_cast<const uint4*>(dlo);
          const uint32_t off128 = ((half * NTH + j8) / 8) * 2048u + c * 16u;
          *reinterpret_cast<uint4*>(sDt + off128) = *reinterpret_cast<const uint4*>(th);
          *reinterpret_cast<uint4*>(sDt + S::kF128 + off128) = *reinterpret_cast<const uint4*>(tl);
        }
      }
    }
    tc::fence_smem_to_async();
    tc::fence_before();
    __syncthreads();
    // [4] scores [G ; P] = [K ; Q] K_l^T   (K_l = hi + lo, MN-major B)
    if (tid == 0) {
      tc::fence_after();
      for (int pass = 0; pass < 2; ++pass)
        for (int kk = 0; kk < D / 16; ++kk)
          tc::mma(t_proj, tc::desc(sKQ + kk * 4096, 2048, 128),
                  tc::desc(sKl + pass * S::kF + kk * 256, 128, S_s), idesc_gp, pass > 0 || kk > 0);
      tc::commit(bar_mma);
    }
    wait_mma();
    // [5] epilogue: decay + causal masks; rows < C are G (strict), C..2C-1 are P (inclusive)
    {
      const bool isG = row < C, isP = row >= C && row < 2 * C;
      const int t = isG ? row : row - C;
      const float gt = (isG || isP) ? sg[t] : 0.f;
#pragma unroll 1
      for (int j8 = 0; j8 < NTH; j8 += 8) {
        float tmp[8];
        tc::ld8(t_proj + lane_base + half * NTH + j8, tmp);
        __half hh[8], ll[8];
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
          const int s_ = half * NTH + j8 + jj;
          float val = 0.f;
          if ((isG && t > s_) || (isP && t >= s_)) val = expf(gt - sg[s_]) * tmp[jj];
          if (isP) {
            tc::split_f16(val, hh[jj], ll[jj]);
          } else {
            hh[jj] = __float2half_rn(val);
            ll[jj] = __float2half_rn(0.f);
          }
        }
        const uint32_t off = ((half * NTH + j8) / 8) * 2048u + row * 16u;
        *reinterpret_cast<uint4*>(sGP + off) = *reinterpret_cast<const uint4*>(hh);
        *reinterpret_cast<uint4*>(sGP + S::kF128 + off) = *reinterpret_cast<const uint4*>(ll);
      }
    }
    tc::fence_smem_to_async();
    tc::fence_before();
    __syncthreads();
    // [6] [R ; O_l] += [G ; P] D_l  and  N_l += Dt_l^T K_l   (3 passes each)
    if (tid == 0) {
      tc::fence_after();
      const int ap[3] = {0, 0, 1}, bp[3] = {0, 1, 0};
      for (int ps = 0; ps < 3; ++ps)
        for (int kk = 0; kk < C / 16; ++kk) {
          const bool acc = l > 0 || ps > 0 || kk > 0;
          tc::mma(t_ro, tc::desc(sGP + ap[ps] * S::kF128 + kk * 4096, 2048, 128),
                  tc::desc(sD + bp[ps] * S::kF + kk * 2 * S_s, S_s, 128), idesc_dd, acc);
          tc::mma(t_n, tc::desc(sDt + ap[ps] * S::kF128 + kk * 4096, 2048, 128),
                  tc::desc(sKl + bp[ps] * S::kF + kk * 2 * S_s, S_s, 128), idesc_dd, acc);
        }
      tc::commit(bar_mma);
    }
  }
  if (L > 0) wait_mma();

  // ================= tail: gated delta rule, state-independent part =================
  const size_t cbase = ((size_t)b * H + h) * NC + chunk;
  float* tAf = reinterpret_cast<float*>(sm + S::tA);
  float* tPf = reinterpret_cast<float*>(sm + S::tP);
  float* tTf = reinterpret_cast<float*>(sm + S::tT);
  float* tYf = reinterpret_cast<float*>(sm + S::tY);
  float* tbeta = reinterpret_cast<float*>(sm + S::tB);
  float* tgam = tbeta + C;
  unsigned char* sTP = sm + S::tTP;
  unsigned char* sKX = sm + S::tKX;
  unsigned char* sTB = sm + S::tTB;
  const uint32_t t_w = t_n;                                     // W / PW columns
  const uint32_t t_x = S::kExtraX ? tmem + 2 * C + 2 * D : tmem; // U / PU columns
  const int s_tok = row;
  const bool tok = s_tok < C;
  const bool tok_valid = tok && s_tok < nv;
  // (a) N = N_l to global (its TMEM columns are reused below)
  if (L > 0) {
    float* nbase = p.Nl + cbase * D * D;      // piece-major: (c, a) at ((a/4)*D + c)*4 + a%4
#pragma unroll 1
    for (int j8 = 0; j8 < D / 2; j8 += 8) {
      float tmp[8];
      tc::ld8(t_n + lane_base + half * (D / 2) + j8, tmp);
      if (cvalid) {
        const int a0 = half * (D / 2) + j8;
        *reinterpret_cast<float4*>(nbase + ((size_t)(a0 / 4) * D + row) * 4) = make_float4(tmp[0], tmp[1], tmp[2], tmp[3]);
        *reinterpret_cast<float4*>(nbase + ((size_t)(a0 / 4 + 1) * D + row) * 4) = make_float4(tmp[4], tmp[5], tmp[6], tmp[7]);
      }
    }
  }
  for (int i = tid; i < C; i += 256) {
    tbeta[i] = i < nv ? p.beta[((size_t)b * T_ + t0 + i) * H + h] : 0.f;
    tgam[i] = expf(sg[i]);
  }
  tc::fence_before();
  __syncthreads();
  // (b) [K K^T ; Q K^T] = [K ; Q] K^T   (B = the K rows of the same tile, K-major)
  if (tid == 0) {
    tc::fence_after();
    for (int kk = 0; kk < D / 16; ++kk)
      tc::mma(t_proj, tc::desc(sKQ + kk * 4096, 2048, 128), tc::desc(sKQ + kk * 4096, 2048, 128),
              idesc_proj, kk > 0);
    tc::commit(bar_mma);
  }
  // (d) meanwhile: X = beta (V - R) and Kb = beta gamma K as the MN-major B tile [Kb | X]:
  //     (s, f) at (f/8)*(16C) + s*16 + (f%8)*2,  f < D: Kb,  f >= D: X
  {
    const float bs = tok ? tbeta[s_tok] : 0.f, gs = tok ? tgam[s_tok] : 0.f;
#pragma unroll 1
    for (int j8 = 0; j8 < D / 2; j8 += 8) {
      const int f0 = half * (D / 2) + j8;
      float rr[8];
      if (L > 0) {
        tc::ld8(t_ro + lane_base + f0, rr);
      } else {
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) rr[jj] = 0.f;
      }
      if (tok) {
        __half xh[8], kh[8];
        uint4 vraw = make_uint4(0u, 0u, 0u, 0u);
        if (tok_valid) vraw = *reinterpret_cast<const uint4*>(p.v + (((size_t)b * T_ + t0 + s_tok) * H + h) * D + f0);
        const __nv_bfloat16* ve = reinterpret_cast<const __nv_bfloat16*>(&vraw);
        const uint4 kraw = *reinterpret_cast<const uint4*>(sKQ + (f0 / 8) * 2048u + s_tok * 16u);
        const __half* ke = reinterpret_cast<const __half*>(&kraw);
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
          xh[jj] = __float2half_rn(tok_valid ? bs * (__bfloat162float(ve[jj]) - rr[jj]) : 0.f);
          kh[jj] = __float2half_rn(bs * gs * __half2float(ke[jj]));
        }
        *reinterpret_cast<uint4*>(sKX + ((D + f0) / 8) * (16u * C) + s_tok * 16u) = *reinterpret_cast<const uint4*>(xh);
        *reinterpret_cast<uint4*>(sKX + (f0 / 8) * (16u * C) + s_tok * 16u) = *reinterpret_cast<const uint4*>(kh);
      }
    }
  }
  wait_mma();
  // (c) A = strict_tril(beta (K K^T) (.) Gamma), P = tril(Q K^T (.) Gamma)   (fp32)
  {
    const bool isA = row < C, isP = row >= C && row < 2 * C;
    const int t = isA ? row : row - C;
#pragma unroll 1
    for (int j8 = 0; j8 < NTH; j8 += 8) {
      float tmp[8];
      tc::ld8(t_proj + lane_base + half * NTH + j8, tmp);
      if (isA || isP) {
        const float gt = sg[t];
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
          const int s_ = half * NTH + j8 + jj;
          if (isA) tAf[t * (C + 1) + s_] = (t > s_) ? tbeta[t] * expf(gt - sg[s_]) * tmp[jj] : 0.f;
          else     tPf[t * (C + 1) + s_] = (t >= s_) ? expf(gt - sg[s_]) * tmp[jj] : 0.f;
        }
      }
    }
  }
  __syncthreads();
  // (e) T = (I + A)^-1 (fp32); then [T ; PT] = [I ; P] T on the tensor core
  solve_tri<C>(tAf, tTf, tYf);
  // A tile [I ; P] (fp16, 128 x C, K-major (r, s) at (s/8)*2048 + r*16 + (s%8)*2), rows >= 2C zero;
  // B tile T (N = j, K = m): (j, m) at (m/8)*(16C) + j*16 + (m%8)*2
  for (int idx = tid; idx < 128 * (C / 8); idx += 256) {
    const int r = idx % 128, s8 = idx / 128;
    __half hv[8];
#pragma unroll
    for (int jj = 0; jj < 8; ++jj) {
      const int j = s8 * 8 + jj;
      float x = 0.f;
      if (r < C) x = (r == j) ? 1.f : 0.f;
      else if (r < 2 * C) x = tPf[(r - C) * (C + 1) + j];
      hv[jj] = __float2half_rn(x);
    }
    *reinterpret_cast<uint4*>(sTP + s8 * 2048u + r * 16u) = *reinterpret_cast<const uint4*>(hv);
  }
  for (int idx = tid; idx < C * (C / 8); idx += 256) {
    const int j = idx % C, m8 = idx / C;
    __half hv[8];
#pragma unroll
    for (int jj = 0; jj < 8; ++jj) hv[jj] = __float2half_rn(tTf[(m8 * 8 + jj) * (C + 1) + j]);
    *reinterpret_cast<uint4*>(sTB + m8 * (16u * C) + j * 16u) = *reinterpret_cast<const uint4*>(hv);
  }
  tc::fence_smem_to_async();
  tc::fence_before();
  __syncthreads();
  if (tid == 0) {
    tc::fence_after();
    for (int kk = 0; kk < C / 16; ++kk)
      tc::mma(t_proj, tc::desc(sTP + kk * 4096, 2048, 128), tc::desc(sTB + kk * 2 * 16 * C, 16 * C, 128),
              idesc_proj, kk > 0);
    tc::commit(bar_mma);
  }
  wait_mma();
  // [T ; PT] back into the A tile (fp16)
#pragma unroll 1
  for (int j8 = 0; j8 < NTH; j8 += 8) {
    float tmp[8];
    tc::ld8(t_proj + lane_base + half * NTH + j8, tmp);
    __half hv[8];
#pragma unroll
    for (int jj = 0; jj < 8; ++jj) hv[jj] = __float2half_rn(tmp[jj]);
    *reinterpret_cast<uint4*>(sTP + ((half * NTH + j8) / 8) * 2048u + row * 16u) = *reinterpret_cast<const uint4*>(hv);
  }
  tc::fence_smem_to_async();
  tc::fence_before();
  __syncthreads();
  // (f) [W ; PW] = [T ; PT] Kb,  [U ; PU] = [T ; PT] X   (B MN-major: LBO = 128, SBO = 16C)
  if (tid == 0) {
    tc::fence_after();
    constexpr uint32_t idesc_tx = tc::idesc_f16(D, false, true);
    for (int kk = 0; kk < C / 16; ++kk) {
      const uint64_t adesc = tc::desc(sTP + kk * 4096, 2048, 128);
      tc::mma(t_w, adesc, tc::desc(sKX + kk * 256, 128, 16 * C), idesc_tx, kk > 0);
      tc::mma(t_x, adesc, tc::desc(sKX + (D / 8) * (16 * C) + kk * 256, 128, 16 * C), idesc_tx, kk > 0);
    }
    tc::commit(bar_mma);
  }
  wait_mma();
  // (g) outputs.  Lanes 0..C-1: W (fp16), U (fp32), Kt (fp16).  Lanes C..2C-1:
  //     Qt = gamma Q - PW (fp16 hi/lo), O_intra = PU + O_l (fp32).
  {
    const bool isT = row < C, isPT = row >= C && row < 2 * C;
    const int t = isT ? row : row - C;
    const size_t cb = cbase * C * D;         // piece-major chunk base
    const int tr = (isT || isPT) ? t : 0;
    const float gt = (isT || isPT) ? tgam[t] : 0.f;
    const float dct = (isT || isPT) ? sdec[t] : 0.f;
#pragma unroll 1
    for (int j8 = 0; j8 < D / 2; j8 += 8) {
      const int f0 = half * (D / 2) + j8;
      float wv[8], xv[8], ov[8];
      tc::ld8(t_w + lane_base + f0, wv);
      tc::ld8(t_x + lane_base + f0, xv);
      if (L > 0) {
        tc::ld8(t_ro + lane_base + f0, ov);
      } else {
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) ov[jj] = 0.f;
      }
      if (isT) {
        __half wh[8], kth[8];
        const uint4 kraw = *reinterpret_cast<const uint4*>(sKQ + (f0 / 8) * 2048u + t * 16u);
        const __half* ke = reinterpret_cast<const __half*>(&kraw);
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
          wh[jj] = __float2half_rn(wv[jj]);
          kth[jj] = __float2half_rn(dct * __half2float(ke[jj]));
        }
        const size_t o16 = cb + ((size_t)(f0 / 8) * C + tr) * 8;     // fp16 piece (8 values)
        *reinterpret_cast<uint4*>(p.Wc + o16) = *reinterpret_cast<const uint4*>(wh);
        *reinterpret_cast<uint4*>(p.Kt + o16) = *reinterpret_cast<const uint4*>(kth);
        *reinterpret_cast<float4*>(p.U + cb + ((size_t)(f0 / 4) * C + tr) * 4) = make_float4(xv[0], xv[1], xv[2], xv[3]);
        *reinterpret_cast<float4*>(p.U + cb + ((size_t)(f0 / 4 + 1) * C + tr) * 4) = make_float4(xv[4], xv[5], xv[6], xv[7]);
      } else if (isPT) {
        __half qh[8], ql[8];
        const uint4 qraw = *reinterpret_cast<const uint4*>(sKQ + (f0 / 8) * 2048u + row * 16u);
        const __half* qe = reinterpret_cast<const __half*>(&qraw);
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) tc::split_f16(gt * __half2float(qe[jj]) - wv[jj], qh[jj], ql[jj]);
        const size_t o16 = cb + ((size_t)(f0 / 8) * C + tr) * 8;
        *reinterpret_cast<uint4*>(p.Qth + o16) = *reinterpret_cast<const uint4*>(qh);
        *reinterpret_cast<uint4*>(p.Qtl + o16) = *reinterpret_cast<const uint4*>(ql);
        *reinterpret_cast<float4*>(p.Oi + cb + ((size_t)(f0 / 4) * C + tr) * 4) =
            make_float4(xv[0] + ov[0], xv[1] + ov[1], xv[2] + ov[2], xv[3] + ov[3]);
        *reinterpret_cast<float4*>(p.Oi + cb + ((size_t)(f0 / 4 + 1) * C + tr) * 4) =
            make_float4(xv[4] + ov[4], xv[5] + ov[5], xv[6] + ov[6], xv[7] + ov[7]);
      }
    }
    if (tid == 0) p.gC[cbase] = tgam[C - 1];
  }
  if (!ok && lane == 0) atomicExch(p.status, 1);
  tc::fence_before();
  __syncthreads();
  if (warp == 0) tc::dealloc(tmem, S::tmem_cols);
}

}  // namespace prism
