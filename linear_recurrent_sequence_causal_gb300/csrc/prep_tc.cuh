// Kernel A (bf16 I/O path): anchor + refinement + the chunk's rank-L write
// summaries, on tcgen05 tensor cores.  ("Technical Summary: PRISM", §2.2
// stages 1-2 and the injection B_t = sum_l beta^(l) delta^(l) k^(l)^T.)
//
// Everything here is state-independent, so it runs fully parallel over chunks.  The
// kernel is persistent: one CTA per SM walks the chunks (b, h, chunk) with a stride of
// the grid size; while a chunk's tail runs, the next chunk's K, Q and v tiles are
// already being copied in and its gates loaded, so a chunk starts without waiting on
// memory.  For the chunk's C tokens it computes the anchor u, the
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

#include <cuda.h>

#include "prism_common.cuh"
#include "tc_common.cuh"

namespace prism {

struct PrepArgs {
  // TMA maps of q, k, v as 4-D bf16 tensors (d, H, T, B); boxes of (d, 1, C, 1) rows for
  // q and k and (d, 1, C + 8, 1) for the v window.
  CUtensorMap tm_q, tm_k, tm_v;
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
  const __nv_bfloat16* vhist;     // [B][H][w][D] (or [B][w][H][D] with flag bit 1) v of the w tokens
                                  // before t = 0 (oldest first), or null
  // Per-chunk outputs, chunk-major [B][H][NC][...].  Inside a chunk each array is
  // stored "piece-major": 16-byte column pieces, rows contiguous within a piece:
  // element (r, f) of an R-row array at ((f / V) * R + r) * V + f % V, V = 16 / elem
  // size.  A warp whose lanes hold consecutive rows then writes 512 contiguous bytes.
  // Two fp16 maps share each piece: WQ holds, per 8-feature piece, the C rows of W
  // then the C rows of Qt_hi ([D/8][2][C][8]); QK the rows of Qt_lo then of Kt.
  //   W  = T diag(beta gamma) K,   Qt = diag(gamma) Q - P W (hi + lo),
  //   Kt = diag(gamma_C / gamma) K
  __half* WQ;                     // [D/8][2][C][8]
  __half* QK;                     // [D/8][2][C][8]
  float* U;                       // [C][D]  U = T diag(beta) (V - R)
  float* Oi;                      // [C][D]  O_intra = P U + O_l
  float* Nt;                      // [D][D]  N^T (d_k x d_v), piece-major over d_v
  float* gC;                      // [1]     gamma_C
  int* status;                    // device error word (bounded waits)
  int* bounds;                    // debug build: word of out-of-bounds accesses (else null)
};

// One weight block: 128 rows (features, zero beyond D) x D columns, fp16,
// K-major with SBO = 128 and LBO = 2048:  (row, c) at (c/8)*2048 + row*16 + (c%8)*2.
template <int D>
struct WeightBlock {
  static constexpr uint32_t bytes = 128u * D * 2u;
  // the conversion kernel: threads of 8 columns, 256 per CTA, kCtas CTAs per block
  static constexpr int kPieces = D / 8, kRowsPerCta = 256 / kPieces, kCtas = 128 / kRowsPerCta;
  // block index of (h, l, which = 0 W_k / 1 W_p, part = 0 hi / 1 lo)
  static __host__ __device__ size_t index(int h, int l, int L, int which, int part) {
    return (((size_t)h * L + l) * 2 + which) * 2 + part;
  }
};

// Converts W_k, W_p (fp32 [H][L][D][D]) into fp16 hi/lo blocks; sets *flag if
// any lo half is significant (|lo| > 2^-22 of its row norm), in which case the
// projections take a third pass with the lo halves.  For 32 <= d < 128 the D rows repeat
// down the block's 128 rows, so the projections land in every TMEM lane quarter (the
// epilogue spreads a chunk's tokens over the copies).
template <int D>
__global__ void __launch_bounds__(256) prep_weights_kernel(const float* Wk, const float* Wp, int H, int L,
                                                           unsigned char* blocks, int* flag) {
  // thread = (row of the block, 8-column piece): two 16-byte loads of the row, one 16-byte
  // store each of hi and lo; the row's P threads are consecutive lanes of one warp
  constexpr int P = WeightBlock<D>::kPieces, ROWS = WeightBlock<D>::kRowsPerCta;
  const int blk = blockIdx.x / WeightBlock<D>::kCtas;   // (h*L + l)*2 + which
  const int row = (blockIdx.x % WeightBlock<D>::kCtas) * ROWS + threadIdx.x / P, c8 = threadIdx.x % P;
  const int which = blk & 1, hl = blk >> 1;
  const float* W = (which == 0 ? Wk : Wp) + (size_t)hl * D * D;
  unsigned char* hi = blocks + (size_t)(blk * 2 + 0) * WeightBlock<D>::bytes;
  unsigned char* lo = blocks + (size_t)(blk * 2 + 1) * WeightBlock<D>::bytes;
  const bool live = D >= 32 || row < D;        // d = 16: one copy (rows 16..127 zero)
  float x[8];
  if (live) {
    const float4* src = reinterpret_cast<const float4*>(W + (size_t)(row % D) * D + c8 * 8);
    const float4 a = src[0], b = src[1];
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w; x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
  } else {
#pragma unroll
    for (int j = 0; j < 8; ++j) x[j] = 0.f;
  }
  float n2 = 0.f;
#pragma unroll
  for (int j = 0; j < 8; ++j) n2 = fmaf(x[j], x[j], n2);
#pragma unroll
  for (int o = P / 2; o > 0; o >>= 1) n2 += __shfl_xor_sync(0xffffffffu, n2, o);
  const float tol = sqrtf(n2) * 0x1p-22f;
  uint4 h, l;
  tc::split8(x, h, l);
  const uint32_t off = c8 * 2048u + row * 16u;
  *reinterpret_cast<uint4*>(hi + off) = h;
  *reinterpret_cast<uint4*>(lo + off) = l;
  const uint32_t lw[4] = {l.x, l.y, l.z, l.w};
  bool need = false;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    __half2 lh;
    memcpy(&lh, &lw[j], 4);
    const float2 lf = __half22float2(lh);
    need |= fabsf(lf.x) > tol || fabsf(lf.y) > tol;
  }
  if (__any_sync(0xffffffffu, need) && (threadIdx.x & 31) == 0) atomicOr(flag, 1);
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
  // Consumer threads: 4 warps per TMEM lane quarter when the column counts allow it;
  // warp w reads lane quarter w % 4 and column group w / 4 of every TMEM tile.  One more
  // warp (the producer) issues the tile copies and the MMAs of the refinement loop.
  // column groups; at d <= 32 one lane quarter holds every feature, so two column groups (8
  // consumer warps) keep the rest of the CTA small enough for two CTAs per SM
  static constexpr int CG = (D <= 32 && C <= 32) ? 2 : (C % 32 == 0 && D % 32 == 0) ? 4 : 2;
  static constexpr int NW = 4 * CG;                      // consumer warps
  static constexpr int NT = 32 * NW;                     // consumer threads
  static constexpr int NTA = NT + 32;                    // all threads (with the producer warp)
  static constexpr int NTH = C / CG;                     // token columns per thread
  // Feature role (anchor, passes A and B): the projections arrive RF times over in TMEM
  // (the weight rows repeat), in whole lane quarters when d >= 32, so replica rf of a
  // feature takes NTF = C / (CG RF) of its column group's tokens (at least 8).
  static constexpr int NQF = D >= 32 ? D / 32 : 1;       // lane quarters per replica
  static constexpr int RF = (D >= 32 && D < 128) ? (128 / D < C / (8 * CG) ? 128 / D : C / (8 * CG)) : 1;
  static constexpr int NTF = C / (CG * RF);
  static constexpr int NFD = D / CG;                     // feature columns per thread
  static constexpr int NQ = (D + 31) / 32;               // lane quarters that hold features
  static constexpr uint32_t kW = WeightBlock<D>::bytes;  // 128 x D
  static constexpr uint32_t kU = C * D * 2;              // tokens x D
  static constexpr uint32_t kKQ = 128 * D * 2;           // 128 rows x D
  static constexpr uint32_t kF = D * C * 2;              // features x tokens
  static constexpr uint32_t kF128 = 128 * C * 2;         // 128 rows x tokens
  static constexpr uint32_t kX = kW > 2 * kF128 ? kW : 2 * kF128;   // W_k, or the [G;P] hi/lo tiles
  // small arrays first
  static constexpr uint32_t oG = 0;                      // f32 g[C]
  static constexpr uint32_t oDec = oG + 4 * C;           // f32 gamma_C/gamma [C]
  static constexpr uint32_t oBeta = oDec + 4 * C;        // f32 beta^(l) [C] (0 past the sequence end)
  static constexpr uint32_t oInv = oBeta + 4 * C;        // f32 1/|k_hat| [C] (0 past the sequence end)
  static constexpr uint32_t oPart = oInv + 4 * C;        // f32 per-quarter partial sums, quarters 1..3:
                                                         //   [3][2][C] (|k_hat|^2, w_beta . u)
  static constexpr uint32_t oBtok = oPart + 24 * C;      // f32 beta_t [C] (0 past the sequence end)
  static constexpr int kBars = 14;
  static constexpr uint32_t oBar = oBtok + 4 * C;        // mbarriers
  static constexpr uint32_t oSlot = oBar + 8 * kBars;
  static constexpr uint32_t oTiles = ((oSlot + 8 + 127) / 128) * 128;
  // refinement-loop tiles
  static constexpr uint32_t oX = oTiles;                 // W_k^(l+1) / [G;P]_l hi, lo
  static constexpr uint32_t oY = oX + kX;                // W_p
  static constexpr uint32_t oU = oY + kW;                // u hi, lo
  static constexpr uint32_t oKQ = oU + 2 * kU;
  static constexpr uint32_t oKl = oKQ + kKQ;             // hi, lo
  static constexpr uint32_t oD = oKl + 2 * kF;           // hi, lo
  static constexpr uint32_t oDt = oD + 2 * kF;           // hi, lo (128 rows)
  static constexpr uint32_t loop_end = oDt + 2 * kF128;
  // tail buffers (after the loop), placed around the [K;Q] tile which stays live
  static constexpr uint32_t sKX = 4 * C * D, sSq = 4 * C * (C + 4), sB = 8 * C;
  static constexpr uint32_t sZ = 4 * 32 * 36;            // block-solve scratch
  static constexpr uint32_t sTB = 2 * C * C;             // f16 T as B operand (C x C)
  // The solve's buffers go where the refinement loop leaves memory free first (W_p and the
  // u tiles: Y and U), then past the loop's footprint, so the solve can run while the last
  // step's MMAs still read X, K_l, D and Dt, and the next chunk's inputs can come into the
  // K_l and D regions meanwhile; [Kb | X] is built in X once those MMAs are done.
  static constexpr Place p0{oY, oKQ, loop_end};
  static constexpr uint32_t tKX = oX;                    // f16 [Kb | X] MN-major, C x 2D
  static_assert(sKX <= kX, "[Kb | X] fits the X region");
  static constexpr uint32_t tTP = p0.where(kF128);       // f16 [I ; P], then [T ; PT], 128 x C
  static constexpr Place p2 = p0.at(kF128);
  static constexpr uint32_t tA = p2.where(sSq);          // f32 A [C][C+4]
  static constexpr Place p3 = p2.at(sSq);
  static constexpr uint32_t tT = p3.where(sSq);          // f32 T [C][C+4]
  static constexpr Place p4 = p3.at(sSq);
  static constexpr uint32_t tZ = p4.where(sZ);           // f32 block-solve scratch
  static constexpr Place p5 = p4.at(sZ);
  static constexpr uint32_t tB = p5.where(sB);           // f32 beta[C], gamma[C]
  static constexpr Place p6 = p5.at(sB);
  static constexpr uint32_t tTB = p6.where(sTB);         // f16 T (B operand)
  static constexpr Place p7 = p6.at(sTB);
  static constexpr uint32_t bytes = p7.o2 > loop_end ? p7.o2 : loop_end;
  // The tail's buffers leave the K_l and D regions free: the next chunk's K, Q rows and v
  // window are copied there while the tail runs.
  static constexpr bool kPrefetch = true;
  // the same condition lets the solve start before the last step's MMAs complete
  static constexpr bool kEarlyTail = kPrefetch;
  // N^T (D x D fp32) leaves through the K_l and D regions (staged by the consumers, copied
  // out by the producer with one bulk store) where the tail leaves them free.
  static constexpr uint32_t kNT = D * D * 4;
  static constexpr bool kStageN = kPrefetch && oKl + kNT <= loop_end;
  static_assert((uint32_t)(2 * C * D * 2) <= 2 * kF && (uint32_t)((C + 8) * D * 2) <= 2 * kF,
                "input tiles fit the K_l and D regions");
  // TMEM columns: k_hat of even / odd steps | p (the u hi and u lo products side by side; the
  // scores [G;P] of K_l hi and lo once p has been read) | [R;O_l] | N_l, and in the tail [W | U] over the first 4C columns
  // (or W over N_l and U after it when D > 2C).
  static constexpr bool kExtraX = D > 4 * C;
  static constexpr uint32_t tmem_cols_needed = 4 * C + 2 * D + (kExtraX ? D : 0);
  static constexpr uint32_t tmem_cols =
      tmem_cols_needed <= 32 ? 32 : tmem_cols_needed <= 64 ? 64 : tmem_cols_needed <= 128 ? 128
                                  : tmem_cols_needed <= 256 ? 256 : 512;
  // CTAs per SM the registers must allow: two where TMEM lets two reside
  static constexpr int kMinBlocks = (NTA <= 288 && tmem_cols <= 256) ? 2 : 1;
  static_assert(NTH % 8 == 0 && NFD % 8 == 0 && NTF % 8 == 0 && RF >= 1, "column groups of 8");
  static_assert(tmem_cols_needed <= 512, "TMEM");
};

// Barrier among the consumer warps only (the producer warp does not take part).
template <int NT>
__device__ __forceinline__ void csync() {
  asm volatile("bar.sync 1, %0;\n" ::"n"(NT) : "memory");
}

// One warp: acc = X[16 x K] Y[K x 16] (fp32, shared memory; row strides ldx and
// ldy, multiples of 4 floats; X 16-byte aligned, Y 8-byte aligned).  Lane
// (rg = lane/8, cg = lane%8) owns rows rg + 4i (i < 4) and columns 2cg, 2cg+1:
// acc[2i + c].  X is read as 4-wide k vectors, Y as column pairs, so one
// shared-memory wavefront feeds 128 FMAs.
__device__ __forceinline__ void warp_blk16(const float* X, int ldx, const float* Y, int ldy, int K,
                                           float (&acc)[8]) {
  const int lane = threadIdx.x & 31, rg = lane >> 3, cg = lane & 7;
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;
#pragma unroll 2
  for (int k = 0; k < K; k += 4) {
    float4 xa[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) xa[i] = *reinterpret_cast<const float4*>(X + (rg + 4 * i) * ldx + k);
    float2 yb[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) yb[q] = *reinterpret_cast<const float2*>(Y + (k + q) * ldy + 2 * cg);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float xv[4] = {xa[i].x, xa[i].y, xa[i].z, xa[i].w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        acc[2 * i] = fmaf(xv[q], yb[q].x, acc[2 * i]);
        acc[2 * i + 1] = fmaf(xv[q], yb[q].y, acc[2 * i + 1]);
      }
    }
  }
}

// Stores -acc of warp_blk16 as block (row0, col0) of T: fp32 into sT (stride ld)
// and fp16 into the B tile sTB ((j, m) -> T[m][j] at (m/8)*16C + j*16 + (m%8)*2).
template <int C>
__device__ __forceinline__ void store_tblk(const float (&acc)[8], float* sT, int ld, unsigned char* sTB,
                                           int row0, int col0) {
  const int lane = threadIdx.x & 31, rg = lane >> 3, cg = lane & 7;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int m = row0 + rg + 4 * i, j = col0 + 2 * cg;
    const float v0 = -acc[2 * i], v1 = -acc[2 * i + 1];
    *reinterpret_cast<float2*>(sT + m * ld + j) = make_float2(v0, v1);
    *reinterpret_cast<__half*>(sTB + (m / 8) * (16u * C) + j * 16u + (m % 8) * 2u) = __float2half_rn(v0);
    *reinterpret_cast<__half*>(sTB + (m / 8) * (16u * C) + (j + 1) * 16u + (m % 8) * 2u) = __float2half_rn(v1);
  }
}

// T = (I + A)^-1 for the strictly lower triangular C x C matrix A (fp32, row
// stride LD = C + 4) by block doubling.  With blocks of 16:
//   diagonal blocks   T_ii = (I + A_ii)^-1, one thread per column: once entry m
//                     of the column is final it is eliminated from all rows
//                     below it (15 dependent steps of independent FMAs);
//   16 -> 32          T_(2p+1)(2p) = -T_(2p+1)(2p+1) (A_(2p+1)(2p) T_(2p)(2p));
//   32 -> 64          [T_20 T_21; T_30 T_31] = -T_hi (A_lo T_lo), with T_lo, T_hi
//                     the 32 x 32 diagonal halves (lower triangular, so the
//                     zero blocks drop out of the sums).
// Each product Y = X Z of 16 x 16 blocks is one warp's job (warp_blk16).
// Results: sT (fp32, stride LD; blocks above the diagonal not written) and sTB,
// T as the fp16 B operand of the [I ; P] T product, K-major: (j, m) -> T[m][j]
// at (m/8)*16C + j*16 + (m%8)*2, zero above the diagonal.  sY: 32 x 36 floats.
template <int C, int NT>
__device__ __forceinline__ void solve_tri(const float* sA, float* sT, unsigned char* sTB, float* sY) {
  constexpr int LD = C + 4, NB = C / 16, LDY = 36;
  const int tid = threadIdx.x, warp = tid >> 5;
  for (int idx = tid; idx < (C / 8) * C; idx += NT) {   // pieces wholly above the diagonal blocks
    const int m8 = idx / C, j = idx % C;
    if (m8 / 2 < j / 16) *reinterpret_cast<uint4*>(sTB + m8 * (16u * C) + j * 16u) = make_uint4(0u, 0u, 0u, 0u);
  }
  if (tid < C) {
    const int o = (tid / 16) * 16, j = tid % 16;
    float col[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) col[i] = (i == j) ? 1.f : 0.f;
#pragma unroll
    for (int m = 0; m < 15; ++m) {
      const float cm = col[m];
#pragma unroll
      for (int i = m + 1; i < 16; ++i) col[i] = fmaf(-sA[(o + i) * LD + o + m], cm, col[i]);
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) sT[(o + i) * LD + o + j] = col[i];
    float a[8], b[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) { a[i] = col[i]; b[i] = col[8 + i]; }
    *reinterpret_cast<uint4*>(sTB + (o / 8) * (16u * C) + (o + j) * 16u) = tc::cvt8(a);
    *reinterpret_cast<uint4*>(sTB + (o / 8 + 1) * (16u * C) + (o + j) * 16u) = tc::cvt8(b);
  }
  if constexpr (NB >= 2) {
    csync<NT>();
    // 16 -> 32: Y_p = A_(2p+1)(2p) T_(2p)(2p), then T_(2p+1)(2p) = -T_(2p+1)(2p+1) Y_p
    float acc[8];
    if (warp < NB / 2) {
      const int p = warp, r = (2 * p + 1) * 16, c = 2 * p * 16;
      warp_blk16(sA + r * LD + c, LD, sT + c * LD + c, LD, 16, acc);
      const int lane = tid & 31, rg = lane >> 3, cg = lane & 7;
#pragma unroll
      for (int i = 0; i < 4; ++i)
        *reinterpret_cast<float2*>(sY + p * 16 * LDY + (rg + 4 * i) * LDY + 2 * cg) = make_float2(acc[2 * i], acc[2 * i + 1]);
    }
    csync<NT>();
    if (warp < NB / 2) {
      const int p = warp, r = (2 * p + 1) * 16, c = 2 * p * 16;
      warp_blk16(sT + r * LD + r, LD, sY + p * 16 * LDY, LDY, 16, acc);
      store_tblk<C>(acc, sT, LD, sTB, r, c);
    }
  }
  if constexpr (NB == 4) {
    csync<NT>();
    // Y = A_lo T_lo  (rows 32..63, cols 0..31):  Y_(bi)(bj) = sum_{k = bj}^{1} A_(bi)(k) T_(k)(bj)
    float acc[8];
    if (warp < 4) {
      const int bi = 2 + (warp >> 1), bj = warp & 1;
      warp_blk16(sA + (bi * 16) * LD + bj * 16, LD, sT + (bj * 16) * LD + bj * 16, LD, 16 * (2 - bj), acc);
      const int lane = tid & 31, rg = lane >> 3, cg = lane & 7;
#pragma unroll
      for (int i = 0; i < 4; ++i)
        *reinterpret_cast<float2*>(sY + ((bi - 2) * 16 + rg + 4 * i) * LDY + bj * 16 + 2 * cg) =
            make_float2(acc[2 * i], acc[2 * i + 1]);
    }
    csync<NT>();
    // T_(bi)(bj) = -sum_{k = 2}^{bi} T_(bi)(k) Y_(k)(bj)
    if (warp < 4) {
      const int bi = 2 + (warp >> 1), bj = warp & 1;
      warp_blk16(sT + (bi * 16) * LD + 32, LD, sY + bj * 16, LDY, 16 * (bi - 1), acc);
      store_tblk<C>(acc, sT, LD, sTB, bi * 16, bj * 16);
    }
  }
}

__device__ __forceinline__ void ld_f8(const float* p, float (&v)[8]) {   // 32-byte aligned
  const float4 a = *reinterpret_cast<const float4*>(p), b = *reinterpret_cast<const float4*>(p + 4);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
__device__ __forceinline__ float u2f(uint32_t x) { return __uint_as_float(x); }
// Eight fp16 values (one 16-byte piece) to fp32.
__device__ __forceinline__ void h8_to_f(uint4 x, float (&f)[8]) {
  const __half2* h = reinterpret_cast<const __half2*>(&x);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 t = __half22float2(h[i]);
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}

template <int D, int C>
__global__ void __launch_bounds__(PrepSmem<D, C>::NTA, PrepSmem<D, C>::kMinBlocks)
    prep_tc_kernel(const __grid_constant__ PrepArgs p) {
  using S = PrepSmem<D, C>;
  constexpr int NT = S::NT, NW = S::NW, NTH = S::NTH, NFD = S::NFD, NQ = S::NQ;
  constexpr int RF = S::RF, NTF = S::NTF, NQF = S::NQF;
  extern __shared__ __align__(1024) unsigned char sm[];
  unsigned char* sX = sm + S::oX;
  unsigned char* sY = sm + S::oY;
  unsigned char* sU = sm + S::oU;
  unsigned char* sKQ = sm + S::oKQ;
  unsigned char* sKl = sm + S::oKl;
  unsigned char* sD = sm + S::oD;
  unsigned char* sDt = sm + S::oDt;
  float* sg = reinterpret_cast<float*>(sm + S::oG);
  float* sdec = reinterpret_cast<float*>(sm + S::oDec);
  float* sbl = reinterpret_cast<float*>(sm + S::oBeta);
  float* sinv = reinterpret_cast<float*>(sm + S::oInv);
  float* spart = reinterpret_cast<float*>(sm + S::oPart);
  float* sbt = reinterpret_cast<float*>(sm + S::oBtok);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + S::oBar);
  // mbarriers.  Tile copies: bar_wk (W_k into X), bar_wp (W_p into Y), bar_in (K, Q, v).
  // MMA completion (tcgen05.commit): bar_k[l % 2] (k_hat^(l)), bar_p (p^(l)), bar_gp (scores
  // of step l), bar_6 (step l's [R;O_l], N_l updates), bar_x (internal), bar_mma (tail).
  // Consumer warps -> producer (one arrival per warp): bar_u (u tiles written), bar_ra
  // (pass A done: K_l tile written, k_hat read), bar_rb (pass B done: D_l tiles written, p
  // read), bar_r5 ([G;P] tiles written).
  uint64_t* bar_mma = bars + 0;
  uint64_t* bar_wk = bars + 1;
  uint64_t* bar_wp = bars + 2;
  uint64_t* bar_in = bars + 3;
  uint64_t* bar_k = bars + 4;                  // [2]
  uint64_t* bar_p = bars + 6;
  uint64_t* bar_gp = bars + 7;
  uint64_t* bar_6 = bars + 8;
  uint64_t* bar_rb = bars + 9;
  uint64_t* bar_r5 = bars + 10;
  uint64_t* bar_x = bars + 11;
  uint64_t* bar_u = bars + 12;
  uint64_t* bar_ra = bars + 13;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + S::oSlot);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool producer = warp == NW;
  const int quarter = warp & 3, cg = warp >> 2;
  const int row = quarter * 32 + lane;         // this thread's TMEM lane
  const int tb0 = cg * NTH;                    // first of this thread's token columns
  const int fb0 = cg * NFD;                    // first of this thread's feature columns
  const int H = p.H, T_ = p.T, L = p.L, w = p.w;
  const int NC = (T_ + C - 1) / C;
  const int total = p.B * H * NC;
  const bool need_lo = *p.wflag != 0;
  const bool cvalid = row < D && !producer;
  // feature role: lane row holds feature cf, replica rf (quarter qf of it) and takes tokens
  // tf0 .. tf0+NTF-1 of its column group
  const int cf = row % D;
  const int rf = D >= 32 ? quarter / NQF : 0, qf = D >= 32 ? quarter % NQF : 0;
  const bool fwarp_f = !producer && quarter < (D >= 32 ? NQF * RF : 1);   // warp-uniform
  const bool fvalid = fwarp_f && (D >= 32 || row < D);
  const int tf0 = (cg * RF + rf) * NTF;
  // extents of the arrays the kernel addresses (the debug build checks each access)
  int* bw = p.bounds;
  const size_t nBTH = (size_t)p.B * T_ * H, nmaps = (size_t)p.B * H * NC;
  const size_t wblock_bytes = (size_t)H * L * 4 * S::kW;
  auto sm_ok = [&](const void* ptr, size_t n) { return within(ptr, n, sm, S::bytes); };
  constexpr int NG = (C + 31) / 32;
  __nv_bfloat16* kqraw = reinterpret_cast<__nv_bfloat16*>(sKl);   // [2C][D]: K rows, then Q rows
  __nv_bfloat16* vwin = reinterpret_cast<__nv_bfloat16*>(sD);     // [C + 8][D]: tokens t0-8 .. t0+C-1
  // Chunks are numbered (b, h, chunk) with a head's chunks consecutive; chunk_of gives the
  // coordinates and the count of tokens before the sequence end (<= 0: padding only).
  auto chunk_of = [&](int id, int& b_, int& h_, int& c_, int& nv_) {
    c_ = id % NC;
    h_ = (id / NC) % H;
    b_ = id / (NC * H);
    const int len_ = p.seq_lens ? min(max(p.seq_lens[b_], 0), T_) : T_;
    nv_ = min(C, len_ - c_ * C);
  };
  auto next_chunk = [&](int id) {              // this CTA's next chunk with tokens, from id on
    for (; id < total; id += gridDim.x) {
      int b_, h_, c_, nv_;
      chunk_of(id, b_, h_, c_, nv_);
      if (nv_ > 0) break;
    }
    return id;
  };
  // (the chunk after `cur` is worked out where it is needed rather than kept live across
  // the chunk: one register fewer through the refinement loop)
  auto next_of = [&](int cur_) { return next_chunk(cur_ + gridDim.x); };
  // One thread: TMA copies of a chunk's K and Q rows and its v window (C + 8 tokens;
  // out-of-range rows arrive as zeros) into the K_l and D regions.
  auto load_inputs = [&](int id) {
    int b_, h_, c_, nv_;
    chunk_of(id, b_, h_, c_, nv_);
    tc::bar_expect_tx(bar_in, (uint32_t)(3 * C + 8) * D * 2);
    tc::tma_load_4d(kqraw, &p.tm_k, 0, h_, c_ * C, b_, bar_in);
    tc::tma_load_4d(kqraw + C * D, &p.tm_q, 0, h_, c_ * C, b_, bar_in);
    tc::tma_load_4d(vwin, &p.tm_v, 0, h_, c_ * C - 8, b_, bar_in);
  };
  // A chunk's gates into shared memory, by the producer warp: log alpha scanned over the
  // chunk (sg) and beta_t (sbt), zero past the sequence end.  The decay factors sdec
  // follow at the chunk's start (the previous chunk's tail still reads its own).
  auto gates_to_smem = [&](int id) {
    int b_, h_, c_, nv_;
    chunk_of(id, b_, h_, c_, nv_);
    float la[NG], be[NG];
#pragma unroll
    for (int q = 0; q < NG; ++q) {
      const int i = q * 32 + lane;
      const size_t g = ((size_t)b_ * T_ + c_ * C + i) * H + h_;
      const bool in = i < nv_ && PRISM_IN_BOUNDS(g < nBTH, bw);
      la[q] = in ? tc::ldg_early(p.log_alpha + g) : 0.f;
      be[q] = in ? tc::ldg_early(p.beta + g) : 0.f;
    }
    float run = 0.f;
#pragma unroll
    for (int q = 0; q < NG; ++q) {
      const int i = q * 32 + lane;
      float x = la[q];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      x += run;
      run = __shfl_sync(0xffffffffu, x, 31);
      if (i < C) {
        sg[i] = x;
        sbt[i] = be[q];
      }
    }
    __syncwarp();
  };

  // ---- once per CTA: barriers, TMEM, the first chunk's tile copies and gates ----
  int cur = next_chunk(blockIdx.x);
  // A CTA with no chunk (all of its chunks lie past their sequence's end: ragged batches
  // launch one CTA per chunk) leaves at once, before it takes TMEM or initialises a
  // barrier; the whole CTA takes this branch.  At d = 128 the check is compiled out:
  // there it cost 0.6 % of the non-ragged step through code generation.
  if constexpr (D < 128)
    if (cur >= total) return;
  if (warp == 0) {
    if (lane == 0) {
      for (int i = 0; i < S::kBars; ++i)
        tc::bar_init(bars + i,
                     (bars + i == bar_u || bars + i == bar_ra || bars + i == bar_rb || bars + i == bar_r5) ? NW : 1);
      tc::bar_fence_init();
      if (cur < total) load_inputs(cur);
    }
    __syncwarp();
    tc::alloc(tslot, S::tmem_cols);
  }
  if (producer && cur < total) gates_to_smem(cur);
  // rows D..127 of the scaled-write tiles stay zero (A operand of the injection); nothing
  // else ever writes them
  if constexpr (D < 128)
    for (int idx = tid; idx < (128 - D) * (C / 8) * 2; idx += S::NTA) {
      const int part = idx / ((128 - D) * (C / 8));
      const int rem = idx % ((128 - D) * (C / 8));
      const int r = D + rem % (128 - D), s8 = rem / (128 - D);
      *reinterpret_cast<uint4*>(sDt + part * S::kF128 + s8 * 2048u + r * 16u) = make_uint4(0u, 0u, 0u, 0u);
    }
  tc::fence_smem_to_async();
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = *tslot;
  // TMEM columns: k_hat (even steps) | k_hat (odd steps) | p (W_p u_hi, W_p u_lo) | [R;O_l] | N_l
  const uint32_t t_k0 = tmem, t_p = tmem + 2 * C;
  const uint32_t t_ro = tmem + 4 * C, t_n = tmem + 4 * C + D;
  const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
  constexpr uint32_t idesc_proj = tc::idesc_f16(C, false, true);   // B = U, MN-major
  constexpr uint32_t idesc_proj2 = tc::idesc_f16(2 * C, false, true);   // B = [u_hi | u_lo]
  constexpr uint32_t idesc_gs = tc::idesc_f16(C, false, true);      // B = K_l (MN-major)
  constexpr uint32_t idesc_cc = tc::idesc_f16(C, false, false);
  constexpr uint32_t idesc_dd = tc::idesc_f16(D, false, false);
  constexpr uint32_t S_s = (D / 8) * 128;      // token step of the feature x token tiles
  bool ok = true;

  // One loop over this CTA's chunks for both roles; the producer warp and the consumer
  // warps split inside it.
  bool have_gates = true;                      // producer: the chunk's gates are in sg / sbt
  for (uint32_t it = 0; cur < total; ++it) {
  int b, h, chunk, nv;
  chunk_of(cur, b, h, chunk, nv);
  const int t0 = chunk * C;
  const int len = p.seq_lens ? min(max(p.seq_lens[b], 0), T_) : T_;
  // parities: bar_k[0] completes ceil(L/2) times per chunk, bar_k[1] floor(L/2) times,
  // bar_p, bar_gp and bar_6 L times, bar_in and bar_u once
  const uint32_t kb0 = it * (uint32_t)((L + 1) / 2), kb1 = it * (uint32_t)(L / 2), sb = it * (uint32_t)L;
  auto kpar = [&](int l) { return (((l & 1) ? kb1 : kb0) + (uint32_t)(l >> 1)) & 1u; };
  auto spar = [&](int l) { return (sb + (uint32_t)l) & 1u; };
  const unsigned char* wsrc = p.wblocks;
  auto wblock = [&](int l, int which, int part) {
    return wsrc + WeightBlock<D>::index(h, l, L, which, part) * S::kW;
  };
  // one weight block into dst, its copy completing on bar (skipped in the debug build if
  // the block or the destination fall outside their arrays: the wait then runs out)
  auto wcopy = [&](unsigned char* dst, const unsigned char* src, uint64_t* bar) {
    if (PRISM_IN_BOUNDS(within(src, S::kW, wsrc, wblock_bytes) && sm_ok(dst, S::kW), bw))
      tc::bulk_g2s(dst, src, S::kW, bar);
  };
  // ---- chunk start: the producer streams W^(0) in (the previous tail is done with X and
  //      Y) and forms the decay factors from the gates it brought in; the consumers fetch
  //      their small parameters ----
  if (producer && lane == 0 && L > 0) {
    tc::bar_expect_tx(bar_wk, S::kW);
    wcopy(sX, wblock(0, 0, 0), bar_wk);
    tc::bar_expect_tx(bar_wp, S::kW);
    wcopy(sY, wblock(0, 1, 0), bar_wp);
  }
  if (producer) {
    if (!have_gates) gates_to_smem(cur);      // first chunk, or no prefetch
    have_gates = false;
    for (int i = lane; i < C; i += 32) sdec[i] = expf(sg[C - 1] - sg[i]);
  }
  // conv taps (ca[m] multiplies v_{t-8+m}) and w_beta^(0) of this thread's feature
  float ca[8];
#pragma unroll
  for (int m = 0; m < 8; ++m) {
    const int j = 8 - m;
    ca[m] = (fvalid && j <= w && PRISM_IN_BOUNDS(((size_t)h * w + (j - 1)) * D + cf < (size_t)H * w * D, bw))
                ? tc::ldg_early(p.conv_w + ((size_t)h * w + (j - 1)) * D + cf) : 0.f;
  }
  float wb_next = (L > 0 && fvalid && PRISM_IN_BOUNDS((size_t)h * L * D + cf < (size_t)H * L * D, bw))
                      ? tc::ldg_early(p.wbeta + (size_t)h * L * D + cf) : 0.f;
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  if (producer) {
    // ================= producer: tile copies and MMAs of the refinement loop =================
    if (lane == 0 && L > 0) {
      // phase counts: per chunk bar_wk and bar_wp complete L times (2L with the lo halves),
      // bar_x 2L times (lo halves only), bar_ra, bar_rb and bar_r5 L times
      const uint32_t nw = need_lo ? 2u * L : (uint32_t)L;
      uint32_t ph_wk = it * nw, ph_wp = it * nw, ph_ra = it * L, ph_rb = it * L, ph_r5 = it * L;
      uint32_t ph_x = need_lo ? it * 2u * L : 0u;
      auto wait = [&](uint64_t* bar, uint32_t parity) {
        ok &= tc::bar_wait(bar, parity);
        tc::fence_after();
      };
      // projection W u^T of step l (which 0: W_k from X into the k_hat columns, 1: W_p from
      // Y into the p columns): hi weights against u hi + lo, then (weights not exact in
      // fp16) the lo weights against u hi; completion on `done`.  k_hat accumulates both
      // halves of u in one set of C columns (two MMAs per K step); p takes [u_hi | u_lo] as
      // one N = 2C operand (one MMA per K step: an MMA costs about the same for any N up
      // to 256) and leaves the two products side by side for the epilogue to add.
      auto proj = [&](int l, int which, uint32_t dst, unsigned char* wbuf, uint64_t* ldbar, uint32_t& ldph,
                      uint64_t* done) {
        if (which == 0) {
          for (int pass = 0; pass < 2; ++pass)
            for (int kk = 0; kk < D / 16; ++kk)
              tc::mma(dst, tc::desc(wbuf + kk * 4096, 2048, 128), tc::desc(sU + pass * S::kU + kk * 256, 128, 16 * D),
                      idesc_proj, pass > 0 || kk > 0);
        } else {
          for (int kk = 0; kk < D / 16; ++kk)
            tc::mma(dst, tc::desc(wbuf + kk * 4096, 2048, 128), tc::desc(sU + kk * 256, 128, 16 * D), idesc_proj2,
                    kk > 0);
        }
        if (need_lo) {
          tc::commit(bar_x);
          wait(bar_x, ph_x++ & 1);
          tc::bar_expect_tx(ldbar, S::kW);
          wcopy(wbuf, wblock(l, which, 1), ldbar);
          wait(ldbar, ldph++ & 1);
          for (int kk = 0; kk < D / 16; ++kk)
            tc::mma(dst, tc::desc(wbuf + kk * 4096, 2048, 128), tc::desc(sU + kk * 256, 128, 16 * D), idesc_proj, true);
        }
        tc::commit(done);
      };
      wait(bar_u, it & 1);
      wait(bar_wk, ph_wk++ & 1);
      proj(0, 0, t_k0, sX, bar_wk, ph_wk, bar_k);
      wait(bar_wp, ph_wp++ & 1);
      proj(0, 1, t_p, sY, bar_wp, ph_wp, bar_p);
      for (int l = 0; l < L; ++l) {
        const uint32_t t_kl = t_k0 + (l & 1) * C;
        if (l + 1 < L) {
          // W_p^(l+1) into Y once p^(l) is done; W_k^(l+1) into X once k_hat^(l) is done and
          // step l-1's [G;P] tiles have been read; then k_hat^(l+1) into the other columns
          wait(bar_p, spar(l));
          tc::bar_expect_tx(bar_wp, S::kW);
          wcopy(sY, wblock(l + 1, 1, 0), bar_wp);
          wait(bar_k + (l & 1), kpar(l));
          if (l > 0) wait(bar_6, spar(l - 1));
          tc::bar_expect_tx(bar_wk, S::kW);
          wcopy(sX, wblock(l + 1, 0, 0), bar_wk);
          wait(bar_wk, ph_wk++ & 1);
          proj(l + 1, 0, t_k0 + ((l + 1) & 1) * C, sX, bar_wk, ph_wk, bar_k + ((l + 1) & 1));
        }
        // [4] scores [G ; P] = [K ; Q] K_l^T into k_hat^(l)'s columns once pass A has read
        //     them and written the K_l tile; the hi and lo halves of K_l accumulate in one set
        //     of C columns, so the scores compute while pass B runs
        wait(bar_ra, ph_ra++ & 1);
        for (int kk = 0; kk < D / 16; ++kk)
          for (int part = 0; part < 2; ++part)
            tc::mma(t_kl, tc::desc(sKQ + kk * 4096, 2048, 128), tc::desc(sKl + part * S::kF + kk * 256, 128, S_s),
                    idesc_gs, kk > 0 || part > 0);
        tc::commit(bar_gp);
        // once pass B has read p^(l) and written the D tiles: p^(l+1) into the p columns, then
        // [6a] N_l^T += K_l^T Dt_l (3 passes; rows of N^T are k features, columns v features)
        wait(bar_rb, ph_rb++ & 1);
        if (l + 1 < L) {
          wait(bar_wp, ph_wp++ & 1);
          proj(l + 1, 1, t_p, sY, bar_wp, ph_wp, bar_p);
        }
        {
          const int ap[3] = {0, 1, 0}, bp[3] = {0, 0, 1};
          for (int ps = 0; ps < 3; ++ps)
            for (int kk = 0; kk < C / 16; ++kk)
              tc::mma(t_n, tc::desc(sKl + ap[ps] * S::kF + kk * 2 * S_s, S_s, 128),
                      tc::desc(sDt + bp[ps] * S::kF128 + kk * 4096, 2048, 128), idesc_dd, l > 0 || ps > 0 || kk > 0);
        }
        // [6b] [R ; O_l] += [G ; P] D_l (3 passes) once the [G;P] tiles are in X
        wait(bar_r5, ph_r5++ & 1);
        {
          const int ap[3] = {0, 0, 1}, bp[3] = {0, 1, 0};
          for (int ps = 0; ps < 3; ++ps)
            for (int kk = 0; kk < C / 16; ++kk)
              tc::mma(t_ro, tc::desc(sX + ap[ps] * S::kF128 + kk * 4096, 2048, 128),
                      tc::desc(sD + bp[ps] * S::kF + kk * 2 * S_s, S_s, 128), idesc_dd, l > 0 || ps > 0 || kk > 0);
        }
        tc::commit(bar_6);
      }
    }
    __syncwarp();
    if constexpr (S::kStageN) {
      // the consumers have staged N^T in the K_l / D regions: copy it out, and once the copy
      // has read it, bring the next chunk's tiles in (they land in the same regions)
      asm volatile("bar.sync 10, %0;\n" ::"n"(S::NTA) : "memory");
      const int nxt = next_of(cur);
      if (lane == 0) {
        const size_t cbase = ((size_t)b * H + h) * NC + chunk;
        if (L > 0) {
          if (PRISM_IN_BOUNDS(within(p.Nt + cbase * D * D, S::kNT, p.Nt, nmaps * D * D * 4) && sm_ok(sKl, S::kNT), bw))
            tc::bulk_s2g(p.Nt + cbase * D * D, sKl, S::kNT);
          tc::bulk_commit();
          tc::bulk_wait_read();
        }
        if (nxt < total) load_inputs(nxt);
      }
      __syncwarp();
      // the consumers have also read this chunk's sg and sbt (sdec stays theirs until the
      // chunk ends): the next chunk's gates come in now
      if (nxt < total) {
        gates_to_smem(nxt);
        have_gates = true;
      }
    }
  } else {
  // ================= consumers =================
  ok &= tc::bar_wait(bar_in, it & 1);
  // v rows past the sequence end are cleared.
  if (t0 + C > len) {
    const int r0 = len - (t0 - 8);             // first v-window row past the end (>= 9)
    for (int idx = tid; idx < (C + 8 - r0) * (D / 8); idx += NT)
      *reinterpret_cast<uint4*>(vwin + (r0 + idx / (D / 8)) * D + (idx % (D / 8)) * 8) = make_uint4(0u, 0u, 0u, 0u);
  }
  if (t0 == 0 && p.vhist) {                    // tokens -w .. -1 of a resumed sequence (rows 8-w .. 7)
    const bool tmaj = p.flags & 2u;
    for (int idx = tid; idx < w * (D / 8); idx += NT) {
      const int rr = idx / (D / 8), pc = idx % (D / 8);
      const __nv_bfloat16* src = p.vhist + (tmaj ? (((size_t)b * w + rr) * H + h) * D : (((size_t)b * H + h) * w + rr) * D) + pc * 8;
      if (PRISM_IN_BOUNDS(within(src, 16, p.vhist, (size_t)p.B * H * w * D * 2) && sm_ok(vwin + (8 - w + rr) * D + pc * 8, 16), bw))
        *reinterpret_cast<uint4*>(vwin + (8 - w + rr) * D + pc * 8) = *reinterpret_cast<const uint4*>(src);
    }
  }
  csync<NT>();
  const int c = cf;
  const bool fwarp = quarter < NQ;             // warp holds feature rows (token-row role: N^T)

  // ---- anchor u = sum_j c_j (.) v_{t-j} (the U tile, hi + lo) and residual r = v - u
  //      (registers); thread (feature c, replica, column group) owns tokens tf0 .. tf0+NTF-1 ----
  float rres[NTF];
  {
#pragma unroll
    for (int j8 = 0; j8 < NTF; j8 += 8) {
      if (fwarp_f) {
        float win[16], uu[8];
#pragma unroll
        for (int i = 0; i < 16; ++i) win[i] = fvalid ? __bfloat162float(vwin[(tf0 + j8 + i) * D + c]) : 0.f;
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
          float u = 0.f;
#pragma unroll
          for (int m = 0; m < 8; ++m) u = fmaf(ca[m], win[jj + m], u);
          uu[jj] = u;
          rres[j8 + jj] = (tf0 + j8 + jj < nv) ? win[jj + 8] - u : 0.f;
        }
        if (fvalid) {
          // U tile, MN-major B operand (K = features, N = tokens): (c, t) at (t/8)*16D + c*16 + (t%8)*2
          uint4 uh, ul;
          tc::split8(uu, uh, ul);
          const uint32_t off = ((tf0 + j8) / 8) * (16u * D) + c * 16u;
          put(reinterpret_cast<uint4*>(sU + off), uh, sU, 2 * S::kU, bw);
          put(reinterpret_cast<uint4*>(sU + S::kU + off), ul, sU, 2 * S::kU, bw);
        }
      } else {
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) rres[j8 + jj] = 0.f;
      }
    }
  }
  // u tiles written: the producer may start the projections.  The barrier keeps every
  // lane's anchor writes ahead of the tail, whose buffers reuse this memory (L = 0).
  tc::fence_smem_to_async();
  tc::fence_before();
  __syncwarp();
  if (lane == 0) tc::bar_arrive(bar_u);
  csync<NT>();
  // [K ; Q] rows as fp16: (row, a) at (a/8)*2048 + row*16 + (a%8)*2; rows of tokens past
  // the sequence end and rows >= 2C zero.  This and the decay mask run while the first
  // projection is on the tensor core (nothing before the scores of step 0 reads them).
  // (the piece index is rotated by the row so that eight consecutive lanes read eight
  //  different bank groups of the raw rows and write eight different ones of the tile)
  for (int idx = tid; idx < 128 * (D / 8); idx += NT) {
    const int r = idx % 128, a8 = (idx / 128 + r) % (D / 8);
    const int t = r < C ? r : r - C;
    uint4 o = make_uint4(0u, 0u, 0u, 0u);
    if (r < 2 * C && t < nv) {
      const uint4 raw = *reinterpret_cast<const uint4*>(kqraw + r * D + a8 * 8);
      const __nv_bfloat16* e = reinterpret_cast<const __nv_bfloat16*>(&raw);
      float f[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) f[j] = __bfloat162float(e[j]);
      o = tc::cvt8(f);
    }
    put(reinterpret_cast<uint4*>(sKQ + a8 * 2048u + r * 16u), o, sKQ, S::kKQ, bw);
  }
  // Decay mask of this thread's token row for the score tiles (fixed for the
  // chunk): rows < C strictly causal (G, A), rows C..2C-1 inclusive (P).
  float gm[NTH];
  {
    const bool isG = row < C, isP = row >= C && row < 2 * C;
    const int t = isG ? row : row - C;
    const float gt = (isG || isP) ? sg[t] : 0.f;
#pragma unroll
    for (int jj = 0; jj < NTH; ++jj) {
      const int s_ = tb0 + jj;
      gm[jj] = ((isG && t > s_) || (isP && t >= s_)) ? __expf(gt - sg[s_]) : 0.f;
    }
  }

  tc::fence_smem_to_async();                   // the [K ; Q] tile is a tensor-core operand
  csync<NT>();                                 // the raw K/Q rows (in the K_l tile) are read

  const bool gelu = !(p.flags & 1u);
  for (int l = 0; l < L; ++l) {
    const uint32_t t_kl = t_k0 + (l & 1) * C;  // k_hat^(l)
    ok &= tc::bar_wait(bar_k + (l & 1), kpar(l));
    tc::fence_after();
    // [3] epilogue.  Pass A: per token |k_hat|^2 and the gate logit w_beta . u,
    //     summed over this warp's 32 features (reduce-scatter over 8-token groups); the
    //     quarter-0 warps keep their sums, the others leave them in shared memory.
    {
      const float wb = wb_next;
      if (l + 1 < L && fvalid && PRISM_IN_BOUNDS(((size_t)h * L + l + 1) * D + c < (size_t)H * L * D, bw))
        wb_next = tc::ldg_early(p.wbeta + ((size_t)h * L + l + 1) * D + c);   // next step's
      float keep_n[NTF / 8], keep_z[NTF / 8];
      float kh[NTF];                           // k_hat of this thread's feature and tokens
      if (fwarp_f) {
#pragma unroll
        for (int j8 = 0; j8 < NTF; j8 += 8) {
          uint32_t kr[8];
          tc::ld8a(t_kl + lane_base + tf0 + j8, kr);
          float uf[8];                            // u = hi + lo from the U tile
          if (fvalid) {
            const uint32_t off = ((tf0 + j8) / 8) * (16u * D) + c * 16u;
            float uh[8], ul[8];
            h8_to_f(*reinterpret_cast<const uint4*>(sU + off), uh);
            h8_to_f(*reinterpret_cast<const uint4*>(sU + S::kU + off), ul);
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) uf[jj] = uh[jj] + ul[jj];
          } else {
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) uf[jj] = 0.f;
          }
          tc::wait_ld(kr);
          float rn[8], rz[8];
#pragma unroll
          for (int jj = 0; jj < 8; ++jj) {
            kh[j8 + jj] = u2f(kr[jj]);
            rn[jj] = kh[j8 + jj] * kh[j8 + jj];
            rz[jj] = wb * uf[jj];
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
          if ((lane & 3) == 0) {                // lane holds token j8 + lane/4 of its group
            const int t = tf0 + j8 + (lane >> 2);
            if (qf == 0) {
              keep_n[j8 / 8] = rn[0];
              keep_z[j8 / 8] = rz[0];
            } else {
              put(spart + (qf - 1) * 2 * C + t, rn[0], spart, 24u * C, bw);
              put(spart + (qf - 1) * 2 * C + C + t, rz[0], spart, 24u * C, bw);
            }
          }
        }
      }
      // the four warps of this column group (one per lane quarter) hold all partial sums
      // of its tokens: they synchronise among themselves
      asm volatile("bar.sync %0, 128;\n" ::"r"(2 + cg) : "memory");
      if (fwarp_f && qf == 0 && (lane & 3) == 0) {   // sums over the quarters, in quarter order
#pragma unroll
        for (int g = 0; g < NTF / 8; ++g) {
          const int t = tf0 + 8 * g + (lane >> 2);
          float ss = keep_n[g], zz = keep_z[g];
#pragma unroll
          for (int q = 1; q < NQF; ++q) {
            ss += spart[(q - 1) * 2 * C + t];
            zz += spart[(q - 1) * 2 * C + C + t];
          }
          const bool tv = t < nv;
          sinv[t] = tv ? rsqrtf(ss + 1e-6f) : 0.f;
          sbl[t] = tv ? __frcp_rn(1.0f + __expf(-zz)) : 0.f;
        }
      }
      asm volatile("bar.sync %0, 128;\n" ::"r"(2 + cg) : "memory");
      // directions k^(l) = k_hat / |k_hat| into the K_l tile (hi, lo) once step l-1's MMAs
      // have read the tiles about to be rewritten; then the producer may score against it
      if (l > 0) ok &= tc::bar_wait(bar_6, spar(l - 1));
      tc::fence_after();
      if (fvalid) {
#pragma unroll
        for (int j8 = 0; j8 < NTF; j8 += 8) {
          const int tb = tf0 + j8;
          float si[8], kd[8];
          ld_f8(sinv + tb, si);
#pragma unroll
          for (int jj = 0; jj < 8; ++jj) kd[jj] = kh[j8 + jj] * si[jj];
          uint4 hi, lo;
          // feature x token tiles: (f, s) at (s/8)*S_s + f*16 + (s%8)*2  (f < D)
          const uint32_t off = (tb / 8) * S_s + c * 16u;
          tc::split8(kd, hi, lo);
          put(reinterpret_cast<uint4*>(sKl + off), hi, sKl, 2 * S::kF, bw);
          put(reinterpret_cast<uint4*>(sKl + S::kF + off), lo, sKl, 2 * S::kF, bw);
        }
      }
      tc::fence_smem_to_async();
      tc::fence_before();
      __syncwarp();
      if (lane == 0) tc::bar_arrive(bar_ra);
      ok &= tc::bar_wait(bar_p, spar(l));       // p^(l) ready
      tc::fence_after();
      // Pass B: residual step and the write values
      if (fwarp_f) {
#pragma unroll
        for (int j8 = 0; j8 < NTF; j8 += 8) {
          uint32_t pr[8], pl[8];
          tc::ld8a(t_p + lane_base + tf0 + j8, pr);
          tc::ld8a(t_p + C + lane_base + tf0 + j8, pl);
          const int tb = tf0 + j8;
          float sb[8], sd[8];
          ld_f8(sbl + tb, sb);
          ld_f8(sdec + tb, sd);
          tc::wait_ld(pr, pl);
          float dv[8], dt[8];
#pragma unroll
          for (int jj = 0; jj < 8; ++jj) {
            const float x = (u2f(pr[jj]) + u2f(pl[jj])) * rres[j8 + jj];
            const float dl = gelu ? gelu_hastings(x) : x;
            rres[j8 + jj] -= dl;
            dv[jj] = sb[jj] * dl;
            dt[jj] = dv[jj] * sd[jj];
          }
          if (fvalid) {
            uint4 hi, lo;
            // feature x token tiles: (f, s) at (s/8)*S_s + f*16 + (s%8)*2  (f < D)
            const uint32_t off = (tb / 8) * S_s + c * 16u;
            const uint32_t off128 = (tb / 8) * 2048u + c * 16u;
            tc::split8(dv, hi, lo);
            put(reinterpret_cast<uint4*>(sD + off), hi, sD, 2 * S::kF, bw);
            put(reinterpret_cast<uint4*>(sD + S::kF + off), lo, sD, 2 * S::kF, bw);
            tc::split8(dt, hi, lo);
            put(reinterpret_cast<uint4*>(sDt + off128), hi, sDt, 2 * S::kF128, bw);
            put(reinterpret_cast<uint4*>(sDt + S::kF128 + off128), lo, sDt, 2 * S::kF128, bw);
          }
        }
      }
    }
    tc::fence_smem_to_async();
    tc::fence_before();
    __syncwarp();
    if (lane == 0) tc::bar_arrive(bar_rb);
    ok &= tc::bar_wait(bar_gp, spar(l));
    tc::fence_after();
    // [5] epilogue: decay and causal mask, then hi/lo split; rows < C are G, C..2C-1 are P
    if (quarter * 32 < 2 * C) {
      uint32_t gr[NTH / 8][8];
#pragma unroll
      for (int g = 0; g < NTH / 8; ++g) tc::ld8a(t_kl + lane_base + tb0 + 8 * g, gr[g]);
      tc::wait_ld();
#pragma unroll
      for (int g = 0; g < NTH / 8; ++g) {
        tc::pin(gr[g]);
        float val[8];
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) val[jj] = gm[8 * g + jj] * u2f(gr[g][jj]);
        uint4 hi, lo;
        tc::split8(val, hi, lo);
        const uint32_t off = ((tb0 + 8 * g) / 8) * 2048u + row * 16u;
        put(reinterpret_cast<uint4*>(sX + off), hi, sX, S::kX, bw);
        put(reinterpret_cast<uint4*>(sX + S::kF128 + off), lo, sX, S::kX, bw);
      }
    }
    tc::fence_smem_to_async();
    tc::fence_before();
    __syncwarp();
    if (lane == 0) tc::bar_arrive(bar_r5);
  }
  uint32_t ph_mma = it * 3u;                   // bar_mma completes three times per chunk
  auto wait_mma = [&]() {
    ok &= tc::bar_wait(bar_mma, ph_mma & 1);
    ++ph_mma;
    tc::fence_after();
  };

  // ================= tail: gated delta rule, state-independent part =================
  const size_t cbase = ((size_t)b * H + h) * NC + chunk;
  float* tAf = reinterpret_cast<float*>(sm + S::tA);
  float* tTf = reinterpret_cast<float*>(sm + S::tT);
  float* tZf = reinterpret_cast<float*>(sm + S::tZ);
  float* tbeta = reinterpret_cast<float*>(sm + S::tB);
  float* tgam = tbeta + C;
  unsigned char* sTP = sm + S::tTP;
  unsigned char* sKX = sm + S::tKX;
  unsigned char* sTB = sm + S::tTB;
  // [W | U] side by side from column 0 when they fit below [R;O_l] (one N = 2D MMA per K
  // step); otherwise W over N_l and U at column 0 (or after N_l when D > 4C)
  constexpr bool kMergeWX = 2 * D <= 4 * C;
  const uint32_t t_w = kMergeWX ? tmem : t_n;                                      // W / PW
  const uint32_t t_x = kMergeWX ? tmem + D : (S::kExtraX ? tmem + 4 * C + 2 * D : tmem);   // U / PU
  const int s_tok = row;
  const bool tok = s_tok < C;
  const bool tok_valid = tok && s_tok < nv;
  // v rows for (d), fetched now so their latency overlaps the solve
  uint4 vr[NFD / 8];
#pragma unroll
  for (int g = 0; g < NFD / 8; ++g)
    vr[g] = (tok_valid && PRISM_IN_BOUNDS((((size_t)b * T_ + t0 + s_tok) * H + h) * D + fb0 + 8 * g + 8 <= nBTH * D, bw))
                ? tc::ldg_early(reinterpret_cast<const uint4*>(p.v + (((size_t)b * T_ + t0 + s_tok) * H + h) * D + fb0 + 8 * g))
                      : make_uint4(0u, 0u, 0u, 0u);
  // Where the solve's buffers avoid the tiles the last step's MMAs read (kEarlyTail), the
  // solve runs before those MMAs are waited for; otherwise after.
  if constexpr (!S::kEarlyTail) {
    if (L > 0) {
      ok &= tc::bar_wait(bar_6, spar(L - 1));
      tc::fence_after();
    }
  }
  // (b) [K K^T ; Q K^T] = [K ; Q] K^T   (B = the K rows of the same tile, K-major), into
  //     the k_hat columns the last refinement step did not use: with the early tail the
  //     last step's scores may still be being read, while the other buffer's (step L-2's)
  //     were read by every warp before its pass A of step L-1, which the producer waited
  //     for before the scores behind bar_gp of step L-1, and this thread has passed that.
  const uint32_t t_kk = t_k0 + (L & 1) * C;
  if (tid == 0) {
    tc::fence_after();
    for (int kk = 0; kk < D / 16; ++kk)
      tc::mma(t_kk, tc::desc(sKQ + kk * 4096, 2048, 128), tc::desc(sKQ + kk * 4096, 2048, 128),
              idesc_cc, kk > 0);
    tc::commit(bar_mma);
  }
  if (tid < C) {
    tbeta[tid] = sbt[tid];
    tgam[tid] = expf(sg[tid]);
  }
  csync<NT>();
  wait_mma();
  // (c) A = strict_tril(beta (K K^T) (.) Gamma) (fp32) and the A tile [I ; P] of the
  //     [T ; PT] product (fp16, K-major (r, s) at (s/8)*2048 + r*16 + (s%8)*2; rows >= 2C zero)
  if (quarter * 32 < 2 * C) {
    const bool isA = row < C;
    const int t = isA ? row : row - C;
    const float bt = isA ? tbeta[t] : 0.f;
    uint32_t ar[NTH / 8][8];
#pragma unroll
    for (int g = 0; g < NTH / 8; ++g) tc::ld8a(t_kk + lane_base + tb0 + 8 * g, ar[g]);
    tc::wait_ld();
#pragma unroll
    for (int g = 0; g < NTH / 8; ++g) {
      tc::pin(ar[g]);
      const int s0 = tb0 + 8 * g;
      float v8[8];
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) v8[jj] = gm[8 * g + jj] * u2f(ar[g][jj]);
      if (isA) {
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
          put(tAf + t * (C + 4) + s0 + jj, bt * v8[jj], tAf, (size_t)S::sSq, bw);
          v8[jj] = (s0 + jj == t) ? 1.f : 0.f;
        }
      }
      put(reinterpret_cast<uint4*>(sTP + (s0 / 8) * 2048u + row * 16u), tc::cvt8(v8), sTP, (size_t)S::kF128, bw);
    }
  } else {
#pragma unroll
    for (int g = 0; g < NTH / 8; ++g)
      *reinterpret_cast<uint4*>(sTP + ((tb0 + 8 * g) / 8) * 2048u + row * 16u) = make_uint4(0u, 0u, 0u, 0u);
  }
  csync<NT>();
  if constexpr (S::kEarlyTail) {
    if (L > 0) {
      ok &= tc::bar_wait(bar_6, spar(L - 1));
      tc::fence_after();
    }
  }
  // (a) N^T to global (its TMEM columns are reused below), piece-major over v:
  //     (k, v) at ((v/4)*D + k)*4 + v%4, so a warp's lanes (consecutive k) write 512
  //     contiguous bytes per piece
  if (L > 0 && fwarp) {
    float* nbase = S::kStageN ? reinterpret_cast<float*>(sKl) : p.Nt + cbase * D * D;
    uint32_t nr[NFD / 8][8];
#pragma unroll
    for (int g = 0; g < NFD / 8; ++g) tc::ld8a(t_n + lane_base + fb0 + 8 * g, nr[g]);
    tc::wait_ld();
#pragma unroll
    for (int g = 0; g < NFD / 8; ++g) {
      tc::pin(nr[g]);
      if (cvalid) {
        const int a0 = fb0 + 8 * g;
        const void* nb0 = S::kStageN ? static_cast<const void*>(sKl) : static_cast<const void*>(p.Nt);
        const size_t nbn = S::kStageN ? (size_t)S::kNT : nmaps * D * D * 4;
        put(reinterpret_cast<float4*>(nbase + ((size_t)(a0 / 4) * D + row) * 4),
            make_float4(u2f(nr[g][0]), u2f(nr[g][1]), u2f(nr[g][2]), u2f(nr[g][3])), nb0, nbn, bw);
        put(reinterpret_cast<float4*>(nbase + ((size_t)(a0 / 4 + 1) * D + row) * 4),
            make_float4(u2f(nr[g][4]), u2f(nr[g][5]), u2f(nr[g][6]), u2f(nr[g][7])), nb0, nbn, bw);
      }
    }
  }
  tc::fence_smem_to_async();
  tc::fence_before();
  // every read of this chunk's K_l / D regions is done (the last step's MMAs have
  // completed, the raw K/Q rows and the v window were read before the loop): with N^T
  // staged there, the producer copies it out and then brings the next chunk's tiles and
  // gates in, while this tail runs
  if constexpr (S::kStageN) {
    asm volatile("bar.sync 10, %0;\n" ::"n"(S::NTA) : "memory");
  } else {
    csync<NT>();
    if (S::kPrefetch && tid == 0) {
      const int nxt = next_of(cur);
      if (nxt < total) load_inputs(nxt);
    }
  }
  // (e) T = (I + A)^-1 (fp32, and the fp16 B tile); then [T ; PT] = [I ; P] T on the tensor core
  solve_tri<C, NT>(tAf, tTf, sTB, tZf);
  tc::fence_smem_to_async();
  tc::fence_before();
  csync<NT>();
  if (tid == 0) {
    tc::fence_after();
    for (int kk = 0; kk < C / 16; ++kk)
      tc::mma(t_k0, tc::desc(sTP + kk * 4096, 2048, 128), tc::desc(sTB + kk * 2 * 16 * C, 16 * C, 128),
              idesc_cc, kk > 0);
    tc::commit(bar_mma);
  }
  wait_mma();
  // [T ; PT] back into the A tile (fp16)
  {
    uint32_t tr[NTH / 8][8];
#pragma unroll
    for (int g = 0; g < NTH / 8; ++g) tc::ld8a(t_k0 + lane_base + tb0 + 8 * g, tr[g]);
    tc::wait_ld();
#pragma unroll
    for (int g = 0; g < NTH / 8; ++g) {
      tc::pin(tr[g]);
      float v8[8];
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) v8[jj] = u2f(tr[g][jj]);
      *reinterpret_cast<uint4*>(sTP + ((tb0 + 8 * g) / 8) * 2048u + row * 16u) = tc::cvt8(v8);
    }
  }
  tc::fence_smem_to_async();
  tc::fence_before();
  csync<NT>();
  // (d) [Kb | X] as the MN-major B tile: (s, f) at (f/8)*(16C) + s*16 + (f%8)*2, f < D: Kb,
  //     f >= D: X.  Rows < C (which hold R in TMEM) write X = beta (V - R) of token row;
  //     rows C..2C-1 write Kb = beta gamma K of token row - C.
  if (quarter * 32 < C) {                      // warps holding rows of R (TMEM loads are warp-wide)
    uint32_t rr[NFD / 8][8];
    if (L > 0) {
#pragma unroll
      for (int g = 0; g < NFD / 8; ++g) tc::ld8a(t_ro + lane_base + fb0 + 8 * g, rr[g]);
      tc::wait_ld();
#pragma unroll
      for (int g = 0; g < NFD / 8; ++g) tc::pin(rr[g]);
    } else {
#pragma unroll
      for (int g = 0; g < NFD / 8; ++g)
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) rr[g][jj] = 0u;
    }
    if (row < C) {
      const float bs = tbeta[row];
#pragma unroll
      for (int g = 0; g < NFD / 8; ++g) {
        const int f0 = fb0 + 8 * g;
        const __nv_bfloat16* ve = reinterpret_cast<const __nv_bfloat16*>(&vr[g]);
        float xf[8];
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) xf[jj] = tok_valid ? bs * (__bfloat162float(ve[jj]) - u2f(rr[g][jj])) : 0.f;
        put(reinterpret_cast<uint4*>(sKX + ((D + f0) / 8) * (16u * C) + row * 16u), tc::cvt8(xf), sKX, (size_t)S::sKX, bw);
      }
    }
  }
  if (row >= C && row < 2 * C) {
    const int sk = row - C;
    const float bg = tbeta[sk] * tgam[sk];
#pragma unroll
    for (int g = 0; g < NFD / 8; ++g) {
      const int f0 = fb0 + 8 * g;
      const uint4 kraw = *reinterpret_cast<const uint4*>(sKQ + (f0 / 8) * 2048u + sk * 16u);
      const __half* ke = reinterpret_cast<const __half*>(&kraw);
      float kf[8];
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) kf[jj] = bg * __half2float(ke[jj]);
      put(reinterpret_cast<uint4*>(sKX + (f0 / 8) * (16u * C) + sk * 16u), tc::cvt8(kf), sKX, (size_t)S::sKX, bw);
    }
  }
  tc::fence_smem_to_async();
  tc::fence_before();
  csync<NT>();
  // (f) [W ; PW] = [T ; PT] Kb,  [U ; PU] = [T ; PT] X   (B MN-major: LBO = 128, SBO = 16C)
  if (tid == 0) {
    tc::fence_after();
    constexpr uint32_t idesc_tx = tc::idesc_f16(D, false, true);
    constexpr uint32_t idesc_tx2 = tc::idesc_f16(kMergeWX ? 2 * D : D, false, true);
    for (int kk = 0; kk < C / 16; ++kk) {
      const uint64_t adesc = tc::desc(sTP + kk * 4096, 2048, 128);
      if constexpr (kMergeWX) {                // B = [Kb | X] as one N = 2D operand
        tc::mma(t_w, adesc, tc::desc(sKX + kk * 256, 128, 16 * C), idesc_tx2, kk > 0);
      } else {
        tc::mma(t_w, adesc, tc::desc(sKX + kk * 256, 128, 16 * C), idesc_tx, kk > 0);
        tc::mma(t_x, adesc, tc::desc(sKX + (D / 8) * (16 * C) + kk * 256, 128, 16 * C), idesc_tx, kk > 0);
      }
    }
    tc::commit(bar_mma);
  }
  wait_mma();
  // (g) outputs.  Lanes 0..C-1: W (fp16), U (fp32), Kt (fp16).  Lanes C..2C-1:
  //     Qt = gamma Q - PW (fp16 hi/lo), O_intra = PU + O_l (fp32).
  __half* oWQ = p.WQ + cbase * 2 * C * D;
  __half* oQK = p.QK + cbase * 2 * C * D;
  float* oU = p.U + cbase * C * D;
  float* oOi = p.Oi + cbase * C * D;
  if (quarter * 32 < 2 * C) {
    const bool isT = row < C, isPT = row >= C && row < 2 * C;
    const int t = isT ? row : row - C;
    const int tr = (isT || isPT) ? t : 0;
    const float gt = (isT || isPT) ? tgam[t] : 0.f;
    const float dct = (isT || isPT) ? sdec[t] : 0.f;
#pragma unroll 1
    for (int j8 = 0; j8 < NFD; j8 += 8) {
      const int f0 = fb0 + j8;
      uint32_t wr[8], xr[8], orr[8];
      tc::ld8a(t_w + lane_base + f0, wr);
      tc::ld8a(t_x + lane_base + f0, xr);
      if (L > 0) {
        tc::ld8a(t_ro + lane_base + f0, orr);
        tc::wait_ld(wr, xr, orr);
      } else {
        tc::wait_ld(wr, xr);
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) orr[jj] = 0u;
      }
      if (isT) {
        const uint4 kraw = *reinterpret_cast<const uint4*>(sKQ + (f0 / 8) * 2048u + t * 16u);
        const __half* ke = reinterpret_cast<const __half*>(&kraw);
        float wv[8], kt[8];
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
          wv[jj] = u2f(wr[jj]);
          kt[jj] = dct * __half2float(ke[jj]);
        }
        const int o16 = ((f0 / 8) * 2 * C + tr) * 8;   // fp16 piece (8 values)
        put(reinterpret_cast<uint4*>(oWQ + o16), tc::cvt8(wv), p.WQ, nmaps * 2 * C * D * 2, bw);
        put(reinterpret_cast<uint4*>(oQK + o16 + C * 8), tc::cvt8(kt), p.QK, nmaps * 2 * C * D * 2, bw);
        put(reinterpret_cast<float4*>(oU + ((f0 / 4) * C + tr) * 4),
            make_float4(u2f(xr[0]), u2f(xr[1]), u2f(xr[2]), u2f(xr[3])), p.U, nmaps * C * D * 4, bw);
        put(reinterpret_cast<float4*>(oU + ((f0 / 4 + 1) * C + tr) * 4),
            make_float4(u2f(xr[4]), u2f(xr[5]), u2f(xr[6]), u2f(xr[7])), p.U, nmaps * C * D * 4, bw);
      } else if (isPT) {
        const uint4 qraw = *reinterpret_cast<const uint4*>(sKQ + (f0 / 8) * 2048u + row * 16u);
        const __half* qe = reinterpret_cast<const __half*>(&qraw);
        float qv[8];
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) qv[jj] = gt * __half2float(qe[jj]) - u2f(wr[jj]);
        uint4 hi, lo;
        tc::split8(qv, hi, lo);
        const int o16 = ((f0 / 8) * 2 * C + tr) * 8;
        put(reinterpret_cast<uint4*>(oWQ + o16 + C * 8), hi, p.WQ, nmaps * 2 * C * D * 2, bw);
        put(reinterpret_cast<uint4*>(oQK + o16), lo, p.QK, nmaps * 2 * C * D * 2, bw);
        put(reinterpret_cast<float4*>(oOi + ((f0 / 4) * C + tr) * 4),
            make_float4(u2f(xr[0]) + u2f(orr[0]), u2f(xr[1]) + u2f(orr[1]), u2f(xr[2]) + u2f(orr[2]),
                        u2f(xr[3]) + u2f(orr[3])), p.Oi, nmaps * C * D * 4, bw);
        put(reinterpret_cast<float4*>(oOi + ((f0 / 4 + 1) * C + tr) * 4),
            make_float4(u2f(xr[4]) + u2f(orr[4]), u2f(xr[5]) + u2f(orr[5]), u2f(xr[6]) + u2f(orr[6]),
                        u2f(xr[7]) + u2f(orr[7])), p.Oi, nmaps * C * D * 4, bw);
      }
    }
  }
  if (tid == 0) put(p.gC + cbase, tgam[C - 1], p.gC, nmaps * 4, bw);
  }  // consumers
  // end of chunk: every role is done with this chunk's shared memory and TMEM
  tc::fence_smem_to_async();
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const int nxt = next_of(cur);
  if (!S::kPrefetch && nxt < total && tid == 0) load_inputs(nxt);
  cur = nxt;
  }  // chunks
  if (!ok) atomicOr(p.status, 1);
  // the last N^T bulk store of this CTA has been read out of shared memory; its writes
  // complete before the CTA exits
  if (producer && lane == 0) tc::bulk_wait_all();
  tc::fence_before();
  __syncthreads();
  if (warp == 0) tc::dealloc(tmem, S::tmem_cols);
}

}  // namespace prism
