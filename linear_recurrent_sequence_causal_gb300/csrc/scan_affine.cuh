// Kernel B (bf16 I/O path): the serial part of the chunkwise scan.
//
// The prep kernel reduces every chunk to its affine state map in factored
// form (see prep_tc.cuh), so what is left is the chain over chunks
// ("Technical Summary: PRISM", §2.1, S_t = S_{t-1} A_t + B_t, composed over a
// chunk):
//   E   = U - W S0^T                      (C x d_v)
//   O   = O_intra + Qt S0^T               (C x d_v), the chunk's outputs o_t = S_t q_t
//   S1  = gamma_C S0 + E^T Kt + N         (d_v x d_k)
// Rows of S evolve independently (A_t acts from the right), so one CTA owns a
// tile of BV rows of S for one (b, h) and walks the chunks in order; W, Qt and
// Kt are shared by the tiles of a head through L2.  The next chunk's operands
// stream in with cp.async while the current one is computed.
//
// The chunk maps arrive piece-major (16-byte column pieces, rows contiguous in
// a piece) and are kept that way in shared memory: every ldmatrix row is one
// 16-byte piece-row, so the copies are linear and the fragment loads are free
// of bank conflicts.
//
// Precision: fp16 operands with fp32 accumulation; the entering state S0 and
// Qt are split into fp16 hi + lo halves (S0 can carry large values written by
// the refinement), so Qt S0^T is formed in three passes and W S0^T in two.
#pragma once

#include "prism_common.cuh"

namespace prism {

struct ScanArgs {
  int B, T, H, L;
  const __half* WQ;      // per chunk [d/8][2][C][8]: W rows, then Qt hi rows
  const __half* QK;      // per chunk [d/8][2][C][8]: Qt lo rows, then Kt rows
  const float* U;
  const float* Oi;
  const float* Nt;       // per chunk N^T piece-major over d_v; null when L == 0
  const float* gC;
  const int* seq_lens;
  float* out;            // [B][T][H][D] fp32
  float* final_state;    // [B][H][D][D] or null
  const float* initial_state;   // [B][H][D][D] entering state, or null (zero)
};

template <int D, int C, int BV>
struct ScanSmem {
  static constexpr int NW = 8;                          // warps per CTA
  static constexpr int LDD = D + 8, LDB = BV + 8;       // padded row-major tiles (S0, E)
  static constexpr uint32_t kTile = C * D * 2;          // one piece-major C x D fp16 map
  static constexpr uint32_t kU = C * BV * 4;            // C x BV fp32, piece-major
  static constexpr uint32_t kN = BV * D * 4;            // BV x D fp32, piece-major
  static constexpr uint32_t kBuf = 4 * kTile + 2 * kU + kN;   // W, Kt, Qt hi, Qt lo, U, O_intra, N
  static constexpr uint32_t oBuf0 = 0;
  static constexpr uint32_t oBuf1 = kBuf;
  static constexpr uint32_t oS0 = 2 * kBuf;             // hi, lo [BV][LDD]
  static constexpr uint32_t oE = oS0 + 2 * BV * LDD * 2;// [C][LDB]
  static constexpr uint32_t bytes = oE + C * LDB * 2;
};

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory"); }

template <int D, int C, int BV>
__global__ void __launch_bounds__(256) scan_affine_kernel(ScanArgs p) {
  using S = ScanSmem<D, C, BV>;
  constexpr int NW = S::NW, LDD = S::LDD, LDB = S::LDB;
  constexpr int NT = D / BV;                            // tiles per head
  extern __shared__ __align__(1024) unsigned char sm[];
  __half* sS0h = reinterpret_cast<__half*>(sm + S::oS0);
  __half* sS0l = sS0h + BV * LDD;
  __half* sE = reinterpret_cast<__half*>(sm + S::oE);

  const int tid = threadIdx.x;
  const int tile = blockIdx.x % NT, bh = blockIdx.x / NT;
  const int h = bh % p.H, b = bh / p.H;
  const int r0 = tile * BV;
  const int H = p.H, T_ = p.T;
  const int NC = (T_ + C - 1) / C;
  const int len = p.seq_lens ? min(max(p.seq_lens[b], 0), T_) : T_;
  const int nchunks = (len + C - 1) / C;
  const size_t cb0 = ((size_t)b * H + h) * NC;          // chunk index base

  using MapE = TileMap<C, BV, NW>;
  using MapS = TileMap<BV, D, NW>;
  Acc16 accS[MapS::kPerWarp];
#pragma unroll
  for (int i = 0; i < MapS::kPerWarp; ++i) accS[i].zero();
  if (p.initial_state) {
    const float* s0 = p.initial_state + ((size_t)b * p.H + h) * D * D;
#pragma unroll
    for (int i = 0; i < MapS::kPerWarp; ++i) {
      if (!MapS::valid(i)) continue;
      const int m0 = MapS::m0(i), n0 = MapS::n0(i);
#pragma unroll
      for (int hh = 0; hh < 2; ++hh)
#pragma unroll
        for (int e = 0; e < 4; ++e) accS[i].v[hh][e] = s0[(size_t)(r0 + m0 + acc_row(e)) * D + n0 + acc_col(hh, e)];
    }
  }

  // Chunk maps are piece-major: fp16 (r, f) at ((f/8)*R + r)*8 + f%8, fp32 at
  // ((f/4)*R + r)*4 + f%4 (R = C for the token-row maps).  The fp16 maps come two to a
  // piece (W then Qt hi, Qt lo then Kt) and are split into one tile each here; N
  // arrives transposed, piece-major over its rows: (a, r) at ((r/4)*D + a)*4 + r%4.
  auto issue_loads = [&](int c, int buf) {
    unsigned char* base = sm + (buf ? S::oBuf1 : S::oBuf0);
    const size_t off = (cb0 + c) * (size_t)C * D;
    // tiles W, Kt, Qt hi, Qt lo: source map and row offset inside its pieces
    const __half* src[4] = {p.WQ + 2 * off, p.QK + 2 * off, p.WQ + 2 * off, p.QK + 2 * off};
    const int roff[4] = {0, C, C, 0};
    constexpr int NP = C * D / 8;                       // 16-byte pieces per map
    for (int idx = tid; idx < 4 * NP; idx += NW * 32) {
      const int m = idx / NP, q = idx % NP;
      cp_async16(base + m * S::kTile + q * 16, src[m] + ((size_t)(q / C) * 2 * C + roff[m] + q % C) * 8);
    }
    // this tile's columns of U and O_intra (pieces r0/4 .. r0/4 + BV/4 - 1, C rows each)
    unsigned char* su = base + 4 * S::kTile;
    constexpr int NU = (BV / 4) * C;
    for (int idx = tid; idx < 2 * NU; idx += NW * 32) {
      const int m = idx / NU, q = idx % NU;
      const float* g = (m == 0 ? p.U : p.Oi) + off + ((size_t)(r0 / 4) * C + q) * 4;
      cp_async16(su + m * S::kU + q * 16, g);
    }
    if (p.Nt) {
      // this tile's rows of N: pieces r0/4 .. r0/4 + BV/4 - 1 of N^T, contiguous
      unsigned char* sn = su + 2 * S::kU;
      const float* g0 = p.Nt + (cb0 + c) * (size_t)D * D + (size_t)(r0 / 4) * D * 4;
      for (int idx = tid; idx < BV * (D / 4); idx += NW * 32) cp_async16(sn + idx * 16, g0 + (size_t)idx * 4);
    }
  };

  if (nchunks > 0) issue_loads(0, 0);
  cp_async_commit();
  for (int c = 0; c < nchunks; ++c) {
    const int buf = c & 1;
    if (c + 1 < nchunks) issue_loads(c + 1, buf ^ 1);
    cp_async_commit();
    const size_t cbase = cb0 + c;
    const int t0 = c * C, nv = min(C, len - t0);
    // entering state of this tile, split into fp16 hi/lo: sS0[r][a]
#pragma unroll
    for (int i = 0; i < MapS::kPerWarp; ++i) {
      if (!MapS::valid(i)) continue;
      const int m0 = MapS::m0(i), n0 = MapS::n0(i);
#pragma unroll
      for (int hh = 0; hh < 2; ++hh)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float x = accS[i].v[hh][e];
          const __half hi = __float2half_rn(x);
          const int o = (m0 + acc_row(e)) * LDD + n0 + acc_col(hh, e);
          sS0h[o] = hi;
          sS0l[o] = __float2half_rn(x - __half2float(hi));
        }
    }
    cp_async_wait<1>();
    __syncthreads();
    const unsigned char* bufp = sm + (buf ? S::oBuf1 : S::oBuf0);
    const unsigned char* sW = bufp;
    const unsigned char* sKt = bufp + S::kTile;
    const unsigned char* sQh = bufp + 2 * S::kTile;
    const unsigned char* sQl = bufp + 3 * S::kTile;
    const float* sUt = reinterpret_cast<const float*>(bufp + 4 * S::kTile);
    const float* sOt = sUt + C * BV;
    const float* sNt = sOt + C * BV;
    // S <- gamma_C S0 + N (the E^T Kt term is added below)
    const float gC = p.gC[cbase];
#pragma unroll
    for (int i = 0; i < MapS::kPerWarp; ++i) {
      if (!MapS::valid(i)) continue;
      const int m0 = MapS::m0(i), n0 = MapS::n0(i);
#pragma unroll
      for (int hh = 0; hh < 2; ++hh)
#pragma unroll
        for (int e = 0; e < 4; e += 2) {
          float2 nn = make_float2(0.f, 0.f);
          const int r = m0 + acc_row(e), a = n0 + acc_col(hh, e);
          if (p.Nt) {                                   // (r, a) of this tile's rows at ((r/4)*D + a)*4 + r%4
            nn.x = sNt[((r / 4) * D + a) * 4 + r % 4];
            nn.y = sNt[((r / 4) * D + a + 1) * 4 + r % 4];
          }
          accS[i].v[hh][e] = fmaf(gC, accS[i].v[hh][e], nn.x);
          accS[i].v[hh][e + 1] = fmaf(gC, accS[i].v[hh][e + 1], nn.y);
        }
    }
    auto pm = [](const unsigned char* base) {           // piece-major C-row fp16 map
      return [base](int row, int col) { return smem_u32(base + ((col / 8) * C + row) * 16); };
    };
    auto rm = [](const __half* base, int ld) {          // padded row-major fp16 tile
      return [base, ld](int row, int col) { return smem_u32(base + row * ld + col); };
    };
    // E = U - W S0^T  and  O = O_intra + Qt S0^T   (tile columns r0 .. r0+BV-1)
#pragma unroll
    for (int i = 0; i < MapE::kPerWarp; ++i) {
      if (!MapE::valid(i)) continue;
      const int m0 = MapE::m0(i), n0 = MapE::n0(i);
      Acc16 e, o;
      e.zero();
      o.zero();
      tile_mma_f16<0, 0>(e, pm(sW), rm(sS0h, LDD), m0, n0, D);
      tile_mma_f16<0, 0>(e, pm(sW), rm(sS0l, LDD), m0, n0, D);
      tile_mma_f16<0, 0>(o, pm(sQh), rm(sS0h, LDD), m0, n0, D);
      tile_mma_f16<0, 0>(o, pm(sQh), rm(sS0l, LDD), m0, n0, D);
      tile_mma_f16<0, 0>(o, pm(sQl), rm(sS0h, LDD), m0, n0, D);
#pragma unroll
      for (int hh = 0; hh < 2; ++hh)
#pragma unroll
        for (int e2 = 0; e2 < 4; e2 += 2) {
          const int t = m0 + acc_row(e2), col = n0 + acc_col(hh, e2);
          const int uo = ((col / 4) * C + t) * 4 + col % 4;
          const float2 u = *reinterpret_cast<const float2*>(sUt + uo);
          const float2 oi = *reinterpret_cast<const float2*>(sOt + uo);
          sE[t * LDB + col] = __float2half_rn(u.x - e.v[hh][e2]);
          sE[t * LDB + col + 1] = __float2half_rn(u.y - e.v[hh][e2 + 1]);
          if (t < nv) {
            float2 ov = make_float2(oi.x + o.v[hh][e2], oi.y + o.v[hh][e2 + 1]);
            *reinterpret_cast<float2*>(p.out + (((size_t)b * T_ + t0 + t) * H + h) * D + r0 + col) = ov;
          }
        }
    }
    __syncthreads();
    // S += E^T Kt
#pragma unroll
    for (int i = 0; i < MapS::kPerWarp; ++i) {
      if (!MapS::valid(i)) continue;
      tile_mma_f16<1, 1>(accS[i], rm(sE, LDB), pm(sKt), MapS::m0(i), MapS::n0(i), C);
    }
    __syncthreads();
  }
  cp_async_wait<0>();
  // padded tokens: zero output columns of this tile
  for (size_t idx = tid; idx < (size_t)(T_ - len) * BV; idx += NW * 32) {
    const int t = len + (int)(idx / BV), col = (int)(idx % BV);
    p.out[(((size_t)b * T_ + t) * H + h) * D + r0 + col] = 0.f;
  }
  if (p.final_state) {
    float* fs = p.final_state + ((size_t)b * H + h) * D * D;
#pragma unroll
    for (int i = 0; i < MapS::kPerWarp; ++i) {
      if (!MapS::valid(i)) continue;
      const int m0 = MapS::m0(i), n0 = MapS::n0(i);
#pragma unroll
      for (int hh = 0; hh < 2; ++hh)
#pragma unroll
        for (int e = 0; e < 4; e += 2)
          *reinterpret_cast<float2*>(fs + (size_t)(r0 + m0 + acc_row(e)) * D + n0 + acc_col(hh, e)) =
              make_float2(accS[i].v[hh][e], accS[i].v[hh][e + 1]);
    }
  }
}

}  // namespace prism
