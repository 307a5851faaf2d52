// Kernel B on tcgen05 (bf16 I/O path, any supported d and chunk): the serial chain of
// the chunkwise scan ("Technical Summary: PRISM", §2.1, S_t = S_{t-1} A_t + B_t
// composed over a chunk), one CTA per (b, h, BV-wide slice of d_v):
//   E   = U - W S0^T                      (C x BV)
//   O   = O_intra + Qt S0^T               (C x BV), the chunk's outputs o_t = S_t q_t
//   S1  = gamma_C S0 + E^T Kt + N         (BV x d_k)
// Both products per chunk run on the tensor core with fp32 accumulators in TMEM:
//   MMA1  [W ; Qt_hi] [S0_hi | S0_lo]^T   (128 x 2BV, K = d_k)
//   MMA2  Kt^T [E_hi | E_lo]               (d_k x 2BV, K = C)
//   MMA1b [Qt_lo ; *] S0_hi^T              (128 x BV), issued after MMA2: it feeds only
//         the outputs, so it runs while the epilogue updates the state
// so W S0^T and Qt S0^T keep ~fp32 accuracy (hi*hi + hi*lo + lo*hi) and E enters
// in two fp16 halves.  The chunk maps arrive in the layout prepare writes (16-byte
// column pieces, in each piece W rows then Qt_hi rows, or Qt_lo rows then Kt rows),
// which is exactly the K-major (resp. MN-major) operand layout, so every chunk is
// five bulk copies into a double buffer.
//
// Sequence split (long sequences with few (b, h) pairs): the chunk chain of a sequence
// is cut into nseg segments of seg_chunks chunks.  Because each chunk acts on the state
// as an affine map, S1 = S0 M + c with M = gamma_C I - W^T Kt and c = U^T Kt + N (the
// state independence of "Technical Summary: PRISM", §2.2, last paragraph), a segment
// composes to one such map.  Phase 1 runs segment 0 in full (its end state is segment
// 1's entering state) and, for every later segment, the same chain twice over: from a
// zero state with U and N (the rows of c) and from the identity without them (the rows
// of M, which evolve exactly like state rows).  scan_seg_chain_kernel then chains the
// entering states S_(s+1) = S_s M_s + c_s, and phase 3 runs segments 1.. in full from
// them.  Rows of the state are independent, so the M rows split over CTAs like S rows.
//
// Threads: warps 0..7 read TMEM lane quarter w % 4 and column half w / 4 (BV / 2 of the
// slice's BV = min(32, d) columns); thread (k, half) keeps those entries of row k of S^T
// (k < d) in fp32 registers across chunks.  Warp 8 issues the copies and the MMAs.  The
// MMAs are M = 128 throughout: where 2C or d is smaller, the extra rows read on into the
// shared memory that follows (the allocation covers it) and their TMEM lanes are ignored.
#pragma once

#include "prism_common.cuh"
#include "tc_common.cuh"

namespace prism {

struct ScanTcArgs {
  int B, T, H;
  const __half* WQ;      // per chunk [d/8][2][C][8]: W rows, then Qt hi rows
  const __half* QK;      // per chunk [d/8][2][C][8]: Qt lo rows, then Kt rows
  const float* U;        // per chunk piece-major [d/4][C][4]
  const float* Oi;       // per chunk piece-major [d/4][C][4]
  const float* Nt;       // per chunk N^T piece-major over d_v: [d/4][d_k][4]; null when L == 0
  const float* gC;       // per chunk gamma_C
  const int* seq_lens;
  float* out;            // [B][T][H][d] fp32
  float* final_state;    // [B][H][d_v][d_k] or null
  const float* initial_state;   // [B][H][d_v][d_k] entering state, or null (zero)
  int* status;           // device error word (bounded waits)
  int* bounds;           // debug build: word of out-of-bounds accesses (else null)
  // Sequence split.  phase 0: one chain per sequence (nseg = 1); phase 1: segment 0 in
  // full plus the affine maps of segments 1..nseg-1; phase 3: segments 1..nseg-1 in full
  // from seg_start.  Arrays [B][H][nseg][D][D], rows d_v (or, for seg_M, d_k) by d_k.
  int nseg, seg_chunks, phase;
  int check_timeout;     // nonzero: a wait that cannot complete first (the failure path, exercised)
  float* seg_start;      // entering state of each segment (slot 0 unused)
  float* seg_c;          // c of each segment (slot 0 unused)
  float* seg_M;          // M of each segment (slot 0 unused)
};

template <int D_, int C>
struct ScanTcSmem {
  static constexpr int D = D_, BV = D < 32 ? D : 32;      // BV columns of d_v (rows of S) per CTA
  static constexpr uint32_t kMap = 2 * C * D * 2;        // one interleaved fp16 map (WQ or QK)
  static constexpr uint32_t kU = C * BV * 4;             // BV columns of U (or O_intra)
  static constexpr uint32_t kN = BV * D * 4;             // BV rows of N
  static constexpr uint32_t oWQ = 0, oQK = kMap, oU = 2 * kMap, oOi = oU + kU, oN = oOi + kU;
  static constexpr uint32_t kBuf = oN + kN;
  static constexpr uint32_t oBuf0 = 0, oBuf1 = kBuf;
  static constexpr uint32_t oS = 2 * kBuf;               // [S_hi | S_lo]^T, MN-major B (K = d_k, N = 2BV)
  static constexpr uint32_t kS = D * 2 * BV * 2;
  static constexpr uint32_t oE = oS + kS;                // [E_hi | E_lo], MN-major B (K = C, N = 2BV)
  static constexpr uint32_t kE = C * 2 * BV * 2;
  static constexpr int LDX = BV + 4;                     // padded row (conflict-free 16-byte accesses)
  static constexpr uint32_t oX = oE + kE;                // Qt_lo S0_hi^T rows, handed to the output rows
  static constexpr uint32_t kX = C * LDX * 4;
  static constexpr uint32_t oBar = oX + kX;              // full[2], mma1, e_ready, mma2, s_ready, mma1b, never
  static constexpr uint32_t oSlot = oBar + 8 * 8;
  // The MMAs run with M = 128; where 2C or d_k is smaller, the rows past them read on into
  // the following shared memory (their TMEM lanes are never read).  The farthest such read:
  // K-major [W ; Qt] or [Qt_lo ; Kt] (128 rows, K = d_k) and MN-major Kt^T (M = 128, K = C)
  // from a chunk map of the second buffer.
  static constexpr uint32_t kRowsA = (D / 8 - 1) * (32u * C) + 128 * 16;
  static constexpr uint32_t kRowsKt = C * 16 + 15 * (32u * C) + (C / 8) * 128;
  static constexpr uint32_t kReach = oBuf1 + oQK + (kRowsA > kRowsKt ? kRowsA : kRowsKt);
  static constexpr uint32_t bytes = (oSlot + 16 > kReach ? oSlot + 16 : kReach);
  static constexpr int NW = 8;                          // epilogue warps
  static constexpr int NT = (NW + 1) * 32;
  // TMEM: the MMA1 and MMA2 accumulators share columns (MMA2 of a chunk is issued once the E
  // epilogue has read MMA1's), then MMA1b's: 3 BV columns; below d = 128 two CTAs share an SM.
  static constexpr uint32_t kTmemCols = 3 * BV <= 64 ? 64 : 3 * BV <= 128 ? 128 : 256;
  static constexpr int kMinBlocks = D < 128 ? 2 : 1;
};

template <int D_, int C>
__global__ void __launch_bounds__(ScanTcSmem<D_, C>::NT, ScanTcSmem<D_, C>::kMinBlocks) scan_tc_kernel(ScanTcArgs p) {
  using S = ScanTcSmem<D_, C>;
  constexpr int D = S::D, BV = S::BV, NSL = D / BV, NW = S::NW, HB = BV / 2, G8 = HB / 8;
  extern __shared__ __align__(1024) unsigned char sm[];
  uint64_t* bar_full = reinterpret_cast<uint64_t*>(sm + S::oBar);   // [2]
  uint64_t* bar_mma1 = bar_full + 2;
  uint64_t* bar_e = bar_full + 3;
  uint64_t* bar_mma2 = bar_full + 4;
  uint64_t* bar_s = bar_full + 5;
  uint64_t* bar_mma1b = bar_full + 6;
  uint64_t* bar_never = bar_full + 7;          // no arrival ever: the timeout check waits on it
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + S::oSlot);
  unsigned char* sS = sm + S::oS;
  unsigned char* sE = sm + S::oE;
  float* sX = reinterpret_cast<float*>(sm + S::oX);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // kind 0: the chain with outputs; 1: the rows of a segment's c; 2: the rows of its M
  int slice = blockIdx.x % NSL, bh = blockIdx.x / NSL, seg = 0, kind = 0;
  const int nseg = p.phase == 0 ? 1 : p.nseg;
  if (p.phase == 1 && bh >= p.B * p.H) {
    const int r = bh - p.B * p.H;
    kind = 1 + r % 2;
    seg = 1 + (r / 2) % (nseg - 1);
    bh = (r / 2) / (nseg - 1);
  } else if (p.phase == 3) {
    seg = 1 + bh % (nseg - 1);
    bh = bh / (nseg - 1);
  }
  const bool outputs = kind == 0, useU = kind != 2;
  const int h = bh % p.H, b = bh / p.H;
  const int v0 = slice * BV;
  const int H = p.H, T_ = p.T;
  const int NC = (T_ + C - 1) / C;
  const int len = p.seq_lens ? min(max(p.seq_lens[b], 0), T_) : T_;
  const int nchunks_seq = (len + C - 1) / C;
  const int c_lo = p.phase == 0 ? 0 : min(seg * p.seg_chunks, nchunks_seq);
  const int c_hi = p.phase == 0 ? nchunks_seq : min(c_lo + p.seg_chunks, nchunks_seq);
  const int nchunks = c_hi - c_lo;             // chunks of this CTA's chain
  const size_t cb0 = ((size_t)b * H + h) * NC + c_lo;
  const bool last_seg = seg == nseg - 1;
  const size_t seg_off = (((size_t)b * H + h) * nseg + seg) * D * D;
  // extents of the arrays the kernel addresses (the debug build checks each access)
  int* bw = p.bounds;
  const size_t nmaps = (size_t)p.B * H * NC, state_bytes = (size_t)p.B * H * D * D * 4;
  const size_t seg_bytes = (size_t)p.B * H * p.nseg * D * D * 4;
  auto copy_in = [&](unsigned char* dst, const void* src, uint32_t bytes, const void* base, size_t extent,
                     uint64_t* bar) {
    if (PRISM_IN_BOUNDS(within(src, bytes, base, extent) && within(dst, bytes, sm, S::bytes), bw))
      tc::bulk_g2s(dst, src, bytes, bar);
  };
  const float* useN = useU ? p.Nt : nullptr;

  if (tid == 0) {
    tc::bar_init(bar_full, 1);
    tc::bar_init(bar_full + 1, 1);
    tc::bar_init(bar_mma1, 1);
    tc::bar_init(bar_e, NW);
    tc::bar_init(bar_mma2, 1);
    tc::bar_init(bar_s, NW);
    tc::bar_init(bar_mma1b, 1);
    tc::bar_init(bar_never, 1);
    tc::bar_fence_init();
  }
  if (warp == 0) tc::alloc(tslot, S::kTmemCols);
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = *tslot;
  const uint32_t t_d1 = tmem, t_d3 = tmem, t_d2 = tmem + 2 * BV;   // 2BV (MMA1, then MMA2) and BV columns
  bool ok = true;
  bool nonfinite = false;                      // a non-finite value written (status bit 1)
  // The failure path on request: nothing is in flight yet (no copy issued, no MMA), so a
  // wait that gives up here leaves nothing behind; it records the error like any other.
  if (p.check_timeout) ok &= tc::bar_wait(bar_never, 0, 1u << 10);

  if (warp == NW) {
    // ================= issuer: chunk copies and MMAs =================
    if (lane == 0) {
      auto load = [&](int c, int buf) {
        unsigned char* base = sm + (buf ? S::oBuf1 : S::oBuf0);
        const size_t cb = cb0 + c;
        tc::bar_expect_tx(bar_full + buf, 2 * S::kMap + (useU ? S::kU : 0) + (outputs ? S::kU : 0) +
                                              (useN ? S::kN : 0));
        copy_in(base + S::oWQ, p.WQ + cb * 2 * C * D, S::kMap, p.WQ, nmaps * 2 * C * D * 2, bar_full + buf);
        copy_in(base + S::oQK, p.QK + cb * 2 * C * D, S::kMap, p.QK, nmaps * 2 * C * D * 2, bar_full + buf);
        if (useU)
          copy_in(base + S::oU, p.U + cb * C * D + (size_t)(v0 / 4) * C * 4, S::kU, p.U, nmaps * C * D * 4,
                  bar_full + buf);
        if (outputs)
          copy_in(base + S::oOi, p.Oi + cb * C * D + (size_t)(v0 / 4) * C * 4, S::kU, p.Oi, nmaps * C * D * 4,
                  bar_full + buf);
        if (useN)
          copy_in(base + S::oN, useN + cb * D * D + (size_t)(v0 / 4) * D * 4, S::kN, useN, nmaps * D * D * 4,
                  bar_full + buf);
      };
      auto wait = [&](uint64_t* bar, uint32_t parity) {
        ok &= tc::bar_wait(bar, parity);
        tc::fence_after();
      };
      constexpr uint32_t idesc_q2 = tc::idesc_f16(2 * BV, false, true);   // [W;Qt_hi] x [S_hi|S_lo]^T
      constexpr uint32_t idesc_q1 = tc::idesc_f16(BV, false, true);       // [Qt_lo;*] x S_hi^T
      constexpr uint32_t idesc_k = tc::idesc_f16(2 * BV, true, true);     // Kt^T x [E_hi|E_lo]
      if (nchunks > 0) load(0, 0);
      if (nchunks > 1) load(1, 1);
      for (int c = 0; c < nchunks; ++c) {
        const int buf = c & 1;
        const unsigned char* base = sm + (buf ? S::oBuf1 : S::oBuf0);
        wait(bar_s, c & 1);                    // state tile of chunk c written, chunk c-1 consumed
        wait(bar_full + buf, (c >> 1) & 1);
        // MMA1a on the state chain; MMA1b (the Qt_lo rows, outputs only) after MMA2, so it
        // runs while the epilogue updates the state
        for (int kk = 0; kk < D / 16; ++kk)
          tc::mma(t_d1, tc::desc(base + S::oWQ + kk * 2 * (2 * C * 16), 2 * C * 16, 128),
                  tc::desc(sS + kk * 256, 128, 16 * D), idesc_q2, kk > 0);
        tc::commit(bar_mma1);
        if (c >= 1 && c + 1 < nchunks) load(c + 1, (c + 1) & 1);   // chunk c-1's buffer is free
        wait(bar_e, c & 1);                    // E tile written
        for (int kk = 0; kk < C / 16; ++kk)
          tc::mma(t_d3, tc::desc(base + S::oQK + C * 16 + kk * 256, 128, 2 * C * 16),
                  tc::desc(sE + kk * 256, 128, 16 * C), idesc_k, kk > 0);
        tc::commit(bar_mma2);
        if (outputs) {
          for (int kk = 0; kk < D / 16; ++kk)
            tc::mma(t_d2, tc::desc(base + S::oQK + kk * 2 * (2 * C * 16), 2 * C * 16, 128),
                    tc::desc(sS + kk * 256, 128, 16 * D), idesc_q1, kk > 0);
          tc::commit(bar_mma1b);
        }
      }
    }
    __syncwarp();
  } else {
    // ================= lanes: epilogues, state in registers =================
    const int k = (warp & 3) * 32 + lane;      // TMEM lane: row of [W;Qt], of E, of S^T
    const int hf = warp >> 2;                  // column half: slice columns hf*16 .. hf*16+15
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const bool krow = k < D;                   // this lane holds a row of S^T
    float st[HB];                              // S^T[k][v0 + hf*HB ..]
    const float* s0 = kind != 0 ? nullptr
                      : seg == 0 ? (p.initial_state ? p.initial_state + ((size_t)b * H + h) * D * D : nullptr)
                                 : p.seg_start + seg_off;
#pragma unroll
    for (int v = 0; v < HB; ++v)
      st[v] = !krow ? 0.f
              : s0  ? get(s0 + (size_t)(v0 + hf * HB + v) * D + k, seg == 0 ? static_cast<const void*>(p.initial_state)
                                                                          : static_cast<const void*>(p.seg_start),
                          seg == 0 ? state_bytes : seg_bytes, bw)
                    : (kind == 2 && v0 + hf * HB + v == k) ? 1.f : 0.f;
    auto write_state = [&]() {                 // [S_hi | S_lo]^T rows: (k, n) at (n/8)*16D + k*16 + (n%8)*2
#pragma unroll
      for (int g = 0; g < HB / 8; ++g) {
        float x[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) x[j] = st[8 * g + j];
        uint4 hi, lo;
        tc::split8(x, hi, lo);
        const int n8 = G8 * hf + g;            // column group of the slice
        if (krow) {
          *reinterpret_cast<uint4*>(sS + n8 * (16u * D) + k * 16u) = hi;
          *reinterpret_cast<uint4*>(sS + (BV / 8 + n8) * (16u * D) + k * 16u) = lo;
        }
      }
      tc::fence_smem_to_async();
      tc::fence_before();
      __syncwarp();
      if (lane == 0) tc::bar_arrive(bar_s);
    };
    write_state();
    for (int c = 0; c < nchunks; ++c) {
      const int buf = c & 1;
      const unsigned char* base = sm + (buf ? S::oBuf1 : S::oBuf0);
      const float* sU = reinterpret_cast<const float*>(base + S::oU);
      const float* sOi = reinterpret_cast<const float*>(base + S::oOi);
      const float* sN = reinterpret_cast<const float*>(base + S::oN);
      const size_t cbase = cb0 + c;
      const int t0 = (c_lo + c) * C, nv = min(C, len - t0);
      const float gC = PRISM_IN_BOUNDS(cbase < nmaps, bw) ? tc::ldg_early(p.gC + cbase) : 0.f;
      ok &= tc::bar_wait(bar_mma1, c & 1);
      tc::fence_after();
      // ---- E = U - W S0^T (lanes < C); O = O_intra + Qt_hi S0^T (lanes C..2C-1) ----
      float ov[HB];
      if ((warp & 3) * 32 < 2 * C) {
        uint32_t d1[2 * G8][8];                // hi columns hf*HB.., lo columns BV + hf*HB..
#pragma unroll
        for (int g = 0; g < G8; ++g) {
          tc::ld8a(t_d1 + lane_base + hf * HB + 8 * g, d1[g]);
          tc::ld8a(t_d1 + lane_base + BV + hf * HB + 8 * g, d1[G8 + g]);
        }
        tc::wait_ld();
        if (k < C) {
#pragma unroll
          for (int g = 0; g < G8; ++g) {
            tc::pin(d1[g]);
            tc::pin(d1[G8 + g]);
            const int pc = (HB / 4) * hf + 2 * g;   // U piece (4 columns) of this group
            float uu[8], e8[8];
            const float4 u0 = useU ? *reinterpret_cast<const float4*>(sU + (pc * C + k) * 4) : make_float4(0.f, 0.f, 0.f, 0.f);
            const float4 u1 = useU ? *reinterpret_cast<const float4*>(sU + ((pc + 1) * C + k) * 4) : make_float4(0.f, 0.f, 0.f, 0.f);
            uu[0] = u0.x; uu[1] = u0.y; uu[2] = u0.z; uu[3] = u0.w;
            uu[4] = u1.x; uu[5] = u1.y; uu[6] = u1.z; uu[7] = u1.w;
#pragma unroll
            for (int j = 0; j < 8; ++j)
              e8[j] = uu[j] - (__uint_as_float(d1[g][j]) + __uint_as_float(d1[G8 + g][j]));
            uint4 hi, lo;
            tc::split8(e8, hi, lo);
            // [E_hi | E_lo]: (r, n) at (n/8)*16C + r*16 + (n%8)*2
            const int n8 = G8 * hf + g;
            *reinterpret_cast<uint4*>(sE + n8 * (16u * C) + k * 16u) = hi;
            *reinterpret_cast<uint4*>(sE + (BV / 8 + n8) * (16u * C) + k * 16u) = lo;
          }
        } else if (outputs && k < 2 * C) {
          const int r = k - C;
#pragma unroll
          for (int g = 0; g < G8; ++g) {
            tc::pin(d1[g]);
            tc::pin(d1[G8 + g]);
            const int pc = (HB / 4) * hf + 2 * g;
            const float4 o0 = *reinterpret_cast<const float4*>(sOi + (pc * C + r) * 4);
            const float4 o1 = *reinterpret_cast<const float4*>(sOi + ((pc + 1) * C + r) * 4);
            const float oi[8] = {o0.x, o0.y, o0.z, o0.w, o1.x, o1.y, o1.z, o1.w};
#pragma unroll
            for (int j = 0; j < 8; ++j)
              ov[8 * g + j] = oi[j] + (__uint_as_float(d1[g][j]) + __uint_as_float(d1[G8 + g][j]));
          }
        }
      }
      tc::fence_smem_to_async();
      tc::fence_before();
      __syncwarp();
      if (lane == 0) tc::bar_arrive(bar_e);
      // ---- S1^T = gamma_C S0^T + Kt^T E + N^T  (lane k, this column half) ----
      ok &= tc::bar_wait(bar_mma2, c & 1);
      tc::fence_after();
      if ((warp & 3) * 32 < D) {                // warps holding rows of S^T (TMEM loads are warp-wide)
        uint32_t d3[2 * G8][8];
#pragma unroll
        for (int g = 0; g < G8; ++g) {
          tc::ld8a(t_d3 + lane_base + hf * HB + 8 * g, d3[g]);
          tc::ld8a(t_d3 + lane_base + BV + hf * HB + 8 * g, d3[G8 + g]);
        }
        tc::wait_ld();
#pragma unroll
        for (int g = 0; g < G8; ++g) {
          tc::pin(d3[g]);
          tc::pin(d3[G8 + g]);
          float nn[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
          if (useN && krow) {
            const int pc = (HB / 4) * hf + 2 * g;
            const float4 n0 = *reinterpret_cast<const float4*>(sN + (pc * D + k) * 4);
            const float4 n1 = *reinterpret_cast<const float4*>(sN + ((pc + 1) * D + k) * 4);
            nn[0] = n0.x; nn[1] = n0.y; nn[2] = n0.z; nn[3] = n0.w;
            nn[4] = n1.x; nn[5] = n1.y; nn[6] = n1.z; nn[7] = n1.w;
          }
#pragma unroll
          for (int j = 0; j < 8; ++j)
            st[8 * g + j] = fmaf(gC, st[8 * g + j],
                                 (__uint_as_float(d3[g][j]) + __uint_as_float(d3[G8 + g][j])) + nn[j]);
        }
      }
      if (!outputs) {                          // affine maps: state rows only
        write_state();
        continue;
      }
      // MMA1b (Qt_lo S0_hi^T) has read the state tile: the new state may replace it; the
      // Qt_lo rows go to the output rows through sX
      ok &= tc::bar_wait(bar_mma1b, c & 1);
      tc::fence_after();
      if ((warp & 3) * 32 < C) {                // TMEM loads are warp-wide; rows k < C are kept
        uint32_t d2[G8][8];
#pragma unroll
        for (int g = 0; g < G8; ++g) tc::ld8a(t_d2 + lane_base + hf * HB + 8 * g, d2[g]);
        tc::wait_ld();
#pragma unroll
        for (int g = 0; g < G8; ++g) {
          tc::pin(d2[g]);
          if (k >= C) continue;
          float* xr = sX + k * S::LDX + hf * HB + 8 * g;
          *reinterpret_cast<float4*>(xr) =
              make_float4(__uint_as_float(d2[g][0]), __uint_as_float(d2[g][1]), __uint_as_float(d2[g][2]), __uint_as_float(d2[g][3]));
          *reinterpret_cast<float4*>(xr + 4) =
              make_float4(__uint_as_float(d2[g][4]), __uint_as_float(d2[g][5]), __uint_as_float(d2[g][6]), __uint_as_float(d2[g][7]));
        }
      }
      write_state();
      asm volatile("bar.sync 1, %0;\n" ::"n"(NW * 32) : "memory");   // the Qt_lo rows are in sX
      if (k >= C && k < 2 * C) {
        const int r = k - C;
        if (r < nv) {
          float* dst = p.out + (((size_t)b * T_ + t0 + r) * H + h) * D + v0 + hf * HB;
#pragma unroll
          for (int g = 0; g < HB / 4; ++g) {
            const float4 x = *reinterpret_cast<const float4*>(sX + r * S::LDX + hf * HB + 4 * g);
            const float4 o = make_float4(ov[4 * g] + x.x, ov[4 * g + 1] + x.y, ov[4 * g + 2] + x.z, ov[4 * g + 3] + x.w);
            nonfinite |= !(isfinite(o.x) && isfinite(o.y) && isfinite(o.z) && isfinite(o.w));
            put(reinterpret_cast<float4*>(dst + 4 * g), o, p.out, (size_t)p.B * T_ * H * D * 4, bw);
          }
        }
      }
    }
    // padded tokens of this chain's token range: zero output columns of this slice
    if (outputs) {
      const int t_lo = max(len, p.phase == 0 ? 0 : seg * p.seg_chunks * C);
      const int t_hi = (p.phase == 0 || last_seg) ? T_ : min(T_, (seg + 1) * p.seg_chunks * C);
      for (size_t idx = tid; idx < (size_t)max(t_hi - t_lo, 0) * BV; idx += NW * 32) {
        const int t = t_lo + (int)(idx / BV), col = (int)(idx % BV);
        put(p.out + (((size_t)b * T_ + t) * H + h) * D + v0 + col, 0.f, p.out, (size_t)p.B * T_ * H * D * 4, bw);
      }
    }
    // end state: the final state (last segment), segment 1's entering state (segment 0 of
    // phase 1), or the rows of c or M
    float* fs = kind == 1 ? p.seg_c + seg_off
              : kind == 2 ? p.seg_M + seg_off
              : (p.phase == 0 || last_seg) ? (p.final_state ? p.final_state + ((size_t)b * H + h) * D * D : nullptr)
              : p.phase == 1 ? p.seg_start + seg_off + (size_t)D * D
              : nullptr;
    if (fs && krow) {
      const void* fbase = (kind == 0 && (p.phase == 0 || last_seg)) ? static_cast<const void*>(p.final_state)
                          : kind == 1 ? static_cast<const void*>(p.seg_c)
                          : kind == 2 ? static_cast<const void*>(p.seg_M)
                                      : static_cast<const void*>(p.seg_start);
      const size_t fext = (kind == 0 && (p.phase == 0 || last_seg)) ? state_bytes : seg_bytes;
#pragma unroll
      for (int v = 0; v < HB; ++v) {
        nonfinite |= !isfinite(st[v]);
        put(fs + (size_t)(v0 + hf * HB + v) * D + k, st[v], fbase, fext, bw);
      }
    }
  }
  // status bit 0: a bounded wait gave up; bit 1: a non-finite value reached an output or
  // an end state (with finite inputs: a value beyond the fp16 range of the tensor-core
  // operands, |delta^(l)| >= 65504, as a diverging refinement chain can reach)
  if (!ok) atomicOr(p.status, 1);
  if (__any_sync(0xffffffffu, nonfinite) && lane == 0) atomicOr(p.status, 2);
  tc::fence_before();
  __syncthreads();
  if (warp == 0) tc::dealloc(tmem, S::kTmemCols);
}

// Phase 2 of the sequence split: the entering state of each segment,
// S_(s+1) = S_s M_s + c_s for s = 1..nseg-2 (S_1 comes from phase 1's segment 0).
// One CTA per (b, h) and 32 rows of the state (rows are independent); the rows stay
// in shared memory from one segment to the next, M_s is staged whole.  fp32 FMA.
constexpr int kSegRows = 32;
template <int D>
struct SegChainSmem {
  static constexpr int LDS = D + 4;            // padded rows: the 4 rows of a warp hit 4 bank groups
  static constexpr size_t bytes = (size_t)(kSegRows * LDS + D * D) * 4;
};
template <int D>
__global__ void __launch_bounds__(256) scan_seg_chain_kernel(ScanTcArgs p) {
  constexpr int LDS = SegChainSmem<D>::LDS, NSL = D >= kSegRows ? D / kSegRows : 1;   // (split only at d = 128)
  extern __shared__ __align__(16) float smc[];
  float* sS = smc;                             // [kSegRows][LDS]
  float* sM = smc + kSegRows * LDS;            // [D][D]
  const int slice = blockIdx.x % NSL, bh = blockIdx.x / NSL;
  const int r0 = slice * kSegRows, tid = threadIdx.x;
  const int row = tid / 8, cg = tid % 8;       // row r0 + row, columns cg + 8 i
  const size_t base = (size_t)bh * p.nseg * D * D;
  int* bw = p.bounds;
  const size_t seg_bytes = (size_t)p.B * p.H * p.nseg * D * D * 4;
  for (int i = tid; i < kSegRows * D / 4; i += 256) {
    const int rr = i / (D / 4), c4 = i % (D / 4);
    *reinterpret_cast<float4*>(sS + rr * LDS + 4 * c4) = get(reinterpret_cast<const float4*>(
        p.seg_start + base + (size_t)D * D + (size_t)(r0 + rr) * D + 4 * c4), p.seg_start, seg_bytes, bw);
  }
  for (int s = 1; s + 1 < p.nseg; ++s) {
    const float* M = p.seg_M + base + (size_t)s * D * D;
    const float* cc = p.seg_c + base + (size_t)s * D * D + (size_t)r0 * D;
    __syncthreads();                           // sS complete; the previous sM fully read
    for (int i = tid; i < D * D / 4; i += 256)
      reinterpret_cast<float4*>(sM)[i] = get(reinterpret_cast<const float4*>(M) + i, p.seg_M, seg_bytes, bw);
    __syncthreads();
    float acc[D / 8];
#pragma unroll
    for (int i = 0; i < D / 8; ++i) acc[i] = get(cc + (size_t)row * D + cg + 8 * i, p.seg_c, seg_bytes, bw);
#pragma unroll 4
    for (int j = 0; j < D; ++j) {
      const float sv = sS[row * LDS + j];
#pragma unroll
      for (int i = 0; i < D / 8; ++i) acc[i] = fmaf(sv, sM[j * D + cg + 8 * i], acc[i]);
    }
    __syncthreads();                           // every thread has read its sS row
    float* dst = p.seg_start + base + (size_t)(s + 1) * D * D + (size_t)r0 * D;
#pragma unroll
    for (int i = 0; i < D / 8; ++i) {
      sS[row * LDS + cg + 8 * i] = acc[i];
      put(dst + (size_t)row * D + cg + 8 * i, acc[i], p.seg_start, seg_bytes, bw);
    }
  }
}

}  // namespace prism
