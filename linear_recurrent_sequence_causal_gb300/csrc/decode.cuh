// Single-token step of the PRISM mixer ("Technical Summary: PRISM", §2.1 and §2.2,
// read token by token): for each (b, h), from the carried state S (d_v x d_k, fp32)
// and the v rows of the w previous tokens,
//   u = sum_j c_j (.) v_{t-j},  r = v_t - u,
//   for l: k^(l) = normalize(W_k^(l) u), p^(l) = W_p^(l) u, beta^(l) = sigmoid(w_beta^(l) . u),
//          delta^(l) = GELU(p^(l) (.) r), r -= delta^(l)
//   S <- alpha (S - beta (S k) k^T) + beta v k^T + sum_l beta^(l) delta^(l) k^(l)^T,   o = S q,
// then the history moves by one token.
//
// Every product of the step is matrix-vector sized, so the step is a chain of memory
// latencies; the kernel is laid out to pay about one of them:
//   - the CTAs of one head h form a cluster of D / RB CTAs; CTA c owns rows
//     [c RB, (c+1) RB) of S, of each W_k^(l), W_p^(l) and of r, delta, for BB sequences
//     at once (the weight rows are read once for the BB sequences);
//   - a thread owns fixed float4 columns of its rows: its part of S stays in registers
//     from the load to the store, and the weight rows it multiplies are copied into
//     shared memory by the same thread (cp.async), so no barrier guards the weight ring;
//   - k_hat^(l) = W_k^(l) u and p^(l) = W_p^(l) u depend on the anchor alone, so every
//     weight slice is requested at the start (as many as the ring holds) and the L
//     refinement steps need one cluster exchange in all: each CTA stores its rows of
//     every k_hat^(l) into the shared memory of every CTA of the cluster (distributed
//     shared memory), and after one cluster barrier each has the whole vectors locally
//     (the norm included); nothing remote is read, so no CTA waits for another to exit;
//   - a row's dot products are summed over the lanes that hold its columns, all of a
//     thread's rows at once (group_sums), which leaves each lane with one (sequence, row)
//     pair: the residual chain and GELU run once per lane, not once per row per lane.
// Everything is fp32 on the CUDA cores.
#pragma once

#include "prism_common.cuh"

namespace prism {

struct DecodeArgs {
  int B, H, w, L;
  int nbuf;                 // weight slices the shared-memory ring holds (2 .. 2L; 0 if L = 0)
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
  int* bounds;              // debug build: word of out-of-bounds accesses (else null)
};

constexpr int kDecodeMaxW = 8;   // longest conv history the entry point accepts

// Geometry and shared-memory layout (offsets in floats) of one CTA.
template <int D, int BB>
struct DecodeGeom {
  static constexpr int RB = D < 32 ? D : 32;        // rows of S per CTA
  static constexpr int NCL = D / RB;                // CTAs per cluster (one head, BB sequences)
  static constexpr int NT = D == 16 ? 64 : 256;     // threads
  static constexpr int GW = D / 4;                  // lanes holding one row (a float4 each)
  static constexpr int J = RB * D / 4 / NT;         // float4s of a row block per thread
  static constexpr int RSTEP = NT / GW;             // row distance between a thread's float4s
  static constexpr int kSlice = RB * D;             // one weight slice
  // [nbuf][RB][D] ring | this CTA's rows of S: [BB][RB][D] | u, k, q, v: [BB][4][D] |
  // w_beta: [L][D] | k_hat^(l), whole: [L][BB][D] | write values of this CTA's rows:
  // [L][BB][RB] | the history on this CTA's columns: [BB][w][RB]
  static __host__ __device__ int oS(int nbuf) { return nbuf * kSlice; }
  static __host__ __device__ int oVec(int nbuf) { return oS(nbuf) + BB * kSlice; }
  static __host__ __device__ int oWb(int nbuf) { return oVec(nbuf) + BB * 4 * D; }
  static __host__ __device__ int oKh(int nbuf, int L) { return oWb(nbuf) + L * D; }
  static __host__ __device__ int oDl(int nbuf, int L) { return oKh(nbuf, L) + L * BB * D; }
  static __host__ __device__ int oHs(int nbuf, int L) { return oDl(nbuf, L) + L * BB * RB; }
  static __host__ __device__ size_t bytes(int nbuf, int L, int w) {
    return sizeof(float) * (size_t)(oHs(nbuf, L) + BB * w * RB);
  }
};

template <int N>
struct Count {
  static constexpr int value = N;
};

// Sum over the GW lanes that hold one row (all lanes of the warp take part).
template <int GW>
__device__ __forceinline__ float row_sum(float x) {
#pragma unroll
  for (int o = GW / 2; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// Sums of NV values over the GW lanes of a row group at once (NV <= GW, powers of two):
// at each of the first log2(NV) butterfly levels a lane keeps half of its values and sends
// the other half, so on return lane g of the group holds, in every one of its GW / NV
// lanes, the full sum of value g / (GW / NV): log2(GW) + NV - 1 shuffles instead of
// NV log2(GW).
template <int NV, int GW>
__device__ __forceinline__ float group_sums(float (&x)[NV]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int lev = 0; (NV >> lev) > 1; ++lev) {
    const int n = NV >> lev, o = (GW / 2) >> lev;
    const bool upper = lane & o;
#pragma unroll
    for (int i = 0; i < n / 2; ++i) {
      const float send = upper ? x[i] : x[i + n / 2];
      const float keep = upper ? x[i + n / 2] : x[i];
      x[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
    }
  }
  float t = x[0];
#pragma unroll
  for (int o = GW / (2 * NV); o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
  return t;
}

__device__ __forceinline__ float dot4(float4 a, float4 b) {
  return fmaf(a.x, b.x, fmaf(a.y, b.y, fmaf(a.z, b.z, a.w * b.w)));
}

// Waits until at most n of this thread's cp.async groups are pending (n clamped to 7,
// which only waits longer).
__device__ __forceinline__ void cp_async_wait_upto(int n) {
  switch (n) {
    case 0: asm volatile("cp.async.wait_group 0;\n" ::: "memory"); break;
    case 1: asm volatile("cp.async.wait_group 1;\n" ::: "memory"); break;
    case 2: asm volatile("cp.async.wait_group 2;\n" ::: "memory"); break;
    case 3: asm volatile("cp.async.wait_group 3;\n" ::: "memory"); break;
    case 4: asm volatile("cp.async.wait_group 4;\n" ::: "memory"); break;
    case 5: asm volatile("cp.async.wait_group 5;\n" ::: "memory"); break;
    case 6: asm volatile("cp.async.wait_group 6;\n" ::: "memory"); break;
    default: asm volatile("cp.async.wait_group 7;\n" ::: "memory"); break;
  }
}

// This thread's float4s of rows r0 .. r0+RB-1 of weight matrix m (W_k^(l) for m = 2l,
// W_p^(l) for m = 2l + 1) into ring slot m % nbuf, as one cp.async group.
template <int D, int BB>
__device__ __forceinline__ void decode_issue_slice(const DecodeArgs& p, int h, int m, int r0,
                                                   float* ring, size_t smem_n) {
  using G = DecodeGeom<D, BB>;
  const int l = m >> 1;
  const float* W = (m & 1) ? p.Wp : p.Wk;
  const float* g = W + (((size_t)h * p.L + l) * D + r0) * D;
  float* dst = ring + (size_t)(m % p.nbuf) * G::kSlice;
  const size_t wbytes = (size_t)p.H * p.L * D * D * sizeof(float);
#pragma unroll
  for (int j = 0; j < G::J; ++j) {
    const int f = threadIdx.x + G::NT * j;
    if (PRISM_IN_BOUNDS(within(g + 4 * (size_t)f, 16, W, wbytes) && within(dst + 4 * f, 16, ring, smem_n), p.bounds))
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(smem_u32(dst + 4 * f)),
                   "l"(g + 4 * (size_t)f) : "memory");
  }
  asm volatile("cp.async.commit_group;\n" ::: "memory");
}

__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;\n" : "=r"(r));
  return r;
}
// Address of the same shared-memory variable in CTA `rank` of the cluster.
__device__ __forceinline__ float* cluster_map_mut(float* p, uint32_t rank) {
  uint64_t out;
  asm volatile("mapa.u64 %0, %1, %2;\n" : "=l"(out) : "l"(reinterpret_cast<uint64_t>(p)), "r"(rank));
  return reinterpret_cast<float*>(out);
}

template <class T, int D, int BB>
__global__ void __cluster_dims__(DecodeGeom<D, BB>::NCL, 1, 1)
    __launch_bounds__(DecodeGeom<D, BB>::NT, D <= 32 ? 4 : 2) decode_kernel(DecodeArgs p) {
  using G = DecodeGeom<D, BB>;
  constexpr int RB = G::RB, NCL = G::NCL, NT = G::NT, GW = G::GW, J = G::J;
  extern __shared__ __align__(128) float smf[];
  const int L = p.L, nbuf = p.nbuf, w = p.w;
  float* ring = smf;
  float* sS = smf + G::oS(nbuf);
  float* svec = smf + G::oVec(nbuf);               // [BB][u, k, q, v][D]
  float* swb = smf + G::oWb(nbuf);
  float* skh = smf + G::oKh(nbuf, L);
  float* sdl = smf + G::oDl(nbuf, L);
  float* shs = smf + G::oHs(nbuf, L);

  const int tid = threadIdx.x;
  const uint32_t crank = cluster_rank();           // which rows of this head
  const int grp = blockIdx.x / NCL;                // (batch group, head)
  const int h = grp % p.H, b0 = (grp / p.H) * BB;
  const int r0 = (int)crank * RB;
  const int c0 = 4 * (tid % GW);                   // this thread's columns c0 .. c0+3
  const int row0 = tid / GW;                       // its rows row0 + RSTEP j (within the block)

  const int nslice = 2 * L;
  const int nfirst = nslice < nbuf ? nslice : nbuf;
  // extents of the arrays this CTA touches (the debug build checks every access)
  int* bw = p.bounds;
  const size_t smem_n = dyn_smem_bytes(), nBH = (size_t)p.B * p.H;
  const size_t tok_bytes = nBH * D * sizeof(T), hist_bytes = nBH * w * D * sizeof(T);
  const size_t state_bytes = nBH * D * D * sizeof(float);
  // another CTA's shared memory may be written only once that CTA runs: this barrier
  // phase (waited for before the first such store) says so
  cluster_arrive_relaxed();

  // the anchor's inputs first, from every warp before any bulk request (they gate the
  // first barrier): thread (bb, c) reads history column c, its taps and the token's
  // k, q, v entries (BB D <= NT threads)
  const int vb = tid / D, vc = tid % D;
  const bool vthread = tid < BB * D && b0 + vb < p.B;
  const size_t vbh = (size_t)(b0 + vb) * p.H + h;
  float hx[kDecodeMaxW], cx[kDecodeMaxW], kv = 0.f, qv = 0.f, vv = 0.f;
  if (vthread) {
    const T* hist = static_cast<const T*>(p.vhist) + vbh * w * D + vc;
#pragma unroll
    for (int t = 0; t < kDecodeMaxW; ++t)
      if (t < w) {
        hx[t] = Elem<T>::to_f(get(hist + (size_t)t * D, p.vhist, hist_bytes, bw));
        cx[t] = get(p.conv_w + ((size_t)h * w + (w - 1 - t)) * D + vc, p.conv_w,
                    (size_t)p.H * w * D * sizeof(float), bw);   // tap j = w - t
      }
    kv = Elem<T>::to_f(get(static_cast<const T*>(p.k) + vbh * D + vc, p.k, tok_bytes, bw));
    qv = Elem<T>::to_f(get(static_cast<const T*>(p.q) + vbh * D + vc, p.q, tok_bytes, bw));
    vv = Elem<T>::to_f(get(static_cast<const T*>(p.v) + vbh * D + vc, p.v, tok_bytes, bw));
  }
  bool valid[BB];
  float la[BB], be[BB];
#pragma unroll
  for (int bb = 0; bb < BB; ++bb) {
    valid[bb] = b0 + bb < p.B;
    const size_t bh = (size_t)(b0 + bb) * p.H + h;
    la[bb] = valid[bb] ? get(p.log_alpha + bh, p.log_alpha, nBH * sizeof(float), bw) : 0.f;
    be[bb] = valid[bb] ? get(p.beta + bh, p.beta, nBH * sizeof(float), bw) : 0.f;
  }
  __syncthreads();
  // cp.async groups, oldest first: w_beta | the first nfirst weight slices | this CTA's
  // rows of S (each thread copies the float4s it later reads) | refills of the ring
  for (int i = tid; i < L * D / 4; i += NT)
    if (PRISM_IN_BOUNDS(within(p.wbeta + (size_t)h * L * D + 4 * (size_t)i, 16, p.wbeta,
                               (size_t)p.H * L * D * sizeof(float)) &&
                        within(swb + 4 * i, 16, smf, smem_n), bw))
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(smem_u32(swb + 4 * i)),
                   "l"(p.wbeta + (size_t)h * L * D + 4 * (size_t)i) : "memory");
  asm volatile("cp.async.commit_group;\n" ::: "memory");
  for (int m = 0; m < nfirst; ++m) decode_issue_slice<D, BB>(p, h, m, r0, ring, smem_n);
#pragma unroll
  for (int bb = 0; bb < BB; ++bb)
    if (valid[bb]) {
      const float* st = p.state + (((size_t)(b0 + bb) * p.H + h) * D + r0) * D;
#pragma unroll
      for (int j = 0; j < J; ++j) {
        const int f = tid + NT * j;
        if (PRISM_IN_BOUNDS(within(st + 4 * (size_t)f, 16, p.state, state_bytes) &&
                            within(sS + bb * G::kSlice + 4 * f, 16, smf, smem_n), bw))
          asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(smem_u32(sS + bb * G::kSlice + 4 * f)),
                       "l"(st + 4 * (size_t)f) : "memory");
      }
    }
  asm volatile("cp.async.commit_group;\n" ::: "memory");

  // anchor u (every CTA forms it in full: w D multiply-adds), and the token's vectors
  if (tid < BB * D) {
    float* vec = svec + vb * 4 * D;
    float u = 0.f;
    if (vthread) {
      const bool own = (unsigned)(vc - r0) < (unsigned)RB;   // kept for the shift at the end
#pragma unroll
      for (int t = kDecodeMaxW - 1; t >= 0; --t)   // j = 1 .. w: the newest row first
        if (t < w) {
          u = fmaf(cx[t], hx[t], u);
          if (own) put(shs + (vb * w + t) * RB + (vc - r0), hx[t], smf, smem_n, bw);
        }
    }
    put(vec + vc, u, smf, smem_n, bw);
    put(vec + D + vc, kv, smf, smem_n, bw);
    put(vec + 2 * D + vc, qv, smf, smem_n, bw);
    put(vec + 3 * D + vc, vv, smf, smem_n, bw);
  }
  cp_async_wait_upto(nfirst + 1);                  // w_beta is in (the rest may still fly)
  __syncthreads();

  // Pair q = bb J + j is (sequence bb, this thread's row j); after group_sums lane g of a
  // row group holds pair g / (GW / NV) and runs its residual chain (every lane of the
  // pair's range alike, the first one stores).
  constexpr int NV = BB * J;
  const int g = tid % GW;
  const int q_own = g / (GW / NV), bb_own = q_own / J;
  const int row_own = row0 + G::RSTEP * (q_own % J);            // within the block
  const bool writer = g % (GW / NV) == 0;
  float4 u4[BB];
#pragma unroll
  for (int bb = 0; bb < BB; ++bb) u4[bb] = get(reinterpret_cast<const float4*>(svec + bb * 4 * D + c0), smf, smem_n, bw);
  float r = get(svec + bb_own * 4 * D + 3 * D + r0 + row_own, smf, smem_n, bw) -
            get(svec + bb_own * 4 * D + r0 + row_own, smf, smem_n, bw);

  const bool gelu = !(p.flags & 1u);
  cluster_wait();                                  // every CTA of the cluster has started
  // NL refinement steps from l: their 2 NL slices are used together (independent sums)
  auto refine = [&](auto count, int l) {
    constexpr int NL = decltype(count)::value;
    // this thread's cp.async groups younger than slice e = 2 (l + NL) - 1: the later first
    // slices, the S group and the refills issued so far, or only later refills
    const int e = 2 * (l + NL) - 1;
    const int refills = max(0, min(2 * l, nslice - nbuf));
    cp_async_wait_upto(e < nfirst ? nfirst - e + refills : refills - (e - nbuf + 1));
    float xk[NL][NV], xp[NL][NV], z[NL][BB];
#pragma unroll
    for (int s = 0; s < NL; ++s) {
      const float* slk = ring + (size_t)((2 * (l + s)) % nbuf) * G::kSlice;
      const float* slp = ring + (size_t)((2 * (l + s) + 1) % nbuf) * G::kSlice;
#pragma unroll
      for (int j = 0; j < J; ++j) {
        const float4 wk = get(reinterpret_cast<const float4*>(slk + 4 * (tid + NT * j)), smf, smem_n, bw);
        const float4 wp = get(reinterpret_cast<const float4*>(slp + 4 * (tid + NT * j)), smf, smem_n, bw);
#pragma unroll
        for (int bb = 0; bb < BB; ++bb) {
          xk[s][bb * J + j] = dot4(wk, u4[bb]);
          xp[s][bb * J + j] = dot4(wp, u4[bb]);
        }
      }
      const float4 wb4 = get(reinterpret_cast<const float4*>(swb + (l + s) * D + c0), smf, smem_n, bw);
#pragma unroll
      for (int bb = 0; bb < BB; ++bb) z[s][bb] = dot4(wb4, u4[bb]);
    }
    float kh[NL], pr[NL], bl[NL];
#pragma unroll
    for (int s = 0; s < NL; ++s) {
      kh[s] = group_sums<NV, GW>(xk[s]);
      pr[s] = group_sums<NV, GW>(xp[s]);
      bl[s] = sigmoidf(group_sums<BB, GW>(z[s]));              // lane g: sequence bb_own
    }
    // the slots' float4s were read by this thread (the sums above consumed them): the
    // same thread refills them
#pragma unroll
    for (int s = 0; s < 2 * NL; ++s)
      if (2 * l + s + nbuf < nslice) decode_issue_slice<D, BB>(p, h, 2 * l + s + nbuf, r0, ring, smem_n);
#pragma unroll
    for (int s = 0; s < NL; ++s) {
      const float x = pr[s] * r;
      const float dl = gelu ? gelu_erf(x) : x;
      r -= dl;
      if (writer) {
        // this CTA's entry of k_hat^(l) into every CTA of the cluster (itself included)
        const int at = ((l + s) * BB + bb_own) * D + r0 + row_own;
        if (PRISM_IN_BOUNDS(at >= 0 && at < L * BB * D && within(skh + at, 4, smf, smem_n), bw))
#pragma unroll
          for (int c = 0; c < NCL; ++c) cluster_map_mut(skh, (uint32_t)c)[at] = kh[s];
        put(sdl + ((l + s) * BB + bb_own) * RB + row_own, bl[s] * dl, smf, smem_n, bw);
      }
    }
  };
  int l = 0;
  if (nbuf >= 4)
    for (; l + 1 < L; l += 2) refine(Count<2>{}, l);
  for (; l < L; ++l) refine(Count<1>{}, l);
  // every CTA's entries of k_hat are stored, and every CTA has read the history (its
  // anchor); after this barrier nothing outside this CTA is touched but global memory
  cluster_arrive();
  cluster_wait();

  // this thread's part of S (its own copies: no barrier needed)
  asm volatile("cp.async.wait_group 0;\n" ::: "memory");
  float4 S[BB][J];
#pragma unroll
  for (int bb = 0; bb < BB; ++bb)
#pragma unroll
    for (int j = 0; j < J; ++j)
      S[bb][j] = valid[bb] ? get(reinterpret_cast<const float4*>(sS + bb * G::kSlice + 4 * (tid + NT * j)), smf,
                                 smem_n, bw)
                           : make_float4(0.f, 0.f, 0.f, 0.f);

  // S <- alpha (S - beta (S k) k^T) + beta v k^T = alpha S + a k^T with
  // a = beta (v - alpha S k), on this thread's part
  {
    float4 k4[BB];
    float x[NV];
#pragma unroll
    for (int bb = 0; bb < BB; ++bb) {
      k4[bb] = get(reinterpret_cast<const float4*>(svec + bb * 4 * D + D + c0), smf, smem_n, bw);
#pragma unroll
      for (int j = 0; j < J; ++j) x[bb * J + j] = dot4(S[bb][j], k4[bb]);
    }
    const float sk = group_sums<NV, GW>(x);
    float al_own = la[0], be_own = be[0];
#pragma unroll
    for (int bb = 1; bb < BB; ++bb)
      if (bb_own == bb) { al_own = la[bb]; be_own = be[bb]; }
    const float a_own = be_own * (get(svec + bb_own * 4 * D + 3 * D + r0 + row_own, smf, smem_n, bw) - expf(al_own) * sk);
    const int base = (threadIdx.x & 31) - g;                      // the row group's first lane
#pragma unroll
    for (int bb = 0; bb < BB; ++bb) {
      const float alpha = expf(la[bb]);
#pragma unroll
      for (int j = 0; j < J; ++j) {
        const float a = __shfl_sync(0xffffffffu, a_own, base + (bb * J + j) * (GW / NV));
        S[bb][j].x = fmaf(a, k4[bb].x, alpha * S[bb][j].x);
        S[bb][j].y = fmaf(a, k4[bb].y, alpha * S[bb][j].y);
        S[bb][j].z = fmaf(a, k4[bb].z, alpha * S[bb][j].z);
        S[bb][j].w = fmaf(a, k4[bb].w, alpha * S[bb][j].w);
      }
    }
  }
  // + sum_l D^(l) k^(l)^T, k^(l) = k_hat^(l) / |k_hat^(l)|: the GW lanes of a row hold all
  // D entries between them, so the norm is a row sum (the same in every lane and CTA)
  for (int l = 0; l < L; ++l) {
#pragma unroll
    for (int bb = 0; bb < BB; ++bb) {
      const int lb = l * BB + bb;
      const float4 kl = get(reinterpret_cast<const float4*>(skh + lb * D + c0), smf, smem_n, bw);
      const float inv = rsqrtf(row_sum<GW>(dot4(kl, kl)) + 1e-6f);
#pragma unroll
      for (int j = 0; j < J; ++j) {
        const float dl = get(sdl + lb * RB + row0 + G::RSTEP * j, smf, smem_n, bw) * inv;
        S[bb][j].x = fmaf(dl, kl.x, S[bb][j].x);
        S[bb][j].y = fmaf(dl, kl.y, S[bb][j].y);
        S[bb][j].z = fmaf(dl, kl.z, S[bb][j].z);
        S[bb][j].w = fmaf(dl, kl.w, S[bb][j].w);
      }
    }
  }

  // store S, and o = S q on this CTA's rows
  {
    float x[NV];
#pragma unroll
    for (int bb = 0; bb < BB; ++bb) {
      const size_t bh = (size_t)(b0 + bb) * p.H + h;
      const float4 q4 = get(reinterpret_cast<const float4*>(svec + bb * 4 * D + 2 * D + c0), smf, smem_n, bw);
      float4* st = reinterpret_cast<float4*>(p.state + (bh * D + r0) * D);
#pragma unroll
      for (int j = 0; j < J; ++j) {
        if (valid[bb]) put(st + tid + NT * j, S[bb][j], p.state, state_bytes, bw);
        x[bb * J + j] = dot4(S[bb][j], q4);
      }
    }
    const float o = group_sums<NV, GW>(x);
    if (writer && b0 + bb_own < p.B)
      put(p.out + ((size_t)(b0 + bb_own) * p.H + h) * D + r0 + row_own, o, p.out, nBH * D * sizeof(float), bw);
  }
  // the history moves by one token: each CTA writes its own columns (read at the start)
  for (int i = tid; i < BB * RB; i += NT) {
    const int bb = i / RB, c = i % RB;
    if (b0 + bb < p.B) {
      const size_t bh = (size_t)(b0 + bb) * p.H + h;
      T* hist = static_cast<T*>(p.vhist) + bh * w * D + r0 + c;
      for (int t = 0; t + 1 < w; ++t)
        put(hist + (size_t)t * D, Elem<T>::from_f(get(shs + (bb * w + t + 1) * RB + c, smf, smem_n, bw)), p.vhist,
            hist_bytes, bw);
      put(hist + (size_t)(w - 1) * D, Elem<T>::from_f(get(svec + bb * 4 * D + 3 * D + r0 + c, smf, smem_n, bw)),
          p.vhist, hist_bytes, bw);
    }
  }
}

}  // namespace prism
