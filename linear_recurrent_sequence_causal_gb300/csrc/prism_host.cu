// Host-to-host forward pass: prism_forward on host buffers, the copies in, the kernels and
// the copies out overlapped piece by piece on three caller-owned streams.
//
// Pieces are groups of whole sequences when B > 1 and chunk-aligned token segments when
// B = 1.  A token segment continues the previous one: it starts from that segment's final
// state and reads the last w v rows before it as the anchor's history (in v's own layout,
// PRISM_FLAG_VHIST_TOKEN_MAJOR), so the pieces give the result of one call.  Only host
// code lives here; every step of the layer runs in the kernels behind prism_forward and
// prism_forward_from.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <vector>

#include "prism.h"

namespace prism {
int forward_from_impl(const prism_dims* dims, const void* q, const void* k, const void* v,
                      const float* log_alpha, const float* beta, const float* conv_w,
                      const float* Wk, const float* Wp, const float* wbeta,
                      const float* initial_state, const void* v_hist, float* out,
                      float* final_state, const int32_t* seq_lens, void* workspace,
                      size_t workspace_bytes, void* stream, bool weights_ready);
}

namespace {

size_t r256(size_t x) { return (x + 255) & ~size_t(255); }
size_t esize(const prism_dims* d) { return d->dtype == PRISM_BF16 ? 2 : 4; }

// Boundaries of the pieces: bounds[0] = 0 < bounds[1] < ... < bounds[n] = B (B > 1) or T.
std::vector<int> plan(const prism_dims* d, int max_pieces, size_t min_piece_bytes) {
  const size_t moved = (size_t)d->B * d->T * d->H * d->d_k * (3 * esize(d) + 4);
  long long pieces = max_pieces;
  if (min_piece_bytes > 0)
    pieces = std::max<long long>(1, std::min<long long>(pieces, (long long)(moved / min_piece_bytes)));
  std::vector<int> b{0};
  if (d->B > 1) {
    // a piece's log_alpha and beta start 16-byte aligned: its first sequence times T*H
    // floats is a multiple of 4
    const long long th = (long long)d->T * d->H;
    const long long m = th % 4 == 0 ? 1 : (th % 2 == 0 ? 2 : 4);
    const long long n = std::min<long long>(pieces, d->B);
    const long long step = ((d->B + n - 1) / n + m - 1) / m * m;
    for (long long a = step; a < d->B; a += step) b.push_back((int)a);
    b.push_back(d->B);
    return b;
  }
  const int C = d->chunk;
  const long long n = std::max<long long>(1, std::min<long long>(pieces, d->T / std::max(C, d->conv_width)));
  long long step = (d->T + n - 1) / n;
  step = (step + C - 1) / C * C;
  for (long long t = step; t < d->T; t += step) b.push_back((int)t);
  b.push_back(d->T);
  return b;
}

// Device arena: inputs, outputs and two states at full size, one seq_lens slot per piece
// and a workspace for the largest piece.
struct Arena {
  size_t q, k, v, la, be, cw, wk, wp, wb, out, st0, st1, lens, lens_slot, ws, ws_bytes, total;
};

Arena arena_layout(const prism_dims* d, const std::vector<int>& b) {
  Arena A{};
  const size_t D = d->d_k, tok = (size_t)d->B * d->T * d->H, L = d->L;
  size_t cur = 0;
  auto take = [&](size_t bytes) {
    const size_t at = cur;
    cur += r256(bytes);
    return at;
  };
  A.q = take(tok * D * esize(d));
  A.k = take(tok * D * esize(d));
  A.v = take(tok * D * esize(d));
  A.la = take(tok * 4);
  A.be = take(tok * 4);
  A.cw = take((size_t)d->H * d->conv_width * D * 4);
  A.wk = take((size_t)d->H * L * D * D * 4);
  A.wp = take((size_t)d->H * L * D * D * 4);
  A.wb = take((size_t)d->H * L * D * 4);
  A.out = take(tok * D * 4);
  A.st0 = take((size_t)d->B * d->H * D * D * 4);
  A.st1 = take((size_t)d->B * d->H * D * D * 4);
  int step = 0;
  for (size_t i = 0; i + 1 < b.size(); ++i) step = std::max(step, b[i + 1] - b[i]);
  A.lens_slot = r256((size_t)step * 4);
  A.lens = take(A.lens_slot * (b.size() - 1));
  prism_dims pd = *d;
  if (d->B > 1) pd.B = step; else { pd.T = step; pd.flags |= PRISM_FLAG_VHIST_TOKEN_MAJOR; }
  A.ws_bytes = prism_workspace_bytes(&pd);
  A.ws = take(A.ws_bytes);
  A.total = cur;
  return A;
}

int check(const prism_dims* d, int max_pieces) {
  size_t offs[PRISM_WS_COUNT];
  const int rc = prism_workspace_layout(d, offs, PRISM_WS_COUNT);   // the dims checks
  if (rc != PRISM_OK) return rc;
  if (d->flags & PRISM_FLAG_VHIST_TOKEN_MAJOR) return PRISM_ERR_INVALID_ARG;   // no history here
  if (max_pieces < 1 || max_pieces > PRISM_HOST_MAX_PIECES) return PRISM_ERR_INVALID_ARG;
  return PRISM_OK;
}

// Events of one call, destroyed when the call returns (CUDA releases a recorded event
// once the device has passed it).
struct Events {
  std::vector<cudaEvent_t> ev;
  ~Events() {
    for (cudaEvent_t e : ev) cudaEventDestroy(e);
  }
  cudaEvent_t make() {
    cudaEvent_t e = nullptr;
    if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) return nullptr;
    ev.push_back(e);
    return e;
  }
};

}  // namespace

extern "C" PRISM_API int prism_host_plan(const prism_dims* dims, int max_pieces,
                                         size_t min_piece_bytes, int* n_pieces, int* bounds) {
  const int rc = check(dims, max_pieces);
  if (rc != PRISM_OK) return rc;
  if (!n_pieces || !bounds) return PRISM_ERR_INVALID_ARG;
  const std::vector<int> b = plan(dims, max_pieces, min_piece_bytes);
  *n_pieces = (int)b.size() - 1;
  std::copy(b.begin(), b.end(), bounds);
  return PRISM_OK;
}

extern "C" PRISM_API size_t prism_host_arena_bytes(const prism_dims* dims, int max_pieces,
                                                   size_t min_piece_bytes) {
  if (check(dims, max_pieces) != PRISM_OK) return 0;
  return arena_layout(dims, plan(dims, max_pieces, min_piece_bytes)).total;
}

extern "C" PRISM_API int prism_forward_host(const prism_dims* dims, const void* q, const void* k,
                                            const void* v, const float* log_alpha,
                                            const float* beta, const float* conv_w,
                                            const float* Wk, const float* Wp, const float* wbeta,
                                            float* out, float* final_state,
                                            const int32_t* seq_lens, int max_pieces,
                                            size_t min_piece_bytes, void* arena,
                                            size_t arena_bytes, void* const* streams) {
  int rc = check(dims, max_pieces);
  if (rc != PRISM_OK) return rc;
  if (!q || !k || !v || !log_alpha || !beta || !out) return PRISM_ERR_INVALID_ARG;
  if (dims->L > 0 && (!conv_w || !Wk || !Wp || !wbeta)) return PRISM_ERR_INVALID_ARG;
  const std::vector<int> b = plan(dims, max_pieces, min_piece_bytes);
  const Arena A = arena_layout(dims, b);
  if (!arena || arena_bytes < A.total) return PRISM_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(arena) & 255) return PRISM_ERR_MISALIGNED;

  const int P = (int)b.size() - 1;
  const int B = dims->B, T = dims->T, H = dims->H, L = dims->L, w = dims->conv_width;
  const size_t D = dims->d_k, es = esize(dims);
  const size_t row_in = (size_t)H * D * es, row_out = (size_t)H * D * 4, row_g = (size_t)H * 4;
  const size_t state_b = (size_t)H * D * D * 4;   // one sequence's states
  unsigned char* base = static_cast<unsigned char*>(arena);
  auto at = [&](size_t off) { return base + off; };
  cudaStream_t s_in = streams ? static_cast<cudaStream_t>(streams[0]) : nullptr;
  cudaStream_t s_comp = streams ? static_cast<cudaStream_t>(streams[1]) : nullptr;
  cudaStream_t s_out = streams ? static_cast<cudaStream_t>(streams[2]) : nullptr;
  Events E;
#define PRISM_CU(call)                       \
  do {                                       \
    if ((call) != cudaSuccess) return PRISM_ERR_CUDA; \
  } while (0)

  // Start after every stream's earlier work: the arena may still be in use by a previous
  // call.  One piece runs on the output stream alone.
  cudaEvent_t e_in = E.make(), e_comp = E.make();
  if (!e_in || !e_comp) return PRISM_ERR_CUDA;
  if (P == 1) s_in = s_comp = s_out;
  PRISM_CU(cudaEventRecord(e_in, streams ? static_cast<cudaStream_t>(streams[0]) : nullptr));
  PRISM_CU(cudaEventRecord(e_comp, streams ? static_cast<cudaStream_t>(streams[1]) : nullptr));
  cudaStream_t first = s_in;
  PRISM_CU(cudaStreamWaitEvent(first, e_in, 0));
  PRISM_CU(cudaStreamWaitEvent(first, e_comp, 0));
  if (P > 1) {
    cudaEvent_t e_out = E.make();
    if (!e_out) return PRISM_ERR_CUDA;
    PRISM_CU(cudaEventRecord(e_out, s_out));
    PRISM_CU(cudaStreamWaitEvent(s_in, e_out, 0));
  }

  // weights, once
  if (conv_w) PRISM_CU(cudaMemcpyAsync(at(A.cw), conv_w, (size_t)H * w * D * 4, cudaMemcpyHostToDevice, s_in));
  if (L > 0) {
    PRISM_CU(cudaMemcpyAsync(at(A.wk), Wk, (size_t)H * L * D * D * 4, cudaMemcpyHostToDevice, s_in));
    PRISM_CU(cudaMemcpyAsync(at(A.wp), Wp, (size_t)H * L * D * D * 4, cudaMemcpyHostToDevice, s_in));
    PRISM_CU(cudaMemcpyAsync(at(A.wb), wbeta, (size_t)H * L * D * 4, cudaMemcpyHostToDevice, s_in));
  }
  const float* d_cw = conv_w ? reinterpret_cast<const float*>(at(A.cw)) : nullptr;
  const float* d_wk = L > 0 ? reinterpret_cast<const float*>(at(A.wk)) : nullptr;
  const float* d_wp = L > 0 ? reinterpret_cast<const float*>(at(A.wp)) : nullptr;
  const float* d_wb = L > 0 ? reinterpret_cast<const float*>(at(A.wb)) : nullptr;

  // B = 1 with a length: the tokens past it are padding; segments are cut there.
  const int len1 = (B == 1 && seq_lens) ? std::max(0, std::min(seq_lens[0], T)) : T;
  int cur = -1;                                  // state buffer holding S (B = 1), -1 = zero
  bool weights_ready = false;                    // the workspace holds the converted weights
  unsigned char* st[2] = {at(A.st0), at(A.st1)};

  for (int i = 0; i < P; ++i) {
    const int a0 = b[i], a1 = b[i + 1];
    // token rows [r0, r1) of the flattened [B*T] token axis
    const size_t r0 = B > 1 ? (size_t)a0 * T : (size_t)a0;
    const size_t r1 = B > 1 ? (size_t)a1 * T : (size_t)a1;
    const size_t nr = r1 - r0;
    PRISM_CU(cudaMemcpyAsync(at(A.q) + r0 * row_in, static_cast<const unsigned char*>(q) + r0 * row_in,
                             nr * row_in, cudaMemcpyHostToDevice, s_in));
    PRISM_CU(cudaMemcpyAsync(at(A.k) + r0 * row_in, static_cast<const unsigned char*>(k) + r0 * row_in,
                             nr * row_in, cudaMemcpyHostToDevice, s_in));
    PRISM_CU(cudaMemcpyAsync(at(A.v) + r0 * row_in, static_cast<const unsigned char*>(v) + r0 * row_in,
                             nr * row_in, cudaMemcpyHostToDevice, s_in));
    PRISM_CU(cudaMemcpyAsync(at(A.la) + r0 * row_g, log_alpha + r0 * H, nr * row_g, cudaMemcpyHostToDevice, s_in));
    PRISM_CU(cudaMemcpyAsync(at(A.be) + r0 * row_g, beta + r0 * H, nr * row_g, cudaMemcpyHostToDevice, s_in));
    int32_t* d_lens = nullptr;
    if (B > 1 && seq_lens) {
      d_lens = reinterpret_cast<int32_t*>(at(A.lens) + (size_t)i * A.lens_slot);
      PRISM_CU(cudaMemcpyAsync(d_lens, seq_lens + a0, (size_t)(a1 - a0) * 4, cudaMemcpyHostToDevice, s_in));
    }
    if (s_in != s_comp) {
      cudaEvent_t e = E.make();
      if (!e) return PRISM_ERR_CUDA;
      PRISM_CU(cudaEventRecord(e, s_in));
      PRISM_CU(cudaStreamWaitEvent(s_comp, e, 0));
    }

    float* d_out = reinterpret_cast<float*>(at(A.out) + r0 * row_out);
    if (B > 1) {
      prism_dims pd = *dims;
      pd.B = a1 - a0;
      float* fs = reinterpret_cast<float*>(at(A.st0) + (size_t)a0 * state_b);
      rc = prism::forward_from_impl(&pd, at(A.q) + r0 * row_in, at(A.k) + r0 * row_in, at(A.v) + r0 * row_in,
                                    reinterpret_cast<const float*>(at(A.la) + r0 * row_g),
                                    reinterpret_cast<const float*>(at(A.be) + r0 * row_g), d_cw, d_wk, d_wp,
                                    d_wb, nullptr, nullptr, d_out, final_state ? fs : nullptr, d_lens,
                                    at(A.ws), A.ws_bytes, s_comp, weights_ready);
      if (rc != PRISM_OK) return rc;
      weights_ready = true;
    } else {
      const int e = std::min(a1, len1);          // valid tokens of this segment: [a0, e)
      if (e > a0) {
        prism_dims pd = *dims;
        pd.T = e - a0;
        pd.flags |= PRISM_FLAG_VHIST_TOKEN_MAJOR;
        const int nxt = cur == 0 ? 1 : 0;
        const void* hist = a0 > 0 ? at(A.v) + ((size_t)a0 - w) * row_in : nullptr;
        rc = prism::forward_from_impl(&pd, at(A.q) + r0 * row_in, at(A.k) + r0 * row_in, at(A.v) + r0 * row_in,
                                      reinterpret_cast<const float*>(at(A.la) + r0 * row_g),
                                      reinterpret_cast<const float*>(at(A.be) + r0 * row_g), d_cw, d_wk,
                                      d_wp, d_wb, cur >= 0 ? reinterpret_cast<const float*>(st[cur]) : nullptr,
                                      hist, d_out, reinterpret_cast<float*>(st[nxt]), nullptr, at(A.ws),
                                      A.ws_bytes, s_comp, weights_ready);
        if (rc != PRISM_OK) return rc;
        weights_ready = true;
        cur = nxt;
      }
      if (e < a1) {                              // padding rows of this segment read 0
        const int z0 = std::max(a0, e);
        PRISM_CU(cudaMemsetAsync(at(A.out) + (size_t)z0 * row_out, 0, (size_t)(a1 - z0) * row_out, s_comp));
      }
    }
    if (s_comp != s_out) {
      cudaEvent_t e = E.make();
      if (!e) return PRISM_ERR_CUDA;
      PRISM_CU(cudaEventRecord(e, s_comp));
      PRISM_CU(cudaStreamWaitEvent(s_out, e, 0));
    }
    PRISM_CU(cudaMemcpyAsync(out + r0 * H * D, d_out, nr * row_out, cudaMemcpyDeviceToHost, s_out));
    if (B > 1 && final_state)
      PRISM_CU(cudaMemcpyAsync(final_state + (size_t)a0 * H * D * D, at(A.st0) + (size_t)a0 * state_b,
                               (size_t)(a1 - a0) * state_b, cudaMemcpyDeviceToHost, s_out));
  }
  if (B == 1 && final_state) {
    if (cur < 0) {                               // no valid token: S stays zero
      cur = 0;
      PRISM_CU(cudaMemsetAsync(st[0], 0, state_b, s_out));
    }
    PRISM_CU(cudaMemcpyAsync(final_state, st[cur], state_b, cudaMemcpyDeviceToHost, s_out));
  }
  // s_out has waited for every piece's kernels, and through them for every copy in.
#undef PRISM_CU
  return PRISM_OK;
}
