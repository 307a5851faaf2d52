// C ABI of the PRISM mixer forward pass: argument checks, workspace layout and
// kernel dispatch.  See include/prism.h for the contract of each entry point.
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/prism.h"
#include "kernels.h"

namespace prism {
cudaError_t launch_k2_bf16_16(int C, const K2Args& a, cudaStream_t s);
cudaError_t launch_k2_bf16_32(int C, const K2Args& a, cudaStream_t s);
cudaError_t launch_k2_bf16_64(int C, const K2Args& a, cudaStream_t s);
cudaError_t launch_k2_bf16_128(int C, const K2Args& a, cudaStream_t s);
cudaError_t launch_k2_f32_16(int C, const K2Args& a, cudaStream_t s);
cudaError_t launch_k2_f32_32(int C, const K2Args& a, cudaStream_t s);
cudaError_t launch_k2_f32_64(int C, const K2Args& a, cudaStream_t s);

cudaError_t launch_k2(int dtype, int D, int C, const K2Args& a, cudaStream_t s) {
  if (dtype == 1) {
    switch (D) {
      case 16: return launch_k2_bf16_16(C, a, s);
      case 32: return launch_k2_bf16_32(C, a, s);
      case 64: return launch_k2_bf16_64(C, a, s);
      case 128: return launch_k2_bf16_128(C, a, s);
    }
  } else {
    switch (D) {
      case 16: return launch_k2_f32_16(C, a, s);
      case 32: return launch_k2_f32_32(C, a, s);
      case 64: return launch_k2_f32_64(C, a, s);
    }
  }
  return cudaErrorInvalidValue;
}
}  // namespace prism

namespace {

constexpr size_t kMaxSmem = 232448;   // 227 KB: opt-in dynamic shared memory per CTA
constexpr int kMaxL = 8, kMaxW = 8;

size_t elem_size(prism_dtype t) { return t == PRISM_BF16 ? 2 : 4; }
size_t round256(size_t x) { return (x + 255) & ~size_t(255); }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Shape checks shared by every entry point.
int check_dims(const prism_dims* d) {
  if (!d) return PRISM_ERR_INVALID_ARG;
  if (d->dtype != PRISM_F32 && d->dtype != PRISM_BF16) return PRISM_ERR_INVALID_ARG;
  if (d->B <= 0 || d->T <= 0 || d->H <= 0 || d->d_k <= 0 || d->d_v <= 0 || d->L < 0 ||
      d->conv_width <= 0 || d->chunk <= 0)
    return PRISM_ERR_INVALID_ARG;
  if (d->d_k != d->d_v) return PRISM_ERR_UNSUPPORTED;
  const int D = d->d_k;
  if (D != 16 && D != 32 && D != 64 && D != 128) return PRISM_ERR_UNSUPPORTED;
  if (d->chunk != 16 && d->chunk != 32 && d->chunk != 64) return PRISM_ERR_UNSUPPORTED;
  if (d->L > kMaxL || d->conv_width > kMaxW) return PRISM_ERR_UNSUPPORTED;
  if (d->flags & ~PRISM_FLAG_NO_GELU) return PRISM_ERR_INVALID_ARG;
  const int dt = d->dtype == PRISM_BF16 ? 1 : 0;
  const size_t s1 = prism::k1_smem_bytes(dt, D), s2 = prism::k2_smem_bytes(dt, D, d->chunk);
  if (s1 == 0 || s2 == 0 || s1 > kMaxSmem || s2 > kMaxSmem) return PRISM_ERR_UNSUPPORTED;
  // index arithmetic is 64-bit; keep per-dimension products within int range
  if ((long long)d->B * d->T > (1LL << 31) - 1) return PRISM_ERR_UNSUPPORTED;
  return PRISM_OK;
}

size_t factor_bytes(const prism_dims* d) {
  return (size_t)d->B * d->T * d->H * d->L * d->d_k * elem_size(d->dtype);
}

}  // namespace

extern "C" PRISM_API size_t prism_workspace_bytes(const prism_dims* dims) {
  if (check_dims(dims) != PRISM_OK) return 0;
  // Kl then Dl (d_k == d_v), each 256-byte aligned.
  return 2 * round256(factor_bytes(dims)) + 256;
}

extern "C" PRISM_API const char* prism_strerror(int code) {
  switch (code) {
    case PRISM_OK: return "success";
    case PRISM_ERR_INVALID_ARG: return "invalid argument (null pointer, non-positive size or bad dtype)";
    case PRISM_ERR_UNSUPPORTED: return "unsupported dims (need d_k == d_v in {16,32,64,128}, chunk in {16,32,64}, L <= 8, conv width <= 8, and a working set that fits in shared memory)";
    case PRISM_ERR_MISALIGNED: return "a tensor pointer is not 16-byte aligned";
    case PRISM_ERR_WORKSPACE: return "workspace missing or smaller than prism_workspace_bytes()";
    case PRISM_ERR_LAUNCH: return "kernel launch failed";
    case PRISM_ERR_CUDA: return "CUDA runtime call failed";
  }
  return "unknown error code";
}

static int run_k1(const prism_dims* dims, const void* v, const float* conv_w, const float* Wk,
                  const float* Wp, const float* wbeta, const int32_t* seq_lens, void* Kl,
                  void* Dl, cudaStream_t s) {
  prism::K1Args a;
  a.B = dims->B; a.T = dims->T; a.H = dims->H; a.w = dims->conv_width; a.L = dims->L;
  a.flags = dims->flags;
  a.v = v; a.conv_w = conv_w; a.Wk = Wk; a.Wp = Wp; a.wbeta = wbeta;
  a.seq_lens = seq_lens; a.Kl = Kl; a.Dl = Dl;
  const int dt = dims->dtype == PRISM_BF16 ? 1 : 0;
  return prism::launch_k1(dt, dims->d_k, a, s) == cudaSuccess ? PRISM_OK : PRISM_ERR_LAUNCH;
}

extern "C" PRISM_API int prism_anchor_refine(const prism_dims* dims, const void* v, const float* conv_w,
                                   const float* Wk, const float* Wp, const float* wbeta,
                                   const int32_t* seq_lens, void* Kl, void* Dl, void* stream) {
  int rc = check_dims(dims);
  if (rc != PRISM_OK) return rc;
  if (dims->L == 0) return PRISM_OK;
  if (!v || !conv_w || !Wk || !Wp || !wbeta || !Kl || !Dl) return PRISM_ERR_INVALID_ARG;
  const void* ptrs[] = {v, conv_w, Wk, Wp, wbeta, Kl, Dl, seq_lens};
  for (const void* p : ptrs)
    if (p && !aligned16(p)) return PRISM_ERR_MISALIGNED;
  return run_k1(dims, v, conv_w, Wk, Wp, wbeta, seq_lens, Kl, Dl,
                static_cast<cudaStream_t>(stream));
}

extern "C" PRISM_API int prism_chunk_scan(const prism_dims* dims, const void* q, const void* k,
                                          const void* v, const float* log_alpha,
                                          const float* beta, const void* Kl, const void* Dl,
                                          void* out, float* final_state, const int32_t* seq_lens,
                                          void* stream);

extern "C" PRISM_API int prism_forward(const prism_dims* dims, const void* q, const void* k, const void* v,
                             const float* log_alpha, const float* beta, const float* conv_w,
                             const float* Wk, const float* Wp, const float* wbeta, void* out,
                             float* final_state, const int32_t* seq_lens, void* workspace,
                             size_t workspace_bytes, void* stream) {
  int rc = check_dims(dims);
  if (rc != PRISM_OK) return rc;
  if (!q || !k || !v || !log_alpha || !beta || !out) return PRISM_ERR_INVALID_ARG;
  if (dims->L > 0 && (!conv_w || !Wk || !Wp || !wbeta)) return PRISM_ERR_INVALID_ARG;
  const void* ptrs[] = {q, k, v, log_alpha, beta, conv_w, Wk, Wp, wbeta, out, final_state,
                        seq_lens, workspace};
  for (const void* p : ptrs)
    if (p && !aligned16(p)) return PRISM_ERR_MISALIGNED;
  const size_t need = prism_workspace_bytes(dims);
  if (dims->L > 0 && (!workspace || workspace_bytes < need)) return PRISM_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  unsigned char* ws = static_cast<unsigned char*>(workspace);
  void* Kl = ws;
  void* Dl = ws ? ws + round256(factor_bytes(dims)) : nullptr;
  if (dims->L > 0) {
    rc = run_k1(dims, v, conv_w, Wk, Wp, wbeta, seq_lens, Kl, Dl, s);
    if (rc != PRISM_OK) return rc;
  }
  return prism_chunk_scan(dims, q, k, v, log_alpha, beta, Kl, Dl, out, final_state, seq_lens,
                          stream);
}

extern "C" PRISM_API int prism_chunk_scan(const prism_dims* dims, const void* q, const void* k,
                                          const void* v, const float* log_alpha,
                                          const float* beta, const void* Kl, const void* Dl,
                                          void* out, float* final_state, const int32_t* seq_lens,
                                          void* stream) {
  int rc = check_dims(dims);
  if (rc != PRISM_OK) return rc;
  if (!q || !k || !v || !log_alpha || !beta || !out) return PRISM_ERR_INVALID_ARG;
  if (dims->L > 0 && (!Kl || !Dl)) return PRISM_ERR_INVALID_ARG;
  const void* ptrs[] = {q, k, v, log_alpha, beta, Kl, Dl, out, final_state, seq_lens};
  for (const void* p : ptrs)
    if (p && !aligned16(p)) return PRISM_ERR_MISALIGNED;
  prism::K2Args a;
  a.B = dims->B; a.T = dims->T; a.H = dims->H; a.L = dims->L;
  a.q = q; a.k = k; a.v = v; a.log_alpha = log_alpha; a.beta = beta;
  a.Kl = Kl; a.Dl = Dl; a.seq_lens = seq_lens; a.out = out; a.final_state = final_state;
  const int dt = dims->dtype == PRISM_BF16 ? 1 : 0;
  return prism::launch_k2(dt, dims->d_k, dims->chunk, a, static_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? PRISM_OK
             : PRISM_ERR_LAUNCH;
}
