// C ABI of the PRISM mixer forward pass: argument checks, workspace layout and
// kernel dispatch.  See include/prism.h for the contract of each entry point.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "../../include/prism.h"
#include "backward.cuh"
#include "decode.cuh"
#include "kernels.h"
#include "kernels_tc.cuh"

namespace prism {
cudaError_t launch_k2_f32_16(int C, const K2Args& a, cudaStream_t s);
cudaError_t launch_k2_f32_32(int C, const K2Args& a, cudaStream_t s);
cudaError_t launch_k2_f32_64(int C, const K2Args& a, cudaStream_t s);
#define PRISM_DECL_TC(D)                                                                        \
  cudaError_t launch_prep_##D(int C, const PrepArgs& a, cudaStream_t s);                       \
  cudaError_t launch_weights_##D(const float* Wk, const float* Wp, int H, int L,                \
                                 unsigned char* blocks, int* flag, cudaStream_t s);             \
  size_t prep_smem_##D(int C);
PRISM_DECL_TC(16)
PRISM_DECL_TC(32)
PRISM_DECL_TC(64)
PRISM_DECL_TC(128)
#undef PRISM_DECL_TC
cudaError_t launch_scan_tc_16(int C, const ScanTcArgs& a, cudaStream_t s);
cudaError_t launch_scan_tc_32(int C, const ScanTcArgs& a, cudaStream_t s);
cudaError_t launch_scan_tc_64(int C, const ScanTcArgs& a, cudaStream_t s);
cudaError_t launch_scan_tc_128(int C, const ScanTcArgs& a, cudaStream_t s);
static cudaError_t launch_scan_tc(int D, int C, const ScanTcArgs& a, cudaStream_t s) {
  switch (D) {
    case 16: return launch_scan_tc_16(C, a, s);
    case 32: return launch_scan_tc_32(C, a, s);
    case 64: return launch_scan_tc_64(C, a, s);
    case 128: return launch_scan_tc_128(C, a, s);
  }
  return cudaErrorInvalidValue;
}
cudaError_t launch_decode(int dtype, int D, const DecodeArgs& a, cudaStream_t s);
cudaError_t launch_backward(int dtype, int D, const BwdArgs& a, cudaStream_t s);

cudaError_t launch_k2(int dtype, int D, int C, const K2Args& a, cudaStream_t s) {
  if (dtype != 0) return cudaErrorInvalidValue;
  switch (D) {
    case 16: return launch_k2_f32_16(C, a, s);
    case 32: return launch_k2_f32_32(C, a, s);
    case 64: return launch_k2_f32_64(C, a, s);
  }
  return cudaErrorInvalidValue;
}
static size_t prep_smem(int D, int C) {
  switch (D) {
    case 16: return prep_smem_16(C);
    case 32: return prep_smem_32(C);
    case 64: return prep_smem_64(C);
    case 128: return prep_smem_128(C);
  }
  return 0;
}
static cudaError_t launch_prep(int D, int C, const PrepArgs& a, cudaStream_t s) {
  switch (D) {
    case 16: return launch_prep_16(C, a, s);
    case 32: return launch_prep_32(C, a, s);
    case 64: return launch_prep_64(C, a, s);
    case 128: return launch_prep_128(C, a, s);
  }
  return cudaErrorInvalidValue;
}
static cudaError_t launch_weights(int D, const float* Wk, const float* Wp, int H, int L,
                                  unsigned char* blocks, int* flag, cudaStream_t s) {
  switch (D) {
    case 16: return launch_weights_16(Wk, Wp, H, L, blocks, flag, s);
    case 32: return launch_weights_32(Wk, Wp, H, L, blocks, flag, s);
    case 64: return launch_weights_64(Wk, Wp, H, L, blocks, flag, s);
    case 128: return launch_weights_128(Wk, Wp, H, L, blocks, flag, s);
  }
  return cudaErrorInvalidValue;
}
}  // namespace prism

#ifdef PRISM_DEBUG_BOUNDS
// the debug build's word of out-of-bounds accesses (prism_debug_bounds), shared by every
// kernel of the library through the pointer each launch passes
__device__ int g_bounds_word;
#endif

namespace {

// the bounds word's device address in the debug build, null otherwise
int* bounds_word() {
#ifdef PRISM_DEBUG_BOUNDS
  void* p = nullptr;
  return cudaGetSymbolAddress(&p, g_bounds_word) == cudaSuccess ? static_cast<int*>(p) : nullptr;
#else
  return nullptr;
#endif
}

constexpr size_t kMaxSmem = 232448;   // 227 KB: opt-in dynamic shared memory per CTA
constexpr int kMaxL = 8, kMaxW = 8;
constexpr size_t kAbsent = ~size_t(0);

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

// cuTensorMapEncodeTiled, looked up once through the runtime (no link to the driver library).
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// TMA map of a bf16 [B][T][H][d] tensor as 4-D (d, H, T, B) with boxes of `rows` tokens
// of one head: (d, 1, rows, 1).
bool make_row_map(CUtensorMap* m, const void* base, const prism_dims* d, int rows) {
  const PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t D = (cuuint64_t)d->d_k, H = (cuuint64_t)d->H, T = (cuuint64_t)d->T;
  const cuuint64_t dim[4] = {D, H, T, (cuuint64_t)d->B};
  const cuuint64_t stride[3] = {D * 2, H * D * 2, T * H * D * 2};
  const cuuint32_t box[4] = {(cuuint32_t)D, 1, (cuuint32_t)rows, 1};
  const cuuint32_t estride[4] = {1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dim, stride, box, estride,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// Shape checks shared by every entry point.
int check_dims(const prism_dims* d) {
  if (!d) return PRISM_ERR_INVALID_ARG;
  if (d->dtype != PRISM_F32 && d->dtype != PRISM_BF16) return PRISM_ERR_INVALID_ARG;
  if (d->B <= 0 || d->T <= 0 || d->H <= 0 || d->d_k <= 0 || d->d_v <= 0 || d->L < 0 ||
      d->conv_width <= 0 || d->chunk <= 0)
    return PRISM_ERR_INVALID_ARG;
  if (d->flags & ~(PRISM_FLAG_NO_GELU | PRISM_FLAG_VHIST_TOKEN_MAJOR | PRISM_FLAG_NO_SEQ_SPLIT |
                   PRISM_FLAG_CHECK_WAIT_TIMEOUT))
    return PRISM_ERR_INVALID_ARG;
  if (d->d_k != d->d_v) return PRISM_ERR_UNSUPPORTED;
  const int D = d->d_k, C = d->chunk;
  if (D != 16 && D != 32 && D != 64 && D != 128) return PRISM_ERR_UNSUPPORTED;
  if (C != 16 && C != 32 && C != 64) return PRISM_ERR_UNSUPPORTED;
  if (d->L > kMaxL || d->conv_width > kMaxW) return PRISM_ERR_UNSUPPORTED;
  if (d->dtype == PRISM_F32) {
    const size_t s1 = prism::k1_smem_bytes(0, D), s2 = prism::k2_smem_bytes(0, D, C);
    if (s1 == 0 || s2 == 0 || s1 > kMaxSmem || s2 > kMaxSmem) return PRISM_ERR_UNSUPPORTED;
  } else {
    const size_t s1 = prism::prep_smem(D, C);
    if (s1 == 0 || s1 > kMaxSmem) return PRISM_ERR_UNSUPPORTED;
  }
  if ((long long)d->B * d->T > (1LL << 31) - 1) return PRISM_ERR_UNSUPPORTED;
  return PRISM_OK;
}

struct Layout {
  size_t off[PRISM_WS_COUNT];
  size_t total;
};

// Segments of the sequence split (1: none).  The first pass runs B*H*4*(2P-1) CTAs of
// one per SM (segment 0 in full, the c and M rows of every later one): it must fit one
// wave of the 152 SMs, and each segment keeps at least kMinSegChunks chunks.  Time goes
// as about 2/P of the serial chain's, so P = 2 gains nothing and is not taken.
constexpr int kScanSMs = 152, kMaxSeg = 16, kMinSegChunks = 8;
int scan_segments(const prism_dims* d) {
  if (d->dtype != PRISM_BF16 || d->d_k != 128 || (d->chunk != 32 && d->chunk != 64)) return 1;
  if (d->flags & PRISM_FLAG_NO_SEQ_SPLIT) return 1;
  const long long ctas = (long long)d->B * d->H * 4;
  const int NC = (d->T + d->chunk - 1) / d->chunk;
  int P = 1;
  for (int q = 3; q <= kMaxSeg; ++q)
    if (ctas * (2 * q - 1) <= kScanSMs && NC >= q * kMinSegChunks) P = q;
  return P;
}

Layout layout(const prism_dims* d) {
  Layout Lo;
  for (auto& o : Lo.off) o = kAbsent;
  size_t cur = 0;
  auto take = [&](int region, size_t bytes) {
    Lo.off[region] = cur;
    cur += round256(bytes);
  };
  const size_t D = d->d_k, C = d->chunk, NC = (d->T + C - 1) / C;
  take(PRISM_WS_STATUS, 256);
  if (d->dtype == PRISM_F32) {
    const size_t f = (size_t)d->B * d->T * d->H * d->L * D * 4;
    if (d->L > 0) {
      take(PRISM_WS_KL, f);
      take(PRISM_WS_DL, f);
    }
  } else {
    const size_t per = (size_t)d->B * d->H * NC * C * D;
    if (d->L > 0) take(PRISM_WS_WBLOCKS, (size_t)d->H * d->L * 4 * 128 * D * 2);
    take(PRISM_WS_WQ, per * 4);
    take(PRISM_WS_QK, per * 4);
    take(PRISM_WS_U, per * 4);
    take(PRISM_WS_OI, per * 4);
    if (d->L > 0) take(PRISM_WS_N, (size_t)d->B * d->H * NC * D * D * 4);
    take(PRISM_WS_GC, (size_t)d->B * d->H * NC * 4);
    const int P = scan_segments(d);
    if (P > 1) take(PRISM_WS_SEG, 3 * (size_t)d->B * d->H * P * D * D * 4);
  }
  Lo.total = cur;
  return Lo;
}

int check_inputs(const prism_dims* dims, const void* q, const void* k, const void* v,
                 const float* log_alpha, const float* beta, const int32_t* seq_lens,
                 const void* workspace, size_t workspace_bytes) {
  if (!q || !k || !v || !log_alpha || !beta) return PRISM_ERR_INVALID_ARG;
  const void* ptrs[] = {q, k, v, log_alpha, beta, seq_lens};
  for (const void* p : ptrs)
    if (p && !aligned(p, 16)) return PRISM_ERR_MISALIGNED;
  if (workspace && !aligned(workspace, 256)) return PRISM_ERR_MISALIGNED;
  if (!workspace || workspace_bytes < layout(dims).total) return PRISM_ERR_WORKSPACE;
  return PRISM_OK;
}

template <class T>
T* region(void* ws, const Layout& Lo, int r) {
  return Lo.off[r] == kAbsent ? nullptr
                              : reinterpret_cast<T*>(static_cast<unsigned char*>(ws) + Lo.off[r]);
}


}  // namespace

extern "C" PRISM_API size_t prism_workspace_bytes(const prism_dims* dims) {
  if (check_dims(dims) != PRISM_OK) return 0;
  return layout(dims).total;
}

extern "C" PRISM_API int prism_scan_segments(const prism_dims* dims) {
  if (check_dims(dims) != PRISM_OK) return 0;
  return scan_segments(dims);
}

extern "C" PRISM_API int prism_workspace_layout(const prism_dims* dims, size_t* offsets, int n) {
  const int rc = check_dims(dims);
  if (rc != PRISM_OK) return rc;
  if (!offsets || n < PRISM_WS_COUNT) return PRISM_ERR_INVALID_ARG;
  const Layout Lo = layout(dims);
  for (int i = 0; i < PRISM_WS_COUNT; ++i) offsets[i] = Lo.off[i];
  return PRISM_OK;
}

extern "C" PRISM_API const char* prism_strerror(int code) {
  switch (code) {
    case PRISM_OK: return "success";
    case PRISM_ERR_INVALID_ARG: return "invalid argument (null pointer, non-positive size, bad dtype or flags)";
    case PRISM_ERR_UNSUPPORTED: return "unsupported dims (need d_k == d_v in {16,32,64,128} (fp32: <= 64), chunk in {16,32,64}, L <= 8, conv width <= 8)";
    case PRISM_ERR_MISALIGNED: return "a tensor pointer is not 16-byte aligned (workspace: 256-byte)";
    case PRISM_ERR_WORKSPACE: return "workspace missing or smaller than prism_workspace_bytes()";
    case PRISM_ERR_LAUNCH: return "kernel launch failed";
    case PRISM_ERR_CUDA: return "CUDA runtime call failed";
    case PRISM_ERR_SCRATCH_LIMIT: return "dims need more scratch than PRISM_STATIC_SCRATCH_BYTES (use prism_forward with a workspace)";
  }
  return "unknown error code";
}

namespace {
// weights_ready: the workspace already holds these weights in the prepare kernel's fp16
// blocks (and the flag saying whether their lo halves matter), converted by an earlier
// call on the same stream; the conversion is skipped and the flag kept.
int prepare_impl(const prism_dims* dims, const void* q, const void* k, const void* v,
                 const float* log_alpha, const float* beta, const float* conv_w, const float* Wk,
                 const float* Wp, const float* wbeta, const int32_t* seq_lens, const void* v_hist,
                 void* workspace, size_t workspace_bytes, void* stream, bool weights_ready = false) {
  int rc = check_dims(dims);
  if (rc != PRISM_OK) return rc;
  rc = check_inputs(dims, q, k, v, log_alpha, beta, seq_lens, workspace, workspace_bytes);
  if (rc != PRISM_OK) return rc;
  if (dims->L > 0 && (!conv_w || !Wk || !Wp || !wbeta)) return PRISM_ERR_INVALID_ARG;
  const void* wp[] = {conv_w, Wk, Wp, wbeta, v_hist};
  for (const void* p : wp)
    if (p && !aligned(p, 16)) return PRISM_ERR_MISALIGNED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const Layout Lo = layout(dims);
  int* status = region<int>(workspace, Lo, PRISM_WS_STATUS);
  const bool keep_weights = weights_ready && dims->dtype == PRISM_BF16 && dims->L > 0;
  if (cudaMemsetAsync(status, 0, keep_weights ? 4 : 8, s) != cudaSuccess) return PRISM_ERR_CUDA;
  const int D = dims->d_k, C = dims->chunk;
  if (dims->dtype == PRISM_F32) {
    if (dims->L == 0) return PRISM_OK;
    prism::K1Args a;
    a.B = dims->B; a.T = dims->T; a.H = dims->H; a.w = dims->conv_width; a.L = dims->L;
    a.flags = dims->flags;
    a.v = v; a.conv_w = conv_w; a.Wk = Wk; a.Wp = Wp; a.wbeta = wbeta;
    a.seq_lens = seq_lens; a.vhist = v_hist;
    a.Kl = region<float>(workspace, Lo, PRISM_WS_KL);
    a.Dl = region<float>(workspace, Lo, PRISM_WS_DL);
    return prism::launch_k1(0, D, a, s) == cudaSuccess ? PRISM_OK : PRISM_ERR_LAUNCH;
  }
  unsigned char* wblocks = region<unsigned char>(workspace, Lo, PRISM_WS_WBLOCKS);
  if (dims->L > 0 && !keep_weights &&
      prism::launch_weights(D, Wk, Wp, dims->H, dims->L, wblocks, status + 1, s) != cudaSuccess)
    return PRISM_ERR_LAUNCH;
  prism::PrepArgs a;
  if (!make_row_map(&a.tm_q, q, dims, C) || !make_row_map(&a.tm_k, k, dims, C) ||
      !make_row_map(&a.tm_v, v, dims, C + 8))
    return PRISM_ERR_CUDA;
  a.B = dims->B; a.T = dims->T; a.H = dims->H; a.w = dims->conv_width; a.L = dims->L;
  a.flags = dims->flags;
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.k = static_cast<const __nv_bfloat16*>(k);
  a.v = static_cast<const __nv_bfloat16*>(v);
  a.log_alpha = log_alpha; a.beta = beta; a.conv_w = conv_w; a.wbeta = wbeta;
  a.wblocks = wblocks; a.wflag = status + 1; a.seq_lens = seq_lens;
  a.vhist = static_cast<const __nv_bfloat16*>(v_hist);
  a.WQ = region<__half>(workspace, Lo, PRISM_WS_WQ);
  a.QK = region<__half>(workspace, Lo, PRISM_WS_QK);
  a.U = region<float>(workspace, Lo, PRISM_WS_U);
  a.Oi = region<float>(workspace, Lo, PRISM_WS_OI);
  a.Nt = region<float>(workspace, Lo, PRISM_WS_N);
  a.gC = region<float>(workspace, Lo, PRISM_WS_GC);
  a.status = status;
  a.bounds = bounds_word();
  return prism::launch_prep(D, C, a, s) == cudaSuccess ? PRISM_OK : PRISM_ERR_LAUNCH;
}
}  // namespace

extern "C" PRISM_API int prism_prepare(const prism_dims* dims, const void* q, const void* k,
                                       const void* v, const float* log_alpha, const float* beta,
                                       const float* conv_w, const float* Wk, const float* Wp,
                                       const float* wbeta, const int32_t* seq_lens,
                                       void* workspace, size_t workspace_bytes, void* stream) {
  return prepare_impl(dims, q, k, v, log_alpha, beta, conv_w, Wk, Wp, wbeta, seq_lens, nullptr,
                      workspace, workspace_bytes, stream);
}

namespace {
int scan_impl(const prism_dims* dims, const void* q, const void* k, const void* v,
              const float* log_alpha, const float* beta, const int32_t* seq_lens,
              const float* initial_state, void* workspace, size_t workspace_bytes, float* out,
              float* final_state, void* stream) {
  int rc = check_dims(dims);
  if (rc != PRISM_OK) return rc;
  rc = check_inputs(dims, q, k, v, log_alpha, beta, seq_lens, workspace, workspace_bytes);
  if (rc != PRISM_OK) return rc;
  if (!out) return PRISM_ERR_INVALID_ARG;
  if (!aligned(out, 16) || (final_state && !aligned(final_state, 16)) ||
      (initial_state && !aligned(initial_state, 16)))
    return PRISM_ERR_MISALIGNED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const Layout Lo = layout(dims);
  const int D = dims->d_k, C = dims->chunk;
  if (dims->dtype == PRISM_F32) {
    prism::K2Args a;
    a.B = dims->B; a.T = dims->T; a.H = dims->H; a.L = dims->L;
    a.q = q; a.k = k; a.v = v; a.log_alpha = log_alpha; a.beta = beta;
    a.Kl = region<float>(workspace, Lo, PRISM_WS_KL);
    a.Dl = region<float>(workspace, Lo, PRISM_WS_DL);
    a.seq_lens = seq_lens; a.out = out; a.final_state = final_state; a.initial_state = initial_state;
    return prism::launch_k2(0, D, C, a, s) == cudaSuccess ? PRISM_OK : PRISM_ERR_LAUNCH;
  }
  // tensor-core scan (every bf16 head dim and chunk)
  {
    prism::ScanTcArgs a;
    a.B = dims->B; a.T = dims->T; a.H = dims->H;
    a.WQ = region<const __half>(workspace, Lo, PRISM_WS_WQ);
    a.QK = region<const __half>(workspace, Lo, PRISM_WS_QK);
    a.U = region<const float>(workspace, Lo, PRISM_WS_U);
    a.Oi = region<const float>(workspace, Lo, PRISM_WS_OI);
    a.Nt = region<const float>(workspace, Lo, PRISM_WS_N);
    a.gC = region<const float>(workspace, Lo, PRISM_WS_GC);
    a.seq_lens = seq_lens; a.out = out; a.final_state = final_state; a.initial_state = initial_state;
    a.status = region<int>(workspace, Lo, PRISM_WS_STATUS);
    a.bounds = bounds_word();
    a.nseg = scan_segments(dims);
    a.phase = 0;
    a.check_timeout = (dims->flags & PRISM_FLAG_CHECK_WAIT_TIMEOUT) ? 1 : 0;
    a.seg_chunks = (int)(((dims->T + C - 1) / C + a.nseg - 1) / a.nseg);
    float* seg = region<float>(workspace, Lo, PRISM_WS_SEG);
    const size_t per = (size_t)dims->B * dims->H * a.nseg * D * D;
    a.seg_start = seg;
    a.seg_c = seg ? seg + per : nullptr;
    a.seg_M = seg ? seg + 2 * per : nullptr;
    return prism::launch_scan_tc(D, C, a, s) == cudaSuccess ? PRISM_OK : PRISM_ERR_LAUNCH;
  }
}
}  // namespace

extern "C" PRISM_API int prism_scan(const prism_dims* dims, const void* q, const void* k,
                                    const void* v, const float* log_alpha, const float* beta,
                                    const int32_t* seq_lens, void* workspace,
                                    size_t workspace_bytes, float* out, float* final_state,
                                    void* stream) {
  return scan_impl(dims, q, k, v, log_alpha, beta, seq_lens, nullptr, workspace, workspace_bytes,
                   out, final_state, stream);
}

namespace prism {
// prism_forward_from; with weights_ready the weight conversion of an earlier call into the
// same workspace is reused (the host pipeline's pieces after the first).
int forward_from_impl(const prism_dims* dims, const void* q, const void* k, const void* v,
                      const float* log_alpha, const float* beta, const float* conv_w,
                      const float* Wk, const float* Wp, const float* wbeta,
                      const float* initial_state, const void* v_hist, float* out,
                      float* final_state, const int32_t* seq_lens, void* workspace,
                      size_t workspace_bytes, void* stream, bool weights_ready) {
  int rc = check_dims(dims);
  if (rc != PRISM_OK) return rc;
  if (!out) return PRISM_ERR_INVALID_ARG;
  if (!aligned(out, 16) || (final_state && !aligned(final_state, 16))) return PRISM_ERR_MISALIGNED;
  rc = prepare_impl(dims, q, k, v, log_alpha, beta, conv_w, Wk, Wp, wbeta, seq_lens, v_hist,
                    workspace, workspace_bytes, stream, weights_ready);
  if (rc != PRISM_OK) return rc;
  return scan_impl(dims, q, k, v, log_alpha, beta, seq_lens, initial_state, workspace,
                   workspace_bytes, out, final_state, stream);
}
}  // namespace prism

extern "C" PRISM_API int prism_forward_from(const prism_dims* dims, const void* q, const void* k,
                                            const void* v, const float* log_alpha,
                                            const float* beta, const float* conv_w,
                                            const float* Wk, const float* Wp, const float* wbeta,
                                            const float* initial_state, const void* v_hist,
                                            float* out, float* final_state,
                                            const int32_t* seq_lens, void* workspace,
                                            size_t workspace_bytes, void* stream) {
  return prism::forward_from_impl(dims, q, k, v, log_alpha, beta, conv_w, Wk, Wp, wbeta,
                                  initial_state, v_hist, out, final_state, seq_lens, workspace,
                                  workspace_bytes, stream, false);
}

extern "C" PRISM_API int prism_forward(const prism_dims* dims, const void* q, const void* k,
                                       const void* v, const float* log_alpha, const float* beta,
                                       const float* conv_w, const float* Wk, const float* Wp,
                                       const float* wbeta, float* out, float* final_state,
                                       const int32_t* seq_lens, void* workspace,
                                       size_t workspace_bytes, void* stream) {
  return prism_forward_from(dims, q, k, v, log_alpha, beta, conv_w, Wk, Wp, wbeta, nullptr, nullptr,
                            out, final_state, seq_lens, workspace, workspace_bytes, stream);
}

namespace prism {
// the bf16 prepare kernel's activation at n points (a diagnostic for tests)
__global__ void debug_activation_kernel(const float* x, float* y, long long n) {
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x)
    y[i] = gelu_hastings(x[i]);
}
}  // namespace prism

extern "C" PRISM_API int prism_debug_activation(const float* x, float* y, long long n, void* stream) {
  if (n < 0 || (n > 0 && (!x || !y))) return PRISM_ERR_INVALID_ARG;
  if (n == 0) return PRISM_OK;
  const long long blocks = (n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096;
  prism::debug_activation_kernel<<<(unsigned)blocks, 256, 0, static_cast<cudaStream_t>(stream)>>>(x, y, n);
  return cudaGetLastError() == cudaSuccess ? PRISM_OK : PRISM_ERR_CUDA;
}

extern "C" PRISM_API int prism_debug_bounds(int* word, int clear) {
  if (!word) return PRISM_ERR_INVALID_ARG;
#ifdef PRISM_DEBUG_BOUNDS
  if (cudaDeviceSynchronize() != cudaSuccess || cudaMemcpyFromSymbol(word, g_bounds_word, sizeof(int)) != cudaSuccess)
    return PRISM_ERR_CUDA;
  if (clear) {
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_bounds_word, &zero, sizeof(int)) != cudaSuccess) return PRISM_ERR_CUDA;
  }
  return PRISM_OK;
#else
  (void)clear;
  *word = 0;
  return PRISM_ERR_UNSUPPORTED;
#endif
}

extern "C" PRISM_API int prism_device_status(const prism_dims* dims, const void* workspace,
                                             size_t workspace_bytes, int* status, void* stream) {
  const int rc = check_dims(dims);
  if (rc != PRISM_OK) return rc;
  if (!status) return PRISM_ERR_INVALID_ARG;
  if (workspace && !aligned(workspace, 256)) return PRISM_ERR_MISALIGNED;
  const Layout Lo = layout(dims);
  if (!workspace || workspace_bytes < Lo.total) return PRISM_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int word = 0;
  const int* src = region<const int>(const_cast<void*>(workspace), Lo, PRISM_WS_STATUS);
  if (cudaMemcpyAsync(&word, src, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return PRISM_ERR_CUDA;
  *status = word;
  return PRISM_OK;
}

extern "C" PRISM_API int prism_decode_step(const prism_dims* dims, const void* q, const void* k,
                                           const void* v, const float* log_alpha,
                                           const float* beta, const float* conv_w,
                                           const float* Wk, const float* Wp, const float* wbeta,
                                           float* state, void* v_hist, float* out, void* stream) {
  if (!dims) return PRISM_ERR_INVALID_ARG;
  if (dims->dtype != PRISM_F32 && dims->dtype != PRISM_BF16) return PRISM_ERR_INVALID_ARG;
  if (dims->B <= 0 || dims->H <= 0 || dims->d_k <= 0 || dims->d_v <= 0 || dims->L < 0 ||
      dims->conv_width <= 0 || dims->T != 1)
    return PRISM_ERR_INVALID_ARG;
  if (dims->flags & ~PRISM_FLAG_NO_GELU) return PRISM_ERR_INVALID_ARG;
  const int D = dims->d_k;
  if (dims->d_k != dims->d_v || (D != 16 && D != 32 && D != 64 && D != 128) || dims->L > kMaxL ||
      dims->conv_width > kMaxW)
    return PRISM_ERR_UNSUPPORTED;
  if (!q || !k || !v || !log_alpha || !beta || !conv_w || !state || !v_hist || !out)
    return PRISM_ERR_INVALID_ARG;
  if (dims->L > 0 && (!Wk || !Wp || !wbeta)) return PRISM_ERR_INVALID_ARG;
  const void* ptrs[] = {q, k, v, log_alpha, beta, conv_w, Wk, Wp, wbeta, state, v_hist, out};
  for (const void* p : ptrs)
    if (p && !aligned(p, 16)) return PRISM_ERR_MISALIGNED;
  prism::DecodeArgs a;
  a.B = dims->B; a.H = dims->H; a.w = dims->conv_width; a.L = dims->L; a.flags = dims->flags;
  a.q = q; a.k = k; a.v = v; a.log_alpha = log_alpha; a.beta = beta; a.conv_w = conv_w;
  a.Wk = Wk; a.Wp = Wp; a.wbeta = wbeta; a.state = state; a.vhist = v_hist; a.out = out;
  a.bounds = bounds_word();
  return prism::launch_decode(dims->dtype == PRISM_F32 ? 0 : 1, D, a, static_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? PRISM_OK
             : PRISM_ERR_LAUNCH;
}

namespace {

// Backward-pass workspace: per token-head factors, then the state checkpoints and the
// block scratch.  Offsets in floats of each region, 256-byte aligned.
struct BwdLayout {
  size_t U, KL, DL, P, NRM, Z, dDL, dKL, dKH, dZ, dU, CK, SCR, PQ, PK, PKL, PB, PA, PW, PSW, total;
  int rs, nsw, nss;
};

BwdLayout bwd_layout(const prism_dims* d) {
  BwdLayout Lo;
  size_t cur = 0;
  auto take = [&](size_t floats) {
    const size_t o = cur;
    cur += round256(floats * 4) / 4;
    return o;
  };
  const size_t D = d->d_k, L = d->L, NTH = (size_t)d->B * d->T * d->H;
  const size_t NCK = (d->T + prism::kBwdCK - 1) / prism::kBwdCK;
  Lo.U = take(NTH * D);
  Lo.KL = take(NTH * L * D);
  Lo.DL = take(NTH * L * D);
  Lo.P = take(NTH * L * D);
  Lo.NRM = take(NTH * L);
  Lo.Z = take(NTH * L);
  Lo.dDL = take(NTH * L * D);
  Lo.dKL = take(NTH * L * D);
  Lo.dKH = take(NTH * L * D);
  Lo.dZ = take(NTH * L);
  Lo.dU = take(NTH * D);
  Lo.CK = take((size_t)d->B * d->H * NCK * D * D);
  Lo.SCR = take((size_t)d->B * d->H * prism::kBwdCK * D * D);
  Lo.rs = prism::bwd_pick_rs((long long)d->B * d->H, (int)D);
  const size_t RSp = Lo.rs > 1 ? (size_t)Lo.rs : 0;   // partial sums only when rows are split
  Lo.PQ = take(RSp * NTH * D);
  Lo.PK = take(RSp * NTH * D);
  Lo.PKL = take(RSp * NTH * L * D);
  Lo.PB = take(RSp * NTH);
  Lo.PA = take(RSp * NTH);
  // token-split partials of the weight gradients (only when split)
  const long long ntok = (long long)d->B * d->T;
  Lo.nsw = L > 0 ? prism::bwd_pick_nsw(ntok) : 1;
  Lo.nss = prism::bwd_pick_nss(ntok);
  Lo.PW = take(Lo.nsw > 1 ? (size_t)Lo.nsw * d->H * 2 * L * D * D : 0);
  Lo.PSW = take(Lo.nss > 1 ? (size_t)Lo.nss * d->H * (L + d->conv_width) * D : 0);
  Lo.total = cur * 4;
  return Lo;
}

int check_bwd_dims(const prism_dims* d) {
  if (!d) return PRISM_ERR_INVALID_ARG;
  if (d->dtype != PRISM_F32 && d->dtype != PRISM_BF16) return PRISM_ERR_INVALID_ARG;
  if (d->B <= 0 || d->T <= 0 || d->H <= 0 || d->d_k <= 0 || d->d_v <= 0 || d->L < 0 || d->conv_width <= 0)
    return PRISM_ERR_INVALID_ARG;
  if (d->flags & ~PRISM_FLAG_NO_GELU) return PRISM_ERR_INVALID_ARG;
  const int D = d->d_k;
  if (d->d_k != d->d_v || (D != 16 && D != 32 && D != 64 && D != 128) || d->L > kMaxL ||
      d->conv_width > kMaxW)
    return PRISM_ERR_UNSUPPORTED;
  if ((long long)d->B * d->T > (1LL << 31) - 1 || d->H > 65535 || d->B > 65535) return PRISM_ERR_UNSUPPORTED;
  return PRISM_OK;
}

}  // namespace

extern "C" PRISM_API size_t prism_backward_workspace_bytes(const prism_dims* dims) {
  if (check_bwd_dims(dims) != PRISM_OK) return 0;
  return bwd_layout(dims).total;
}

extern "C" PRISM_API int prism_backward(const prism_dims* dims, const void* q, const void* k,
                                        const void* v, const float* log_alpha, const float* beta,
                                        const float* conv_w, const float* Wk, const float* Wp,
                                        const float* wbeta, const float* d_out,
                                        const float* d_final_state, float* dq, float* dk, float* dv,
                                        float* dlog_alpha, float* dbeta, float* dconv_w, float* dWk,
                                        float* dWp, float* dwbeta, const int32_t* seq_lens,
                                        void* workspace, size_t workspace_bytes, void* stream) {
  int rc = check_bwd_dims(dims);
  if (rc != PRISM_OK) return rc;
  const bool hasL = dims->L > 0;
  if (!q || !k || !v || !log_alpha || !beta || !conv_w || !d_out || !dq || !dk || !dv || !dlog_alpha ||
      !dbeta || !dconv_w)
    return PRISM_ERR_INVALID_ARG;
  if (hasL && (!Wk || !Wp || !wbeta || !dWk || !dWp || !dwbeta)) return PRISM_ERR_INVALID_ARG;
  const void* ptrs[] = {q, k, v, log_alpha, beta, conv_w, Wk, Wp, wbeta, d_out, d_final_state, dq, dk, dv,
                        dlog_alpha, dbeta, dconv_w, dWk, dWp, dwbeta, seq_lens};
  for (const void* p : ptrs)
    if (p && !aligned(p, 16)) return PRISM_ERR_MISALIGNED;
  if (workspace && !aligned(workspace, 256)) return PRISM_ERR_MISALIGNED;
  const BwdLayout Lo = bwd_layout(dims);
  if (!workspace || workspace_bytes < Lo.total) return PRISM_ERR_WORKSPACE;
  float* ws = static_cast<float*>(workspace);
  prism::BwdArgs a;
  a.B = dims->B; a.T = dims->T; a.H = dims->H; a.L = dims->L; a.w = dims->conv_width;
  a.flags = dims->flags;
  a.q = q; a.k = k; a.v = v; a.log_alpha = log_alpha; a.beta = beta; a.conv_w = conv_w;
  a.Wk = Wk; a.Wp = Wp; a.wbeta = wbeta; a.d_out = d_out; a.d_fs = d_final_state;
  a.seq_lens = seq_lens;
  a.dq = dq; a.dk = dk; a.dv = dv; a.dla = dlog_alpha; a.dbeta = dbeta; a.dconv = dconv_w;
  a.dWk = dWk; a.dWp = dWp; a.dwb = dwbeta;
  a.U = ws + Lo.U; a.KL = ws + Lo.KL; a.DL = ws + Lo.DL; a.P = ws + Lo.P; a.NRM = ws + Lo.NRM;
  a.Z = ws + Lo.Z; a.dDL = ws + Lo.dDL; a.dKL = ws + Lo.dKL; a.dKH = ws + Lo.dKH; a.dZ = ws + Lo.dZ;
  a.dU = ws + Lo.dU; a.CK = ws + Lo.CK; a.SCR = ws + Lo.SCR;
  a.rs = Lo.rs;
  a.PQ = ws + Lo.PQ; a.PK = ws + Lo.PK; a.PKL = ws + Lo.PKL; a.PB = ws + Lo.PB; a.PA = ws + Lo.PA;
  a.nsw = Lo.nsw; a.nss = Lo.nss; a.PW = ws + Lo.PW; a.PSW = ws + Lo.PSW;
  return prism::launch_backward(dims->dtype == PRISM_F32 ? 0 : 1, dims->d_k, a,
                                static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? PRISM_OK
             : PRISM_ERR_LAUNCH;
}
