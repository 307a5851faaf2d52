/*
 * prism.h — C ABI of the PRISM mixer forward pass on GB300 (sm_103a).
 *
 * The operation ("Technical Summary: PRISM (Parallel Residual Iterative
 * Sequence Model)", gist.science/paper/2602.10796):
 *
 *   §2.1  S_t = S_{t-1} A_t + B_t,  A_t = alpha_t (I - beta_t k_t k_t^T)
 *         (the forget operator "identical to Gated DeltaNet"),
 *         alpha_t = exp(log_alpha_t)
 *   §2.2  stage 1: u_t = sum_{j=1..w} c_j (.) v_{t-j}    (causal ShortConv)
 *         stage 2, l = 1..L, r^(1) = v_t - u_t:
 *           k^(l) = normalize(W_k^(l) u_t),  p^(l) = W_p^(l) u_t,
 *           delta^(l) = GELU(p^(l) (.) r^(l)),  r^(l+1) = r^(l) - delta^(l),
 *           beta^(l) = sigmoid(w_beta^(l) . u_t)
 *         write: B_t = beta_t v_t k_t^T + sum_l beta^(l) delta^(l) k^(l)^T
 *   readout o_t = S_t q_t,  S_0 = 0.
 *
 * The Gated DeltaNet term beta_t v_t k_t^T of B_t is what makes L = 0 reduce to
 * Gated DeltaNet (§3.3); normalize(x) = x / sqrt(|x|^2 + 1e-6); GELU is the
 * exact erf form.
 *
 * Conventions for every entry point:
 *   - Tensor pointers are DEVICE pointers, row-major and contiguous, owned by
 *     the caller; the library allocates nothing and keeps no state.
 *   - Every tensor pointer must be 16-byte aligned; the workspace 256-byte.
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = the legacy default
 *     stream) and runs asynchronously; errors found before launch are
 *     returned synchronously and nothing is launched.
 *   - Shapes (dims fields): q, k [B,T,H,d_k]; v [B,T,H,d_v] in `dtype`;
 *     log_alpha, beta [B,T,H] fp32; conv_w [H,w,d_v] fp32 (row j-1 multiplies
 *     v_{t-j}); Wk [H,L,d_k,d_v], Wp [H,L,d_v,d_v], wbeta [H,L,d_v] fp32;
 *     out [B,T,H,d_v] fp32 (always fp32: the refinement makes outputs
 *     heavy-tailed, and a 16-bit output rounding alone would exceed the
 *     accuracy this library is checked to); final_state [B,H,d_v,d_k] fp32;
 *     seq_lens [B] int32.
 *   - dtype PRISM_BF16 runs the tensor-core path (tcgen05 prepare kernel,
 *     fp16/fp32 split-precision products); PRISM_F32 runs an fp32 path for
 *     small head dims (d <= 64).
 */
#ifndef PRISM_H
#define PRISM_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define PRISM_API __attribute__((visibility("default")))
#else
#define PRISM_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { PRISM_F32 = 0, PRISM_BF16 = 1 } prism_dtype;

/* flags */
#define PRISM_FLAG_NO_GELU 1u   /* ablation: delta^(l) = p^(l) (.) r^(l) (identity activation) */
#define PRISM_FLAG_VHIST_TOKEN_MAJOR 2u  /* prism_forward_from: v_hist is [B,w,H,d_v], the layout of
                                            v itself (so the last w token rows of the previous
                                            segment's v serve directly when B = 1) */
#define PRISM_FLAG_NO_SEQ_SPLIT 4u  /* run the scan as one serial chain per sequence even where
                                       prism_scan_segments() would cut it (see there) */
#define PRISM_FLAG_CHECK_WAIT_TIMEOUT 8u  /* diagnostic of the failure path: on the PRISM_BF16 path
                                             (ignored on the PRISM_F32 path, refused by
                                             prism_decode_step), every CTA of the scan
                                             first waits, with a short poll limit, on an mbarrier
                                             that nothing completes (no copy or MMA is in flight
                                             then); the wait gives up and the status word is set,
                                             as a real timeout would set it, and the outputs are
                                             then computed as without the flag.  prism_device_status
                                             must read nonzero after such a call. */

typedef struct {
    int B, T, H;          /* batch, sequence length, heads */
    int d_k, d_v;         /* key / value head dims (supported: d_k == d_v in {16,32,64,128};
                             PRISM_F32: d <= 64) */
    int conv_width;       /* w, ShortConv taps, 1..8 */
    int L;                /* refinement steps, 0..8 */
    int chunk;            /* scan chunk length C in {16, 32, 64} */
    prism_dtype dtype;    /* I/O type of q and k and v */
    unsigned flags;       /* PRISM_FLAG_* */
} prism_dims;

enum {
    PRISM_OK = 0,
    PRISM_ERR_INVALID_ARG = 1,   /* null required pointer, non-positive size, bad dtype */
    PRISM_ERR_UNSUPPORTED = 2,   /* dims outside the supported set */
    PRISM_ERR_MISALIGNED = 3,    /* a tensor pointer is not 16-byte aligned (workspace: 256) */
    PRISM_ERR_WORKSPACE = 4,     /* workspace NULL or smaller than prism_workspace_bytes() */
    PRISM_ERR_LAUNCH = 5,        /* a kernel launch failed (cudaGetLastError) */
    PRISM_ERR_CUDA = 6,          /* another CUDA runtime call failed */
    PRISM_ERR_SCRATCH_LIMIT = 7  /* prism_forward_static: the dims need more scratch than
                                    PRISM_STATIC_SCRATCH_BYTES */
};

/* Workspace regions (see prism_workspace_layout). */
enum {
    PRISM_WS_STATUS = 0,   /* int32[2]: device status word (nonzero = a bounded wait gave up), flag */
    PRISM_WS_KL = 1,       /* PRISM_F32: k^(l)              [B,T,H,L,d_k] fp32 */
    PRISM_WS_DL = 2,       /* PRISM_F32: beta^(l) delta^(l) [B,T,H,L,d_v] fp32 */
    PRISM_WS_WBLOCKS = 3,  /* PRISM_BF16: fp16 hi/lo weight blocks */
    PRISM_WS_WQ = 4,       /* PRISM_BF16, per chunk [B,H,NC,2C,d]: W = T diag(beta gamma) K and
                              Qt = diag(gamma) Q - P W (hi half), fp16, interleaved (below) */
    PRISM_WS_QK = 5,       /*   Qt lo half and Kt = diag(gamma_C/gamma) K, fp16, interleaved   */
    PRISM_WS_U = 6,        /*   U = T diag(beta)(V - R)                          [C,d]  fp32 */
    PRISM_WS_OI = 7,       /*   O_intra = P U + O_l                              [C,d]  fp32 */
    PRISM_WS_N = 8,        /*   N^T, N = sum_l D_l^T diag(gamma_C/gamma) K_l     [d,d]  fp32 */
    PRISM_WS_GC = 9,       /*   gamma_C, [B,H,NC]                                       fp32 */
    PRISM_WS_SEG = 10,     /* sequence split only (prism_scan_segments() = P > 1): three arrays
                              [B,H,P,d,d] fp32 — each segment's entering state, and the c and M
                              of its affine map S_end = S_start M + c */
    PRISM_WS_COUNT = 11
};

/* Inside one chunk, the PRISM_BF16 per-chunk arrays (R rows x d features) are
 * stored in 16-byte column pieces: element (r, f) at ((f / V) * R + r) * V + f % V
 * with V = 16 / element size (8 for fp16, 4 for fp32).  U and O_intra use R = C; N^T
 * (rows k, features v) uses R = d.  WQ and QK hold two fp16 maps each, sharing the
 * pieces: in piece f / 8, first the C rows of W (resp. Qt lo), then the C rows of
 * Qt hi (resp. Kt), so W(r, f) is at ((f / 8) * 2C + r) * 8 + f % 8 and
 * Qt_hi(r, f) at ((f / 8) * 2C + C + r) * 8 + f % 8. */

/* Bytes of device workspace for these dims (0 if the dims are invalid).  The
 * workspace holds each chunk's factored state map: the chunkwise form of the
 * recurrence S_t = S_{t-1} A_t + B_t ("Technical Summary: PRISM", §2.1), whose
 * state-independent part (§2.2, last paragraph) is what allows a parallel scan. */
PRISM_API size_t prism_workspace_bytes(const prism_dims* dims);

/* Byte offset of each PRISM_WS_* region inside the workspace (SIZE_MAX when the
 * region is absent for these dims).  offsets must hold n >= PRISM_WS_COUNT
 * entries.  Returns PRISM_OK or an error code. */
PRISM_API int prism_workspace_layout(const prism_dims* dims, size_t* offsets, int n);

/* The full mixer forward pass (anchor, refinement, write, chunkwise scan,
 * readout) over B sequences = prism_prepare followed by prism_scan.
 *   seq_lens    NULL: every sequence has length T.  Otherwise tokens
 *               t >= seq_lens[b] are padding: out is 0 there, they do not
 *               touch the state, and their input values are never used
 *               (NaN in padding cannot reach any output).  0 <= len <= T.
 *   final_state NULL: not written.  Else S after each sequence's last token.
 *   workspace   device buffer of at least prism_workspace_bytes(dims) bytes,
 *               256-byte aligned; its contents are scratch.
 * Returns PRISM_OK after enqueueing, or an error code (nothing launched). */
PRISM_API int prism_forward(const prism_dims* dims,
                            const void* q, const void* k, const void* v,
                            const float* log_alpha, const float* beta,
                            const float* conv_w, const float* Wk, const float* Wp,
                            const float* wbeta,
                            float* out, float* final_state, const int32_t* seq_lens,
                            void* workspace, size_t workspace_bytes, void* stream);

/* prism_forward resuming sequences (for instance a long sequence processed in
 * pieces): the chunkwise scan starts from initial_state [B,H,d_v,d_k] fp32 (NULL:
 * zero), and the anchor of tokens 0..w-1 reads v_hist [B,H,w,d_v] in `dtype` — the
 * v rows of the w tokens before t = 0, oldest first (NULL: zeros).  Running a
 * sequence in two pieces, the second from the first's final_state and last w v
 * rows, gives the one-piece result up to rounding.  The pages' layer has S_0 = 0
 * and no history; these arguments only extend it to sequences that continue. */
PRISM_API int prism_forward_from(const prism_dims* dims,
                                 const void* q, const void* k, const void* v,
                                 const float* log_alpha, const float* beta,
                                 const float* conv_w, const float* Wk, const float* Wp,
                                 const float* wbeta,
                                 const float* initial_state, const void* v_hist,
                                 float* out, float* final_state, const int32_t* seq_lens,
                                 void* workspace, size_t workspace_bytes, void* stream);

/* (No counterpart in the pages: failure detection of this library.)
 * The device status word of the last prism_forward / prism_forward_from /
 * prism_prepare + prism_scan call that used this workspace (same dims).  Every
 * wait those kernels make on an mbarrier is bounded; one that gives up writes a
 * nonzero word instead of hanging, and that call's outputs are then invalid.
 *   *status = 0 when every wait completed and, on the PRISM_BF16 path, every value
 *   written to out and final_state is finite.  Bit 0 (1): a wait gave up.  Bit 1 (2,
 *   PRISM_BF16 path): a non-finite value reached out or final_state.  With finite
 *   inputs this means a value beyond the fp16 range of the tensor-core operands: a
 *   refinement chain that diverges until |delta^(l)| >= 65504, which long chains (L near
 *   8) with large gains can reach.  The outputs are then invalid; the fp32 path
 *   (PRISM_F32) is not limited this way.
 * Waits for `stream` (it copies 4 bytes from the workspace and synchronises), so
 * call it on the stream the forward pass ran on, after it.  The word is cleared
 * at the start of each forward call.  Errors: as for prism_forward's dims and
 * workspace checks; PRISM_ERR_INVALID_ARG for a NULL status; PRISM_ERR_CUDA when
 * the copy or the synchronisation fails.  prism_forward_static keeps its word in
 * the library's own scratch: prism_static_status reads that one. */
PRISM_API int prism_device_status(const prism_dims* dims, const void* workspace,
                                  size_t workspace_bytes, int* status, void* stream);

/* (No counterpart in the pages: a debugging aid of this library.)
 * In the bounds-checked debug build of the library (every translation unit compiled
 * with -DPRISM_DEBUG_BOUNDS; build.py's build_debug() makes _build/debug/libprism.so),
 * the tensor-core forward kernels (prepare, scan, the sequence split's chain) and the
 * decode kernel check each index of their plain loads and stores, of their shared-memory
 * tile writes and of the source ranges of their bulk copies against the extent of the
 * array it addresses; an access that would fall outside is skipped and bit value 2 of a
 * library-wide word is set.  This call synchronises the device and returns that word in
 * *word (0: no violation since the last clear), clearing it when `clear` is nonzero.  In
 * the normal build it writes 0 and returns PRISM_ERR_UNSUPPORTED.  Errors:
 * PRISM_ERR_INVALID_ARG for a NULL word; PRISM_ERR_CUDA when the synchronisation or the
 * copy fails.  Not covered: the fp32 path's kernels and the backward pass. */
PRISM_API int prism_debug_bounds(int* word, int clear);

/* (No counterpart in the pages: a debugging aid of this library.)
 * y[i] = GELU(x[i]) for i < n as the bf16 path's prepare kernel evaluates it in its
 * refinement loop: x Phi(x) with erf by Hastings' rational approximation (Abramowitz and
 * Stegun 7.1.26), within about 4e-7 max(|x|, 1) of the exact GELU of "Technical Summary:
 * PRISM", §2.2.  x and y are device arrays of n fp32 values (caller-owned, may not
 * overlap); the work is enqueued on `stream` (a cudaStream_t; NULL = the legacy default
 * stream).  Errors: PRISM_ERR_INVALID_ARG for n < 0 or a NULL array with n > 0;
 * PRISM_ERR_CUDA when the launch fails.  n = 0 does nothing. */
PRISM_API int prism_debug_activation(const float* x, float* y, long long n, void* stream);

/* One token of every sequence (dims->T must be 1; chunk is ignored): the
 * recurrence of §2.1-2.2 of "Technical Summary: PRISM" applied to a single token,
 * for streaming generation after a prism_forward_from / prism_forward prefix.
 *   q, k, v     [B,H,d] in `dtype` (the token's rows)
 *   log_alpha, beta [B,H] fp32
 *   state       [B,H,d_v,d_k] fp32: S before the token on entry, after it on return
 *   v_hist      [B,H,w,d_v] in `dtype`: the v rows of the w previous tokens, oldest
 *               first; on return it has moved by one token (v appended)
 *   out         [B,H,d_v] fp32, o_t = S_t q_t
 * No workspace; every sequence advances (no seq_lens).  Arithmetic is fp32 on the
 * CUDA cores.  The pages describe no decoding procedure; this entry point has no
 * counterpart there beyond the recurrence itself. */
PRISM_API int prism_decode_step(const prism_dims* dims,
                                const void* q, const void* k, const void* v,
                                const float* log_alpha, const float* beta,
                                const float* conv_w, const float* Wk, const float* Wp,
                                const float* wbeta,
                                float* state, void* v_hist, float* out, void* stream);

/* State-independent stage (fully parallel over chunks; "Technical Summary:
 * PRISM", §2.2 stages 1-2 and the state-independence noted at its end):
 * anchor, refinement and,
 * on the PRISM_BF16 path, each chunk's factored affine state map; results go
 * to the workspace regions listed above. */
PRISM_API int prism_prepare(const prism_dims* dims,
                            const void* q, const void* k, const void* v,
                            const float* log_alpha, const float* beta,
                            const float* conv_w, const float* Wk, const float* Wp,
                            const float* wbeta, const int32_t* seq_lens,
                            void* workspace, size_t workspace_bytes, void* stream);

/* Number of segments P the scan cuts each sequence into (1: one serial chain).
 * The chunk chain is serial in time, so few long sequences (a small B*H) leave most
 * of the GPU idle.  Each chunk acts on the state as an affine map S1 = S0 M + c
 * ("Technical Summary: PRISM", §2.2, last paragraph: the update is state-independent,
 * the condition for parallel prefix scanning), so a segment of chunks composes to
 * one such map.  With P > 1 the scan runs: segment 0 in full and, in parallel, the
 * (M, c) of every later segment; the entering states chained segment to segment;
 * segments 1..P-1 in full from them.  About twice the chain work, P-fold shorter.
 * P > 1 only on the PRISM_BF16 path with d = 128 and chunk 32 or 64, without
 * PRISM_FLAG_NO_SEQ_SPLIT, when the first pass fits one wave of CTAs
 * (B*H*4*(2P-1) <= 152) with P >= 3 and at least 8 chunks per segment; P <= 16.
 * A function of the dims alone.  Returns 0 for invalid dims. */
PRISM_API int prism_scan_segments(const prism_dims* dims);

/* Serial stage ("Technical Summary: PRISM", §2.1: S_t = S_{t-1} A_t + B_t,
 * composed chunk to chunk): the state chain and the outputs, from a
 * workspace filled by prism_prepare with the same dims and inputs. */
PRISM_API int prism_scan(const prism_dims* dims,
                         const void* q, const void* k, const void* v,
                         const float* log_alpha, const float* beta,
                         const int32_t* seq_lens, void* workspace, size_t workspace_bytes,
                         float* out, float* final_state, void* stream);

/* Size of the library's own device scratch array used by prism_forward_static. */
#define PRISM_STATIC_SCRATCH_BYTES (32u << 20)

/* prism_forward without a caller-provided workspace.  (The paper has no
 * counterpart: this is a deployment convenience of this library.)
 *
 * For callers that cannot allocate device memory where they run the layer
 * (pre-planned memory arenas, frameworks that forbid allocation on the hot
 * path, plugins handed only input and output buffers).  The scratch is a
 * fixed array of PRISM_STATIC_SCRATCH_BYTES in the library's device memory;
 * every GPU that loads the library holds it until the process exits.  Inputs
 * and outputs are as for prism_forward.
 *   - Dims whose prism_workspace_bytes() exceeds PRISM_STATIC_SCRATCH_BYTES
 *     are rejected with PRISM_ERR_SCRATCH_LIMIT before anything is launched.
 *   - Nothing is allocated: no cudaMalloc, cudaFree or allocating library call.
 *   - Every call looks up the array's device address with the caller's device
 *     current (cudaGetSymbolAddress; not cached, so a device reset or a new
 *     context cannot leave a stale address behind).  The first call on a
 *     device may load the library's device code: make it before any stream
 *     capture on that device.
 *   - The bounded-wait status word of these calls lives in the library's own
 *     array; prism_device_status does not read it.
 *   - All calls on a device share the array and it keeps the last call's
 *     contents.  Calls that overlap on the GPU (other streams, or threads
 *     without ordering between their launches) race on it: serialise them. */
/* (No counterpart in the pages: failure detection of this library.)
 * prism_device_status for prism_forward_static: the device status word of the last
 * static call with these dims on the current device (0: every bounded wait completed),
 * read from the library's scratch array.  Waits for `stream` like prism_device_status.
 * Calls on the device share the array, so the word is that of whichever static call ran
 * last.  Errors: as for prism_forward_static's dims checks; PRISM_ERR_INVALID_ARG for a
 * NULL status; PRISM_ERR_CUDA when the lookup, the copy or the synchronisation fails. */
PRISM_API int prism_static_status(const prism_dims* dims, int* status, void* stream);

PRISM_API int prism_forward_static(const prism_dims* dims,
                                   const void* q, const void* k, const void* v,
                                   const float* log_alpha, const float* beta,
                                   const float* conv_w, const float* Wk, const float* Wp,
                                   const float* wbeta,
                                   float* out, float* final_state, const int32_t* seq_lens,
                                   void* stream);

/* ---- Backward pass ----
 * Gradients of a scalar loss through prism_forward ("Technical Summary: PRISM",
 * §2.1-2.2: the anchor, the refinement, the rank-L write and the gated delta-rule
 * recurrence from a zero state), given
 *   d_out          [B,T,H,d_v] fp32: dLoss/d out (ignored at padding tokens)
 *   d_final_state  [B,H,d_v,d_k] fp32: dLoss/d final_state, or NULL (zero)
 * Outputs (fp32, every element overwritten; zero at padding tokens):
 *   dq, dk, dv     [B,T,H,d]
 *   dlog_alpha, dbeta [B,T,H]
 *   dconv_w        [H,w,d_v]
 *   dWk, dWp       [H,L,d,d]      (not written when L = 0)
 *   dwbeta         [H,L,d_v]      (not written when L = 0)
 * Inputs are those of prism_forward; d_k must equal d_v.  dims->chunk is ignored.
 * Arithmetic is fp32 on the CUDA cores: the refinement per token (recomputed), the
 * state forward with a checkpoint every 16 tokens and then backwards block by block
 * (the block's states recomputed from its checkpoint), the refinement chain backwards,
 * and token sums for the weight gradients.  Deterministic (no atomics).  The workspace
 * (prism_backward_workspace_bytes) holds per-token factors and the checkpoints; it is
 * caller-owned, 256-byte aligned, and needs no initialisation.  Errors as for
 * prism_forward; asynchronous on `stream`. */
PRISM_API size_t prism_backward_workspace_bytes(const prism_dims* dims);
PRISM_API int prism_backward(const prism_dims* dims,
                             const void* q, const void* k, const void* v,
                             const float* log_alpha, const float* beta,
                             const float* conv_w, const float* Wk, const float* Wp,
                             const float* wbeta,
                             const float* d_out, const float* d_final_state,
                             float* dq, float* dk, float* dv,
                             float* dlog_alpha, float* dbeta,
                             float* dconv_w, float* dWk, float* dWp, float* dwbeta,
                             const int32_t* seq_lens, void* workspace, size_t workspace_bytes,
                             void* stream);

/* ---- Host-to-host forward pass ----
 * prism_forward on HOST buffers: q, k, v, log_alpha, beta, conv_w, Wk, Wp, wbeta,
 * seq_lens are read from host memory and out, final_state written to host memory
 * (same shapes and meaning as prism_forward; final_state and seq_lens may be NULL,
 * conv_w and the weights too when L = 0).  The work is cut into pieces, and piece i's
 * kernels run while piece i+1 is copied in and piece i-1 copied out:
 *   streams[0] copies in, streams[1] runs the kernels, streams[2] copies out
 *   (caller-owned cudaStream_t handles; streams = NULL runs all on the legacy default
 *   stream; a single piece runs on streams[2] alone).
 * Pieces are groups of whole sequences when B > 1 and chunk-aligned token segments
 * when B = 1 (a segment starts from the previous one's final state and reads the v rows
 * before it as the anchor's history, so the result equals one prism_forward call).  At
 * most max_pieces (1..PRISM_HOST_MAX_PIECES) pieces, each moving at least
 * min_piece_bytes of q, k, v and out (0: no minimum).
 *   arena  DEVICE buffer of at least prism_host_arena_bytes(dims, max_pieces,
 *          min_piece_bytes) bytes, 256-byte aligned: device copies of the inputs and
 *          outputs and a workspace; its contents are scratch.
 * Ordering: the call's work starts after the work already enqueued on all three
 * streams and is complete when streams[2] gets past it (synchronise on streams[2], or
 * wait on an event recorded there, before reading out or final_state).  Overlap needs
 * page-locked host memory; pageable buffers work but the copies then block.  When
 * B = 1, seq_lens[0] is read on the host during the call.  Errors: those of
 * prism_forward's dims checks; PRISM_ERR_INVALID_ARG for a NULL required pointer,
 * max_pieces out of range or PRISM_FLAG_VHIST_TOKEN_MAJOR in dims->flags;
 * PRISM_ERR_WORKSPACE / PRISM_ERR_MISALIGNED for the arena; PRISM_ERR_CUDA when a copy,
 * event or stream call fails (part of the work may then be enqueued and the outputs are
 * undefined).  The pages describe the layer, not its data movement: this entry point
 * has no counterpart there. */
#define PRISM_HOST_MAX_PIECES 16

/* The pieces prism_forward_host cuts these dims into: *n_pieces and their boundaries
 * bounds[0] = 0 < bounds[1] < ... < bounds[*n_pieces] (= B when B > 1, else T); bounds
 * must hold max_pieces + 1 ints. */
PRISM_API int prism_host_plan(const prism_dims* dims, int max_pieces, size_t min_piece_bytes,
                              int* n_pieces, int* bounds);
/* Device arena bytes for prism_forward_host (0 if the arguments are invalid). */
PRISM_API size_t prism_host_arena_bytes(const prism_dims* dims, int max_pieces,
                                        size_t min_piece_bytes);
PRISM_API int prism_forward_host(const prism_dims* dims,
                                 const void* q, const void* k, const void* v,
                                 const float* log_alpha, const float* beta,
                                 const float* conv_w, const float* Wk, const float* Wp,
                                 const float* wbeta,
                                 float* out, float* final_state, const int32_t* seq_lens,
                                 int max_pieces, size_t min_piece_bytes,
                                 void* arena, size_t arena_bytes, void* const* streams);

/* Static description of an error code. */
PRISM_API const char* prism_strerror(int code);

#ifdef __cplusplus
}
#endif
#endif /* PRISM_H */
