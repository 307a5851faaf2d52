/*
 * PRISM mixer forward pass: CPU oracle interface (fp64).
 * TEST INFRASTRUCTURE ONLY: used by the tests, the smoke check and the
 * benchmark's CPU-baseline leg; never by the CUDA path.
 *
 * All arrays are row-major fp64 unless stated:
 *   q, k [B,T,H,dk]; v [B,T,H,dv]; log_alpha, beta [B,T,H];
 *   conv_w [H,w,dv] (row j-1 multiplies v_{t-j});
 *   Wk [H,L,dk,dv]; Wp [H,L,dv,dv]; wbeta [H,L,dv];
 *   seq_lens [B] int32 or NULL (all sequences have length T);
 *   out [B,T,H,dv]; final_state [B,H,dv,dk] or NULL;
 *   initial_state [B,H,dv,dk] or NULL (S_0 = 0);
 *   v_hist [B,H,w,dv] or NULL: v of the w tokens before t = 0, oldest first, which
 *   the anchor of the first tokens reads (zero history when NULL).
 */
#ifndef PRISM_ORACLE_H
#define PRISM_ORACLE_H

#ifdef __cplusplus
extern "C" {
#endif

/* Optional per-token intermediates (any pointer may be NULL). */
typedef struct {
    double* u;        /* [B,T,H,dv]      anchor u_t */
    double* r1;       /* [B,T,H,dv]      r^(1) = v_t - u_t */
    double* r_final;  /* [B,T,H,dv]      r^(L+1) */
    double* kl;       /* [B,T,H,L,dk]    k^(l) (normalised) */
    double* pl;       /* [B,T,H,L,dv]    p^(l) */
    double* delta;    /* [B,T,H,L,dv]    delta^(l) */
    double* betal;    /* [B,T,H,L]       beta^(l) */
    double* dl;       /* [B,T,H,L,dv]    beta^(l) delta^(l) */
    double* Bt;       /* [B,T,H,dv,dk]   the full write B_t (tiny problems only) */
} oracle_trace;

typedef struct {
    int B, T, H, dk, dv, w, L;
    int identity_act;   /* 0: GELU (erf form); 1: identity (no-GELU ablation) */
    const double *q, *k, *v, *log_alpha, *beta, *conv_w, *Wk, *Wp, *wbeta;
    const int* seq_lens;
    double* out;
    double* final_state;
    const oracle_trace* trace;
    const double* initial_state;
    const double* v_hist;
} oracle_problem;

/* Runs the (b,h) sequences listed in bh_items (index b*H+h; NULL = all) on
 * n_threads threads.  Rows of out/final_state for unlisted pairs are untouched.
 * Returns 0, -1 on allocation failure, -2 on invalid arguments. */
int prism_oracle_forward(const oracle_problem* P, const int* bh_items, int n_items,
                         int n_threads);

#ifdef __cplusplus
}
#endif
#endif
