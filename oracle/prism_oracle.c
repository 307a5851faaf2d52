/*
 * PRISM mixer forward pass: the CPU oracle.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the package's smoke check and
 * the benchmark's CPU-baseline leg may build, load or call this file.  It
 * shares no code, header or constant with the CUDA path.
 *
 * A plain, slow, token-by-token fp64 restatement of the method described in
 * "Technical Summary: PRISM (Parallel Residual Iterative Sequence Model)"
 * (gist.science/paper/2602.10796):
 *
 *   §2.1 Write-Forget Decoupling:   S_t = S_{t-1} A_t + B_t,
 *        A_t rank-1 "identical to Gated DeltaNet": A_t = alpha_t (I - beta_t k_t k_t^T)
 *   §2.2 Input-Anchored Loop Unrolling, stage 1 (anchor):
 *        u_t = sum_{j=1..w} c_j (.) v_{t-j}      (strictly causal ShortConv on v)
 *   §2.2 stage 2 (refinement), l = 1..L:
 *        k^(l) = normalize(W_k^(l) u_t)          (direction)
 *        p^(l) = W_p^(l) u_t                      (gain)
 *        delta^(l) = GELU(p^(l) (.) r^(l)),  r^(l+1) = r^(l) - delta^(l)
 *        beta^(l) = sigmoid(w_beta^(l) . u_t)     (confidence gate)
 *   §2.2 final injection: B_t = sum_l beta^(l) delta^(l) k^(l)^T
 *   §3.3 (contribution 3): at L = 0 the model is Gated DeltaNet.
 *
 * Readings where the summary is silent:
 *   - r^(1) = v_t - u_t.
 *   - The Gated DeltaNet write beta_t v_t k_t^T is always part of B_t and the
 *     L refinement terms add to it; otherwise B_t is empty at L = 0 and the
 *     model could not reduce to Gated DeltaNet there.
 *   - normalize(x) = x / sqrt(|x|^2 + 1e-6); GELU is the exact erf form.
 *   - beta^(l) = sigmoid(w_beta^(l) . u_t) without bias; alpha_t = exp(log_alpha_t).
 *   - Readout o_t = S_t q_t (post-update, no scaling); S_0 = 0 unless an initial
 *     state is given, and the anchor of the first tokens reads zeros before t = 0
 *     unless the v rows of the preceding tokens are given (resuming a sequence).
 *   - Right padding: for t >= len_b the output is 0 and the state is frozen.
 *
 * S is d_v x d_k.  The product S_{t-1} A_t is formed as
 * alpha_t (S - beta_t (S k_t) k_t^T), which is the matrix product with
 * A_t = alpha_t (I - beta_t k_t k_t^T) expanded by distributivity.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include "prism_oracle.h"

#define NORM_EPS 1e-6

static double gelu_erf(double x) { return 0.5 * x * (1.0 + erf(x / sqrt(2.0))); }
static double sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

typedef struct {
    const oracle_problem* P;
    const int* items;        /* (b*H + h) indices to process */
    int n_items;
    int next;                /* shared work counter */
    pthread_mutex_t lock;
    int status;
} job_t;

/* Offsets into [B,T,H,X] and [B,T,H,L,X] row-major arrays. */
static size_t off_bthx(const oracle_problem* P, int b, int t, int h, int X) {
    return (((size_t)b * P->T + t) * P->H + h) * (size_t)X;
}
static size_t off_bthlx(const oracle_problem* P, int b, int t, int h, int l, int X) {
    return ((((size_t)b * P->T + t) * P->H + h) * (size_t)P->L + l) * (size_t)X;
}

/* One (b, h) sequence, token by token. */
static int run_sequence(const oracle_problem* P, int b, int h) {
    const int T = P->T, dk = P->dk, dv = P->dv, w = P->w, L = P->L;
    const int len = P->seq_lens ? P->seq_lens[b] : T;
    double* S = calloc((size_t)dv * dk, sizeof(double));
    double* Bw = malloc((size_t)dv * dk * sizeof(double));
    double* u = malloc(sizeof(double) * dv);
    double* r = malloc(sizeof(double) * dv);
    double* p = malloc(sizeof(double) * dv);
    double* dl = malloc(sizeof(double) * dv);
    double* kk = malloc(sizeof(double) * dk);
    double* Sk = malloc(sizeof(double) * dv);
    if (!S || !Bw || !u || !r || !p || !dl || !kk || !Sk) {
        free(S); free(Bw); free(u); free(r); free(p); free(dl); free(kk); free(Sk);
        return -1;
    }
    const oracle_trace* tr = P->trace;
    if (P->initial_state)
        memcpy(S, P->initial_state + ((size_t)b * P->H + h) * dv * dk, sizeof(double) * dv * dk);

    for (int t = 0; t < T; ++t) {
        double* o = P->out + off_bthx(P, b, t, h, dv);
        if (t >= len) {                 /* padding: output 0, state frozen */
            for (int i = 0; i < dv; ++i) o[i] = 0.0;
            continue;
        }
        const double* vt = P->v + off_bthx(P, b, t, h, dv);
        const double* kt = P->k + off_bthx(P, b, t, h, dk);
        const double* qt = P->q + off_bthx(P, b, t, h, dk);
        const double alpha = exp(P->log_alpha[((size_t)b * T + t) * P->H + h]);
        const double beta = P->beta[((size_t)b * T + t) * P->H + h];

        /* Stage 1: anchor u_t = sum_{j=1..w} c_j (.) v_{t-j}; before t = 0 the given
           history (row w + t - j of v_hist), else zero. */
        for (int i = 0; i < dv; ++i) u[i] = 0.0;
        for (int j = 1; j <= w; ++j) {
            const double* vp;
            if (t - j >= 0)
                vp = P->v + off_bthx(P, b, t - j, h, dv);
            else if (P->v_hist)
                vp = P->v_hist + (((size_t)b * P->H + h) * w + (w + t - j)) * dv;
            else
                break;
            const double* c = P->conv_w + ((size_t)h * w + (j - 1)) * dv;
            for (int i = 0; i < dv; ++i) u[i] += c[i] * vp[i];
        }
        /* r^(1) = v_t - u_t */
        for (int i = 0; i < dv; ++i) r[i] = vt[i] - u[i];
        if (tr && tr->u) memcpy(tr->u + off_bthx(P, b, t, h, dv), u, sizeof(double) * dv);
        if (tr && tr->r1) memcpy(tr->r1 + off_bthx(P, b, t, h, dv), r, sizeof(double) * dv);

        /* Gated DeltaNet base write beta_t v_t k_t^T. */
        for (int i = 0; i < dv; ++i)
            for (int j = 0; j < dk; ++j) Bw[(size_t)i * dk + j] = beta * vt[i] * kt[j];

        /* Stage 2: refinement loop. */
        for (int l = 0; l < L; ++l) {
            const double* Wk = P->Wk + ((size_t)h * L + l) * dk * dv;   /* [dk, dv] */
            const double* Wp = P->Wp + ((size_t)h * L + l) * dv * dv;   /* [dv, dv] */
            const double* wb = P->wbeta + ((size_t)h * L + l) * dv;     /* [dv] */
            double nrm2 = 0.0;
            for (int a = 0; a < dk; ++a) {
                double s = 0.0;
                for (int c = 0; c < dv; ++c) s += Wk[(size_t)a * dv + c] * u[c];
                kk[a] = s;
                nrm2 += s * s;
            }
            const double inv = 1.0 / sqrt(nrm2 + NORM_EPS);
            for (int a = 0; a < dk; ++a) kk[a] *= inv;
            for (int a = 0; a < dv; ++a) {
                double s = 0.0;
                for (int c = 0; c < dv; ++c) s += Wp[(size_t)a * dv + c] * u[c];
                p[a] = s;
            }
            double z = 0.0;
            for (int c = 0; c < dv; ++c) z += wb[c] * u[c];
            const double bl = sigmoid(z);
            for (int i = 0; i < dv; ++i) {
                const double x = p[i] * r[i];
                dl[i] = P->identity_act ? x : gelu_erf(x);
                r[i] -= dl[i];
            }
            for (int i = 0; i < dv; ++i)
                for (int j = 0; j < dk; ++j) Bw[(size_t)i * dk + j] += bl * dl[i] * kk[j];
            if (tr) {
                if (tr->kl) memcpy(tr->kl + off_bthlx(P, b, t, h, l, dk), kk, sizeof(double) * dk);
                if (tr->pl) memcpy(tr->pl + off_bthlx(P, b, t, h, l, dv), p, sizeof(double) * dv);
                if (tr->delta) memcpy(tr->delta + off_bthlx(P, b, t, h, l, dv), dl, sizeof(double) * dv);
                if (tr->betal) tr->betal[(((size_t)b * T + t) * P->H + h) * L + l] = bl;
                if (tr->dl) {
                    double* dst = tr->dl + off_bthlx(P, b, t, h, l, dv);
                    for (int i = 0; i < dv; ++i) dst[i] = bl * dl[i];
                }
            }
        }
        if (tr && tr->r_final) memcpy(tr->r_final + off_bthx(P, b, t, h, dv), r, sizeof(double) * dv);
        if (tr && tr->Bt) memcpy(tr->Bt + off_bthx(P, b, t, h, dv * dk), Bw, sizeof(double) * dv * dk);

        /* S <- S A_t + B_t, with S A_t = alpha (S - beta (S k) k^T). */
        for (int i = 0; i < dv; ++i) {
            double s = 0.0;
            for (int j = 0; j < dk; ++j) s += S[(size_t)i * dk + j] * kt[j];
            Sk[i] = s;
        }
        for (int i = 0; i < dv; ++i)
            for (int j = 0; j < dk; ++j) {
                double* sij = &S[(size_t)i * dk + j];
                *sij = alpha * (*sij - beta * Sk[i] * kt[j]) + Bw[(size_t)i * dk + j];
            }
        /* o_t = S_t q_t */
        for (int i = 0; i < dv; ++i) {
            double s = 0.0;
            for (int j = 0; j < dk; ++j) s += S[(size_t)i * dk + j] * qt[j];
            o[i] = s;
        }
    }
    if (P->final_state)
        memcpy(P->final_state + ((size_t)b * P->H + h) * dv * dk, S, sizeof(double) * dv * dk);
    free(S); free(Bw); free(u); free(r); free(p); free(dl); free(kk); free(Sk);
    return 0;
}

static void* worker(void* arg) {
    job_t* J = (job_t*)arg;
    for (;;) {
        pthread_mutex_lock(&J->lock);
        const int i = J->next++;
        pthread_mutex_unlock(&J->lock);
        if (i >= J->n_items) break;
        const int bh = J->items[i];
        if (run_sequence(J->P, bh / J->P->H, bh % J->P->H) != 0) {
            pthread_mutex_lock(&J->lock);
            J->status = -1;
            pthread_mutex_unlock(&J->lock);
        }
    }
    return NULL;
}

int prism_oracle_forward(const oracle_problem* P, const int* bh_items, int n_items,
                         int n_threads) {
    if (!P || P->B <= 0 || P->T <= 0 || P->H <= 0 || P->dk <= 0 || P->dv <= 0 ||
        P->w < 0 || P->L < 0 || !P->q || !P->k || !P->v || !P->log_alpha || !P->beta ||
        !P->out || (P->w > 0 && !P->conv_w) ||
        (P->L > 0 && (!P->Wk || !P->Wp || !P->wbeta)))
        return -2;
    int* all = NULL;
    if (!bh_items) {
        n_items = P->B * P->H;
        all = malloc(sizeof(int) * (size_t)n_items);
        if (!all) return -1;
        for (int i = 0; i < n_items; ++i) all[i] = i;
        bh_items = all;
    }
    job_t J;
    J.P = P; J.items = bh_items; J.n_items = n_items; J.next = 0; J.status = 0;
    pthread_mutex_init(&J.lock, NULL);
    if (n_threads < 1) n_threads = 1;
    if (n_threads > n_items) n_threads = n_items > 0 ? n_items : 1;
    pthread_t* th = malloc(sizeof(pthread_t) * (size_t)n_threads);
    if (!th) { free(all); return -1; }
    for (int i = 0; i < n_threads; ++i) pthread_create(&th[i], NULL, worker, &J);
    for (int i = 0; i < n_threads; ++i) pthread_join(th[i], NULL);
    free(th);
    pthread_mutex_destroy(&J.lock);
    free(all);
    return J.status;
}
