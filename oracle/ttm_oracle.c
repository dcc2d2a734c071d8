/*
 * Float64 CPU oracle for the chunked test-time-training memory scan.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, plain reference that the
 * GPU library is compared against.  Only the test suite, the smoke check and
 * the benchmark's CPU-baseline leg may load it.  It shares no code, header,
 * table or helper with the CUDA path.
 *
 * What it computes is the token-by-token ("primal") recurrence, written out
 * exactly as the pages define it:
 *
 *   inner loss      l(W; k, v) = || f(k; W) - v ||^2
 *                   ("TTT layers 与 fast weights", eq (2); "论文速览 | Titans" §3.6)
 *   gradient        linear f(k;W) = W k:  grad = 2 (W k - v) k^T
 *                   ("TTT layers 与 fast weights", eq (4))
 *   mini-batch      every gradient of a chunk of b tokens is taken at the
 *                   state left by the previous chunk
 *                   ("TTT layers 与 fast weights", eq (6), mini-batch GD;
 *                    "论文速览 | Titans" §4.2)
 *   momentum        S_t = eta_t S_{t-1} - theta_t grad
 *   forgetting      M_t = (1 - alpha_t) M_{t-1} + S_t
 *                   ("论文速览 | Titans" §3.4 and §3.7;
 *                    "Continual Learning: From Attention to Neural Memory" §5.2)
 *   read            z_t = f(q_t; M_t), after token t's own write
 *                   ("TTT layers 与 fast weights", eq (3); "Continual Learning:
 *                    From Attention to Neural Memory" §4.2 and §4.7)
 *
 * Plain TTT-Linear is the same loop with eta = alpha = 0 (then S_t is just
 * -theta_t grad and W_t = W_{t-1} - theta_t grad).
 *
 * The deep memory is f(k) = W2 GELU(W1 k) with exact GELU
 * x/2 (1 + erf(x / sqrt 2)); its gradients are the chain rule written out:
 *   h = W1 k, a = GELU(h), y = W2 a, e = 2 (y - v)
 *   dl/dW2 = e a^T,   dl/dW1 = ((W2^T e) * GELU'(h)) k^T
 * ("论文速览 | Titans" §3.9; "Continual Learning: From Attention to Neural
 *  Memory" §4.2).  The pages name no activation; exact GELU is the reading
 * taken here.
 *
 * Layouts (all float64, row-major, contiguous):
 *   q, k      [B][H][T][dk]          v, z  [B][H][T][dv]
 *   eta, theta, alpha  [B][H][T]     (eta or alpha NULL means all zero)
 *   W0, S0    [B or 1][H][dv][dk]    (1 when shared_over_batch != 0; S0 NULL = 0)
 *   W_out, S_out [B][H][dv][dk]      (S_out may be NULL)
 * Deep memory: W1 [.][H][hidden][d], W2 [.][H][d][hidden], same for S1, S2.
 *
 * The gradient of the linear / Titans scan (oracle_linear_primal_bwd) is the
 * reverse-mode derivative of the same token loop, taken step by step in the
 * opposite order ("Continual Learning: From Attention to Neural Memory" §4.5:
 * the outer gradient follows the chain of state transitions backward; the
 * update is ordinary arithmetic and every step of it is differentiated, the
 * chunk-start snapshot included).  For a scalar outer loss L with adjoints
 * dz_t = dL/dz_t, dW_T = dL/dW_T, dS_T = dL/dS_T it returns dL/d of every
 * input: q, k, v, eta, theta, alpha, W0, S0.
 *
 * The DGD memory (oracle_dgd_primal) is the update of "Nested Learning" §8.1
 * eq (88) with the matrix memory and the L2 objective of eq (93), taken
 * chunk-wise as in §8.2 (the gradient at the state left by the previous
 * chunk):
 *   M_t = M_{t-1} (alpha_t I - eta_t k_t k_t^T) - eta_t (Mc k_t - v_t) k_t^T
 * with alpha_t a retention factor (alpha = 1 keeps everything) and eta_t the
 * step, both as printed (no factor 2 on the gradient, as eq (93) writes it).
 * The read is the one eq (86) prints, y_t = M_{t-1} q_t: the memory as it
 * stands before token t's own write (unlike the other memories here, whose
 * pages read after the write).
 *
 * The (b, h) sequences are independent, so they are spread over POSIX
 * threads; each one runs the plain loop below.
 */
#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

/* ------------------------------------------------------------------ */
/* linear memory                                                      */
/* ------------------------------------------------------------------ */

typedef struct {
    int B, H, T, dk, dv, chunk;
    const double *q, *k, *v, *eta, *theta, *alpha, *W0, *S0;
    int shared;
    double *z, *W_out, *S_out;
} lin_args;

/* one (b, h) sequence of the linear / Titans recurrence */
static void lin_one(const lin_args* a, int b, int h) {
    const int T = a->T, dk = a->dk, dv = a->dv;
    const size_t seq = (size_t)b * a->H + h;
    const size_t init = (size_t)(a->shared ? 0 : b) * a->H + h;
    const size_t nstate = (size_t)dv * dk;

    double* W = (double*)malloc(nstate * sizeof(double));
    double* S = (double*)malloc(nstate * sizeof(double));
    double* Wc = (double*)malloc(nstate * sizeof(double)); /* chunk-start snapshot */
    double* e = (double*)malloc((size_t)dv * sizeof(double));

    memcpy(W, a->W0 + init * nstate, nstate * sizeof(double));
    if (a->S0) memcpy(S, a->S0 + init * nstate, nstate * sizeof(double));
    else memset(S, 0, nstate * sizeof(double));

    for (int t = 0; t < T; ++t) {
        const double* kt = a->k + (seq * T + t) * dk;
        const double* qt = a->q + (seq * T + t) * dk;
        const double* vt = a->v + (seq * T + t) * dv;
        const double th = a->theta[seq * T + t];
        const double et = a->eta ? a->eta[seq * T + t] : 0.0;
        const double al = a->alpha ? a->alpha[seq * T + t] : 0.0;

        if (t % a->chunk == 0) memcpy(Wc, W, nstate * sizeof(double));

        /* prediction error at the chunk-start state: e = Wc k - v */
        for (int i = 0; i < dv; ++i) {
            double acc = 0.0;
            for (int j = 0; j < dk; ++j) acc += Wc[(size_t)i * dk + j] * kt[j];
            e[i] = acc - vt[i];
        }
        /* grad_ij = 2 e_i k_j; momentum, then forgetting */
        for (int i = 0; i < dv; ++i) {
            for (int j = 0; j < dk; ++j) {
                const size_t ij = (size_t)i * dk + j;
                const double g = 2.0 * e[i] * kt[j];
                S[ij] = et * S[ij] - th * g;
                W[ij] = (1.0 - al) * W[ij] + S[ij];
            }
        }
        /* read after the write: z = W q */
        double* zt = a->z + (seq * T + t) * dv;
        for (int i = 0; i < dv; ++i) {
            double acc = 0.0;
            for (int j = 0; j < dk; ++j) acc += W[(size_t)i * dk + j] * qt[j];
            zt[i] = acc;
        }
    }
    memcpy(a->W_out + seq * nstate, W, nstate * sizeof(double));
    if (a->S_out) memcpy(a->S_out + seq * nstate, S, nstate * sizeof(double));
    free(W); free(S); free(Wc); free(e);
}

/* ------------------------------------------------------------------ */
/* deep (2-layer MLP) memory                                          */
/* ------------------------------------------------------------------ */

static double gelu(double x) { return 0.5 * x * (1.0 + erf(x / sqrt(2.0))); }

/* d/dx GELU(x) = Phi(x) + x phi(x) */
static double gelu_grad(double x) {
    const double Phi = 0.5 * (1.0 + erf(x / sqrt(2.0)));
    const double phi = exp(-0.5 * x * x) / sqrt(2.0 * M_PI);
    return Phi + x * phi;
}

/* f(x) = W2 GELU(W1 x); W1 [hid][d], W2 [d][hid]; scratch hbuf/abuf [hid] */
static void mlp_apply(int d, int hid, const double* W1, const double* W2, const double* x,
                      double* hbuf, double* abuf, double* y) {
    for (int u = 0; u < hid; ++u) {
        double acc = 0.0;
        for (int j = 0; j < d; ++j) acc += W1[(size_t)u * d + j] * x[j];
        hbuf[u] = acc;
        abuf[u] = gelu(acc);
    }
    for (int i = 0; i < d; ++i) {
        double acc = 0.0;
        for (int u = 0; u < hid; ++u) acc += W2[(size_t)i * hid + u] * abuf[u];
        y[i] = acc;
    }
}

/* Gradient of ||W2 GELU(W1 k) - v||^2 with respect to W1 and W2. */
void oracle_mlp_grad(int d, int hid, const double* W1, const double* W2, const double* k,
                     const double* v, double* gW1, double* gW2) {
    double* hb = (double*)malloc((size_t)hid * sizeof(double));
    double* ab = (double*)malloc((size_t)hid * sizeof(double));
    double* y = (double*)malloc((size_t)d * sizeof(double));
    double* e = (double*)malloc((size_t)d * sizeof(double));
    mlp_apply(d, hid, W1, W2, k, hb, ab, y);
    for (int i = 0; i < d; ++i) e[i] = 2.0 * (y[i] - v[i]);
    for (int i = 0; i < d; ++i)
        for (int u = 0; u < hid; ++u) gW2[(size_t)i * hid + u] = e[i] * ab[u];
    for (int u = 0; u < hid; ++u) {
        double back = 0.0; /* (W2^T e)_u */
        for (int i = 0; i < d; ++i) back += W2[(size_t)i * hid + u] * e[i];
        const double delta = back * gelu_grad(hb[u]);
        for (int j = 0; j < d; ++j) gW1[(size_t)u * d + j] = delta * k[j];
    }
    free(hb); free(ab); free(y); free(e);
}

/* The loss itself, so that the gradient above can be checked by differences. */
double oracle_mlp_loss(int d, int hid, const double* W1, const double* W2, const double* k,
                       const double* v) {
    double* hb = (double*)malloc((size_t)hid * sizeof(double));
    double* ab = (double*)malloc((size_t)hid * sizeof(double));
    double* y = (double*)malloc((size_t)d * sizeof(double));
    mlp_apply(d, hid, W1, W2, k, hb, ab, y);
    double l = 0.0;
    for (int i = 0; i < d; ++i) l += (y[i] - v[i]) * (y[i] - v[i]);
    free(hb); free(ab); free(y);
    return l;
}

double oracle_gelu(double x) { return gelu(x); }
double oracle_gelu_grad(double x) { return gelu_grad(x); }

typedef struct {
    int B, H, T, d, hid, chunk;
    const double *q, *k, *v, *eta, *theta, *alpha, *W1_0, *W2_0, *S1_0, *S2_0;
    int shared;
    double *z, *W1_out, *W2_out, *S1_out, *S2_out;
} mlp_args;

static void mlp_one(const mlp_args* a, int b, int h) {
    const int T = a->T, d = a->d, hid = a->hid;
    const size_t seq = (size_t)b * a->H + h;
    const size_t init = (size_t)(a->shared ? 0 : b) * a->H + h;
    const size_t n = (size_t)hid * d; /* both W1 and W2 hold hid*d numbers */

    double* W1 = (double*)malloc(n * sizeof(double));
    double* W2 = (double*)malloc(n * sizeof(double));
    double* S1 = (double*)malloc(n * sizeof(double));
    double* S2 = (double*)malloc(n * sizeof(double));
    double* W1c = (double*)malloc(n * sizeof(double));
    double* W2c = (double*)malloc(n * sizeof(double));
    double* g1 = (double*)malloc(n * sizeof(double));
    double* g2 = (double*)malloc(n * sizeof(double));
    double* hb = (double*)malloc((size_t)hid * sizeof(double));
    double* ab = (double*)malloc((size_t)hid * sizeof(double));

    memcpy(W1, a->W1_0 + init * n, n * sizeof(double));
    memcpy(W2, a->W2_0 + init * n, n * sizeof(double));
    if (a->S1_0) memcpy(S1, a->S1_0 + init * n, n * sizeof(double));
    else memset(S1, 0, n * sizeof(double));
    if (a->S2_0) memcpy(S2, a->S2_0 + init * n, n * sizeof(double));
    else memset(S2, 0, n * sizeof(double));

    for (int t = 0; t < T; ++t) {
        const double* kt = a->k + (seq * T + t) * d;
        const double* qt = a->q + (seq * T + t) * d;
        const double* vt = a->v + (seq * T + t) * d;
        const double th = a->theta[seq * T + t];
        const double et = a->eta ? a->eta[seq * T + t] : 0.0;
        const double al = a->alpha ? a->alpha[seq * T + t] : 0.0;

        if (t % a->chunk == 0) {
            memcpy(W1c, W1, n * sizeof(double));
            memcpy(W2c, W2, n * sizeof(double));
        }
        oracle_mlp_grad(d, hid, W1c, W2c, kt, vt, g1, g2);
        for (size_t x = 0; x < n; ++x) {
            S1[x] = et * S1[x] - th * g1[x];
            W1[x] = (1.0 - al) * W1[x] + S1[x];
            S2[x] = et * S2[x] - th * g2[x];
            W2[x] = (1.0 - al) * W2[x] + S2[x];
        }
        mlp_apply(d, hid, W1, W2, qt, hb, ab, a->z + (seq * T + t) * d);
    }
    memcpy(a->W1_out + seq * n, W1, n * sizeof(double));
    memcpy(a->W2_out + seq * n, W2, n * sizeof(double));
    if (a->S1_out) memcpy(a->S1_out + seq * n, S1, n * sizeof(double));
    if (a->S2_out) memcpy(a->S2_out + seq * n, S2, n * sizeof(double));
    free(W1); free(W2); free(S1); free(S2); free(W1c); free(W2c);
    free(g1); free(g2); free(hb); free(ab);
}

/* ------------------------------------------------------------------ */
/* gradient of the linear / Titans memory (reverse mode)              */
/* ------------------------------------------------------------------ */

typedef struct {
    int B, H, T, dk, dv, chunk;
    const double *q, *k, *v, *eta, *theta, *alpha, *W0, *S0;
    int shared;
    const double *dz, *dWT, *dST;              /* adjoints of the outputs (dWT, dST may be NULL) */
    double *dq, *dk_, *dv_, *deta, *dtheta, *dalpha; /* deta / dalpha NULL when the gate is */
    double *dW0, *dS0;                          /* [B][H][dv][dk], per sequence */
} lin_bwd_args;

/* one token of the forward loop, from (W, S) = state before token t and the
   chunk snapshot Wc; leaves the state after the token in (W, S) */
static void lin_token(int dk, int dv, const double* Wc, double* W, double* S, const double* kt,
                      const double* vt, double th, double et, double al, double* e) {
    for (int i = 0; i < dv; ++i) {
        double acc = 0.0;
        for (int j = 0; j < dk; ++j) acc += Wc[(size_t)i * dk + j] * kt[j];
        e[i] = acc - vt[i];
    }
    for (int i = 0; i < dv; ++i)
        for (int j = 0; j < dk; ++j) {
            const size_t ij = (size_t)i * dk + j;
            S[ij] = et * S[ij] - th * 2.0 * e[i] * kt[j];
            W[ij] = (1.0 - al) * W[ij] + S[ij];
        }
}

static void lin_bwd_one(const lin_bwd_args* a, int b, int h) {
    const int T = a->T, dk = a->dk, dv = a->dv, bc = a->chunk;
    const size_t seq = (size_t)b * a->H + h;
    const size_t init = (size_t)(a->shared ? 0 : b) * a->H + h;
    const size_t ns = (size_t)dv * dk, nsb = ns * sizeof(double);
    const int nchunks = (T + bc - 1) / bc;

    /* forward once, keeping the state at every chunk start */
    double* Wck = (double*)malloc((size_t)(nchunks + 1) * nsb);
    double* Sck = (double*)malloc((size_t)(nchunks + 1) * nsb);
    double* W = (double*)malloc(nsb);
    double* S = (double*)malloc(nsb);
    double* e = (double*)malloc((size_t)dv * sizeof(double));
    memcpy(W, a->W0 + init * ns, nsb);
    if (a->S0) memcpy(S, a->S0 + init * ns, nsb);
    else memset(S, 0, nsb);
    for (int c = 0; c < nchunks; ++c) {
        memcpy(Wck + (size_t)c * ns, W, nsb);
        memcpy(Sck + (size_t)c * ns, S, nsb);
        for (int t = c * bc; t < T && t < (c + 1) * bc; ++t) {
            const size_t ti = seq * T + t;
            lin_token(dk, dv, Wck + (size_t)c * ns, W, S, a->k + ti * dk, a->v + ti * dv,
                      a->theta[ti], a->eta ? a->eta[ti] : 0.0, a->alpha ? a->alpha[ti] : 0.0, e);
        }
    }

    /* adjoints of the current state and of the current chunk's snapshot */
    double* dW = (double*)calloc(ns, sizeof(double));
    double* dS = (double*)calloc(ns, sizeof(double));
    double* dWc = (double*)calloc(ns, sizeof(double));
    double* dSt = (double*)malloc(nsb);
    double* de = (double*)malloc((size_t)dv * sizeof(double));
    if (a->dWT) memcpy(dW, a->dWT + seq * ns, nsb);
    if (a->dST) memcpy(dS, a->dST + seq * ns, nsb);
    /* per-token states of one chunk: Wh[u] / Sh[u] = state before its token u, Wh[n] after the last */
    double* Wh = (double*)malloc((size_t)(bc + 1) * nsb);
    double* Sh = (double*)malloc((size_t)(bc + 1) * nsb);

    for (int c = nchunks - 1; c >= 0; --c) {
        const int t0 = c * bc, n = (T - t0 < bc) ? T - t0 : bc;
        const double* Wc = Wck + (size_t)c * ns;
        memcpy(Wh, Wc, nsb);
        memcpy(Sh, Sck + (size_t)c * ns, nsb);
        for (int u = 0; u < n; ++u) {
            const size_t ti = seq * T + t0 + u;
            memcpy(Wh + (size_t)(u + 1) * ns, Wh + (size_t)u * ns, nsb);
            memcpy(Sh + (size_t)(u + 1) * ns, Sh + (size_t)u * ns, nsb);
            lin_token(dk, dv, Wc, Wh + (size_t)(u + 1) * ns, Sh + (size_t)(u + 1) * ns,
                      a->k + ti * dk, a->v + ti * dv, a->theta[ti], a->eta ? a->eta[ti] : 0.0,
                      a->alpha ? a->alpha[ti] : 0.0, e);
        }
        for (int u = n - 1; u >= 0; --u) {
            const size_t ti = seq * T + t0 + u;
            const double* kt = a->k + ti * dk;
            const double* qt = a->q + ti * dk;
            const double* vt = a->v + ti * dv;
            const double* dzt = a->dz + ti * dv;
            const double th = a->theta[ti];
            const double et = a->eta ? a->eta[ti] : 0.0;
            const double al = a->alpha ? a->alpha[ti] : 0.0;
            const double* Wprev = Wh + (size_t)u * ns;   /* W_{t-1} */
            const double* Sprev = Sh + (size_t)u * ns;   /* S_{t-1} */
            const double* Wnow = Wh + (size_t)(u + 1) * ns; /* W_t */
            double* dqt = a->dq + ti * dk;
            double* dkt = a->dk_ + ti * dk;
            double* dvt = a->dv_ + ti * dv;

            /* read z_t = W_t q_t */
            for (int j = 0; j < dk; ++j) {
                double acc = 0.0;
                for (int i = 0; i < dv; ++i) acc += Wnow[(size_t)i * dk + j] * dzt[i];
                dqt[j] = acc;
            }
            for (int i = 0; i < dv; ++i)
                for (int j = 0; j < dk; ++j) dW[(size_t)i * dk + j] += dzt[i] * qt[j];

            /* forgetting W_t = (1 - alpha_t) W_{t-1} + S_t */
            double dal = 0.0;
            for (size_t ij = 0; ij < ns; ++ij) {
                dal -= dW[ij] * Wprev[ij];
                dSt[ij] = dS[ij] + dW[ij];   /* S_t feeds W_t and S_{t+1} */
                dW[ij] *= (1.0 - al);        /* now the adjoint of W_{t-1} */
            }
            if (a->dalpha) a->dalpha[ti] = dal;

            /* error at the snapshot, e = Wc k_t - v_t (recomputed) */
            for (int i = 0; i < dv; ++i) {
                double acc = 0.0;
                for (int j = 0; j < dk; ++j) acc += Wc[(size_t)i * dk + j] * kt[j];
                e[i] = acc - vt[i];
            }
            /* momentum S_t = eta_t S_{t-1} - theta_t g_t, g_t = 2 e k_t^T */
            double det = 0.0, dth = 0.0;
            for (int i = 0; i < dv; ++i) de[i] = 0.0;
            for (int j = 0; j < dk; ++j) dkt[j] = 0.0;
            for (int i = 0; i < dv; ++i)
                for (int j = 0; j < dk; ++j) {
                    const size_t ij = (size_t)i * dk + j;
                    det += dSt[ij] * Sprev[ij];
                    dth -= dSt[ij] * 2.0 * e[i] * kt[j];
                    const double dg = -th * dSt[ij];  /* adjoint of g_t[i][j] */
                    de[i] += 2.0 * dg * kt[j];
                    dkt[j] += 2.0 * dg * e[i];
                    dS[ij] = et * dSt[ij];            /* adjoint of S_{t-1} */
                }
            if (a->deta) a->deta[ti] = det;
            a->dtheta[ti] = dth;

            /* e = Wc k_t - v_t */
            for (int i = 0; i < dv; ++i) {
                dvt[i] = -de[i];
                for (int j = 0; j < dk; ++j) {
                    dWc[(size_t)i * dk + j] += de[i] * kt[j];
                    dkt[j] += Wc[(size_t)i * dk + j] * de[i];
                }
            }
        }
        /* the chunk's first token took its snapshot: Wc = W before it */
        for (size_t ij = 0; ij < ns; ++ij) {
            dW[ij] += dWc[ij];
            dWc[ij] = 0.0;
        }
    }
    memcpy(a->dW0 + seq * ns, dW, nsb);
    if (a->dS0) memcpy(a->dS0 + seq * ns, dS, nsb);
    free(Wck); free(Sck); free(W); free(S); free(e); free(dW); free(dS); free(dWc); free(dSt);
    free(de); free(Wh); free(Sh);
}

/* ------------------------------------------------------------------ */
/* DGD memory                                                         */
/* ------------------------------------------------------------------ */

typedef struct {
    int B, H, T, dk, dv, chunk;
    const double *q, *k, *v, *eta, *alpha, *W0;
    int shared;
    double *z, *W_out;
} dgd_args;

static void dgd_one(const dgd_args* a, int b, int h) {
    const int T = a->T, dk = a->dk, dv = a->dv;
    const size_t seq = (size_t)b * a->H + h;
    const size_t init = (size_t)(a->shared ? 0 : b) * a->H + h;
    const size_t ns = (size_t)dv * dk;
    double* M = (double*)malloc(ns * sizeof(double));
    double* Mc = (double*)malloc(ns * sizeof(double));
    double* u = (double*)malloc((size_t)dv * sizeof(double));
    double* e = (double*)malloc((size_t)dv * sizeof(double));
    memcpy(M, a->W0 + init * ns, ns * sizeof(double));
    for (int t = 0; t < T; ++t) {
        const double* kt = a->k + (seq * T + t) * dk;
        const double* qt = a->q + (seq * T + t) * dk;
        const double* vt = a->v + (seq * T + t) * dv;
        const double et = a->eta[seq * T + t];
        const double al = a->alpha[seq * T + t];
        if (t % a->chunk == 0) memcpy(Mc, M, ns * sizeof(double));
        /* read before the write: y_t = M_{t-1} q_t (eq (86)) */
        double* zt = a->z + (seq * T + t) * dv;
        for (int i = 0; i < dv; ++i) {
            double acc = 0.0;
            for (int j = 0; j < dk; ++j) acc += M[(size_t)i * dk + j] * qt[j];
            zt[i] = acc;
        }
        /* u = M_{t-1} k_t (the k k^T term) and e = Mc k_t - v_t (the gradient) */
        for (int i = 0; i < dv; ++i) {
            double mu = 0.0, mc = 0.0;
            for (int j = 0; j < dk; ++j) {
                mu += M[(size_t)i * dk + j] * kt[j];
                mc += Mc[(size_t)i * dk + j] * kt[j];
            }
            u[i] = mu;
            e[i] = mc - vt[i];
        }
        /* M (alpha I - eta k k^T) - eta e k^T */
        for (int i = 0; i < dv; ++i)
            for (int j = 0; j < dk; ++j) {
                const size_t ij = (size_t)i * dk + j;
                M[ij] = al * M[ij] - et * u[i] * kt[j] - et * e[i] * kt[j];
            }
    }
    memcpy(a->W_out + seq * ns, M, ns * sizeof(double));
    free(M); free(Mc); free(u); free(e);
}

/* ------------------------------------------------------------------ */
/* thread pool over the independent (b, h) sequences                  */
/* ------------------------------------------------------------------ */

typedef struct {
    int kind; /* 0 linear, 1 mlp, 2 linear gradient, 3 DGD */
    const void* args;
    int units, next;
    pthread_mutex_t lock;
} pool_t;

static void* worker(void* p) {
    pool_t* pool = (pool_t*)p;
    for (;;) {
        pthread_mutex_lock(&pool->lock);
        const int u = pool->next++;
        pthread_mutex_unlock(&pool->lock);
        if (u >= pool->units) break;
        if (pool->kind == 0) {
            const lin_args* a = (const lin_args*)pool->args;
            lin_one(a, u / a->H, u % a->H);
        } else if (pool->kind == 1) {
            const mlp_args* a = (const mlp_args*)pool->args;
            mlp_one(a, u / a->H, u % a->H);
        } else if (pool->kind == 2) {
            const lin_bwd_args* a = (const lin_bwd_args*)pool->args;
            lin_bwd_one(a, u / a->H, u % a->H);
        } else {
            const dgd_args* a = (const dgd_args*)pool->args;
            dgd_one(a, u / a->H, u % a->H);
        }
    }
    return NULL;
}

/* Runs the sequences on nthreads threads (0: every online core).
   Returns the number of threads actually used. */
static int run_pool(int kind, const void* args, int units, int nthreads) {
    if (nthreads <= 0) nthreads = (int)sysconf(_SC_NPROCESSORS_ONLN);
    if (nthreads < 1) nthreads = 1;
    if (nthreads > units) nthreads = units;
    pool_t pool;
    pool.kind = kind; pool.args = args; pool.units = units; pool.next = 0;
    pthread_mutex_init(&pool.lock, NULL);
    pthread_t* th = (pthread_t*)malloc((size_t)nthreads * sizeof(pthread_t));
    for (int i = 0; i < nthreads; ++i) pthread_create(&th[i], NULL, worker, &pool);
    for (int i = 0; i < nthreads; ++i) pthread_join(th[i], NULL);
    free(th);
    pthread_mutex_destroy(&pool.lock);
    return nthreads;
}

int oracle_linear_primal(int B, int H, int T, int dk, int dv, int chunk,
                         const double* q, const double* k, const double* v,
                         const double* eta, const double* theta, const double* alpha,
                         const double* W0, const double* S0, int shared_over_batch,
                         double* z, double* W_out, double* S_out, int nthreads) {
    if (B < 1 || H < 1 || T < 0 || dk < 1 || dv < 1 || chunk < 1) return -1;
    lin_args a = {B, H, T, dk, dv, chunk, q, k, v, eta, theta, alpha, W0, S0,
                  shared_over_batch, z, W_out, S_out};
    return run_pool(0, &a, B * H, nthreads);
}

int oracle_mlp_primal(int B, int H, int T, int d, int hidden, int chunk,
                      const double* q, const double* k, const double* v,
                      const double* eta, const double* theta, const double* alpha,
                      const double* W1_0, const double* W2_0, const double* S1_0,
                      const double* S2_0, int shared_over_batch,
                      double* z, double* W1_out, double* W2_out, double* S1_out,
                      double* S2_out, int nthreads) {
    if (B < 1 || H < 1 || T < 0 || d < 1 || hidden < 1 || chunk < 1) return -1;
    mlp_args a = {B, H, T, d, hidden, chunk, q, k, v, eta, theta, alpha, W1_0, W2_0,
                  S1_0, S2_0, shared_over_batch, z, W1_out, W2_out, S1_out, S2_out};
    return run_pool(1, &a, B * H, nthreads);
}

/* Gradient of the linear / Titans scan.  dz [B][H][T][dv]; dWT, dST
   [B][H][dv][dk] or NULL (= 0).  Outputs dq, dk [B][H][T][dk], dv [B][H][T][dv],
   deta, dtheta, dalpha [B][H][T] (deta / dalpha may be NULL and must be when
   eta / alpha are), dW0 and dS0 [B][H][dv][dk] per sequence (the caller sums
   over the batch when W0 is shared; dS0 may be NULL). */
int oracle_linear_primal_bwd(int B, int H, int T, int dk, int dv, int chunk,
                             const double* q, const double* k, const double* v,
                             const double* eta, const double* theta, const double* alpha,
                             const double* W0, const double* S0, int shared_over_batch,
                             const double* dz, const double* dWT, const double* dST,
                             double* dq, double* dk_, double* dv_, double* deta, double* dtheta,
                             double* dalpha, double* dW0, double* dS0, int nthreads) {
    if (B < 1 || H < 1 || T < 0 || dk < 1 || dv < 1 || chunk < 1) return -1;
    if ((deta && !eta) || (dalpha && !alpha)) return -1;
    lin_bwd_args a = {B, H, T, dk, dv, chunk, q, k, v, eta, theta, alpha, W0, S0,
                      shared_over_batch, dz, dWT, dST, dq, dk_, dv_, deta, dtheta, dalpha,
                      dW0, dS0};
    return run_pool(2, &a, B * H, nthreads);
}

/* DGD memory scan (see the header).  q, k [B][H][T][dk], v [B][H][T][dv],
   eta (step) and alpha (retention) [B][H][T], W0 [B or 1][H][dv][dk];
   z [B][H][T][dv] and W_out [B][H][dv][dk] written. */
int oracle_dgd_primal(int B, int H, int T, int dk, int dv, int chunk, const double* q,
                      const double* k, const double* v, const double* eta, const double* alpha,
                      const double* W0, int shared_over_batch, double* z, double* W_out,
                      int nthreads) {
    if (B < 1 || H < 1 || T < 0 || dk < 1 || dv < 1 || chunk < 1 || !eta || !alpha) return -1;
    dgd_args a = {B, H, T, dk, dv, chunk, q, k, v, eta, alpha, W0, shared_over_batch, z, W_out};
    return run_pool(3, &a, B * H, nthreads);
}
