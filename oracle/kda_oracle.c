/*
 * kda_oracle.c -- plain fp64 CPU oracle for the Kimi Delta Attention (KDA)
 * forward pass.  TEST INFRASTRUCTURE ONLY: nothing in the product path may
 * link, load or call this file.  Only the tests, the smoke check and the
 * CPU-baseline leg of the benchmark use it.  It shares no code, header,
 * table or constant with the CUDA library.
 *
 * Sources (web pages, cited by title and section):
 *   [lshu]   "Kimi K3" article, lshu.cn/news/263999
 *              §二.1  linear memory: S_t in R^{dk x dv}; read o_t = S_t^T q_t
 *              §三    delta rule: predict v^_t = S_{t-1}^T k_t, error
 *                     e_t = v_t - v^_t, write S_t = S_{t-1} + beta_t k_t e_t^T,
 *                     i.e. S_t = (I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T
 *              §四    KDA: S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1}
 *                                + beta_t k_t v_t^T,  alpha_t in [0,1]^{dk}
 *              §六    chunking ([1,C], [C+1,2C], ...; recurrent between
 *                     chunks, parallel inside) and the WY form P = D - K W^T
 *   [hubwiz] "Kimi K3 混合线性注意力", §3: state of 128 x 128 per head,
 *              independent of the sequence length; §5: state snapshots.
 *
 * Readings taken where the pages are silent or garbled (page 3 lost its
 * '=' and '+' signs in extraction):
 *   - operator order: the decay Diag(alpha_t) acts first, the delta-rule
 *     prediction reads the decayed state (the §四 operator order);
 *   - the read o_t = S_t^T q_t happens after token t's update (§二.1);
 *   - no 1/sqrt(d) scale and no normalisation inside the operator;
 *   - alpha_t = exp(log_alpha_t), log_alpha given per key channel.
 *
 * Parity: every function here is pinned by tests/test_oracle_pins.py
 * (special cases with closed forms, the pages' overwrite example, brute
 * force matrix products on tiny inputs, and recurrent == chunked).
 *
 * bf16-stored state ("Kimi K3 混合线性注意力", §3 sizes the state in bf16): the
 * variant kda_oracle_recurrent_bf16state keeps every step's arithmetic in fp64
 * but rounds the state to bf16 (round to nearest, ties to even) after each
 * token's update and read, as a decode step that stores its state in bf16
 * does.  kda_oracle_round_bf16 exposes that rounding.
 *
 * Backward (reverse mode of the same per-token recurrence; the pages give none, so it
 * is derived here step by step from the forward definition above):
 * kda_oracle_recurrent_bwd takes the loss L = sum_t <do_t, o_t> + <dS_T, S_T> and
 * returns dL/dq, dL/dk, dL/dv, dL/dlog_alpha, dL/dbeta and dL/dS0.  It stores every
 * state of the forward sweep and walks the tokens backwards, undoing one operation
 * of the step at a time (read, rank-one write, error, prediction, decay).
 *
 * Layouts (all contiguous, head-major; "n" = independent heads):
 *   q, k, log_alpha : [n][T][dk]  double  (bf16 / fp32 inputs upcast exactly)
 *   v               : [n][T][dv]  double
 *   beta            : [n][T]      double
 *   S0              : [n][dk][dv] double  (NULL = zero state)
 *   out             : [n][T][dv]  double
 *   S_final         : [n][dk][dv] double
 *   snaps           : [n][T / interval][dk][dv] double (state after token
 *                     m*interval, m = 1..T/interval), or NULL
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#if defined(ORACLE_MUTANT)
/* Planted mistakes, compiled only by the mutation test (never by build()). */
#define MUT(n) (ORACLE_MUTANT == (n))
#else
#define MUT(n) 0
#endif

typedef struct {
    int64_t n, T;
    int dk, dv, C;
    const double *q, *k, *v, *la, *beta;
    const double* S0;
    double *out, *S_final;
    int64_t interval;
    double* snaps;
    int colblk; /* value columns per work unit */
    int state_bf16; /* round the state to bf16 after every token */
    /* backward: cotangents in, gradients out ([n][T][..] like the inputs) */
    const double *dout, *dSf;
    double *g_q, *g_k, *g_v, *g_la, *g_beta, *g_S0;
    int bwd;
    int64_t n_units;
    int64_t next; /* shared unit counter, guarded by mu */
    pthread_mutex_t mu;
    int err;
} job_t;

/* Nearest bf16 value (8 significant bits, fp32's exponent range), ties to even. */
static double round_bf16(double x) {
    if (x == 0.0 || !isfinite(x)) return x;
    int e;
    frexp(x, &e); /* |x| in [2^(e-1), 2^e) */
    if (e < -125) e = -125; /* below 2^-126 the spacing stays 2^-133 (subnormals) */
    const double quantum = ldexp(1.0, e - 8);
    const double y = nearbyint(x / quantum) * quantum; /* default rounding: to nearest, ties to even */
    if (fabs(y) > 3.3895313892515355e38) return copysign(INFINITY, x); /* beyond the largest bf16 */
    return y;
}

static int64_t grab_unit(job_t* J) {
    pthread_mutex_lock(&J->mu);
    int64_t u = J->next++;
    pthread_mutex_unlock(&J->mu);
    return u < J->n_units ? u : -1;
}

/* ------------------------------------------------------------------------
 * Per-token recurrence for one head h and value columns [j0, j0+nj).
 * The columns of S evolve independently (column j only ever meets v[:, j]),
 * so splitting them across threads is exact.
 * ---------------------------------------------------------------------- */
static void recurrent_unit(job_t* J, int64_t h, int j0, int nj) {
    const int dk = J->dk, dv = J->dv;
    const int64_t T = J->T;
    double* S = (double*)malloc(sizeof(double) * (size_t)dk * nj); /* S[i][j] */
    double* p = (double*)malloc(sizeof(double) * nj);
    double* u = (double*)malloc(sizeof(double) * nj);
    double* o = (double*)malloc(sizeof(double) * nj);
    if (!S || !p || !u || !o) { J->err = 1; free(S); free(p); free(u); free(o); return; }

    for (int i = 0; i < dk; ++i)
        for (int j = 0; j < nj; ++j)
            S[(size_t)i * nj + j] = J->S0 ? J->S0[((size_t)h * dk + i) * dv + j0 + j] : 0.0;

    for (int64_t t = 0; t < T; ++t) {
        const double* qt = J->q + ((size_t)h * T + t) * dk;
        const double* kt = J->k + ((size_t)h * T + t) * dk;
        const double* vt = J->v + ((size_t)h * T + t) * dv + j0;
        const double* lat = J->la + ((size_t)h * T + t) * dk;
        const double bt = (double)J->beta[(size_t)h * T + t];

        /* Diag(alpha_t) S_{t-1}, then the prediction p = S'^T k_t (§四, §三). */
        for (int j = 0; j < nj; ++j) p[j] = 0.0;
        for (int i = 0; i < dk; ++i) {
            const double a = MUT(1) ? 1.0 : exp((double)lat[i]);
            const double ki = (double)kt[i];
            double* Si = S + (size_t)i * nj;
            for (int j = 0; j < nj; ++j) {
                if (!MUT(2)) Si[j] *= a;
                p[j] += ki * Si[j];
            }
            if (MUT(2))
                for (int j = 0; j < nj; ++j) Si[j] *= a; /* predicts from the undecayed state */
        }
        /* e_t = v_t - p;  write beta_t k_t e_t^T  (§三). */
        for (int j = 0; j < nj; ++j) u[j] = bt * ((double)vt[j] - (MUT(3) ? -p[j] : p[j]));
        /* S_t = S' + k_t u^T, then o_t = S_t^T q_t (§二.1). */
        for (int j = 0; j < nj; ++j) o[j] = 0.0;
        for (int i = 0; i < dk; ++i) {
            const double ki = (double)kt[i];
            const double qi = (double)(MUT(4) ? kt[i] : qt[i]);
            double* Si = S + (size_t)i * nj;
            for (int j = 0; j < nj; ++j) {
                if (MUT(5)) o[j] += qi * Si[j]; /* reads before the write */
                Si[j] += ki * u[j];
                if (!MUT(5)) o[j] += qi * Si[j];
            }
        }
        double* ot = J->out + ((size_t)h * T + t) * dv + j0;
        for (int j = 0; j < nj; ++j) ot[j] = o[j];
        if (J->state_bf16) /* the state is stored in bf16 between tokens */
            for (size_t i = 0; i < (size_t)dk * nj; ++i) S[i] = round_bf16(S[i]);

        if (J->snaps && J->interval > 0 && (t + 1) % J->interval == 0) {
            const int64_t m = (t + 1) / J->interval - 1;
            const int64_t nsnap = T / J->interval;
            double* dst = J->snaps + (((size_t)h * nsnap + m) * dk) * dv;
            for (int i = 0; i < dk; ++i)
                for (int j = 0; j < nj; ++j) dst[(size_t)i * dv + j0 + j] = S[(size_t)i * nj + j];
        }
    }
    if (J->S_final)
        for (int i = 0; i < dk; ++i)
            for (int j = 0; j < nj; ++j)
                J->S_final[((size_t)h * dk + i) * dv + j0 + j] = S[(size_t)i * nj + j];
    free(S); free(p); free(u); free(o);
}

/* ------------------------------------------------------------------------
 * Naive chunked rewrite (§六).  For one chunk of C rows starting from
 * state S0, with g_r = sum_{s<=r} log alpha_s (per key channel):
 *   A[r][i]  = beta_r sum_c k_r[c] k_i[c] exp(g_r[c] - g_i[c])    (i < r)
 *   Tinv     = (I + A)^{-1}                         (unit lower triangular)
 *   W        = Tinv diag(beta) Ktil,   Ktil[r][c] = k_r[c] exp(g_r[c])
 *   U'       = Tinv diag(beta) V
 *   U        = U' - W S0
 *   O        = Qtil S0 + lower_incl(Qtil Khat^T) U,  with Qtil = q exp(g),
 *              (Qtil Khat^T)[r][i] = sum_c q_r[c] k_i[c] exp(g_r[c] - g_i[c])
 *   S_C      = P S0 + Kend^T U',  P = D - Kend^T W,  D = Diag(exp(g_C)),
 *              Kend[r][c] = k_r[c] exp(g_C[c] - g_r[c])
 * This is the pages' "P = D - K W^T" transition; it is derived from the
 * §四 recurrence by unrolling it over the chunk.  All pairwise decays are
 * taken directly in fp64 (never as a ratio), so nothing overflows.
 * One work unit = one whole head (the chunked form mixes all columns).
 * ---------------------------------------------------------------------- */
static void chunked_head(job_t* J, int64_t h) {
    const int dk = J->dk, dv = J->dv, C = J->C;
    const int64_t T = J->T;
    size_t sz_S = (size_t)dk * dv;
    double* S = (double*)calloc(sz_S, sizeof(double));
    double* g = (double*)malloc(sizeof(double) * (size_t)C * dk);
    double* A = (double*)malloc(sizeof(double) * (size_t)C * C);
    double* Tinv = (double*)malloc(sizeof(double) * (size_t)C * C);
    double* QK = (double*)malloc(sizeof(double) * (size_t)C * C);
    double* W = (double*)malloc(sizeof(double) * (size_t)C * dk);
    double* Up = (double*)malloc(sizeof(double) * (size_t)C * dv);
    double* U = (double*)malloc(sizeof(double) * (size_t)C * dv);
    double* Ke = (double*)malloc(sizeof(double) * (size_t)C * dk);
    double* P = (double*)malloc(sizeof(double) * (size_t)dk * dk);
    double* Sn = (double*)malloc(sizeof(double) * sz_S);
    if (!S || !g || !A || !Tinv || !QK || !W || !Up || !U || !Ke || !P || !Sn) {
        J->err = 1;
        goto done;
    }
    if (J->S0) memcpy(S, J->S0 + (size_t)h * sz_S, sizeof(double) * sz_S);

    for (int64_t t0 = 0; t0 < T; t0 += C) {
        const int n = (int)((T - t0) < C ? (T - t0) : C); /* ragged last chunk */
        const double* q = J->q + ((size_t)h * T + t0) * dk;
        const double* k = J->k + ((size_t)h * T + t0) * dk;
        const double* v = J->v + ((size_t)h * T + t0) * dv;
        const double* la = J->la + ((size_t)h * T + t0) * dk;
        const double* be = J->beta + (size_t)h * T + t0;

        /* cumulative log decay per channel */
        for (int c = 0; c < dk; ++c) {
            double s = 0.0;
            for (int r = 0; r < n; ++r) {
                s += (double)la[(size_t)r * dk + c];
                g[(size_t)r * dk + c] = s;
            }
        }
        /* A (strictly lower) and Qtil Khat^T (lower incl. diagonal) */
        for (int r = 0; r < n; ++r)
            for (int i = 0; i < n; ++i) {
                double a = 0.0, b = 0.0;
                if (i <= r)
                    for (int c = 0; c < dk; ++c) {
                        const double dec = exp(g[(size_t)r * dk + c] - g[(size_t)i * dk + c]);
                        a += (double)k[(size_t)r * dk + c] * (double)k[(size_t)i * dk + c] * dec;
                        b += (double)q[(size_t)r * dk + c] * (double)k[(size_t)i * dk + c] * dec;
                    }
                A[(size_t)r * n + i] = (i < r) ? (double)be[r] * a : 0.0;
                QK[(size_t)r * n + i] = (i <= r) ? b : 0.0;
            }
        /* Tinv = (I + A)^{-1} by forward substitution, one column at a time */
        for (int j = 0; j < n; ++j)
            for (int r = 0; r < n; ++r) {
                double x = (r == j) ? 1.0 : 0.0;
                for (int i = 0; i < r; ++i) x -= A[(size_t)r * n + i] * Tinv[(size_t)i * n + j];
                Tinv[(size_t)r * n + j] = x;
            }
        /* W = Tinv diag(beta) Ktil,  U' = Tinv diag(beta) V,  Kend */
        for (int r = 0; r < n; ++r) {
            for (int c = 0; c < dk; ++c) {
                double w = 0.0;
                for (int i = 0; i <= r; ++i)
                    w += Tinv[(size_t)r * n + i] * (double)be[i] * (double)k[(size_t)i * dk + c] *
                         exp(g[(size_t)i * dk + c]);
                W[(size_t)r * dk + c] = w;
                Ke[(size_t)r * dk + c] =
                    (double)k[(size_t)r * dk + c] * exp(g[(size_t)(n - 1) * dk + c] - g[(size_t)r * dk + c]);
            }
            for (int j = 0; j < dv; ++j) {
                double w = 0.0;
                for (int i = 0; i <= r; ++i)
                    w += Tinv[(size_t)r * n + i] * (double)be[i] * (double)v[(size_t)i * dv + j];
                Up[(size_t)r * dv + j] = w;
            }
        }
        /* U = U' - W S0 */
        for (int r = 0; r < n; ++r)
            for (int j = 0; j < dv; ++j) {
                double s = Up[(size_t)r * dv + j];
                for (int c = 0; c < dk; ++c) s -= W[(size_t)r * dk + c] * S[(size_t)c * dv + j];
                U[(size_t)r * dv + j] = s;
            }
        /* O = Qtil S0 + lower_incl(Qtil Khat^T) U */
        for (int r = 0; r < n; ++r) {
            double* o = J->out + ((size_t)h * T + t0 + r) * dv;
            for (int j = 0; j < dv; ++j) {
                double s = 0.0;
                for (int c = 0; c < dk; ++c)
                    s += (double)q[(size_t)r * dk + c] * exp(g[(size_t)r * dk + c]) * S[(size_t)c * dv + j];
                for (int i = 0; i <= r; ++i) s += QK[(size_t)r * n + i] * U[(size_t)i * dv + j];
                o[j] = s;
            }
        }
        /* P = D - Kend^T W;  S_C = P S0 + Kend^T U' */
        for (int a = 0; a < dk; ++a)
            for (int c = 0; c < dk; ++c) {
                double s = (a == c) ? exp(g[(size_t)(n - 1) * dk + a]) : 0.0;
                for (int r = 0; r < n; ++r) s -= Ke[(size_t)r * dk + a] * W[(size_t)r * dk + c];
                P[(size_t)a * dk + c] = s;
            }
        for (int a = 0; a < dk; ++a)
            for (int j = 0; j < dv; ++j) {
                double s = 0.0;
                for (int c = 0; c < dk; ++c) s += P[(size_t)a * dk + c] * S[(size_t)c * dv + j];
                for (int r = 0; r < n; ++r) s += Ke[(size_t)r * dk + a] * Up[(size_t)r * dv + j];
                Sn[(size_t)a * dv + j] = s;
            }
        memcpy(S, Sn, sizeof(double) * sz_S);

        if (J->snaps && J->interval > 0 && (t0 + n) % J->interval == 0) {
            const int64_t m = (t0 + n) / J->interval - 1;
            const int64_t nsnap = T / J->interval;
            memcpy(J->snaps + ((size_t)h * nsnap + m) * sz_S, S, sizeof(double) * sz_S);
        }
    }
    if (J->S_final) memcpy(J->S_final + (size_t)h * sz_S, S, sizeof(double) * sz_S);
done:
    free(S); free(g); free(A); free(Tinv); free(QK); free(W); free(Up); free(U); free(Ke); free(P); free(Sn);
}

/* ------------------------------------------------------------------------
 * Reverse mode of the per-token recurrence for head h.  Forward step t, from
 * S = S_{t-1}:
 *     a = exp(log_alpha_t)       S' = Diag(a) S        p = S'^T k
 *     e = v - p                  u = beta e            S_t = S' + k u^T
 *     o_t = S_t^T q
 * Backward step t, with dS = dL/dS_t (from the later tokens) and do = dL/do_t:
 *     o_t = S_t^T q        ->  dS += q do^T,            dq = S_t do
 *     S_t = S' + k u^T     ->  dS' = dS,  dk = dS u,     du = dS^T k
 *     u = beta e           ->  dbeta = du . e,           de = beta du
 *     e = v - p            ->  dv = de,                  dp = -de
 *     p = S'^T k           ->  dS' += k dp^T,            dk += S' dp
 *     S' = Diag(a) S       ->  dS_{t-1} = Diag(a) dS',   dlog_alpha_i = a_i sum_j dS'_ij S_ij
 * ---------------------------------------------------------------------- */
static void backward_head(job_t* J, int64_t h) {
    const int dk = J->dk, dv = J->dv;
    const int64_t T = J->T;
    const size_t sz_S = (size_t)dk * dv;
    double* St = (double*)malloc(sizeof(double) * sz_S * (size_t)(T > 0 ? T : 1)); /* S_{t-1}, t = 0..T-1 */
    double* S = (double*)malloc(sizeof(double) * sz_S);
    double* Sp = (double*)malloc(sizeof(double) * sz_S);
    double* dS = (double*)malloc(sizeof(double) * sz_S);
    double* dSp = (double*)malloc(sizeof(double) * sz_S);
    double* vec = (double*)malloc(sizeof(double) * (size_t)(3 * dk + 4 * dv));
    if (!St || !S || !Sp || !dS || !dSp || !vec) { J->err = 1; goto done; }
    double *a = vec, *p = a + dk, *e = p + dv, *u = e + dv, *du = u + dv, *gk = du + dv, *da = gk + dk;
    (void)da;

    for (size_t x = 0; x < sz_S; ++x) S[x] = J->S0 ? J->S0[(size_t)h * sz_S + x] : 0.0;
    for (int64_t t = 0; t < T; ++t) { /* forward sweep, keeping S_{t-1} */
        const size_t r = (size_t)h * T + t;
        const double* kt = J->k + r * dk;
        memcpy(St + (size_t)t * sz_S, S, sizeof(double) * sz_S);
        for (int i = 0; i < dk; ++i) a[i] = exp(J->la[r * dk + i]);
        for (int j = 0; j < dv; ++j) p[j] = 0.0;
        for (int i = 0; i < dk; ++i)
            for (int j = 0; j < dv; ++j) {
                S[(size_t)i * dv + j] *= a[i];
                p[j] += kt[i] * S[(size_t)i * dv + j];
            }
        for (int j = 0; j < dv; ++j) u[j] = J->beta[r] * (J->v[r * dv + j] - p[j]);
        for (int i = 0; i < dk; ++i)
            for (int j = 0; j < dv; ++j) S[(size_t)i * dv + j] += kt[i] * u[j];
    }

    for (size_t x = 0; x < sz_S; ++x) dS[x] = J->dSf ? J->dSf[(size_t)h * sz_S + x] : 0.0;
    for (int64_t t = T - 1; t >= 0; --t) {
        const size_t r = (size_t)h * T + t;
        const double *qt = J->q + r * dk, *kt = J->k + r * dk, *vt = J->v + r * dv, *dot = J->dout + r * dv;
        const double bt = J->beta[r];
        const double* Sprev = St + (size_t)t * sz_S;
        /* recompute the step */
        for (int i = 0; i < dk; ++i) a[i] = exp(J->la[r * dk + i]);
        for (int j = 0; j < dv; ++j) p[j] = 0.0;
        for (int i = 0; i < dk; ++i)
            for (int j = 0; j < dv; ++j) {
                Sp[(size_t)i * dv + j] = a[i] * Sprev[(size_t)i * dv + j];
                p[j] += kt[i] * Sp[(size_t)i * dv + j];
            }
        for (int j = 0; j < dv; ++j) {
            e[j] = vt[j] - p[j];
            u[j] = bt * e[j];
        }
        /* o_t = S_t^T q: dS += q do^T, dq = S_t do (S_t = S' + k u^T) */
        for (int i = 0; i < dk; ++i) {
            double acc = 0.0;
            for (int j = 0; j < dv; ++j) {
                dS[(size_t)i * dv + j] += qt[i] * dot[j];
                acc += (Sp[(size_t)i * dv + j] + kt[i] * u[j]) * dot[j];
            }
            J->g_q[r * dk + i] = acc;
        }
        /* S_t = S' + k u^T: dS' = dS, dk = dS u, du = dS^T k */
        for (int j = 0; j < dv; ++j) du[j] = 0.0;
        for (int i = 0; i < dk; ++i) {
            double acc = 0.0;
            for (int j = 0; j < dv; ++j) {
                const double d = dS[(size_t)i * dv + j];
                dSp[(size_t)i * dv + j] = d;
                acc += d * u[j];
                du[j] += d * kt[i];
            }
            gk[i] = acc;
        }
        /* u = beta e, e = v - p */
        double gb = 0.0;
        for (int j = 0; j < dv; ++j) {
            gb += du[j] * e[j];
            J->g_v[r * dv + j] = bt * du[j];
            p[j] = -bt * du[j]; /* p now holds dp */
        }
        J->g_beta[r] = gb;
        /* p = S'^T k: dS' += k dp^T, dk += S' dp */
        for (int i = 0; i < dk; ++i) {
            double acc = 0.0;
            for (int j = 0; j < dv; ++j) {
                dSp[(size_t)i * dv + j] += kt[i] * p[j];
                acc += Sp[(size_t)i * dv + j] * p[j];
            }
            J->g_k[r * dk + i] = MUT(6) ? gk[i] : gk[i] + acc;
        }
        /* S' = Diag(a) S_{t-1} */
        for (int i = 0; i < dk; ++i) {
            double acc = 0.0;
            for (int j = 0; j < dv; ++j) {
                acc += dSp[(size_t)i * dv + j] * Sprev[(size_t)i * dv + j];
                dS[(size_t)i * dv + j] = MUT(7) ? dSp[(size_t)i * dv + j] : a[i] * dSp[(size_t)i * dv + j];
            }
            J->g_la[r * dk + i] = a[i] * acc;
        }
    }
    if (J->g_S0) memcpy(J->g_S0 + (size_t)h * sz_S, dS, sizeof(double) * sz_S);
done:
    free(St); free(S); free(Sp); free(dS); free(dSp); free(vec);
}

static void* worker(void* arg) {
    job_t* J = (job_t*)arg;
    for (int64_t u; (u = grab_unit(J)) >= 0;) {
        if (J->bwd) {
            backward_head(J, u);
        } else if (J->C > 0) {
            chunked_head(J, u);
        } else {
            const int nblk = (J->dv + J->colblk - 1) / J->colblk;
            const int64_t h = u / nblk;
            const int j0 = (int)(u % nblk) * J->colblk;
            const int nj = (J->dv - j0) < J->colblk ? (J->dv - j0) : J->colblk;
            recurrent_unit(J, h, j0, nj);
        }
    }
    return NULL;
}

static int run(job_t* J, int n_threads) {
    if (J->n < 0 || J->T < 0 || J->dk <= 0 || J->dv <= 0) return 1;
    pthread_mutex_init(&J->mu, NULL);
    if (n_threads < 1) n_threads = 1;
    if (n_threads > 1024) n_threads = 1024;
    pthread_t th[1024];
    int started = 0;
    for (int i = 1; i < n_threads; ++i)
        if (pthread_create(&th[started], NULL, worker, J) == 0) ++started;
    worker(J);
    for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
    pthread_mutex_destroy(&J->mu);
    return J->err;
}

/* Per-token fp64 recurrence.  Returns 0 on success. */
int kda_oracle_recurrent(int64_t n, int64_t T, int dk, int dv, const double* q, const double* k,
                         const double* v, const double* log_alpha, const double* beta, const double* S0, double* out,
                         double* S_final, int64_t snap_interval, double* snaps, int n_threads) {
    job_t J;
    memset(&J, 0, sizeof J);
    J.n = n; J.T = T; J.dk = dk; J.dv = dv; J.C = 0;
    J.q = q; J.k = k; J.v = v; J.la = log_alpha; J.beta = beta; J.S0 = S0;
    J.out = out; J.S_final = S_final; J.interval = snap_interval; J.snaps = snaps;
    J.colblk = 16;
    J.n_units = n * (int64_t)((dv + J.colblk - 1) / J.colblk);
    return run(&J, n_threads);
}

/* The same with the state rounded to bf16 after every token (S0 should hold bf16 values). */
int kda_oracle_recurrent_bf16state(int64_t n, int64_t T, int dk, int dv, const double* q, const double* k,
                                   const double* v, const double* log_alpha, const double* beta, const double* S0,
                                   double* out, double* S_final, int n_threads) {
    job_t J;
    memset(&J, 0, sizeof J);
    J.n = n; J.T = T; J.dk = dk; J.dv = dv; J.C = 0;
    J.q = q; J.k = k; J.v = v; J.la = log_alpha; J.beta = beta; J.S0 = S0;
    J.out = out; J.S_final = S_final;
    J.colblk = 16;
    J.state_bf16 = 1;
    J.n_units = n * (int64_t)((dv + J.colblk - 1) / J.colblk);
    return run(&J, n_threads);
}

/* round_bf16 over an array (exposed so that the rounding itself can be checked). */
void kda_oracle_round_bf16(const double* x, double* y, int64_t count) {
    for (int64_t i = 0; i < count; ++i) y[i] = round_bf16(x[i]);
}

/* Naive chunked rewrite in fp64 (chunk length C >= 1). Returns 0 on success. */
int kda_oracle_chunked(int64_t n, int64_t T, int dk, int dv, int C, const double* q, const double* k,
                       const double* v, const double* log_alpha, const double* beta, const double* S0,
                       double* out, double* S_final, int64_t snap_interval, double* snaps, int n_threads) {
    if (C < 1) return 1;
    if (snaps && snap_interval > 0 && snap_interval % C != 0) return 1; /* snapshots sit on chunk ends */
    job_t J;
    memset(&J, 0, sizeof J);
    J.n = n; J.T = T; J.dk = dk; J.dv = dv; J.C = C;
    J.q = q; J.k = k; J.v = v; J.la = log_alpha; J.beta = beta; J.S0 = S0;
    J.out = out; J.S_final = S_final; J.interval = snap_interval; J.snaps = snaps;
    J.n_units = n;
    return run(&J, n_threads);
}

/* Gradients of L = sum_t <dout_t, o_t> + <dS_final, S_T> (dS_final may be NULL) with
 * respect to q, k, v, log_alpha, beta and S0, each in the layout of its input.  Holds
 * T * dk * dv doubles per head in flight.  Returns 0 on success. */
int kda_oracle_recurrent_bwd(int64_t n, int64_t T, int dk, int dv, const double* q, const double* k,
                             const double* v, const double* log_alpha, const double* beta, const double* S0,
                             const double* dout, const double* dS_final, double* dq, double* dk_out, double* dv_out,
                             double* dlog_alpha, double* dbeta, double* dS0, int n_threads) {
    job_t J;
    memset(&J, 0, sizeof J);
    J.n = n; J.T = T; J.dk = dk; J.dv = dv; J.C = 0;
    J.q = q; J.k = k; J.v = v; J.la = log_alpha; J.beta = beta; J.S0 = S0;
    J.dout = dout; J.dSf = dS_final;
    J.g_q = dq; J.g_k = dk_out; J.g_v = dv_out; J.g_la = dlog_alpha; J.g_beta = dbeta; J.g_S0 = dS0;
    J.bwd = 1;
    J.n_units = n;
    if (!dout || !dq || !dk_out || !dv_out || !dlog_alpha || !dbeta) return 1;
    return run(&J, n_threads);
}
