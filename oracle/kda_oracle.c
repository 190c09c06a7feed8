/*
 * kda_oracle.c -- plain FP64 CPU oracle for Kimi Delta Attention (KDA) prefill.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the smoke check and the CPU
 * baseline leg of the benchmark load this file's library. The product path
 * (the CUDA library) never links, calls or shares code with it.
 *
 * Two independent formulations of the same operation live here; they share
 * no helper (each has its own L2 normalisation) so that one can check the
 * other:
 *
 *  1. kda_oracle_token -- the per-token gated delta rule.  For one sequence and
 *     one head, with the state S a dv x dk matrix (rows = value channels,
 *     columns = key channels):
 *         S <- S Diag(alpha_t)                alpha_t = exp(g_t), per key channel
 *         u_t = beta_t (v_t - S khat_t)       delta-rule error
 *         S <- S + u_t khat_t^T
 *         o_t = s S qhat_t
 *     This is the chunkwise system of "FlashKDA column split", section 1
 *     (equations for U_c, O_c, S_{c+1}) taken with one-token chunks: with C=1,
 *     D_{0:0} = Diag(alpha_t), K^end = k^T, A^kk = 1 and A^qk = s <k|q>, so
 *     O = s (S D_0 + U k^T) q, i.e. the output reads the state after the write.
 *     The in-kernel L2 normalisation of q and k follows the flashinfer
 *     kda_prefill page, "Optimized Blackwell prefill subset"
 *     (use_qk_l2norm_in_kernel): xhat = x / sqrt(sum x^2 + eps).
 *
 *  2. kda_oracle_chunk -- the chunkwise form of "FlashKDA column split",
 *     section 1, for any chunk length C:
 *         D_{0:i}  = D_0 ... D_i                        (products of alpha)
 *         K^start  column i = D_{0:i} khat_i ;  Q^start column i = D_{0:i} qhat_i
 *         K^end    row i    = khat_i^T D_{i+1:C-1}
 *         (R)_ij   = beta_i <khat_j| D_{j+1:i} |khat_i>,  j < i
 *         A^kk     = (I + R)^{-1}
 *         (A^qk)_ij = s <khat_j| D_{j+1:i} |qhat_i>,     j <= i
 *         U = (V - S K^start) B (A^kk)^T
 *         O = s S Q^start + U (A^qk)^T
 *         S <- S D_{0:C-1} + U K^end
 *     A^kk is formed either by forward substitution on (I + R) X = I or by
 *     the repeated-squaring Neumann product of "K3's KDA precision problem",
 *     section "Matrix inversion in FlashKDA":
 *         (I + L)^{-1} = (I - L)(I + L^2)(I + L^4)(I + L^8)...   (L nilpotent)
 *
 * Layouts (all row-major, FP64):
 *   q, k, g : [tokens, H, dk]     v, out : [tokens, H, dv]     beta : [tokens, H]
 *   init_state, final_state : [N, H, dv, dk]
 *   Fixed layout (cu_seqlens == NULL): N sequences of T tokens, tokens = N*T.
 *   Packed layout: tokens = T, sequence n is [cu_seqlens[n], cu_seqlens[n+1]).
 * init_state may be NULL (zero state).  Every (sequence, head) is independent.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define KDA_ORACLE_OK 0
#define KDA_ORACLE_EBADARG (-1)
#define KDA_ORACLE_ENOMEM (-2)

int kda_oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

static int seq_bounds(const int64_t* cu, int64_t n, int64_t T, int64_t* start, int64_t* end) {
    if (cu) {
        *start = cu[n];
        *end = cu[n + 1];
    } else {
        *start = n * T;
        *end = n * T + T;
    }
    return *end >= *start;
}

static int check_cu(const int64_t* cu, int64_t N, int64_t T) {
    if (!cu) return 1;
    if (cu[0] != 0 || cu[N] != T) return 0;
    for (int64_t n = 0; n < N; ++n)
        if (cu[n + 1] < cu[n]) return 0;
    return 1;
}

/* ------------------------------------------------------------------------- */
/* 1. Per-token recurrence.                                                   */
/* ------------------------------------------------------------------------- */

/* L2 normalisation used by the token form. */
static void token_l2norm(const double* x, double* y, int64_t d, double eps, int enable) {
    if (!enable) {
        for (int64_t c = 0; c < d; ++c) y[c] = x[c];
        return;
    }
    double ss = 0.0;
    for (int64_t c = 0; c < d; ++c) ss += x[c] * x[c];
    double inv = 1.0 / sqrt(ss + eps);
    for (int64_t c = 0; c < d; ++c) y[c] = x[c] * inv;
}

/*
 * Value rows of one (sequence, head) are independent recurrences that share
 * q, k, g and beta, so the work is split over (sequence, head, block of value
 * rows).  Every row still runs its tokens strictly in order.
 */
int kda_oracle_token(const double* q, const double* k, const double* v, const double* g,
                     const double* beta, const double* init_state, double* out,
                     double* final_state, int64_t N, int64_t T, int64_t H, int64_t dk,
                     int64_t dv, const int64_t* cu_seqlens, double scale, double eps,
                     int l2norm) {
    if (!q || !k || !v || !g || !beta || !out || N <= 0 || T < 0 || H <= 0 || dk <= 0 ||
        dv <= 0)
        return KDA_ORACLE_EBADARG;
    if (!check_cu(cu_seqlens, N, T)) return KDA_ORACLE_EBADARG;

    int nthreads = kda_oracle_num_threads();
    int64_t tasks_nh = N * H;
    int64_t nblk = 1;
    if (tasks_nh < nthreads) nblk = (nthreads + tasks_nh - 1) / tasks_nh;
    if (nblk > dv) nblk = dv;
    int64_t rows_per = (dv + nblk - 1) / nblk;
    int64_t ntask = tasks_nh * nblk;
    int failed = 0;

#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t task = 0; task < ntask; ++task) {
        int64_t blk = task % nblk;
        int64_t nh = task / nblk;
        int64_t n = nh / H, h = nh % H;
        int64_t r0 = blk * rows_per, r1 = r0 + rows_per;
        if (r1 > dv) r1 = dv;
        if (r0 >= r1) continue;
        int64_t nrows = r1 - r0;
        int64_t start, end;
        seq_bounds(cu_seqlens, n, T, &start, &end);

        double* S = (double*)malloc(sizeof(double) * (size_t)(nrows * dk));
        double* kh = (double*)malloc(sizeof(double) * (size_t)dk);
        double* qh = (double*)malloc(sizeof(double) * (size_t)dk);
        double* alpha = (double*)malloc(sizeof(double) * (size_t)dk);
        if (!S || !kh || !qh || !alpha) {
            free(S); free(kh); free(qh); free(alpha);
#pragma omp atomic write
            failed = 1;
            continue;
        }
        for (int64_t r = 0; r < nrows; ++r)
            for (int64_t c = 0; c < dk; ++c)
                S[r * dk + c] =
                    init_state ? init_state[((n * H + h) * dv + (r0 + r)) * dk + c] : 0.0;

        for (int64_t t = start; t < end; ++t) {
            const int64_t th = t * H + h;
            token_l2norm(k + th * dk, kh, dk, eps, l2norm);
            token_l2norm(q + th * dk, qh, dk, eps, l2norm);
            for (int64_t c = 0; c < dk; ++c) alpha[c] = exp(g[th * dk + c]);
            const double b = beta[th];
            for (int64_t r = 0; r < nrows; ++r) {
                double* s = S + r * dk;
                /* S <- S Diag(alpha): scale key column c by alpha[c]. */
                for (int64_t c = 0; c < dk; ++c) s[c] *= alpha[c];
                /* Prediction of v_t from the decayed state, then the error. */
                double pred = 0.0;
                for (int64_t c = 0; c < dk; ++c) pred += s[c] * kh[c];
                double u = b * (v[th * dv + r0 + r] - pred);
                /* Rank-one write along khat. */
                for (int64_t c = 0; c < dk; ++c) s[c] += u * kh[c];
                /* Read-out after the write. */
                double o = 0.0;
                for (int64_t c = 0; c < dk; ++c) o += s[c] * qh[c];
                out[th * dv + r0 + r] = scale * o;
            }
        }
        if (final_state)
            for (int64_t r = 0; r < nrows; ++r)
                for (int64_t c = 0; c < dk; ++c)
                    final_state[((n * H + h) * dv + (r0 + r)) * dk + c] = S[r * dk + c];
        free(S); free(kh); free(qh); free(alpha);
    }
    return failed ? KDA_ORACLE_ENOMEM : KDA_ORACLE_OK;
}

/* ------------------------------------------------------------------------- */
/* 2. Chunkwise form.                                                         */
/* ------------------------------------------------------------------------- */

/* L2 normalisation used by the chunkwise form (kept separate on purpose). */
static void chunk_normalise(const double* x, double* y, int64_t d, double eps, int enable) {
    double ss = 0.0;
    for (int64_t c = 0; c < d; ++c) ss += x[c] * x[c];
    double f = enable ? 1.0 / sqrt(ss + eps) : 1.0;
    for (int64_t c = 0; c < d; ++c) y[c] = f * x[c];
}

/* X = (I + R)^{-1} by forward substitution; R strictly lower triangular, C x C. */
static void inverse_forward(const double* R, double* X, int64_t C) {
    for (int64_t m = 0; m < C; ++m) {        /* column m of X */
        for (int64_t i = 0; i < C; ++i) {    /* row i: X_im = delta_im - sum_{j<i} R_ij X_jm */
            double acc = (i == m) ? 1.0 : 0.0;
            for (int64_t j = 0; j < i; ++j) acc -= R[i * C + j] * X[j * C + m];
            X[i * C + m] = acc;
        }
    }
}

static void matmul_sq(const double* A, const double* B, double* Cm, int64_t n) {
    for (int64_t i = 0; i < n; ++i)
        for (int64_t j = 0; j < n; ++j) {
            double acc = 0.0;
            for (int64_t l = 0; l < n; ++l) acc += A[i * n + l] * B[l * n + j];
            Cm[i * n + j] = acc;
        }
}

/*
 * X = (I + L)^{-1} by the repeated-squaring Neumann product
 *   (I - L)(I + L^2)(I + L^4) ... (I + L^(2^p)),  2^(p+1) >= C,
 * which is exact because the strictly lower-triangular L satisfies L^C = 0.
 */
static int inverse_neumann(const double* L, double* X, int64_t C) {
    size_t sz = sizeof(double) * (size_t)(C * C);
    double* P = (double*)malloc(sz);   /* current power L^(2^q) */
    double* T1 = (double*)malloc(sz);
    double* T2 = (double*)malloc(sz);
    if (!P || !T1 || !T2) {
        free(P); free(T1); free(T2);
        return 0;
    }
    for (int64_t i = 0; i < C; ++i)
        for (int64_t j = 0; j < C; ++j) {
            X[i * C + j] = ((i == j) ? 1.0 : 0.0) - L[i * C + j];
            P[i * C + j] = L[i * C + j];
        }
    for (int64_t e = 2; e < C; e *= 2) {
        matmul_sq(P, P, T1, C);             /* L^e */
        memcpy(P, T1, sz);
        matmul_sq(X, P, T2, C);             /* X (I + L^e) = X + X L^e */
        for (int64_t i = 0; i < C * C; ++i) X[i] += T2[i];
    }
    free(P); free(T1); free(T2);
    return 1;
}

/*
 * Per-chunk quantities of one (sequence, head), for chunk c of length Cc (the
 * last chunk of a sequence may be shorter than C).  Arrays are written for the
 * chunk only; caller provides storage:
 *   Kst[dk*C], Qst[dk*C]  (column i = D_{0:i} x_i, stored [channel][i])
 *   Kend[C*dk]            (row i = x_i^T D_{i+1:Cc-1})
 *   Dtot[dk]              (D_{0:Cc-1})
 *   R[C*C], Akk[C*C], Aqk[C*C]   (row-major [i][j])
 */
typedef struct {
    int64_t dk, C;
    double *kh, *qh;      /* [C][dk] normalised keys / queries of the chunk */
    double *alpha;        /* [C][dk] per-token decay alpha = exp(g) */
    double *Dpre;         /* [C][dk] D_{0:i} */
    double *Dpair;        /* [C][C][dk] D_{j+1:i} for j < i (j == i gives identity) */
} chunk_scratch;

static void chunk_quantities(const chunk_scratch* w, int64_t Cc, const double* betac,
                             double scale, double* Kst, double* Qst, double* Kend,
                             double* Dtot, double* R, double* Akk, double* Aqk,
                             int inv_mode) {
    const int64_t dk = w->dk, C = w->C;
    /* D_{0:i} = D_0 D_1 ... D_i (product of per-token decays, inclusive). */
    for (int64_t c = 0; c < dk; ++c) {
        double p = 1.0;
        for (int64_t i = 0; i < Cc; ++i) {
            p *= w->alpha[i * dk + c];
            w->Dpre[i * dk + c] = p;
        }
    }
    /* D_{j+1:i} = D_{j+1} ... D_i, the empty product being the identity. */
    for (int64_t j = 0; j < Cc; ++j)
        for (int64_t c = 0; c < dk; ++c) {
            double p = 1.0;
            w->Dpair[(j * C + j) * dk + c] = 1.0;
            for (int64_t i = j + 1; i < Cc; ++i) {
                p *= w->alpha[i * dk + c];
                w->Dpair[(i * C + j) * dk + c] = p;
            }
        }
    for (int64_t c = 0; c < dk; ++c) Dtot[c] = w->Dpre[(Cc - 1) * dk + c];
    for (int64_t i = 0; i < Cc; ++i)
        for (int64_t c = 0; c < dk; ++c) {
            Kst[c * C + i] = w->Dpre[i * dk + c] * w->kh[i * dk + c];
            Qst[c * C + i] = w->Dpre[i * dk + c] * w->qh[i * dk + c];
            /* D_{i+1:Cc-1}: the pair product from i to the chunk's last token. */
            Kend[i * dk + c] = w->kh[i * dk + c] * w->Dpair[((Cc - 1) * C + i) * dk + c];
        }
    for (int64_t i = 0; i < Cc; ++i)
        for (int64_t j = 0; j < Cc; ++j) {
            double rkk = 0.0, rqk = 0.0;
            if (j <= i) {
                for (int64_t c = 0; c < dk; ++c) {
                    double d = w->Dpair[(i * C + j) * dk + c];
                    rkk += w->kh[j * dk + c] * d * w->kh[i * dk + c];
                    rqk += w->kh[j * dk + c] * d * w->qh[i * dk + c];
                }
            }
            R[i * Cc + j] = (j < i) ? betac[i] * rkk : 0.0;
            Aqk[i * Cc + j] = (j <= i) ? scale * rqk : 0.0;
        }
    if (inv_mode == 1)
        inverse_neumann(R, Akk, Cc);
    else
        inverse_forward(R, Akk, Cc);
}

static int chunk_scratch_init(chunk_scratch* w, int64_t C, int64_t dk) {
    w->dk = dk;
    w->C = C;
    w->kh = (double*)malloc(sizeof(double) * (size_t)(C * dk));
    w->qh = (double*)malloc(sizeof(double) * (size_t)(C * dk));
    w->alpha = (double*)malloc(sizeof(double) * (size_t)(C * dk));
    w->Dpre = (double*)malloc(sizeof(double) * (size_t)(C * dk));
    w->Dpair = (double*)malloc(sizeof(double) * (size_t)(C * C * dk));
    return w->kh && w->qh && w->alpha && w->Dpre && w->Dpair;
}

static void chunk_scratch_free(chunk_scratch* w) {
    free(w->kh); free(w->qh); free(w->alpha); free(w->Dpre); free(w->Dpair);
}

static void chunk_load(chunk_scratch* w, const double* q, const double* k, const double* g,
                       int64_t t0, int64_t Cc, int64_t H, int64_t h, double eps, int l2norm) {
    const int64_t dk = w->dk;
    for (int64_t i = 0; i < Cc; ++i) {
        const int64_t th = (t0 + i) * H + h;
        chunk_normalise(k + th * dk, w->kh + i * dk, dk, eps, l2norm);
        chunk_normalise(q + th * dk, w->qh + i * dk, dk, eps, l2norm);
        for (int64_t c = 0; c < dk; ++c) w->alpha[i * dk + c] = exp(g[th * dk + c]);
    }
}

int kda_oracle_chunk(const double* q, const double* k, const double* v, const double* g,
                     const double* beta, const double* init_state, double* out,
                     double* final_state, int64_t N, int64_t T, int64_t H, int64_t dk,
                     int64_t dv, const int64_t* cu_seqlens, double scale, double eps,
                     int l2norm, int64_t C, int inv_mode) {
    if (!q || !k || !v || !g || !beta || !out || N <= 0 || T < 0 || H <= 0 || dk <= 0 ||
        dv <= 0 || C <= 0)
        return KDA_ORACLE_EBADARG;
    if (!check_cu(cu_seqlens, N, T)) return KDA_ORACLE_EBADARG;
    int failed = 0;

#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t nh = 0; nh < N * H; ++nh) {
        int64_t n = nh / H, h = nh % H;
        int64_t start, end;
        seq_bounds(cu_seqlens, n, T, &start, &end);
        chunk_scratch w;
        int ok = chunk_scratch_init(&w, C, dk);
        double* S = (double*)malloc(sizeof(double) * (size_t)(dv * dk));
        double* Snew = (double*)malloc(sizeof(double) * (size_t)(dv * dk));
        double* Kst = (double*)malloc(sizeof(double) * (size_t)(dk * C));
        double* Qst = (double*)malloc(sizeof(double) * (size_t)(dk * C));
        double* Kend = (double*)malloc(sizeof(double) * (size_t)(C * dk));
        double* Dtot = (double*)malloc(sizeof(double) * (size_t)dk);
        double* R = (double*)malloc(sizeof(double) * (size_t)(C * C));
        double* Akk = (double*)malloc(sizeof(double) * (size_t)(C * C));
        double* Aqk = (double*)malloc(sizeof(double) * (size_t)(C * C));
        double* E = (double*)malloc(sizeof(double) * (size_t)(dv * C));   /* (V - S K^start) B */
        double* U = (double*)malloc(sizeof(double) * (size_t)(dv * C));
        double* bc = (double*)malloc(sizeof(double) * (size_t)C);
        if (!ok || !S || !Snew || !Kst || !Qst || !Kend || !Dtot || !R || !Akk || !Aqk || !E ||
            !U || !bc) {
#pragma omp atomic write
            failed = 1;
        } else {
            for (int64_t r = 0; r < dv; ++r)
                for (int64_t c = 0; c < dk; ++c)
                    S[r * dk + c] =
                        init_state ? init_state[((n * H + h) * dv + r) * dk + c] : 0.0;
            for (int64_t t0 = start; t0 < end; t0 += C) {
                int64_t Cc = (end - t0 < C) ? (end - t0) : C;
                chunk_load(&w, q, k, g, t0, Cc, H, h, eps, l2norm);
                for (int64_t i = 0; i < Cc; ++i) bc[i] = beta[(t0 + i) * H + h];
                chunk_quantities(&w, Cc, bc, scale, Kst, Qst, Kend, Dtot, R, Akk, Aqk,
                                 inv_mode);
                /* E = (V - S K^start) B : value rows x tokens. */
                for (int64_t r = 0; r < dv; ++r)
                    for (int64_t i = 0; i < Cc; ++i) {
                        double sk = 0.0;
                        for (int64_t c = 0; c < dk; ++c) sk += S[r * dk + c] * Kst[c * C + i];
                        E[r * C + i] = (v[((t0 + i) * H + h) * dv + r] - sk) * bc[i];
                    }
                /* U = E (A^kk)^T. */
                for (int64_t r = 0; r < dv; ++r)
                    for (int64_t i = 0; i < Cc; ++i) {
                        double acc = 0.0;
                        for (int64_t j = 0; j < Cc; ++j) acc += E[r * C + j] * Akk[i * Cc + j];
                        U[r * C + i] = acc;
                    }
                /* O = s S Q^start + U (A^qk)^T. */
                for (int64_t r = 0; r < dv; ++r)
                    for (int64_t i = 0; i < Cc; ++i) {
                        double sq = 0.0, ua = 0.0;
                        for (int64_t c = 0; c < dk; ++c) sq += S[r * dk + c] * Qst[c * C + i];
                        for (int64_t j = 0; j < Cc; ++j) ua += U[r * C + j] * Aqk[i * Cc + j];
                        out[((t0 + i) * H + h) * dv + r] = scale * sq + ua;
                    }
                /* S <- S D_{0:Cc-1} + U K^end. */
                for (int64_t r = 0; r < dv; ++r)
                    for (int64_t c = 0; c < dk; ++c) {
                        double acc = S[r * dk + c] * Dtot[c];
                        for (int64_t i = 0; i < Cc; ++i) acc += U[r * C + i] * Kend[i * dk + c];
                        Snew[r * dk + c] = acc;
                    }
                memcpy(S, Snew, sizeof(double) * (size_t)(dv * dk));
            }
            if (final_state)
                memcpy(final_state + (n * H + h) * dv * dk, S, sizeof(double) * (size_t)(dv * dk));
        }
        chunk_scratch_free(&w);
        free(S); free(Snew); free(Kst); free(Qst); free(Kend); free(Dtot);
        free(R); free(Akk); free(Aqk); free(E); free(U); free(bc);
    }
    return failed ? KDA_ORACLE_ENOMEM : KDA_ORACLE_OK;
}

/*
 * Per-chunk intermediates of the chunkwise form for every (chunk, head), for
 * checking a chunk-preparation stage.  Chunks are numbered per sequence from
 * the sequence's first token; chunk index space is the concatenation over
 * sequences (sequence n owns ceil(len_n / C) chunks).  Outputs, per chunk x
 * head (index ch * H + h), with chunk length C (entries of a short last chunk
 * beyond its length are zero):
 *   Kst, Qst : [.., C, dk]  row i = D_{0:i} xhat_i   (the columns of K^start/Q^start)
 *   Kend     : [.., C, dk]  row i = khat_i^T D_{i+1:Cc-1}
 *   Dtot     : [.., dk]
 *   Akk, Aqk : [.., C, C]   (Aqk includes the scale s)
 */
int kda_oracle_chunk_intermediates(const double* q, const double* k, const double* g,
                                   const double* beta, double* Kst_o, double* Qst_o,
                                   double* Kend_o, double* Dtot_o, double* Akk_o,
                                   double* Aqk_o, int64_t N, int64_t T, int64_t H,
                                   int64_t dk, const int64_t* cu_seqlens, double scale,
                                   double eps, int l2norm, int64_t C, int inv_mode) {
    if (!q || !k || !g || !beta || N <= 0 || T < 0 || H <= 0 || dk <= 0 || C <= 0)
        return KDA_ORACLE_EBADARG;
    if (!check_cu(cu_seqlens, N, T)) return KDA_ORACLE_EBADARG;
    /* First chunk index of every sequence. */
    int64_t* first = (int64_t*)malloc(sizeof(int64_t) * (size_t)(N + 1));
    if (!first) return KDA_ORACLE_ENOMEM;
    first[0] = 0;
    for (int64_t n = 0; n < N; ++n) {
        int64_t s0, s1;
        seq_bounds(cu_seqlens, n, T, &s0, &s1);
        first[n + 1] = first[n] + (s1 - s0 + C - 1) / C;
    }
    int failed = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t nh = 0; nh < N * H; ++nh) {
        int64_t n = nh / H, h = nh % H;
        int64_t start, end;
        seq_bounds(cu_seqlens, n, T, &start, &end);
        chunk_scratch w;
        int ok = chunk_scratch_init(&w, C, dk);
        double* Kst = (double*)malloc(sizeof(double) * (size_t)(dk * C));
        double* Qst = (double*)malloc(sizeof(double) * (size_t)(dk * C));
        double* Kend = (double*)malloc(sizeof(double) * (size_t)(C * dk));
        double* Dtot = (double*)malloc(sizeof(double) * (size_t)dk);
        double* R = (double*)malloc(sizeof(double) * (size_t)(C * C));
        double* Akk = (double*)malloc(sizeof(double) * (size_t)(C * C));
        double* Aqk = (double*)malloc(sizeof(double) * (size_t)(C * C));
        double* bc = (double*)malloc(sizeof(double) * (size_t)C);
        if (!ok || !Kst || !Qst || !Kend || !Dtot || !R || !Akk || !Aqk || !bc) {
#pragma omp atomic write
            failed = 1;
        } else {
            int64_t ch = first[n];
            for (int64_t t0 = start; t0 < end; t0 += C, ++ch) {
                int64_t Cc = (end - t0 < C) ? (end - t0) : C;
                chunk_load(&w, q, k, g, t0, Cc, H, h, eps, l2norm);
                for (int64_t i = 0; i < Cc; ++i) bc[i] = beta[(t0 + i) * H + h];
                chunk_quantities(&w, Cc, bc, scale, Kst, Qst, Kend, Dtot, R, Akk, Aqk,
                                 inv_mode);
                int64_t base = ch * H + h;
                for (int64_t i = 0; i < C; ++i)
                    for (int64_t c = 0; c < dk; ++c) {
                        int64_t o = (base * C + i) * dk + c;
                        Kst_o[o] = (i < Cc) ? Kst[c * C + i] : 0.0;
                        Qst_o[o] = (i < Cc) ? Qst[c * C + i] : 0.0;
                        Kend_o[o] = (i < Cc) ? Kend[i * dk + c] : 0.0;
                    }
                for (int64_t c = 0; c < dk; ++c) Dtot_o[base * dk + c] = Dtot[c];
                for (int64_t i = 0; i < C; ++i)
                    for (int64_t j = 0; j < C; ++j) {
                        int64_t o = (base * C + i) * C + j;
                        Akk_o[o] = (i < Cc && j < Cc) ? Akk[i * Cc + j] : (i == j ? 1.0 : 0.0);
                        Aqk_o[o] = (i < Cc && j < Cc) ? Aqk[i * Cc + j] : 0.0;
                    }
            }
        }
        chunk_scratch_free(&w);
        free(Kst); free(Qst); free(Kend); free(Dtot); free(R); free(Akk); free(Aqk); free(bc);
    }
    free(first);
    return failed ? KDA_ORACLE_ENOMEM : KDA_ORACLE_OK;
}

/*
 * The inverse alone, for tests: X = (I + L)^{-1} for a strictly lower
 * triangular C x C matrix L, by forward substitution (mode 0) or the Neumann
 * product (mode 1).
 */
int kda_oracle_unitri_inverse(const double* L, double* X, int64_t C, int mode) {
    if (!L || !X || C <= 0) return KDA_ORACLE_EBADARG;
    if (mode == 1) return inverse_neumann(L, X, C) ? KDA_ORACLE_OK : KDA_ORACLE_ENOMEM;
    inverse_forward(L, X, C);
    return KDA_ORACLE_OK;
}

/*
 * beta from a logit: beta = sigmoid(x) = 1 / (1 + exp(-x)), elementwise, n
 * values.  The flashinfer kda_prefill page ("Optimized Blackwell prefill
 * subset": beta_is_logit=True, and the N16 schedule's list of rounding points,
 * which names "sigmoid beta") takes beta as a logit and applies the sigmoid
 * inside the operation; the page gives no other formula, so this is the plain
 * logistic function, in FP64.  For x < 0 it is evaluated as exp(x) / (1 +
 * exp(x)), the same function, so that exp never overflows.
 */
int kda_oracle_sigmoid(const double* x, double* y, int64_t n) {
    if (n < 0 || (n > 0 && (!x || !y))) return KDA_ORACLE_EBADARG;
    for (int64_t i = 0; i < n; ++i) {
        if (x[i] >= 0.0) {
            y[i] = 1.0 / (1.0 + exp(-x[i]));
        } else {
            const double e = exp(x[i]);
            y[i] = e / (1.0 + e);
        }
    }
    return KDA_ORACLE_OK;
}
