/*
 * Native Hybrid Attention (NHA) -- plain fp64 CPU oracle.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the tests, the package's smoke() check and the CPU
 * baseline leg of bench.py use it.  It shares no code, header, table or
 * helper with the CUDA library.
 *
 * What it computes (source: "Native Hybrid Attention for Efficient Sequence
 * Modeling", Paper-Notes page, section "关键设计 / 层内混合", the K^long_t
 * recurrence and the o_t = softmax(q_t K^H_t^T / sqrt(d)) V^H_t equation;
 * same page, "整体框架" for the memory shapes K^long in R^{m x d},
 * K^short in R^{w x d}; same section's design-motivation paragraph for the
 * token shift and for RoPE applied only inside the window):
 *
 *   per (b,h), slot states S^K, S^V in R^{m x d}, zero at the start;
 *   for t = 0..T-1:
 *     if t >= w:  token j = t-w leaves the window and is absorbed
 *        S^K[i] = alpha_j[i] * S^K[i] + (1 - alpha_j[i]) * k_j  (S^V likewise)
 *        slot logit   L_i = q_t . S^K[i] / sqrt(d)      (no position encoding)
 *     else:      all m slot logits are masked (-inf)
 *     window logit  S_s = rope(q_t, t) . rope(k_s, s) / sqrt(d),
 *                   s in [max(0, t-w+1), t]
 *     one softmax over the m + n_win logits; lse_t = log of its partition
 *     o_t = sum_i p_i S^V[i] + sum_s p_s v_s
 *
 * Optional initial slot states (h0k, h0v in R^{m x d} per head; the ai.info
 * page, Future Directions, names learned initial slot states): the long memory before
 * token 0 is h0 instead of zero, and because it is then never empty the
 * slot logits are not masked for t < w (query t < w reads h0 itself).
 * The backward returns dh0 = the state adjoint carried back past token 0.
 *
 * Readings of points the pages leave open:
 *   - token j is absorbed with its own gate alpha_j, and the query at t reads
 *     the state after token t-w (the token shift);
 *   - the window holds the w most recent tokens including t itself, so w = 0
 *     gives a pure slot RNN and w >= T gives causal attention;
 *   - the slot mask is positional: all slots are masked iff t < w;
 *   - the 1/sqrt(d) scale applies to slot and window logits alike;
 *   - RoPE is the rotate-half form with theta_i = base^(-2i/d), i < d/2,
 *     at absolute 0-based positions;
 *   - 1 - alpha is evaluated as -expm1(log_alpha).
 *
 * The backward pass is a hand-derived reverse sweep of exactly that
 * program: the adjoints of S^K and S^V are carried backwards through each
 * state update S_j = diag(alpha_j) S_{j-1} + u_j (x) k_j.  States are
 * checkpointed every CKPT tokens and recomputed segment by segment.
 *
 * Build: gcc -O2 -fopenmp -shared -fPIC nha_oracle.c -lm
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define CKPT 64

typedef struct {
    long T, d, m, w;
    double base;
} shape_t;

/* cos/sin of pos * theta_i for every position and frequency; theta_i =
 * base^(-2i/d).  tab has T * (d/2) entries. */
static void rope_tables(const shape_t* sh, double* cs, double* sn) {
    long h = sh->d / 2;
    for (long i = 0; i < h; i++) {
        double theta = pow(sh->base, -2.0 * (double)i / (double)sh->d);
        for (long t = 0; t < sh->T; t++) {
            double a = (double)t * theta;
            cs[t * h + i] = cos(a);
            sn[t * h + i] = sin(a);
        }
    }
}

/* y = R_pos x  (rotate-half pairing i <-> i + d/2) */
static void rope_apply(const double* x, double* y, long d, const double* c, const double* s) {
    long h = d / 2;
    for (long i = 0; i < h; i++) {
        double a = x[i], b = x[i + h];
        y[i] = a * c[i] - b * s[i];
        y[i + h] = b * c[i] + a * s[i];
    }
}

/* y += R_pos^T g  (the transpose rotates by -angle) */
static void rope_apply_t_acc(const double* g, double* y, long d, const double* c, const double* s) {
    long h = d / 2;
    for (long i = 0; i < h; i++) {
        double a = g[i], b = g[i + h];
        y[i] += a * c[i] + b * s[i];
        y[i + h] += b * c[i] - a * s[i];
    }
}

static double dot(const double* a, const double* b, long n) {
    double acc = 0.0;
    for (long i = 0; i < n; i++) acc += a[i] * b[i];
    return acc;
}

/* Absorb token j: S = diag(alpha_j) S + u_j (x) x_j, for one state. */
static void absorb(double* S, const double* la, const double* x, long m, long d) {
    for (long i = 0; i < m; i++) {
        double a = exp(la[i]);
        double u = -expm1(la[i]);
        double* row = S + i * d;
        for (long c = 0; c < d; c++) row[c] = a * row[c] + u * x[c];
    }
}

/* Logits, max and partition for query t given the current states.
 * Fills L[m] (slot logits, only if have_slots) and S[n_win] (window logits,
 * keys lo..t).  Returns lse. */
static double query_logits(const shape_t* sh, long t, const double* q_t, const double* qr_t,
                           const double* kr, const double* SK, int have_slots,
                           double* L, double* Sw, long lo) {
    long d = sh->d, m = sh->m;
    double sigma = 1.0 / sqrt((double)d);
    double M = -INFINITY;
    if (have_slots) {
        for (long i = 0; i < m; i++) {
            L[i] = sigma * dot(q_t, SK + i * d, d);
            if (L[i] > M) M = L[i];
        }
    }
    for (long s = lo; s <= t; s++) {
        double v = sigma * dot(qr_t, kr + s * d, d);
        Sw[s - lo] = v;
        if (v > M) M = v;
    }
    double Z = 0.0;
    if (have_slots)
        for (long i = 0; i < m; i++) Z += exp(L[i] - M);
    for (long s = lo; s <= t; s++) Z += exp(Sw[s - lo] - M);
    return M + log(Z);
}

static long window_lo(long t, long w) {
    long lo = t - w + 1;
    return lo < 0 ? 0 : lo;
}

/* One (b,h) head, forward.  h0k, h0v: initial states [m][d] or NULL; hTk,
 * hTv: [m][d] outputs (or NULL) for the final states, the long memory after the
 * last token that left the window (token T - w - 1; h0, or zero, when none
 * has). */
static void head_forward(const shape_t* sh, const double* q, const double* k, const double* v,
                         const double* la, double* o, double* lse, double* omega,
                         const double* cs, const double* sn, const double* h0k, const double* h0v,
                         double* hTk, double* hTv) {
    long T = sh->T, d = sh->d, m = sh->m, w = sh->w, h = d / 2;
    double* SK = calloc((size_t)(m * d), sizeof(double));
    double* SV = calloc((size_t)(m * d), sizeof(double));
    if (h0k) memcpy(SK, h0k, sizeof(double) * (size_t)(m * d));
    if (h0v) memcpy(SV, h0v, sizeof(double) * (size_t)(m * d));
    double* kr = malloc(sizeof(double) * (size_t)(T * d));
    double* qr = malloc(sizeof(double) * (size_t)d);
    double* L = malloc(sizeof(double) * (size_t)(m > 0 ? m : 1));
    double* Sw = malloc(sizeof(double) * (size_t)(T + 1));
    for (long s = 0; s < T; s++) rope_apply(k + s * d, kr + s * d, d, cs + s * h, sn + s * h);
    for (long t = 0; t < T; t++) {
        int have_slots = (t >= w) || h0k != NULL;
        if (t >= w) {
            long j = t - w;
            absorb(SK, la + j * m, k + j * d, m, d);
            absorb(SV, la + j * m, v + j * d, m, d);
        }
        rope_apply(q + t * d, qr, d, cs + t * h, sn + t * h);
        long lo = window_lo(t, w);
        double l = query_logits(sh, t, q + t * d, qr, kr, SK, have_slots, L, Sw, lo);
        lse[t] = l;
        double* ot = o + t * d;
        for (long c = 0; c < d; c++) ot[c] = 0.0;
        double wl = 0.0;
        if (have_slots) {
            for (long i = 0; i < m; i++) {
                double p = exp(L[i] - l);
                wl += p;
                for (long c = 0; c < d; c++) ot[c] += p * SV[i * d + c];
            }
        }
        for (long s = lo; s <= t; s++) {
            double p = exp(Sw[s - lo] - l);
            for (long c = 0; c < d; c++) ot[c] += p * v[s * d + c];
        }
        if (omega) omega[t] = wl;
    }
    if (hTk) memcpy(hTk, SK, sizeof(double) * (size_t)(m * d));
    if (hTv) memcpy(hTv, SV, sizeof(double) * (size_t)(m * d));
    free(SK); free(SV); free(kr); free(qr); free(L); free(Sw);
}

/* One (b,h) head, backward (reverse sweep with state adjoints).  h0k, h0v:
 * initial states or NULL; dh0k, dh0v (written when h0k is given): their
 * gradients.  dhTk, dhTv: [m][d] or NULL: the gradient of the loss with
 * respect to the final states (the loss is then sum(o * dout) + <hT, dhT>);
 * it is the state adjoint the reverse sweep starts from. */
static void head_backward(const shape_t* sh, const double* q, const double* k, const double* v,
                          const double* la, const double* dout, double* dq, double* dk,
                          double* dv, double* dla, const double* cs, const double* sn,
                          const double* h0k, const double* h0v, double* dh0k, double* dh0v,
                          const double* dhTk, const double* dhTv) {
    long T = sh->T, d = sh->d, m = sh->m, w = sh->w, h = d / 2;
    long md = m * d;
    double sigma = 1.0 / sqrt((double)d);
    long R = T - w; /* number of absorbed tokens that some query reads */
    if (R < 0) R = 0;
    long nseg = (R + CKPT - 1) / CKPT;

    double* kr = malloc(sizeof(double) * (size_t)(T * d));
    double* dkr = calloc((size_t)(T * d), sizeof(double));
    double* qr = malloc(sizeof(double) * (size_t)d);
    double* dqr = malloc(sizeof(double) * (size_t)d);
    double* L = malloc(sizeof(double) * (size_t)(m > 0 ? m : 1));
    double* Sw = malloc(sizeof(double) * (size_t)(T + 1));
    double* o_t = malloc(sizeof(double) * (size_t)d);
    /* checkpoints: state before segment c, i.e. after tokens 0..c*CKPT-1 */
    double* ckK = calloc((size_t)((nseg + 1) * md), sizeof(double));
    double* ckV = calloc((size_t)((nseg + 1) * md), sizeof(double));
    /* states inside one segment: seg[r] = state after token c*CKPT + r - 1 */
    double* segK = malloc(sizeof(double) * (size_t)((CKPT + 1) * md));
    double* segV = malloc(sizeof(double) * (size_t)((CKPT + 1) * md));
    double* dSK = calloc((size_t)md, sizeof(double));
    double* dSV = calloc((size_t)md, sizeof(double));
    if (dhTk) memcpy(dSK, dhTk, sizeof(double) * (size_t)md);
    if (dhTv) memcpy(dSV, dhTv, sizeof(double) * (size_t)md);

    memset(dq, 0, sizeof(double) * (size_t)(T * d));
    memset(dk, 0, sizeof(double) * (size_t)(T * d));
    memset(dv, 0, sizeof(double) * (size_t)(T * d));
    memset(dla, 0, sizeof(double) * (size_t)(T * m));

    for (long s = 0; s < T; s++) rope_apply(k + s * d, kr + s * d, d, cs + s * h, sn + s * h);

    /* forward over absorbed tokens only, saving checkpoints */
    {
        double* SK = calloc((size_t)md, sizeof(double));
        double* SV = calloc((size_t)md, sizeof(double));
        if (h0k) memcpy(SK, h0k, sizeof(double) * (size_t)md);
        if (h0v) memcpy(SV, h0v, sizeof(double) * (size_t)md);
        for (long j = 0; j < R; j++) {
            if (j % CKPT == 0) {
                memcpy(ckK + (j / CKPT) * md, SK, sizeof(double) * (size_t)md);
                memcpy(ckV + (j / CKPT) * md, SV, sizeof(double) * (size_t)md);
            }
            absorb(SK, la + j * m, k + j * d, m, d);
            absorb(SV, la + j * m, v + j * d, m, d);
        }
        free(SK); free(SV);
    }

    /* One query's contribution; SKj/SVj are the states it reads (NULL when
     * t < w).  Adds to dq, dkr, dv and to the state adjoints. */
#define QUERY_BACKWARD(t, SKj, SVj)                                                         \
    do {                                                                                    \
        long tt = (t);                                                                      \
        int hs = ((SKj) != NULL);                                                           \
        rope_apply(q + tt * d, qr, d, cs + tt * h, sn + tt * h);                            \
        long lo = window_lo(tt, w);                                                         \
        double l = query_logits(sh, tt, q + tt * d, qr, kr, (SKj), hs, L, Sw, lo);          \
        const double* g = dout + tt * d;                                                    \
        for (long c = 0; c < d; c++) o_t[c] = 0.0;                                          \
        if (hs)                                                                             \
            for (long i = 0; i < m; i++) {                                                  \
                double p = exp(L[i] - l);                                                   \
                for (long c = 0; c < d; c++) o_t[c] += p * (SVj)[i * d + c];                \
            }                                                                               \
        for (long s = lo; s <= tt; s++) {                                                   \
            double p = exp(Sw[s - lo] - l);                                                 \
            for (long c = 0; c < d; c++) o_t[c] += p * v[s * d + c];                        \
        }                                                                                   \
        double D = dot(g, o_t, d);                                                          \
        for (long c = 0; c < d; c++) dqr[c] = 0.0;                                          \
        if (hs)                                                                             \
            for (long i = 0; i < m; i++) {                                                  \
                double p = exp(L[i] - l);                                                   \
                double dP = dot(g, (SVj) + i * d, d);                                       \
                double dL = p * (dP - D);                                                   \
                for (long c = 0; c < d; c++) {                                              \
                    dq[tt * d + c] += sigma * dL * (SKj)[i * d + c];                        \
                    dSK[i * d + c] += sigma * dL * q[tt * d + c];                           \
                    dSV[i * d + c] += p * g[c];                                             \
                }                                                                           \
            }                                                                               \
        for (long s = lo; s <= tt; s++) {                                                   \
            double p = exp(Sw[s - lo] - l);                                                 \
            double dP = dot(g, v + s * d, d);                                               \
            double dS = p * (dP - D);                                                       \
            for (long c = 0; c < d; c++) {                                                  \
                dqr[c] += sigma * dS * kr[s * d + c];                                       \
                dkr[s * d + c] += sigma * dS * qr[c];                                       \
                dv[s * d + c] += p * g[c];                                                  \
            }                                                                               \
        }                                                                                   \
        rope_apply_t_acc(dqr, dq + tt * d, d, cs + tt * h, sn + tt * h);                    \
    } while (0)

    /* queries t >= w, in reverse, segment by segment of j = t - w */
    for (long c = nseg - 1; c >= 0; c--) {
        long j0 = c * CKPT;
        long j1 = j0 + CKPT < R ? j0 + CKPT : R;
        memcpy(segK, ckK + c * md, sizeof(double) * (size_t)md);
        memcpy(segV, ckV + c * md, sizeof(double) * (size_t)md);
        for (long j = j0; j < j1; j++) {
            long r = j - j0;
            memcpy(segK + (r + 1) * md, segK + r * md, sizeof(double) * (size_t)md);
            memcpy(segV + (r + 1) * md, segV + r * md, sizeof(double) * (size_t)md);
            absorb(segK + (r + 1) * md, la + j * m, k + j * d, m, d);
            absorb(segV + (r + 1) * md, la + j * m, v + j * d, m, d);
        }
        for (long j = j1 - 1; j >= j0; j--) {
            long r = j - j0;
            const double* SKj = segK + (r + 1) * md;
            const double* SVj = segV + (r + 1) * md;
            const double* SKp = segK + r * md; /* state before token j */
            const double* SVp = segV + r * md;
            QUERY_BACKWARD(j + w, SKj, SVj);
            /* back through S_j = diag(alpha_j) S_{j-1} + u_j (x) x_j */
            for (long i = 0; i < m; i++) {
                double lg = la[j * m + i];
                double a = exp(lg);
                double u = -expm1(lg);
                double dA = dot(dSK + i * d, SKp + i * d, d) + dot(dSV + i * d, SVp + i * d, d);
                double dU = dot(dSK + i * d, k + j * d, d) + dot(dSV + i * d, v + j * d, d);
                for (long cc = 0; cc < d; cc++) {
                    dk[j * d + cc] += u * dSK[i * d + cc];
                    dv[j * d + cc] += u * dSV[i * d + cc];
                    dSK[i * d + cc] *= a;
                    dSV[i * d + cc] *= a;
                }
                /* alpha = exp(l): d alpha/dl = alpha; u = -expm1(l): du/dl = -alpha */
                dla[j * m + i] += a * dA - a * dU;
            }
        }
    }
    /* queries t < w: window only, or (with initial states) reading h0; dSK,
     * dSV now hold the adjoint of the state before token 0, which is h0 */
    {
        long tw = w < T ? w : T;
        for (long t = tw - 1; t >= 0; t--) QUERY_BACKWARD(t, h0k, h0v);
    }
    if (h0k) {
        memcpy(dh0k, dSK, sizeof(double) * (size_t)md);
        memcpy(dh0v, dSV, sizeof(double) * (size_t)md);
    }
#undef QUERY_BACKWARD
    for (long s = 0; s < T; s++) rope_apply_t_acc(dkr + s * d, dk + s * d, d, cs + s * h, sn + s * h);

    free(kr); free(dkr); free(qr); free(dqr); free(L); free(Sw); free(o_t);
    free(ckK); free(ckV); free(segK); free(segV); free(dSK); free(dSV);
}

static int check_shape(long B, long H, long T, long d, long m, long w) {
    if (B < 0 || H < 0 || T < 0 || d <= 0 || (d % 2) != 0 || m < 0 || w < 0) return -1;
    return 0;
}

/* o[B,H,T,d], lse[B,H,T], omega[B,H,T] (optional, may be NULL): the share of
 * softmax mass on the long-memory slots (the omega_L diagnostic of the same
 * section). */
/* h0k, h0v [B,H,m,d]: optional initial slot states (both or neither); hTk,
 * hTv [B,H,m,d]: optional final states (both or neither). */
int nha_oracle_forward(const double* q, const double* k, const double* v, const double* log_alpha,
                       double* o, double* lse, double* omega, long B, long H, long T, long d,
                       long m, long w, double rope_base, int nthreads, const double* h0k,
                       const double* h0v, double* hTk, double* hTv) {
    if ((h0k == NULL) != (h0v == NULL)) return -1;
    if ((hTk == NULL) != (hTv == NULL)) return -1;
    if (hTk && B * H > 0 && (T == 0 || w >= T)) {
        /* no token leaves the window: the final states are the initial ones */
        for (long e = 0; e < B * H * m * d; e++) {
            hTk[e] = h0k ? h0k[e] : 0.0;
            hTv[e] = h0v ? h0v[e] : 0.0;
        }
    }
    if (check_shape(B, H, T, d, m, w)) return -1;
    if (T == 0 || B * H == 0) return 0;
    shape_t sh = {T, d, m, w > T ? T : w, rope_base};
    long h = d / 2;
    double* cs = malloc(sizeof(double) * (size_t)(T * h));
    double* sn = malloc(sizeof(double) * (size_t)(T * h));
    rope_tables(&sh, cs, sn);
    long nbh = B * H;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
#endif
    for (long bh = 0; bh < nbh; bh++) {
        head_forward(&sh, q + bh * T * d, k + bh * T * d, v + bh * T * d, log_alpha + bh * T * m,
                     o + bh * T * d, lse + bh * T, omega ? omega + bh * T : NULL, cs, sn,
                     h0k ? h0k + bh * m * d : NULL, h0v ? h0v + bh * m * d : NULL,
                     hTk ? hTk + bh * m * d : NULL, hTv ? hTv + bh * m * d : NULL);
    }
    (void)nthreads;
    free(cs); free(sn);
    return 0;
}

/* h0k, h0v [B,H,m,d]: optional initial slot states; dh0k, dh0v [B,H,m,d]
 * receive their gradients (all four given, or none).  dhTk, dhTv [B,H,m,d]:
 * optional gradient with respect to the final states (both or neither). */
int nha_oracle_backward(const double* q, const double* k, const double* v, const double* log_alpha,
                        const double* dout, double* dq, double* dk, double* dv, double* dlog_alpha,
                        long B, long H, long T, long d, long m, long w, double rope_base,
                        int nthreads, const double* h0k, const double* h0v, double* dh0k,
                        double* dh0v, const double* dhTk, const double* dhTv) {
    int given = (h0k != NULL) + (h0v != NULL) + (dh0k != NULL) + (dh0v != NULL);
    if (given != 0 && given != 4) return -1;
    if ((dhTk == NULL) != (dhTv == NULL)) return -1;
    if (check_shape(B, H, T, d, m, w)) return -1;
    if (B * H > 0 && T == 0 && dh0k) {  /* no query: the final states are the initial ones */
        for (long e = 0; e < B * H * m * d; e++) {
            dh0k[e] = dhTk ? dhTk[e] : 0.0;
            dh0v[e] = dhTv ? dhTv[e] : 0.0;
        }
    }
    if (T == 0 || B * H == 0) return 0;
    shape_t sh = {T, d, m, w > T ? T : w, rope_base};
    long h = d / 2;
    double* cs = malloc(sizeof(double) * (size_t)(T * h));
    double* sn = malloc(sizeof(double) * (size_t)(T * h));
    rope_tables(&sh, cs, sn);
    long nbh = B * H;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
#endif
    for (long bh = 0; bh < nbh; bh++) {
        head_backward(&sh, q + bh * T * d, k + bh * T * d, v + bh * T * d, log_alpha + bh * T * m,
                      dout + bh * T * d, dq + bh * T * d, dk + bh * T * d, dv + bh * T * d,
                      dlog_alpha + bh * T * m, cs, sn, h0k ? h0k + bh * m * d : NULL,
                      h0v ? h0v + bh * m * d : NULL, dh0k ? dh0k + bh * m * d : NULL,
                      dh0v ? dh0v + bh * m * d : NULL, dhTk ? dhTk + bh * m * d : NULL,
                      dhTv ? dhTv + bh * m * d : NULL);
    }
    (void)nthreads;
    free(cs); free(sn);
    return 0;
}

int nha_oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
