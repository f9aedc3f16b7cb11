/*
 * gdn_oracle.c -- plain, slow fp64 CPU oracle for the gated delta rule.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file; only the test suite, the smoke check and the bench's CPU
 * baseline leg use it.  It shares no code, header, table or helper with the
 * CUDA library.
 *
 * What it computes (per batch b and head h, one independent recurrence):
 *
 *   "GDN & MLA Mechanism Deep-Dive", Step 4 (Gated delta rule):
 *       alpha_t[i] = exp(g_t * A[i]),   A[i] = -exp(A_log[h, i])
 *       gated mode:  h_t = alpha_t (.)rows h_{t-1} + b_t v_t^T
 *                    o_t = h_t^T c_t                    (read after write)
 *   "HyMo-434M -- documentation portal", card 01 (GDN recurrence, delta rule):
 *       delta mode:  h'  = alpha_t (.)rows h_{t-1}
 *                    u_t = beta_t (v_t - h'^T b_t)
 *                    h_t = h' + b_t u_t^T
 *                    o_t = h_t^T c_t
 *     i.e. h_t = (I - beta_t b_t b_t^T) diag(alpha_t) h_{t-1} + beta_t b_t v_t^T,
 *     the decay applied first and the erase made with the write key b.
 *
 * The state h is [d_k, d_v] with rows indexed by the key/state index i that
 * A and alpha act on (the page's "(S, D)" state shape, Worked example).
 *
 * Tensor layouts (all fp64, contiguous):
 *   v, b, c, o, dO, dv, db, dc : [B, T, H, d]   (d = d_k for b, c; d_v for v, o)
 *   g, beta, dg, dbeta         : [B, T, H]
 *   A_log                      : [H, d_k]
 *   h0, hT, dhT, dh0           : [B, H, d_k, d_v]
 *   dA_log_unit                : [B*H, d_k]  per-(b,h) partial of dA_log;
 *                                the caller sums over b.
 *
 * Every function processes the (b,h) units u = b*H + h with
 * unit_begin <= u < unit_end, so a caller can spread units over threads.
 * Each function returns 0 on success and -1 on bad arguments or when a
 * scratch allocation fails.
 */
#include <math.h>
#include <stddef.h>
#include <stdlib.h>
#include <string.h>

#define MODE_GATED 0
#define MODE_DELTA 1

static size_t at_btHd(int b, int t, int h, int k, int T, int H, int d)
{
    return (((size_t)b * T + t) * H + h) * d + k;
}

static size_t at_btH(int b, int t, int h, int T, int H)
{
    return ((size_t)b * T + t) * H + h;
}

static int bad_args(int B, int H, int T, int dk, int dv, int mode,
                    int unit_begin, int unit_end)
{
    if (B < 1 || H < 1 || T < 0 || dk < 1 || dv < 1) return 1;
    if (mode != MODE_GATED && mode != MODE_DELTA) return 1;
    if (unit_begin < 0 || unit_end > B * H || unit_begin > unit_end) return 1;
    return 0;
}

/*
 * One recurrence step on the state S [dk, dv] (row-major), in place.
 * Step 4 of "GDN & MLA Mechanism Deep-Dive" (gated) and the delta-rule card
 * of the documentation portal (delta).  On return S holds h_t.  If hp_out is
 * not NULL it receives h' = alpha (.) h_{t-1}; if r_out/u_out are not NULL
 * they receive r = h'^T b and the written value u (u = v in gated mode).
 */
static void step(int dk, int dv, int mode, double* S,
                 const double* A, double g, double beta,
                 const double* bvec, const double* vvec,
                 double* hp_out, double* r_out, double* u_out)
{
    for (int i = 0; i < dk; i++) {
        double alpha = exp(g * A[i]);
        for (int j = 0; j < dv; j++) S[i * dv + j] *= alpha;
    }
    if (hp_out) memcpy(hp_out, S, sizeof(double) * (size_t)dk * dv);
    for (int j = 0; j < dv; j++) {
        double u;
        if (mode == MODE_DELTA) {
            double r = 0.0;
            for (int i = 0; i < dk; i++) r += S[i * dv + j] * bvec[i];
            if (r_out) r_out[j] = r;
            u = beta * (vvec[j] - r);
        } else {
            if (r_out) r_out[j] = 0.0;
            u = vvec[j];
        }
        if (u_out) u_out[j] = u;
        for (int i = 0; i < dk; i++) S[i * dv + j] += bvec[i] * u;
    }
}

/* Serial forward: the recurrence exactly as written, one token at a time. */
int oracle_gdn_fwd(int B, int H, int T, int dk, int dv, int mode,
                   const double* v, const double* bk, const double* c,
                   const double* g, const double* beta, const double* A_log,
                   const double* h0, double* o, double* hT,
                   int unit_begin, int unit_end)
{
    if (bad_args(B, H, T, dk, dv, mode, unit_begin, unit_end)) return -1;
    if (mode == MODE_DELTA && !beta) return -1;
    double* S = (double*)malloc(sizeof(double) * (size_t)dk * dv);
    double* A = (double*)malloc(sizeof(double) * (size_t)dk);
    double* bv = (double*)malloc(sizeof(double) * (size_t)dk);
    double* vv = (double*)malloc(sizeof(double) * (size_t)dv);
    if (!S || !A || !bv || !vv) { free(S); free(A); free(bv); free(vv); return -1; }

    for (int u = unit_begin; u < unit_end; u++) {
        int b = u / H, h = u % H;
        for (int i = 0; i < dk; i++) A[i] = -exp(A_log[(size_t)h * dk + i]);
        if (h0) memcpy(S, h0 + (size_t)u * dk * dv, sizeof(double) * (size_t)dk * dv);
        else memset(S, 0, sizeof(double) * (size_t)dk * dv);
        for (int t = 0; t < T; t++) {
            for (int i = 0; i < dk; i++) bv[i] = bk[at_btHd(b, t, h, i, T, H, dk)];
            for (int j = 0; j < dv; j++) vv[j] = v[at_btHd(b, t, h, j, T, H, dv)];
            double gt = g[at_btH(b, t, h, T, H)];
            double bt = (mode == MODE_DELTA) ? beta[at_btH(b, t, h, T, H)] : 0.0;
            step(dk, dv, mode, S, A, gt, bt, bv, vv, NULL, NULL, NULL);
            for (int j = 0; j < dv; j++) {
                double acc = 0.0;
                for (int i = 0; i < dk; i++) acc += S[i * dv + j] * c[at_btHd(b, t, h, i, T, H, dk)];
                o[at_btHd(b, t, h, j, T, H, dv)] = acc;
            }
        }
        if (hT) memcpy(hT + (size_t)u * dk * dv, S, sizeof(double) * (size_t)dk * dv);
    }
    free(S); free(A); free(bv); free(vv);
    return 0;
}

/*
 * Serial backward: reverse-mode differentiation of oracle_gdn_fwd, by hand.
 * States are kept at every `seg`-th token and each segment is recomputed
 * forward before it is walked in reverse.  For t = T-1 ... 0:
 *   dh  += c_t dO_t^T;            dc_t = h_t dO_t
 *   du   = dh^T b_t;              db_t = dh u_t;   dh' = dh
 *   gated: dv_t = du
 *   delta: dbeta_t = du . (v_t - r_t);  dv_t = beta_t du;  dr = -beta_t du
 *          dh' += b_t dr^T;             db_t += h' dr
 *   q[i] = sum_j dh'[i,j] h'[i,j]   (= d(alpha_t[i]) * alpha_t[i])
 *   dg_t = sum_i q[i] A[i];   dA[i] += q[i] g_t;   dh = alpha_t (.)rows dh'
 * and at the end dh0 = dh, dA_log = dA (.) A  (dA/dA_log = -exp(A_log) = A).
 * dbeta may be NULL in gated mode; dhT, h0 may be NULL (zeros); dh0 may be NULL.
 */
int oracle_gdn_bwd(int B, int H, int T, int dk, int dv, int mode,
                   const double* v, const double* bk, const double* c,
                   const double* g, const double* beta, const double* A_log,
                   const double* h0, const double* dO, const double* dhT,
                   double* dv_out, double* db_out, double* dc_out,
                   double* dg_out, double* dbeta_out, double* dA_log_unit,
                   double* dh0, int seg, int unit_begin, int unit_end)
{
    if (bad_args(B, H, T, dk, dv, mode, unit_begin, unit_end)) return -1;
    if (mode == MODE_DELTA && (!beta || !dbeta_out)) return -1;
    if (seg < 1) return -1;
    const size_t SZ = (size_t)dk * dv;
    int nseg = (T + seg - 1) / seg;
    double* ck = (double*)malloc(sizeof(double) * SZ * (size_t)(nseg > 0 ? nseg : 1));
    double* prev = (double*)malloc(sizeof(double) * SZ * (size_t)seg); /* h_{t-1} per t in segment */
    double* S = (double*)malloc(sizeof(double) * SZ);
    double* hp = (double*)malloc(sizeof(double) * SZ);
    double* dS = (double*)malloc(sizeof(double) * SZ);
    double* A = (double*)malloc(sizeof(double) * (size_t)dk);
    double* dA = (double*)malloc(sizeof(double) * (size_t)dk);
    double* bv = (double*)malloc(sizeof(double) * (size_t)dk);
    double* cv = (double*)malloc(sizeof(double) * (size_t)dk);
    double* vv = (double*)malloc(sizeof(double) * (size_t)dv);
    double* r = (double*)malloc(sizeof(double) * (size_t)dv);
    double* uu = (double*)malloc(sizeof(double) * (size_t)dv);
    double* du = (double*)malloc(sizeof(double) * (size_t)dv);
    double* dov = (double*)malloc(sizeof(double) * (size_t)dv);
    int ok = ck && prev && S && hp && dS && A && dA && bv && cv && vv && r && uu && du && dov;
    if (!ok) goto done;

    for (int u = unit_begin; u < unit_end; u++) {
        int b = u / H, h = u % H;
        for (int i = 0; i < dk; i++) { A[i] = -exp(A_log[(size_t)h * dk + i]); dA[i] = 0.0; }
        /* forward sweep: keep the state entering each segment */
        if (h0) memcpy(S, h0 + (size_t)u * SZ, sizeof(double) * SZ);
        else memset(S, 0, sizeof(double) * SZ);
        for (int t = 0; t < T; t++) {
            if (t % seg == 0) memcpy(ck + (size_t)(t / seg) * SZ, S, sizeof(double) * SZ);
            for (int i = 0; i < dk; i++) bv[i] = bk[at_btHd(b, t, h, i, T, H, dk)];
            for (int j = 0; j < dv; j++) vv[j] = v[at_btHd(b, t, h, j, T, H, dv)];
            double bt = (mode == MODE_DELTA) ? beta[at_btH(b, t, h, T, H)] : 0.0;
            step(dk, dv, mode, S, A, g[at_btH(b, t, h, T, H)], bt, bv, vv, NULL, NULL, NULL);
        }
        if (dhT) memcpy(dS, dhT + (size_t)u * SZ, sizeof(double) * SZ);
        else memset(dS, 0, sizeof(double) * SZ);

        for (int n = nseg - 1; n >= 0; n--) {
            int t0 = n * seg, t1 = (t0 + seg < T) ? t0 + seg : T;
            /* recompute the segment forward, keeping h_{t-1} for every t */
            memcpy(S, ck + (size_t)n * SZ, sizeof(double) * SZ);
            for (int t = t0; t < t1; t++) {
                memcpy(prev + (size_t)(t - t0) * SZ, S, sizeof(double) * SZ);
                for (int i = 0; i < dk; i++) bv[i] = bk[at_btHd(b, t, h, i, T, H, dk)];
                for (int j = 0; j < dv; j++) vv[j] = v[at_btHd(b, t, h, j, T, H, dv)];
                double bt = (mode == MODE_DELTA) ? beta[at_btH(b, t, h, T, H)] : 0.0;
                step(dk, dv, mode, S, A, g[at_btH(b, t, h, T, H)], bt, bv, vv, NULL, NULL, NULL);
            }
            for (int t = t1 - 1; t >= t0; t--) {
                double gt = g[at_btH(b, t, h, T, H)];
                double bt = (mode == MODE_DELTA) ? beta[at_btH(b, t, h, T, H)] : 0.0;
                for (int i = 0; i < dk; i++) {
                    bv[i] = bk[at_btHd(b, t, h, i, T, H, dk)];
                    cv[i] = c[at_btHd(b, t, h, i, T, H, dk)];
                }
                for (int j = 0; j < dv; j++) {
                    vv[j] = v[at_btHd(b, t, h, j, T, H, dv)];
                    dov[j] = dO[at_btHd(b, t, h, j, T, H, dv)];
                }
                /* rebuild h', r, u and h_t from h_{t-1} */
                memcpy(S, prev + (size_t)(t - t0) * SZ, sizeof(double) * SZ);
                step(dk, dv, mode, S, A, gt, bt, bv, vv, hp, r, uu);
                /* read: o_t = h_t^T c_t */
                for (int i = 0; i < dk; i++) {
                    double acc = 0.0;
                    for (int j = 0; j < dv; j++) {
                        dS[i * dv + j] += cv[i] * dov[j];
                        acc += S[i * dv + j] * dov[j];
                    }
                    dc_out[at_btHd(b, t, h, i, T, H, dk)] = acc;
                }
                /* write: h_t = h' + b u^T */
                for (int j = 0; j < dv; j++) {
                    double acc = 0.0;
                    for (int i = 0; i < dk; i++) acc += dS[i * dv + j] * bv[i];
                    du[j] = acc;
                }
                for (int i = 0; i < dk; i++) {
                    double acc = 0.0;
                    for (int j = 0; j < dv; j++) acc += dS[i * dv + j] * uu[j];
                    db_out[at_btHd(b, t, h, i, T, H, dk)] = acc;
                }
                if (mode == MODE_DELTA) {
                    double dbt = 0.0;
                    for (int j = 0; j < dv; j++) {
                        dbt += du[j] * (vv[j] - r[j]);
                        dv_out[at_btHd(b, t, h, j, T, H, dv)] = bt * du[j];
                    }
                    dbeta_out[at_btH(b, t, h, T, H)] = dbt;
                    /* r = h'^T b: dr = -beta du */
                    for (int i = 0; i < dk; i++) {
                        double acc = 0.0;
                        for (int j = 0; j < dv; j++) {
                            double drj = -bt * du[j];
                            acc += hp[i * dv + j] * drj;
                            dS[i * dv + j] += bv[i] * drj;
                        }
                        db_out[at_btHd(b, t, h, i, T, H, dk)] += acc;
                    }
                } else {
                    for (int j = 0; j < dv; j++) dv_out[at_btHd(b, t, h, j, T, H, dv)] = du[j];
                    if (dbeta_out) dbeta_out[at_btH(b, t, h, T, H)] = 0.0;
                }
                /* decay: h' = alpha (.) h_{t-1}; alpha = exp(g A) */
                double dgt = 0.0;
                for (int i = 0; i < dk; i++) {
                    double q = 0.0;
                    for (int j = 0; j < dv; j++) q += dS[i * dv + j] * hp[i * dv + j];
                    dgt += q * A[i];
                    dA[i] += q * gt;
                    double alpha = exp(gt * A[i]);
                    for (int j = 0; j < dv; j++) dS[i * dv + j] *= alpha;
                }
                dg_out[at_btH(b, t, h, T, H)] = dgt;
            }
        }
        if (dh0) memcpy(dh0 + (size_t)u * SZ, dS, sizeof(double) * SZ);
        for (int i = 0; i < dk; i++) dA_log_unit[(size_t)u * dk + i] = dA[i] * A[i];
    }
done:
    free(ck); free(prev); free(S); free(hp); free(dS); free(A); free(dA);
    free(bv); free(cv); free(vv); free(r); free(uu); free(du); free(dov);
    return ok ? 0 : -1;
}

/*
 * Chunked restatement of the forward ("GDN & MLA Mechanism Deep-Dive",
 * Step 5: split the sequence into chunks, solve each chunk in closed form
 * with chunk x chunk matrices and carry the state between chunks).  Written
 * separately from the serial loop so the two pin each other.  Per chunk of
 * n tokens starting at t0, with G_t = sum_{r=t0..t} g_r and
 * Gam_t[i] = A[i] G_t:
 *   P[t,s] = sum_i c_t[i] b_s[i] exp(Gam_t[i] - Gam_s[i])          (s <= t)
 *   M[t,s] = beta_t sum_i b_t[i] b_s[i] exp(Gam_t[i] - Gam_s[i])   (s <  t)
 *   gated: U = V
 *   delta: (I + M) U = diag(beta) (V - Btil S),  Btil_t = b_t (.) exp(Gam_t)
 *          solved by forward substitution
 *   O  = Ctil S + P U,                Ctil_t = c_t (.) exp(Gam_t)
 *   S' = exp(Gam_last) (.)rows S + sum_s (b_s (.) exp(Gam_last - Gam_s)) u_s^T
 */
int oracle_gdn_fwd_chunked(int B, int H, int T, int dk, int dv, int mode,
                           const double* v, const double* bk, const double* c,
                           const double* g, const double* beta, const double* A_log,
                           const double* h0, double* o, double* hT, int chunk,
                           int unit_begin, int unit_end)
{
    if (bad_args(B, H, T, dk, dv, mode, unit_begin, unit_end)) return -1;
    if (mode == MODE_DELTA && !beta) return -1;
    if (chunk < 1) return -1;
    const size_t SZ = (size_t)dk * dv;
    int C = chunk;
    double* S = (double*)malloc(sizeof(double) * SZ);
    double* Sn = (double*)malloc(sizeof(double) * SZ);
    double* A = (double*)malloc(sizeof(double) * (size_t)dk);
    double* G = (double*)malloc(sizeof(double) * (size_t)C);
    double* P = (double*)malloc(sizeof(double) * (size_t)C * C);
    double* M = (double*)malloc(sizeof(double) * (size_t)C * C);
    double* U = (double*)malloc(sizeof(double) * (size_t)C * dv);
    int ok = S && Sn && A && G && P && M && U;
    if (!ok) goto done;

    for (int u = unit_begin; u < unit_end; u++) {
        int b = u / H, h = u % H;
        for (int i = 0; i < dk; i++) A[i] = -exp(A_log[(size_t)h * dk + i]);
        if (h0) memcpy(S, h0 + (size_t)u * SZ, sizeof(double) * SZ);
        else memset(S, 0, sizeof(double) * SZ);
        for (int t0 = 0; t0 < T; t0 += C) {
            int n = (t0 + C <= T) ? C : T - t0;
            double run = 0.0;
            for (int k = 0; k < n; k++) { run += g[at_btH(b, t0 + k, h, T, H)]; G[k] = run; }
            /* intra-chunk decay-masked scores */
            for (int t = 0; t < n; t++)
                for (int s = 0; s < n; s++) {
                    double p = 0.0, m = 0.0;
                    if (s <= t) {
                        for (int i = 0; i < dk; i++) {
                            double e = exp(A[i] * (G[t] - G[s]));
                            double bs = bk[at_btHd(b, t0 + s, h, i, T, H, dk)];
                            p += c[at_btHd(b, t0 + t, h, i, T, H, dk)] * bs * e;
                            if (s < t) m += bk[at_btHd(b, t0 + t, h, i, T, H, dk)] * bs * e;
                        }
                        if (mode == MODE_DELTA) m *= beta[at_btH(b, t0 + t, h, T, H)];
                    }
                    P[t * C + s] = p;
                    M[t * C + s] = (s < t) ? m : 0.0;
                }
            /* values written into the state */
            for (int t = 0; t < n; t++)
                for (int j = 0; j < dv; j++) {
                    double vt = v[at_btHd(b, t0 + t, h, j, T, H, dv)];
                    if (mode == MODE_DELTA) {
                        double bts = 0.0;
                        for (int i = 0; i < dk; i++)
                            bts += bk[at_btHd(b, t0 + t, h, i, T, H, dk)] * exp(A[i] * G[t]) * S[i * dv + j];
                        double rhs = beta[at_btH(b, t0 + t, h, T, H)] * (vt - bts);
                        for (int s = 0; s < t; s++) rhs -= M[t * C + s] * U[s * dv + j];
                        U[t * dv + j] = rhs;
                    } else {
                        U[t * dv + j] = vt;
                    }
                }
            /* outputs */
            for (int t = 0; t < n; t++)
                for (int j = 0; j < dv; j++) {
                    double acc = 0.0;
                    for (int i = 0; i < dk; i++)
                        acc += c[at_btHd(b, t0 + t, h, i, T, H, dk)] * exp(A[i] * G[t]) * S[i * dv + j];
                    for (int s = 0; s <= t; s++) acc += P[t * C + s] * U[s * dv + j];
                    o[at_btHd(b, t0 + t, h, j, T, H, dv)] = acc;
                }
            /* carry the state to the next chunk */
            for (int i = 0; i < dk; i++) {
                double dec = exp(A[i] * G[n - 1]);
                for (int j = 0; j < dv; j++) {
                    double acc = dec * S[i * dv + j];
                    for (int s = 0; s < n; s++)
                        acc += bk[at_btHd(b, t0 + s, h, i, T, H, dk)] * exp(A[i] * (G[n - 1] - G[s])) * U[s * dv + j];
                    Sn[i * dv + j] = acc;
                }
            }
            memcpy(S, Sn, sizeof(double) * SZ);
        }
        if (hT) memcpy(hT + (size_t)u * SZ, S, sizeof(double) * SZ);
    }
done:
    free(S); free(Sn); free(A); free(G); free(P); free(M); free(U);
    return ok ? 0 : -1;
}
