/*
 * favor_oracle.c -- plain, slow, float64 CPU statement of the FAVOR+ forward
 * pass.  TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the CPU
 * baseline leg of the benchmark load this; the product path never does.  It
 * shares no code, header or constant with the CUDA library.
 *
 * What it computes, and where the pages define it:
 *
 *  - feature maps (one vector x in R^d, r outputs):
 *      positive (FAVOR+):  phi(x) = exp(-|x|^2/2)/sqrt(m) [exp(w_1.x) ... exp(w_m.x)]
 *          -- "Performer: Unbiased Softmax Approximation", the phi(x) equation,
 *             and "Kernel Feature Maps", section 4 "Positive Random Features".
 *      trig (random Fourier): phi(x) = 1/sqrt(m) [sin(w_1.x), cos(w_1.x), ...,
 *             sin(w_m.x), cos(w_m.x)]  (r = 2m, interleaved as printed)
 *          -- "Kernel Feature Maps", section 3 "Random Fourier Features".
 *      elu1: phi(x)_j = x_j + 1 if x_j > 0, exp(x_j) otherwise  (r = d, no w)
 *          -- "Kernel Feature Maps", section 1 "ELU + 1".
 *  - non-causal contraction (eps = 0):
 *      KV = phi(K)^T V,  z = sum_j phi(k_j),  out_i = phi(q_i)^T KV / phi(q_i)^T z
 *          -- "Performer: Unbiased Softmax Approximation", In[25] (the
 *             performer_attention statement of the math), and the Performer
 *             study notes, "Core points" steps 4-5 (reordering, linear
 *             denominator).
 *  - causal form, the literal token recurrence:
 *      S_i = S_{i-1} + phi(k_i) v_i^T,  z_i = z_{i-1} + phi(k_i),
 *      out_i = phi(q_i)^T S_i / phi(q_i)^T z_i   (diagonal j = i included)
 *          -- Performer study notes, "Case 2: the causal version" (prefix sum),
 *             with the denominator of "Core points" step 5.
 *  - carried state and one decode step (the same recurrence, one token at
 *    a time): state(K, V) = (S_L, z_L) after L keys; a step takes (S, z) and
 *    one (q, k, v), forms S + phi(k) v^T, z + phi(k), and returns them with
 *    out = phi(q)^T S' / phi(q)^T z'
 *          -- Performer study notes, "Case 2" (S_i, z_i are running sums;
 *             each step costs O(r d)).
 *
 * No stabiliser, no blocking, no reordering: every value is the definition
 * evaluated in float64.  Exponents are checked against |t| < 700.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_MAP_POSITIVE 0
#define ORACLE_MAP_TRIG 1
#define ORACLE_MAP_ELU1 2

/* feature count r for a map */
int oracle_feature_dim(int map, int d, int m)
{
    if (map == ORACLE_MAP_TRIG) return 2 * m;
    if (map == ORACLE_MAP_ELU1) return d;
    return m;
}

/* phi of n vectors x[n][d] with projection omega[m][d] -> phi[n][r].
 * Returns 0, or -1 for an unknown map, -2 if an exponent left |t| < 700. */
int oracle_features(const double *x, const double *omega, int n, int d, int m,
                    int map, double *phi)
{
    int r = oracle_feature_dim(map, d, m);
    for (int t = 0; t < n; ++t) {
        const double *xt = x + (size_t)t * d;
        double *pt = phi + (size_t)t * r;
        if (map == ORACLE_MAP_ELU1) {
            for (int j = 0; j < d; ++j) {
                double v = xt[j];
                if (v < -700.0) return -2;
                pt[j] = v > 0.0 ? v + 1.0 : exp(v);
            }
            continue;
        }
        double norm2 = 0.0;
        for (int j = 0; j < d; ++j) norm2 += xt[j] * xt[j];
        double scale = 1.0 / sqrt((double)m);
        double pref = exp(-norm2 / 2.0) * scale;
        for (int i = 0; i < m; ++i) {
            const double *wi = omega + (size_t)i * d;
            double proj = 0.0;
            for (int j = 0; j < d; ++j) proj += wi[j] * xt[j];
            if (map == ORACLE_MAP_POSITIVE) {
                if (fabs(proj) >= 700.0 || norm2 / 2.0 >= 700.0) return -2;
                pt[i] = pref * exp(proj);
            } else if (map == ORACLE_MAP_TRIG) {
                pt[2 * i] = scale * sin(proj);
                pt[2 * i + 1] = scale * cos(proj);
            } else {
                return -1;
            }
        }
    }
    return 0;
}

/* One head: q[L][d], k[L][d], v[L][dv], omega[m][d] -> out[L][dv].
 * den_out (optional, may be NULL) receives the denominator of each row. */
static int oracle_head(const double *q, const double *k, const double *v,
                       const double *omega, double *out, double *den_out,
                       int L, int d, int dv, int m, int causal, int map)
{
    int r = oracle_feature_dim(map, d, m);
    double *phik = (double *)malloc(sizeof(double) * (size_t)r);
    double *phiq = (double *)malloc(sizeof(double) * (size_t)r);
    double *S = (double *)calloc((size_t)r * dv, sizeof(double));
    double *z = (double *)calloc((size_t)r, sizeof(double));
    int rc = 0;
    if (!phik || !phiq || !S || !z) { rc = -3; goto done; }

    if (!causal) {
        /* KV = phi(K)^T V, z = phi(K)^T 1 over all L keys */
        for (int j = 0; j < L; ++j) {
            rc = oracle_features(k + (size_t)j * d, omega, 1, d, m, map, phik);
            if (rc) goto done;
            const double *vj = v + (size_t)j * dv;
            for (int f = 0; f < r; ++f) {
                double a = phik[f];
                double *Sf = S + (size_t)f * dv;
                for (int c = 0; c < dv; ++c) Sf[c] += a * vj[c];
                z[f] += a;
            }
        }
    }
    for (int i = 0; i < L; ++i) {
        if (causal) {
            /* S_i = S_{i-1} + phi(k_i) v_i^T ; z_i = z_{i-1} + phi(k_i) */
            rc = oracle_features(k + (size_t)i * d, omega, 1, d, m, map, phik);
            if (rc) goto done;
            const double *vi = v + (size_t)i * dv;
            for (int f = 0; f < r; ++f) {
                double a = phik[f];
                double *Sf = S + (size_t)f * dv;
                for (int c = 0; c < dv; ++c) Sf[c] += a * vi[c];
                z[f] += a;
            }
        }
        rc = oracle_features(q + (size_t)i * d, omega, 1, d, m, map, phiq);
        if (rc) goto done;
        double den = 0.0;
        for (int f = 0; f < r; ++f) den += phiq[f] * z[f];
        double *oi = out + (size_t)i * dv;
        for (int c = 0; c < dv; ++c) oi[c] = 0.0;
        for (int f = 0; f < r; ++f) {
            double a = phiq[f];
            const double *Sf = S + (size_t)f * dv;
            for (int c = 0; c < dv; ++c) oi[c] += a * Sf[c];
        }
        for (int c = 0; c < dv; ++c) oi[c] = oi[c] / den;
        if (den_out) den_out[i] = den;
    }
done:
    free(phik); free(phiq); free(S); free(z);
    return rc;
}

/* Full forward over B*H heads.  q,k [B][H][L][d], v/out [B][H][L][dv],
 * omega [H][m][d] (ignored for elu1).  heads: optional list of n_heads flat
 * head indices (b*H + h) to evaluate; NULL means all.  Only the rows of the
 * listed heads are written.  den (optional) is [B][H][L].
 * Returns 0, or the first non-zero head status. */
int oracle_forward(const double *q, const double *k, const double *v,
                   const double *omega, double *out, double *den,
                   int B, int H, int L, int d, int dv, int m, int causal, int map,
                   const int *heads, int n_heads)
{
    int total = heads ? n_heads : B * H;
    int status = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (int t = 0; t < total; ++t) {
        int bh = heads ? heads[t] : t;
        int h = bh % H;
        size_t xo = (size_t)bh * L * d, vo = (size_t)bh * L * dv;
        const double *om = omega ? omega + (size_t)h * m * d : NULL;
        int rc = oracle_head(q + xo, k + xo, v + vo, om, out + vo,
                             den ? den + (size_t)bh * L : NULL,
                             L, d, dv, m, causal, map);
        if (rc) {
#pragma omp critical
            { if (!status) status = rc; }
        }
    }
    return status;
}

/* Carried state after the L keys of every head: S[B][H][r][dv] = sum_j
 * phi(k_j) v_j^T, z[B][H][r] = sum_j phi(k_j) (Performer study notes,
 * "Case 2": the prefix sums at i = L).  Returns 0 or the first head status. */
int oracle_state(const double *k, const double *v, const double *omega, double *S, double *z,
                 int B, int H, int L, int d, int dv, int m, int map)
{
    int r = oracle_feature_dim(map, d, m);
    int status = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (int bh = 0; bh < B * H; ++bh) {
        const double *om = omega ? omega + (size_t)(bh % H) * m * d : NULL;
        double *Sh = S + (size_t)bh * r * dv, *zh = z + (size_t)bh * r;
        double *phik = (double *)malloc(sizeof(double) * (size_t)r);
        int rc = phik ? 0 : -3;
        for (size_t i = 0; i < (size_t)r * dv; ++i) Sh[i] = 0.0;
        for (int f = 0; f < r; ++f) zh[f] = 0.0;
        for (int j = 0; j < L && !rc; ++j) {
            rc = oracle_features(k + ((size_t)bh * L + j) * d, om, 1, d, m, map, phik);
            if (rc) break;
            const double *vj = v + ((size_t)bh * L + j) * dv;
            for (int f = 0; f < r; ++f) {
                for (int c = 0; c < dv; ++c) Sh[(size_t)f * dv + c] += phik[f] * vj[c];
                zh[f] += phik[f];
            }
        }
        free(phik);
        if (rc) {
#pragma omp critical
            { if (!status) status = rc; }
        }
    }
    return status;
}

/* One decode step for every head, in place: S += phi(k) v^T, z += phi(k),
 * then out = phi(q)^T S / phi(q)^T z with the updated state (the diagonal
 * term included, as in the causal recurrence).  q, k [B][H][d], v, out
 * [B][H][dv], S [B][H][r][dv], z [B][H][r]. */
int oracle_decode_step(const double *q, const double *k, const double *v, const double *omega,
                       double *S, double *z, double *out, int B, int H, int d, int dv, int m, int map)
{
    int r = oracle_feature_dim(map, d, m);
    double *phik = (double *)malloc(sizeof(double) * (size_t)r);
    double *phiq = (double *)malloc(sizeof(double) * (size_t)r);
    int rc = (phik && phiq) ? 0 : -3;
    for (int bh = 0; bh < B * H && !rc; ++bh) {
        const double *om = omega ? omega + (size_t)(bh % H) * m * d : NULL;
        double *Sh = S + (size_t)bh * r * dv, *zh = z + (size_t)bh * r;
        const double *vh = v + (size_t)bh * dv;
        double *oh = out + (size_t)bh * dv;
        rc = oracle_features(k + (size_t)bh * d, om, 1, d, m, map, phik);
        if (!rc) rc = oracle_features(q + (size_t)bh * d, om, 1, d, m, map, phiq);
        if (rc) break;
        for (int f = 0; f < r; ++f) {
            for (int c = 0; c < dv; ++c) Sh[(size_t)f * dv + c] += phik[f] * vh[c];
            zh[f] += phik[f];
        }
        double den = 0.0;
        for (int f = 0; f < r; ++f) den += phiq[f] * zh[f];
        for (int c = 0; c < dv; ++c) {
            double num = 0.0;
            for (int f = 0; f < r; ++f) num += phiq[f] * Sh[(size_t)f * dv + c];
            oh[c] = num / den;
        }
    }
    free(phik); free(phiq);
    return rc;
}
