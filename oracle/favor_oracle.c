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
 *      relu: phi(x)_j = max(0, x_j)  (r = d, no w)
 *          -- "Kernel Feature Maps", section 2 "ReLU".
 *      softmax-scaled trig: exp(|x|^2/2) times the trig map, so that
 *          E[phi(q).phi(k)] = exp(|q|^2/2 + |k|^2/2 - |q-k|^2/2) = exp(q.k)
 *          -- "Kernel Feature Maps", section 3 (the remark that with an
 *             additional scaling the Fourier features approximate the
 *             softmax kernel; the scaling read as the Gaussian identity).
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
 *  - random projections drawn from a counter-based generator (the draw the
 *    library also makes on the device; the pages leave the generator open):
 *      Philox4x64-10 -- Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers:
 *        As Easy as 1, 2, 3" (SC 2011): ten rounds of two 64x64->128-bit
 *        products with the counter words crossed and the key xored in, the
 *        key bumped by the Weyl constants between rounds;
 *      Box-Muller normals from pairs of 53-bit uniforms in (0, 1);
 *      iid rows w_i ~ N(0, I_d) ("Performer: Unbiased Softmax Approximation",
 *        the w ~ N(0, I) draw), or block-orthogonal rows: per head ceil(m/d)
 *        Gaussian d x d blocks, rows orthonormalised by modified Gram-Schmidt
 *        and scaled by the norm of an independent N(0, I_d) vector, the last
 *        block truncated (the orthogonal random features the Performer study
 *        notes name, read as in the block construction).
 *  - the backward pass of the forward above (gradients of a loss given
 *    g = dloss/dout), the reverse sweep of the prefix sums the Performer study
 *    notes ask for ("Case 2"; the prefix sums accumulated in reverse):
 *      dnum_i = g_i / den_i,  dden_i = -(g_i . out_i) / den_i
 *      dphi(q_i) = S_i dnum_i + z_i dden_i             (S_i, z_i as above)
 *      R_j = sum_{i >= j} phi(q_i) dnum_i^T,  rho_j = sum_{i >= j} phi(q_i) dden_i
 *      dphi(k_j) = R_j v_j + rho_j,  dv_j = R_j^T phi(k_j)
 *    (non-causal: S, z, R, rho over all rows), then through each feature
 *    map's derivative to dq, dk and dw (w shared by the batch: summed).
 *
 * No stabiliser, no blocking, no reordering: every value is the definition
 * evaluated in float64.  Exponents are checked against |t| < 700.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_MAP_POSITIVE 0
#define ORACLE_MAP_TRIG 1
#define ORACLE_MAP_ELU1 2
#define ORACLE_MAP_RELU 3
#define ORACLE_MAP_TRIG_SOFTMAX 4

/* feature count r for a map */
int oracle_feature_dim(int map, int d, int m)
{
    if (map == ORACLE_MAP_TRIG || map == ORACLE_MAP_TRIG_SOFTMAX) return 2 * m;
    if (map == ORACLE_MAP_ELU1 || map == ORACLE_MAP_RELU) return d;
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
        if (map == ORACLE_MAP_RELU) {
            for (int j = 0; j < d; ++j) pt[j] = xt[j] > 0.0 ? xt[j] : 0.0;
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
            } else if (map == ORACLE_MAP_TRIG_SOFTMAX) {
                if (norm2 / 2.0 >= 700.0) return -2;
                const double g = exp(norm2 / 2.0) * scale;
                pt[2 * i] = g * sin(proj);
                pt[2 * i + 1] = g * cos(proj);
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

/* ---- random projections ------------------------------------------------ */

/* one Philox4x64-10 block: out = f_key(ctr) */
void oracle_philox4x64(const uint64_t ctr[4], const uint64_t key[2], uint64_t out[4])
{
    const uint64_t M0 = 0xD2E7470EE14C6C93ULL, M1 = 0xCA5A826395121157ULL;
    const uint64_t W0 = 0x9E3779B97F4A7C15ULL, W1 = 0xBB67AE8584CAA73BULL;
    uint64_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
    uint64_t k0 = key[0], k1 = key[1];
    for (int round = 0; round < 10; ++round) {
        if (round > 0) { k0 += W0; k1 += W1; }
        unsigned __int128 p0 = (unsigned __int128)M0 * c0;
        unsigned __int128 p1 = (unsigned __int128)M1 * c2;
        uint64_t hi0 = (uint64_t)(p0 >> 64), lo0 = (uint64_t)p0;
        uint64_t hi1 = (uint64_t)(p1 >> 64), lo1 = (uint64_t)p1;
        uint64_t n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
        c0 = n0; c1 = lo1; c2 = n2; c3 = lo0;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* normal number e of stream s: block (e / 4, s, 0, 0) under key (seed, 0);
 * words (x0, x1) give normals 0, 1 and (x2, x3) normals 2, 3 by Box-Muller
 * with u = (x / 2^11 + 1/2) 2^-53 */
double oracle_normal(uint64_t seed, uint64_t stream, uint64_t e)
{
    const uint64_t ctr[4] = {e >> 2, stream, 0, 0}, key[2] = {seed, 0};
    uint64_t x[4];
    oracle_philox4x64(ctr, key, x);
    const int pair = (int)((e >> 1) & 1), which = (int)(e & 1);
    const double u1 = ((double)(x[2 * pair] >> 11) + 0.5) * 0x1p-53;
    const double u2 = ((double)(x[2 * pair + 1] >> 11) + 0.5) * 0x1p-53;
    const double rad = sqrt(-2.0 * log(u1)), ang = 2.0 * 3.14159265358979323846 * u2;
    return which ? rad * sin(ang) : rad * cos(ang);
}

/* omega [H][m][d] in float64: kind 0 iid, kind 1 block-orthogonal.
 * Returns 0, -1 for bad arguments, -3 on allocation failure. */
int oracle_draw_omega(double *omega, int H, int m, int d, int kind, uint64_t seed)
{
    if (H < 1 || m < 1 || d < 1 || (kind != 0 && kind != 1)) return -1;
    if (kind == 0) {
        for (uint64_t e = 0; e < (uint64_t)H * m * d; ++e) omega[e] = oracle_normal(seed, 0, e);
        return 0;
    }
    const int nb = (m + d - 1) / d;
    double *G = (double *)malloc(sizeof(double) * (size_t)d * d);
    if (!G) return -3;
    for (int h = 0; h < H; ++h)
        for (int b = 0; b < nb; ++b) {
            const uint64_t base = ((uint64_t)h * nb + b) * d * d;
            for (int i = 0; i < d * d; ++i) G[i] = oracle_normal(seed, 0, base + i);
            /* modified Gram-Schmidt on the rows, in row order */
            for (int i = 0; i < d; ++i) {
                double *v = G + (size_t)i * d;
                for (int j = 0; j < i; ++j) {
                    const double *qj = G + (size_t)j * d;
                    double dot = 0.0;
                    for (int t = 0; t < d; ++t) dot += v[t] * qj[t];
                    for (int t = 0; t < d; ++t) v[t] -= dot * qj[t];
                }
                double nrm = 0.0;
                for (int t = 0; t < d; ++t) nrm += v[t] * v[t];
                nrm = sqrt(nrm);
                for (int t = 0; t < d; ++t) v[t] /= nrm;
            }
            for (int i = 0; i < d && b * d + i < m; ++i) {
                double ss = 0.0;
                for (int t = 0; t < d; ++t) {
                    const double g = oracle_normal(seed, 1, base + (uint64_t)i * d + t);
                    ss += g * g;
                }
                const double chi = sqrt(ss);
                double *dst = omega + ((size_t)h * m + (size_t)b * d + i) * d;
                for (int t = 0; t < d; ++t) dst[t] = G[(size_t)i * d + t] * chi;
            }
        }
    free(G);
    return 0;
}

/* ---- backward ------------------------------------------------------------ */

/* dphi (r values) -> dx (d values) for one vector x; dw [m][d] += the
 * projection rows' gradient.  Feature derivatives:
 *   positive:  dphi_i/dx = phi_i (w_i - x),  dphi_i/dw_i = phi_i x
 *   trig:      phi_{2i} = sin(a)/sqrt(m), phi_{2i+1} = cos(a)/sqrt(m), a = w_i.x
 *   softmax-scaled trig: exp(|x|^2/2) times trig: adds x (sum_f dphi_f phi_f)
 *   elu1:      1 (x > 0), exp(x);   relu: 1 (x > 0), 0 */
static int feature_backward(const double *x, const double *omega, const double *dphi, double *dx,
                            double *dw, int d, int m, int map)
{
    int r = oracle_feature_dim(map, d, m);
    double *phi = (double *)malloc(sizeof(double) * (size_t)r);
    if (!phi) return -3;
    int rc = oracle_features(x, omega, 1, d, m, map, phi);
    if (rc) { free(phi); return rc; }
    for (int j = 0; j < d; ++j) dx[j] = 0.0;
    if (map == ORACLE_MAP_ELU1 || map == ORACLE_MAP_RELU) {
        for (int j = 0; j < d; ++j) {
            double der = x[j] > 0.0 ? 1.0 : (map == ORACLE_MAP_ELU1 ? exp(x[j]) : 0.0);
            dx[j] = dphi[j] * der;
        }
        free(phi);
        return 0;
    }
    if (map == ORACLE_MAP_POSITIVE) {
        double tot = 0.0;
        for (int i = 0; i < m; ++i) {
            double c = dphi[i] * phi[i];
            tot += c;
            const double *wi = omega + (size_t)i * d;
            for (int j = 0; j < d; ++j) {
                dx[j] += c * wi[j];
                dw[(size_t)i * d + j] += c * x[j];
            }
        }
        for (int j = 0; j < d; ++j) dx[j] -= tot * x[j];
        free(phi);
        return 0;
    }
    /* trig and its softmax-scaled form: phi = s [sin a_i, cos a_i] with
     * s = 1/sqrt(m) (times exp(|x|^2/2) when scaled) */
    double norm2 = 0.0;
    for (int j = 0; j < d; ++j) norm2 += x[j] * x[j];
    double s = 1.0 / sqrt((double)m);
    if (map == ORACLE_MAP_TRIG_SOFTMAX) s *= exp(norm2 / 2.0);
    double tot = 0.0;
    for (int i = 0; i < m; ++i) {
        const double *wi = omega + (size_t)i * d;
        double a = 0.0;
        for (int j = 0; j < d; ++j) a += wi[j] * x[j];
        double c = s * (dphi[2 * i] * cos(a) - dphi[2 * i + 1] * sin(a));
        tot += dphi[2 * i] * phi[2 * i] + dphi[2 * i + 1] * phi[2 * i + 1];
        for (int j = 0; j < d; ++j) {
            dx[j] += c * wi[j];
            dw[(size_t)i * d + j] += c * x[j];
        }
    }
    if (map == ORACLE_MAP_TRIG_SOFTMAX)
        for (int j = 0; j < d; ++j) dx[j] += tot * x[j];
    free(phi);
    return 0;
}

/* One head: gradients dq, dk [L][d], dv [L][dv] and dw [m][d] (accumulated). */
static int oracle_head_backward(const double *q, const double *k, const double *v, const double *omega,
                                const double *g, double *dq, double *dk, double *dv, double *dw,
                                int L, int d, int dvd, int m, int causal, int map)
{
    int r = oracle_feature_dim(map, d, m);
    double *pk = (double *)malloc(sizeof(double) * (size_t)L * r);
    double *pq = (double *)malloc(sizeof(double) * (size_t)L * r);
    double *S = (double *)calloc((size_t)r * dvd, sizeof(double));
    double *z = (double *)calloc((size_t)r, sizeof(double));
    double *dnum = (double *)malloc(sizeof(double) * (size_t)L * dvd);
    double *dden = (double *)malloc(sizeof(double) * (size_t)L);
    double *dphi = (double *)malloc(sizeof(double) * (size_t)r);
    double *R = (double *)calloc((size_t)r * dvd, sizeof(double));
    double *rho = (double *)calloc((size_t)r, sizeof(double));
    int rc = 0;
    if (!pk || !pq || !S || !z || !dnum || !dden || !dphi || !R || !rho) { rc = -3; goto done; }
    if ((rc = oracle_features(k, omega, L, d, m, map, pk))) goto done;
    if ((rc = oracle_features(q, omega, L, d, m, map, pq))) goto done;
    if (!causal)
        for (int j = 0; j < L; ++j)
            for (int f = 0; f < r; ++f) {
                for (int c = 0; c < dvd; ++c) S[(size_t)f * dvd + c] += pk[(size_t)j * r + f] * v[(size_t)j * dvd + c];
                z[f] += pk[(size_t)j * r + f];
            }
    /* forward sweep: out_i, dnum_i, dden_i and dphi(q_i) */
    for (int i = 0; i < L; ++i) {
        if (causal)
            for (int f = 0; f < r; ++f) {
                for (int c = 0; c < dvd; ++c) S[(size_t)f * dvd + c] += pk[(size_t)i * r + f] * v[(size_t)i * dvd + c];
                z[f] += pk[(size_t)i * r + f];
            }
        const double *ph = pq + (size_t)i * r;
        double den = 0.0;
        for (int f = 0; f < r; ++f) den += ph[f] * z[f];
        double gdo = 0.0;
        for (int c = 0; c < dvd; ++c) {
            double num = 0.0;
            for (int f = 0; f < r; ++f) num += ph[f] * S[(size_t)f * dvd + c];
            gdo += g[(size_t)i * dvd + c] * (num / den);
            dnum[(size_t)i * dvd + c] = g[(size_t)i * dvd + c] / den;
        }
        dden[i] = -gdo / den;
        for (int f = 0; f < r; ++f) {
            double acc = z[f] * dden[i];
            for (int c = 0; c < dvd; ++c) acc += S[(size_t)f * dvd + c] * dnum[(size_t)i * dvd + c];
            dphi[f] = acc;
        }
        if ((rc = feature_backward(q + (size_t)i * d, omega, dphi, dq + (size_t)i * d, dw, d, m, map))) goto done;
    }
    /* reverse sweep: R_j, rho_j; dphi(k_j) and dv_j */
    if (!causal)
        for (int i = 0; i < L; ++i)
            for (int f = 0; f < r; ++f) {
                for (int c = 0; c < dvd; ++c) R[(size_t)f * dvd + c] += pq[(size_t)i * r + f] * dnum[(size_t)i * dvd + c];
                rho[f] += pq[(size_t)i * r + f] * dden[i];
            }
    for (int j = L - 1; j >= 0; --j) {
        if (causal)
            for (int f = 0; f < r; ++f) {
                for (int c = 0; c < dvd; ++c) R[(size_t)f * dvd + c] += pq[(size_t)j * r + f] * dnum[(size_t)j * dvd + c];
                rho[f] += pq[(size_t)j * r + f] * dden[j];
            }
        for (int f = 0; f < r; ++f) {
            double acc = rho[f];
            for (int c = 0; c < dvd; ++c) acc += R[(size_t)f * dvd + c] * v[(size_t)j * dvd + c];
            dphi[f] = acc;
        }
        for (int c = 0; c < dvd; ++c) {
            double acc = 0.0;
            for (int f = 0; f < r; ++f) acc += R[(size_t)f * dvd + c] * pk[(size_t)j * r + f];
            dv[(size_t)j * dvd + c] = acc;
        }
        if ((rc = feature_backward(k + (size_t)j * d, omega, dphi, dk + (size_t)j * d, dw, d, m, map))) goto done;
    }
done:
    free(pk); free(pq); free(S); free(z); free(dnum); free(dden); free(dphi); free(R); free(rho);
    return rc;
}

/* Backward over B*H heads: g [B][H][L][dv] -> dq, dk [B][H][L][d],
 * dv [B][H][L][dv], dw [H][m][d] (summed over the batch; may be NULL for the
 * elementwise maps). */
int oracle_backward(const double *q, const double *k, const double *v, const double *omega,
                    const double *g, double *dq, double *dk, double *dv, double *dw,
                    int B, int H, int L, int d, int dvd, int m, int causal, int map)
{
    int status = 0;
    const int has_w = !(map == ORACLE_MAP_ELU1 || map == ORACLE_MAP_RELU);
    if (has_w) memset(dw, 0, sizeof(double) * (size_t)H * m * d);
    /* heads of one h share dw: parallel over h, sequential over b */
#pragma omp parallel for schedule(dynamic, 1)
    for (int h = 0; h < H; ++h) {
        double *dwh = has_w ? dw + (size_t)h * m * d : NULL;
        double *scratch = has_w ? NULL : (double *)calloc((size_t)m * d, sizeof(double));
        for (int b = 0; b < B; ++b) {
            size_t bh = (size_t)b * H + h;
            size_t xo = bh * L * d, vo = bh * L * dvd;
            const double *om = has_w ? omega + (size_t)h * m * d : NULL;
            int rc = oracle_head_backward(q + xo, k + xo, v + vo, om, g + vo, dq + xo, dk + xo, dv + vo,
                                          has_w ? dwh : scratch, L, d, dvd, m, causal, map);
            if (rc) {
#pragma omp critical
                { if (!status) status = rc; }
            }
        }
        free(scratch);
    }
    return status;
}
