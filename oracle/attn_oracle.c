/*
 * attn_oracle.c -- fp64 CPU oracle for exact scaled-dot-product attention.
 *
 * TEST INFRASTRUCTURE ONLY (see attn_oracle.h). Plain, slow, obviously correct:
 * every score row is materialised in fp64 and the softmax is taken over it.
 *
 * Definition followed ([Streaming] = "FlashAttention: Exact Attention as an
 * IO-Aware Streaming Computation", section "Problem setting"; [Glossary] =
 * "FlashAttention", section "Move less data"):
 *     s_ij = scale * <q_i, k_j> + M[i][j]     (-inf where causality excludes j)
 *     o_i  = sum_j exp(s_ij) v_j / sum_j exp(s_ij)
 * evaluated with the row maximum subtracted ([Streaming], "Mathematical
 * structure": m_i is the stabilising row maximum), and lse_i = m_i + ln l_i.
 */
#include "attn_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Is key j visible to query i? Causal alignment puts the last query on the last
 * key, which for Nq == Nk is j <= i. */
static int key_allowed(int64_t i, int64_t j, int64_t Nq, int64_t Nk, int causal) {
    if (!causal) return 1;
    return j <= i + (Nk - Nq);
}

/* Scaled, masked scores of query row (b, h, i) against all Nk keys. */
static void score_row(const double *q, const double *k, const double *mask, int64_t H, int64_t Nq,
                      int64_t Nk, int64_t d, double scale, int causal, int64_t b, int64_t h, int64_t i,
                      double *s) {
    const double *qi = q + ((b * H + h) * Nq + i) * d;
    const double *kb = k + (b * H + h) * Nk * d;
    for (int64_t j = 0; j < Nk; ++j) {
        if (!key_allowed(i, j, Nq, Nk, causal)) {
            s[j] = -INFINITY;
            continue;
        }
        double dot = 0.0;
        for (int64_t t = 0; t < d; ++t) dot += qi[t] * kb[j * d + t];
        double sij = scale * dot;
        if (mask) sij += mask[(b * Nq + i) * Nk + j];
        s[j] = sij;
    }
}

/* Softmax-weighted sum over the materialised row s[0..Nk). */
static void attend_row(const double *v, int64_t H, int64_t Nk, int64_t d, int64_t b, int64_t h,
                       const double *s, double *o, double *lse) {
    const double *vb = v + (b * H + h) * Nk * d;
    double m = -INFINITY;
    for (int64_t j = 0; j < Nk; ++j)
        if (s[j] > m) m = s[j];
    for (int64_t t = 0; t < d; ++t) o[t] = 0.0;
    if (m == -INFINITY) { /* every key masked: the convention is o = 0, lse = -inf */
        *lse = -INFINITY;
        return;
    }
    double l = 0.0;
    for (int64_t j = 0; j < Nk; ++j) {
        double p = exp(s[j] - m);
        if (p == 0.0) continue;
        l += p;
        for (int64_t t = 0; t < d; ++t) o[t] += p * vb[j * d + t];
    }
    for (int64_t t = 0; t < d; ++t) o[t] /= l;
    *lse = m + log(l);
}

static int bad_args(const double *q, const double *k, const double *v, int64_t B, int64_t H,
                    int64_t Nq, int64_t Nk, int64_t d) {
    return !q || !k || !v || B < 0 || H < 0 || Nq < 0 || Nk < 0 || d < 1;
}

int oracle_attn_rows_f64(const double *q, const double *k, const double *v, const double *mask,
                         double *out, double *lse, int64_t B, int64_t H, int64_t Nq, int64_t Nk,
                         int64_t d, double scale, int causal, const int64_t *rows, int64_t nrows) {
    if (bad_args(q, k, v, B, H, Nq, Nk, d) || !out || !lse || (nrows > 0 && !rows)) return -1;
    const int64_t total = B * H * Nq;
    for (int64_t r = 0; r < nrows; ++r)
        if (rows[r] < 0 || rows[r] >= total) return -1;
    int err = 0;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(Nk > 0 ? Nk : 1));
        if (!s) {
#pragma omp atomic write
            err = 1;
        }
#pragma omp for schedule(dynamic, 8)
        for (int64_t r = 0; r < nrows; ++r) {
            if (!s) continue;
            const int64_t row = rows[r];
            const int64_t i = row % Nq, bh = row / Nq;
            const int64_t b = bh / H, h = bh % H;
            score_row(q, k, mask, H, Nq, Nk, d, scale, causal, b, h, i, s);
            attend_row(v, H, Nk, d, b, h, s, out + r * d, lse + r);
        }
        free(s);
    }
    return err ? -1 : 0;
}

int oracle_attn_f64(const double *q, const double *k, const double *v, const double *mask,
                    double *out, double *lse, int64_t B, int64_t H, int64_t Nq, int64_t Nk,
                    int64_t d, double scale, int causal) {
    if (bad_args(q, k, v, B, H, Nq, Nk, d) || !out || !lse) return -1;
    const int64_t total = B * H * Nq;
    int64_t *rows = (int64_t *)malloc(sizeof(int64_t) * (size_t)(total > 0 ? total : 1));
    if (!rows) return -1;
    for (int64_t r = 0; r < total; ++r) rows[r] = r;
    int rc = oracle_attn_rows_f64(q, k, v, mask, out, lse, B, H, Nq, Nk, d, scale, causal, rows, total);
    free(rows);
    return rc;
}

/* ---- blockwise summaries and their merge ([Glossary], "Why a tile can be
 * discarded" and "One row, checked two ways") ---------------------------- */

void oracle_block_summary_f64(const double *s, const double *vals, int64_t n, int64_t dv, double *m,
                              double *l, double *u) {
    double mx = -INFINITY;
    for (int64_t j = 0; j < n; ++j)
        if (s[j] > mx) mx = s[j];
    for (int64_t t = 0; t < dv; ++t) u[t] = 0.0;
    *m = mx;
    *l = 0.0;
    if (mx == -INFINITY) return; /* a fully masked block contributes nothing */
    for (int64_t j = 0; j < n; ++j) {
        double p = exp(s[j] - mx);
        *l += p;
        for (int64_t t = 0; t < dv; ++t) u[t] += p * vals[j * dv + t];
    }
}

void oracle_merge_f64(double mA, double lA, const double *uA, double mB, double lB, const double *uB,
                      int64_t dv, double *m, double *l, double *u) {
    double mx = mA > mB ? mA : mB;
    if (mx == -INFINITY) { /* both empty: never form (-inf) - (-inf) */
        *m = -INFINITY;
        *l = 0.0;
        for (int64_t t = 0; t < dv; ++t) u[t] = 0.0;
        return;
    }
    /* Each side is re-expressed relative to the common maximum. */
    double fa = (mA == -INFINITY) ? 0.0 : exp(mA - mx);
    double fb = (mB == -INFINITY) ? 0.0 : exp(mB - mx);
    *l = fa * lA + fb * lB;
    for (int64_t t = 0; t < dv; ++t) u[t] = fa * uA[t] + fb * uB[t];
    *m = mx;
}

int oracle_attn_blockwise_f64(const double *q, const double *k, const double *v, const double *mask,
                              double *out, double *lse, int64_t B, int64_t H, int64_t Nq, int64_t Nk,
                              int64_t d, double scale, int causal, int64_t block) {
    if (bad_args(q, k, v, B, H, Nq, Nk, d) || !out || !lse || block < 1) return -1;
    const int64_t total = B * H * Nq;
    int err = 0;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(Nk > 0 ? Nk : 1));
        double *ub = (double *)malloc(sizeof(double) * (size_t)d);
        double *ur = (double *)malloc(sizeof(double) * (size_t)d);
        if (!s || !ub || !ur) {
#pragma omp atomic write
            err = 1;
        }
#pragma omp for schedule(dynamic, 8)
        for (int64_t row = 0; row < total; ++row) {
            if (!s || !ub || !ur) continue;
            const int64_t i = row % Nq, bh = row / Nq;
            const int64_t b = bh / H, h = bh % H;
            const double *vb = v + bh * Nk * d;
            score_row(q, k, mask, H, Nq, Nk, d, scale, causal, b, h, i, s);
            double mr = -INFINITY, lr = 0.0;
            for (int64_t t = 0; t < d; ++t) ur[t] = 0.0;
            for (int64_t j0 = 0; j0 < Nk; j0 += block) {
                int64_t n = (Nk - j0 < block) ? Nk - j0 : block;
                double mb, lb;
                oracle_block_summary_f64(s + j0, vb + j0 * d, n, d, &mb, &lb, ub);
                oracle_merge_f64(mr, lr, ur, mb, lb, ub, d, &mr, &lr, ur);
            }
            double *o = out + row * d;
            if (lr == 0.0) {
                for (int64_t t = 0; t < d; ++t) o[t] = 0.0;
                lse[row] = -INFINITY;
            } else {
                for (int64_t t = 0; t < d; ++t) o[t] = ur[t] / lr;
                lse[row] = mr + log(lr);
            }
        }
        free(s);
        free(ub);
        free(ur);
    }
    return err ? -1 : 0;
}

/* ---- backward of the materialised definition ------------------------------
 * With P = softmax(S) row-wise and O = P V, for the scalar sum(dO * O):
 *   dV = P^T dO,  dP = dO V^T,  dS_ij = P_ij (dP_ij - sum_t P_it dP_it),
 *   dQ = scale * dS K,  dK = scale * dS^T Q.
 * Each (b, h) is one task, so dk and dv accumulate without races. */
int oracle_attn_bwd_f64(const double *q, const double *k, const double *v, const double *mask,
                        const double *dout, double *dq, double *dk, double *dv, int64_t B, int64_t H,
                        int64_t Nq, int64_t Nk, int64_t d, double scale, int causal) {
    if (bad_args(q, k, v, B, H, Nq, Nk, d) || !dout || !dq || !dk || !dv) return -1;
    int err = 0;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(Nk > 0 ? Nk : 1));
        double *dp = (double *)malloc(sizeof(double) * (size_t)(Nk > 0 ? Nk : 1));
        if (!s || !dp) {
#pragma omp atomic write
            err = 1;
        }
#pragma omp for schedule(dynamic, 1)
        for (int64_t bh = 0; bh < B * H; ++bh) {
            if (!s || !dp) continue;
            const int64_t b = bh / H, h = bh % H;
            const double *kb = k + bh * Nk * d, *vb = v + bh * Nk * d;
            double *dkb = dk + bh * Nk * d, *dvb = dv + bh * Nk * d;
            memset(dkb, 0, sizeof(double) * (size_t)(Nk * d));
            memset(dvb, 0, sizeof(double) * (size_t)(Nk * d));
            for (int64_t i = 0; i < Nq; ++i) {
                const double *qi = q + (bh * Nq + i) * d;
                const double *doi = dout + (bh * Nq + i) * d;
                double *dqi = dq + (bh * Nq + i) * d;
                for (int64_t t = 0; t < d; ++t) dqi[t] = 0.0;
                score_row(q, k, mask, H, Nq, Nk, d, scale, causal, b, h, i, s);
                double m = -INFINITY;
                for (int64_t j = 0; j < Nk; ++j)
                    if (s[j] > m) m = s[j];
                if (m == -INFINITY) continue; /* o_i = 0 is constant: no gradient flows */
                double l = 0.0;
                for (int64_t j = 0; j < Nk; ++j) {
                    s[j] = exp(s[j] - m); /* s now holds the unnormalised weights */
                    l += s[j];
                }
                double rowdot = 0.0; /* sum_j P_ij dP_ij */
                for (int64_t j = 0; j < Nk; ++j) {
                    double pij = s[j] / l, dpij = 0.0;
                    for (int64_t t = 0; t < d; ++t) dpij += doi[t] * vb[j * d + t];
                    s[j] = pij;
                    dp[j] = dpij;
                    rowdot += pij * dpij;
                }
                for (int64_t j = 0; j < Nk; ++j) {
                    double pij = s[j];
                    if (pij == 0.0) continue;
                    double dsij = pij * (dp[j] - rowdot);
                    for (int64_t t = 0; t < d; ++t) {
                        dqi[t] += scale * dsij * kb[j * d + t];
                        dkb[j * d + t] += scale * dsij * qi[t];
                        dvb[j * d + t] += pij * doi[t];
                    }
                }
            }
        }
        free(s);
        free(dp);
    }
    return err ? -1 : 0;
}

/* ---- dropout (see attn_oracle.h) ---------------------------------------------
 * Philox4x64-10 (Salmon et al., SC 2011): a round multiplies counter words 0 and
 * 2 by the two multipliers, and the new counter is (hi(M1 x2) ^ x1 ^ k0,
 * lo(M1 x2), hi(M0 x0) ^ x3 ^ k1, lo(M0 x0)); the key is bumped by the two Weyl
 * constants (the golden ratio and sqrt(3) - 1 in 64-bit fixed point) after
 * every round. */
static const uint64_t PHILOX_M0 = 0xD2E7470EE14C6C93ull;
static const uint64_t PHILOX_M1 = 0xCA5A826395121157ull;
static const uint64_t PHILOX_W0 = 0x9E3779B97F4A7C15ull;
static const uint64_t PHILOX_W1 = 0xBB67AE8584CAA73Bull;

void oracle_philox4x64_10(const uint64_t ctr[4], const uint64_t key[2], uint64_t out[4]) {
    uint64_t x0 = ctr[0], x1 = ctr[1], x2 = ctr[2], x3 = ctr[3];
    uint64_t k0 = key[0], k1 = key[1];
    for (int round = 0; round < 10; ++round) {
        const unsigned __int128 p0 = (unsigned __int128)PHILOX_M0 * x0;
        const unsigned __int128 p1 = (unsigned __int128)PHILOX_M1 * x2;
        const uint64_t hi0 = (uint64_t)(p0 >> 64), lo0 = (uint64_t)p0;
        const uint64_t hi1 = (uint64_t)(p1 >> 64), lo1 = (uint64_t)p1;
        x0 = hi1 ^ x1 ^ k0;
        x1 = lo1;
        x2 = hi0 ^ x3 ^ k1;
        x3 = lo0;
        k0 += PHILOX_W0;
        k1 += PHILOX_W1;
    }
    out[0] = x0;
    out[1] = x1;
    out[2] = x2;
    out[3] = x3;
}

/* keep decisions of row (b, h, i) for keys 0 .. Nk-1 */
static void keep_row(uint8_t *keep, int64_t H, int64_t Nk, int threshold, uint64_t seed, uint64_t offset,
                     int64_t b, int64_t h, int64_t i) {
    const uint64_t key[2] = {seed, 0};
    for (int64_t g = 0; g * 32 < Nk; ++g) {
        const uint64_t ctr[4] = {(uint64_t)i, (uint64_t)g, (uint64_t)(b * H + h), offset};
        uint64_t w[4];
        oracle_philox4x64_10(ctr, key, w);
        for (int64_t t = 0; t < 32 && g * 32 + t < Nk; ++t) {
            const unsigned byte = (unsigned)((w[t / 8] >> (8 * (t % 8))) & 0xFFu);
            keep[g * 32 + t] = byte < (unsigned)threshold ? 1 : 0;
        }
    }
}

int oracle_dropout_keep(uint8_t *keep, int64_t B, int64_t H, int64_t Nq, int64_t Nk, int threshold,
                        uint64_t seed, uint64_t offset) {
    if (!keep || B < 0 || H < 0 || Nq < 0 || Nk < 0 || threshold < 1 || threshold > 256) return -1;
#pragma omp parallel for schedule(dynamic, 8)
    for (int64_t row = 0; row < B * H * Nq; ++row) {
        const int64_t i = row % Nq, bh = row / Nq;
        keep_row(keep + row * Nk, H, Nk, threshold, seed, offset, bh / H, bh % H, i);
    }
    return 0;
}

/* Softmax over the materialised row s, as attend_row; then each kept key's
 * probability, scaled by 1/q, weights its value row. */
static void attend_row_dropout(const double *v, int64_t H, int64_t Nk, int64_t d, int64_t b, int64_t h,
                               const double *s, const uint8_t *keep, double inv_q, double *o, double *lse) {
    const double *vb = v + (b * H + h) * Nk * d;
    double m = -INFINITY;
    for (int64_t j = 0; j < Nk; ++j)
        if (s[j] > m) m = s[j];
    for (int64_t t = 0; t < d; ++t) o[t] = 0.0;
    if (m == -INFINITY) {
        *lse = -INFINITY;
        return;
    }
    double l = 0.0;
    for (int64_t j = 0; j < Nk; ++j) {
        double p = exp(s[j] - m);
        if (p == 0.0) continue;
        l += p;
        if (keep[j])
            for (int64_t t = 0; t < d; ++t) o[t] += p * vb[j * d + t];
    }
    for (int64_t t = 0; t < d; ++t) o[t] = (o[t] / l) * inv_q;
    *lse = m + log(l);
}

int oracle_attn_dropout_f64(const double *q, const double *k, const double *v, double *out, double *lse,
                            int64_t B, int64_t H, int64_t Nq, int64_t Nk, int64_t d, double scale,
                            int causal, int threshold, uint64_t seed, uint64_t offset) {
    if (bad_args(q, k, v, B, H, Nq, Nk, d) || !out || !lse || threshold < 1 || threshold > 256) return -1;
    const double inv_q = 256.0 / (double)threshold;
    int err = 0;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(Nk > 0 ? Nk : 1));
        uint8_t *keep = (uint8_t *)malloc((size_t)(Nk > 0 ? Nk : 1));
        if (!s || !keep) {
#pragma omp atomic write
            err = 1;
        }
#pragma omp for schedule(dynamic, 8)
        for (int64_t row = 0; row < B * H * Nq; ++row) {
            if (!s || !keep) continue;
            const int64_t i = row % Nq, bh = row / Nq;
            const int64_t b = bh / H, h = bh % H;
            score_row(q, k, NULL, H, Nq, Nk, d, scale, causal, b, h, i, s);
            keep_row(keep, H, Nk, threshold, seed, offset, b, h, i);
            attend_row_dropout(v, H, Nk, d, b, h, s, keep, inv_q, out + row * d, lse + row);
        }
        free(s);
        free(keep);
    }
    return err ? -1 : 0;
}
