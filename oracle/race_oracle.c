/*
 * race_oracle.c -- float64 CPU oracle for one RACE attention layer (forward and backward).
 *
 * TEST INFRASTRUCTURE ONLY. This file is the slow, plain statement of what the GPU library
 * computes. Only the test-suite, the smoke check and the CPU-baseline leg of the benchmark load
 * it; the product path (the C-ABI library and its Python binding) never links, imports or calls
 * it, and it shares no code, header, table or constant with the GPU path.
 *
 * Sources (page titles as printed):
 *  - "RACE Attention" slides (arXiv:2510.04008v5 reading deck), frames "Soft corner assignments
 *    make hashing differentiable" (paper Algorithm 1: u = tanh(W x), phi_r = softmax_r(beta u.v_r)),
 *    "Each bucket stores mass and a weighted value sum" (per-table sketches), "Normalize after
 *    combining the tables" (global ratio of summed numerators and denominators) and "Causality is
 *    a prefix update of the same statistics" (paper Algorithm 2: update, then read).
 *  - "RACE Attention: reading notes" (zh), sections 2.2 (notation), 2.4 (soft buckets),
 *    2.5 (aggregate and read) and 2.6 (causal prefix buckets).
 *
 * Readings taken where the pages are silent (each is listed in the design notes):
 *  - Each Q and K row is L2-normalised before projection (the theory assumes unit rows); a zero
 *    row maps to the zero vector, so its buckets are uniform.  `normalize = 0` turns this off.
 *  - Vertex r has coordinates v_{r,t} = +1 if bit t of r is set, else -1.
 *  - Naming: A = Phi_K^T V (content, R x d) and B = Phi_K^T 1 (mass, R); the packed per-table
 *    sketch is [A | B], R rows of d+1 numbers.  The 1/L factors cancel in the ratio.
 *  - The backward pass is the chain rule through these steps (the pages print none).
 *  - beta = +infinity is the hard-hashing limit the slides name ("beta -> infinity: hard
 *    hashing"; reading notes 2.3): each bit is the sign of the projection, so a row falls in one
 *    corner with probability 1.  A projection that is exactly zero keeps the limit of the soft
 *    bit, sigma(0) = 1/2, so it splits the row's mass evenly over both corners (a zero row is
 *    uniform over all R).  Gradients through the hash are zero there (the limit of the soft
 *    gradient away from ties); values still receive theirs.
 *  - W is either one [L, P, d] array shared by every head, or one per head, [H, L, P, d] (the
 *    pages are silent on this; `per_head` selects it).
 *
 * Element types of the token tensors: 0 = float64, 1 = float32, 2 = bfloat16 (raw 16-bit
 * patterns).  Every value is widened exactly to double before use.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_MAX_P 12

static double widen(const void *p, int elem, int64_t i)
{
    if (elem == 0) return ((const double *)p)[i];
    if (elem == 1) return (double)((const float *)p)[i];
    uint32_t bits = ((uint32_t)((const uint16_t *)p)[i]) << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

static void load_row(const void *p, int elem, int64_t off, int64_t d, double *out)
{
    for (int64_t k = 0; k < d; ++k) out[k] = widen(p, elem, off + k);
}

/* Coordinate t of hypercube vertex r. */
static double vertex(int r, int t) { return ((r >> t) & 1) ? 1.0 : -1.0; }

/*
 * Soft bucket features of one row x (length d) for all L tables: Algorithm 1 of the paper,
 * written out step by step.  Outputs: xhat (d), u (L*P, the tanh projections) and phi (L*R).
 */
static void features(const double *x, int64_t d, const double *W, int L, int P, double beta,
                     int normalize, double *xhat, double *u, double *phi)
{
    const int R = 1 << P;
    double n2 = 0.0;
    for (int64_t k = 0; k < d; ++k) n2 += x[k] * x[k];
    double nrm = sqrt(n2);
    for (int64_t k = 0; k < d; ++k)
        xhat[k] = normalize ? (nrm > 0.0 ? x[k] / nrm : 0.0) : x[k];

    double logit[1 << ORACLE_MAX_P];
    for (int l = 0; l < L; ++l) {
        double *ul = u + (int64_t)l * P;
        for (int t = 0; t < P; ++t) {
            const double *w = W + ((int64_t)l * P + t) * d;
            double z = 0.0;
            for (int64_t k = 0; k < d; ++k) z += w[k] * xhat[k];
            ul[t] = tanh(z);
        }
        if (isinf(beta) && beta > 0) {
            /* hard hash: corner r takes the row iff every coordinate of v_r has the sign of u
             * (tanh keeps the sign of z); a zero coordinate halves the mass of both corners */
            for (int r = 0; r < R; ++r) {
                double pr = 1.0;
                for (int t = 0; t < P; ++t) {
                    if (ul[t] == 0.0) pr *= 0.5;
                    else if ((ul[t] > 0.0) != (vertex(r, t) > 0.0)) pr = 0.0;
                }
                phi[(int64_t)l * R + r] = pr;
            }
            continue;
        }
        /* beta-sharpened softmax over the R corners v_r of the hypercube */
        double m = -INFINITY;
        for (int r = 0; r < R; ++r) {
            double s = 0.0;
            for (int t = 0; t < P; ++t) s += ul[t] * vertex(r, t);
            logit[r] = beta * s;
            if (logit[r] > m) m = logit[r];
        }
        double Z = 0.0;
        for (int r = 0; r < R; ++r) Z += exp(logit[r] - m);
        for (int r = 0; r < R; ++r) phi[(int64_t)l * R + r] = exp(logit[r] - m) / Z;
    }
}

/*
 * Chain rule back through `features`: given dphi (L*R), returns dx (d).
 * softmax: ds_r = phi_r (dphi_r - sum_r' phi_r' dphi_r'); logits: du_t = beta sum_r ds_r v_{r,t};
 * tanh: dz = du (1 - u^2); projection: dxhat = sum_l W^(l)^T dz^(l);
 * normalisation: dx = (dxhat - xhat (xhat . dxhat)) / |x|  (zero row: dx = 0).
 */
static void features_backward(const double *x, const double *xhat, const double *u,
                              const double *phi, const double *dphi, int64_t d, const double *W,
                              int L, int P, double beta, int normalize, double *dxhat, double *dx,
                              double *dz_out)
{
    const int R = 1 << P;
    for (int64_t k = 0; k < d; ++k) dxhat[k] = 0.0;
    for (int l = 0; l < L; ++l) {
        const double *ph = phi + (int64_t)l * R;
        const double *dph = dphi + (int64_t)l * R;
        double c = 0.0;
        for (int r = 0; r < R; ++r) c += ph[r] * dph[r];
        for (int t = 0; t < P; ++t) {
            double du = 0.0;
            for (int r = 0; r < R; ++r) du += ph[r] * (dph[r] - c) * vertex(r, t);
            du = isinf(beta) ? 0.0 : du * beta;  /* a hard hash passes no gradient */
            double ut = u[(int64_t)l * P + t];
            double dz = du * (1.0 - ut * ut);
            if (dz_out) dz_out[(int64_t)l * P + t] = dz;
            const double *w = W + ((int64_t)l * P + t) * d;
            for (int64_t k = 0; k < d; ++k) dxhat[k] += dz * w[k];
        }
    }
    if (!normalize) {
        for (int64_t k = 0; k < d; ++k) dx[k] = dxhat[k];
        return;
    }
    double n2 = 0.0;
    for (int64_t k = 0; k < d; ++k) n2 += x[k] * x[k];
    double nrm = sqrt(n2);
    if (!(nrm > 0.0)) {
        for (int64_t k = 0; k < d; ++k) dx[k] = 0.0;
        return;
    }
    double proj = 0.0;
    for (int64_t k = 0; k < d; ++k) proj += xhat[k] * dxhat[k];
    for (int64_t k = 0; k < d; ++k) dx[k] = (dxhat[k] - xhat[k] * proj) / nrm;
}

/*
 * d(loss)/d(beta) from one row's features: the logits are beta (u . v_r), so with the softmax
 * gradient ds_r = phi_r (dphi_r - sum_r' phi_r' dphi_r') the row adds sum_l sum_r ds_r (u . v_r).
 */
static double features_dbeta(const double *u, const double *phi, const double *dphi, int L, int P,
                            double beta)
{
    const int R = 1 << P;
    double acc = 0.0;
    if (isinf(beta)) return 0.0;  /* saturated corners: the limit of the soft sum is zero */
    for (int l = 0; l < L; ++l) {
        const double *ph = phi + (int64_t)l * R;
        const double *dph = dphi + (int64_t)l * R;
        const double *ul = u + (int64_t)l * P;
        double c = 0.0;
        for (int r = 0; r < R; ++r) c += ph[r] * dph[r];
        for (int r = 0; r < R; ++r) {
            double uv = 0.0;
            for (int t = 0; t < P; ++t) uv += ul[t] * vertex(r, t);
            acc += ph[r] * (dph[r] - c) * uv;
        }
    }
    return acc;
}

/*
 * d(loss)/d(W) from one row: z^(l)_t = w^(l)_t . xhat, so the row adds dz^(l)_t xhat to the
 * gradient of hyperplane row (l, t).  dW: [L*P, d].
 */
static void add_dW(double *dW, const double *dz, const double *xhat, int64_t d, int L, int P)
{
    for (int64_t j = 0; j < (int64_t)L * P; ++j)
        for (int64_t k = 0; k < d; ++k) dW[j * d + k] += dz[j] * xhat[k];
}

/* Sketch update with one key: S[j][c] += phi_j * v_c for the d value columns, S[j][d] += phi_j. */
static void sketch_add(double *S, const double *phi, int64_t nfeat, const double *v, int64_t d)
{
    for (int64_t j = 0; j < nfeat; ++j) {
        double *row = S + j * (d + 1);
        for (int64_t c = 0; c < d; ++c) row[c] += phi[j] * v[c];
        row[d] += phi[j];
    }
}

/* Read-out of one query: num_c = sum_j phi_j S[j][c], den = sum_j phi_j S[j][d]. */
static double sketch_read(const double *S, const double *phi, int64_t nfeat, int64_t d, double *num)
{
    double den = 0.0;
    for (int64_t c = 0; c < d; ++c) num[c] = 0.0;
    for (int64_t j = 0; j < nfeat; ++j) {
        const double *row = S + j * (d + 1);
        for (int64_t c = 0; c < d; ++c) num[c] += phi[j] * row[c];
        den += phi[j] * row[d];
    }
    return den;
}

/* ---------------------------------------------------------------- exported entry points */

int race_oracle_max_p(void) { return ORACLE_MAX_P; }

/* Features of M rows x (float64, [M, d]) for L tables: phi [M, L*R], u [M, L*P] (nullable). */
int race_oracle_features(int64_t M, int64_t d, const double *X, const double *W, int L, int P,
                         double beta, int normalize, double *phi, double *u_out)
{
    if (P < 1 || P > ORACLE_MAX_P || L < 1 || d < 1 || M < 0) return -1;
    const int64_t R = (int64_t)1 << P;
    double *xhat = malloc(sizeof(double) * d);
    double *u = malloc(sizeof(double) * L * P);
    if (!xhat || !u) { free(xhat); free(u); return -2; }
    for (int64_t i = 0; i < M; ++i) {
        features(X + i * d, d, W, L, P, beta, normalize, xhat, u, phi + i * L * R);
        if (u_out) memcpy(u_out + i * L * P, u, sizeof(double) * L * P);
    }
    free(xhat);
    free(u);
    return 0;
}

/*
 * Sketch and read-out with the bucket probabilities given directly (no hashing):
 * phiK [L, N, R], V [N, dv], phiQ [L, M, R].  Non-causal: every query reads the full sketch.
 * Causal (M == N): query t reads the sketch after key t was added.  Outputs O [M, dv] and,
 * when non-null, the final per-table mass [L, R] and content [L, R, dv].
 */
int race_oracle_readout_given_phi(int64_t N, int64_t M, int64_t dv, int L, int R,
                                  const double *phiK, const double *V, const double *phiQ,
                                  int causal, double *O, double *mass, double *content)
{
    if (causal && M != N) return -1;
    const int64_t nfeat = (int64_t)L * R;
    double *S = calloc((size_t)(nfeat * (dv + 1)), sizeof(double));
    double *fk = malloc(sizeof(double) * nfeat);
    double *fq = malloc(sizeof(double) * nfeat);
    double *num = malloc(sizeof(double) * dv);
    if (!S || !fk || !fq || !num) { free(S); free(fk); free(fq); free(num); return -2; }
    /* gather the concatenated L*R feature vector of row i */
#define GATHER(dst, src, rows, i) \
    for (int l_ = 0; l_ < L; ++l_) for (int r_ = 0; r_ < R; ++r_) \
        (dst)[(int64_t)l_ * R + r_] = (src)[((int64_t)l_ * (rows) + (i)) * R + r_]
    if (!causal) {
        for (int64_t j = 0; j < N; ++j) { GATHER(fk, phiK, N, j); sketch_add(S, fk, nfeat, V + j * dv, dv); }
        for (int64_t i = 0; i < M; ++i) {
            GATHER(fq, phiQ, M, i);
            double den = sketch_read(S, fq, nfeat, dv, num);
            for (int64_t c = 0; c < dv; ++c) O[i * dv + c] = num[c] / den;
        }
    } else {
        for (int64_t t = 0; t < N; ++t) {
            GATHER(fk, phiK, N, t);
            sketch_add(S, fk, nfeat, V + t * dv, dv);
            GATHER(fq, phiQ, M, t);
            double den = sketch_read(S, fq, nfeat, dv, num);
            for (int64_t c = 0; c < dv; ++c) O[t * dv + c] = num[c] / den;
        }
    }
#undef GATHER
    for (int64_t j = 0; j < nfeat; ++j) {
        if (mass) mass[j] = S[j * (dv + 1) + dv];
        if (content) for (int64_t c = 0; c < dv; ++c) content[j * dv + c] = S[j * (dv + 1) + c];
    }
    free(S); free(fk); free(fq); free(num);
    return 0;
}

static int check_args(int64_t B, int64_t H, int64_t N, int64_t d, int elem, int L, int P,
                      const int64_t *rows, int64_t nrows)
{
    if (B < 1 || H < 1 || N < 1 || d < 1) return -1;
    if (elem < 0 || elem > 2) return -1;
    if (L < 1 || P < 1 || P > ORACLE_MAX_P) return -1;
    if (rows) {
        if (nrows < 1) return -1;
        for (int64_t i = 0; i < nrows; ++i) {
            if (rows[i] < 0 || rows[i] >= N) return -1;
            if (i > 0 && rows[i] <= rows[i - 1]) return -1; /* strictly increasing */
        }
    }
    return 0;
}

/*
 * One causal decode step per (b, h) (the recurrent form of paper Algorithm 2, "Causality is a
 * prefix update of the same statistics"): the new key is added to the prefix sketch, then the
 * new query reads it.  q, k, v: [B, H, d] of element type `elem`; S: [B, H, L*R, d+1] float64,
 * updated in place (zeros for an empty prefix, or the non-causal sketch [A | B] of a prefix);
 * o: [B, H, d] float64.
 */
int race_oracle_decode_step(int64_t B, int64_t H, int64_t d, int elem, const void *q, const void *k,
                            const void *v, const double *W, int per_head, int L, int P, double beta,
                            int normalize, double *S, double *o)
{
    if (check_args(B, H, 1, d, elem, L, P, NULL, 0)) return -1;
    const int64_t R = (int64_t)1 << P, nfeat = (int64_t)L * R;
    double *x = malloc(sizeof(double) * d), *xhat = malloc(sizeof(double) * d);
    double *vv = malloc(sizeof(double) * d), *num = malloc(sizeof(double) * d);
    double *u = malloc(sizeof(double) * L * P), *phi = malloc(sizeof(double) * nfeat);
    int status = 0;
    if (!x || !xhat || !vv || !num || !u || !phi) {
        status = -2;
    } else {
        for (int64_t bh = 0; bh < B * H; ++bh) {
            double *Sbh = S + bh * nfeat * (d + 1);
            const double *Wh = W + (per_head ? (bh % H) * (int64_t)L * P * d : 0);
            load_row(k, elem, bh * d, d, x);
            features(x, d, Wh, L, P, beta, normalize, xhat, u, phi);
            load_row(v, elem, bh * d, d, vv);
            sketch_add(Sbh, phi, nfeat, vv, d);
            load_row(q, elem, bh * d, d, x);
            features(x, d, Wh, L, P, beta, normalize, xhat, u, phi);
            double den = sketch_read(Sbh, phi, nfeat, d, num);
            for (int64_t c = 0; c < d; ++c) o[bh * d + c] = num[c] / den;
        }
    }
    free(x); free(xhat); free(vv); free(num); free(u); free(phi);
    return status;
}

/*
 * Forward pass.  Q, K, V: [B, H, N, d] of element type `elem`; W: [L, P, d] float64, or
 * [H, L, P, d] with `per_head` (head h hashes with W[h]).
 * rows == NULL: O is [B, H, N, d].  Otherwise O is [B, H, nrows, d] and holds only the listed
 * token rows (strictly increasing, the same for every (b, h)).
 * sketch (nullable, non-causal only): the final [A | B] per (b, h), [B, H, L*R, d+1].
 */
int race_oracle_forward(int64_t B, int64_t H, int64_t N, int64_t d, int elem,
                        const void *Q, const void *K, const void *V, const double *W,
                        int per_head, int L, int P, double beta, int causal, int normalize,
                        const int64_t *rows, int64_t nrows, double *O, double *sketch,
                        int nthreads)
{
    if (check_args(B, H, N, d, elem, L, P, rows, nrows)) return -1;
    const int64_t R = (int64_t)1 << P, nfeat = (int64_t)L * R;
    const int64_t nout = rows ? nrows : N;
    int status = 0;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t bh = 0; bh < B * H; ++bh) {
        double *S = calloc((size_t)(nfeat * (d + 1)), sizeof(double));
        double *x = malloc(sizeof(double) * d), *xhat = malloc(sizeof(double) * d);
        double *v = malloc(sizeof(double) * d), *num = malloc(sizeof(double) * d);
        double *u = malloc(sizeof(double) * L * P), *phi = malloc(sizeof(double) * nfeat);
        if (!S || !x || !xhat || !v || !num || !u || !phi) {
#pragma omp atomic write
            status = -2;
        } else {
            const int64_t base = bh * N * d;
            const double *Wh = W + (per_head ? (bh % H) * (int64_t)L * P * d : 0);
            double *Obh = O + bh * nout * d;
            if (!causal) {
                for (int64_t j = 0; j < N; ++j) {
                    load_row(K, elem, base + j * d, d, x);
                    features(x, d, Wh, L, P, beta, normalize, xhat, u, phi);
                    load_row(V, elem, base + j * d, d, v);
                    sketch_add(S, phi, nfeat, v, d);
                }
                for (int64_t o = 0; o < nout; ++o) {
                    int64_t i = rows ? rows[o] : o;
                    load_row(Q, elem, base + i * d, d, x);
                    features(x, d, Wh, L, P, beta, normalize, xhat, u, phi);
                    double den = sketch_read(S, phi, nfeat, d, num);
                    for (int64_t c = 0; c < d; ++c) Obh[o * d + c] = num[c] / den;
                }
                if (sketch) memcpy(sketch + bh * nfeat * (d + 1), S, sizeof(double) * nfeat * (d + 1));
            } else {
                int64_t o = 0;
                for (int64_t t = 0; t < N && o < nout; ++t) {
                    /* Algorithm 2: add key t to the prefix sketch, then read it with query t */
                    load_row(K, elem, base + t * d, d, x);
                    features(x, d, Wh, L, P, beta, normalize, xhat, u, phi);
                    load_row(V, elem, base + t * d, d, v);
                    sketch_add(S, phi, nfeat, v, d);
                    if (rows && rows[o] != t) continue;
                    load_row(Q, elem, base + t * d, d, x);
                    features(x, d, Wh, L, P, beta, normalize, xhat, u, phi);
                    double den = sketch_read(S, phi, nfeat, d, num);
                    for (int64_t c = 0; c < d; ++c) Obh[o * d + c] = num[c] / den;
                    ++o;
                }
            }
        }
        free(S); free(x); free(xhat); free(v); free(num); free(u); free(phi);
    }
    return status;
}

/*
 * Backward pass of the loss-free output O: given dO, returns dQ, dK, dV (float64); W as in
 * `race_oracle_forward`.
 * rows == NULL: all [B, H, N, d].  Otherwise only the listed rows, [B, H, nrows, d].
 *
 * Chain rule (O_i = num_i / den_i):
 *   dnum_i = dO_i / den_i,  dden_i = -(dO_i . O_i) / den_i,
 *   dphi_Q(i) = [A | B] [dnum_i ; dden_i]                         (sketch seen by query i),
 *   G = sum_i phi_Q(i) [dnum_i | dden_i]   (non-causal: all i; causal: suffix over i >= j),
 *   dV_j = G_A^T phi_K(j),   dphi_K(j) = G_A V_j + G_B,
 * followed by `features_backward` for each side.  When `dbeta` is given (B * H values) every
 * token's query and key features also contribute d(loss)/d(beta) (`features_dbeta`), and when
 * `dW` is given ([B * H, L * P * d], zeroed by the caller) every token also adds dz xhat to the
 * rows of the hyperplanes it was hashed with (`add_dW`), whatever `rows` selects for dQ, dK, dV.
 * Both are per (b, h); the gradient of a shared W is their sum over (b, h), of a per-head W
 * the sum over b.
 */
int race_oracle_backward(int64_t B, int64_t H, int64_t N, int64_t d, int elem,
                         const void *Q, const void *K, const void *V, const void *dO,
                         const double *W, int per_head, int L, int P, double beta, int causal,
                         int normalize,
                         const int64_t *rows, int64_t nrows, double *dQ, double *dK, double *dV,
                         double *dbeta, double *dW, int nthreads)
{
    if (check_args(B, H, N, d, elem, L, P, rows, nrows)) return -1;
    const int64_t R = (int64_t)1 << P, nfeat = (int64_t)L * R;
    const int64_t nout = rows ? nrows : N;
    const int wantg = dbeta != NULL || dW != NULL;  /* every token's features count */
    int status = 0;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t bh = 0; bh < B * H; ++bh) {
        const int64_t sz = nfeat * (d + 1);
        double *S = calloc((size_t)sz, sizeof(double)), *G = calloc((size_t)sz, sizeof(double));
        double *x = malloc(sizeof(double) * d), *xhat = malloc(sizeof(double) * d);
        double *v = malloc(sizeof(double) * d), *num = malloc(sizeof(double) * d);
        double *g = malloc(sizeof(double) * d), *dnum = malloc(sizeof(double) * d);
        double *dxhat = malloc(sizeof(double) * d), *dx = malloc(sizeof(double) * d);
        double *u = malloc(sizeof(double) * L * P), *phi = malloc(sizeof(double) * nfeat);
        double *dphi = malloc(sizeof(double) * nfeat), *dz = malloc(sizeof(double) * L * P);
        /* per-token den_i and (dO_i . O_i), needed by the key side */
        double *den_all = malloc(sizeof(double) * N), *dOO_all = malloc(sizeof(double) * N);
        if (!S || !G || !x || !xhat || !v || !num || !g || !dnum || !dxhat || !dx || !u ||
            !phi || !dphi || !dz || !den_all || !dOO_all) {
#pragma omp atomic write
            status = -2;
        } else {
            const int64_t base = bh * N * d;
            const double *Wh = W + (per_head ? (bh % H) * (int64_t)L * P * d : 0);
            double *dQbh = dQ + bh * nout * d, *dKbh = dK + bh * nout * d, *dVbh = dV + bh * nout * d;
            if (!causal) {
                /* sketch of all keys */
                for (int64_t j = 0; j < N; ++j) {
                    load_row(K, elem, base + j * d, d, x);
                    features(x, d, Wh, L, P, beta, normalize, xhat, u, phi);
                    load_row(V, elem, base + j * d, d, v);
                    sketch_add(S, phi, nfeat, v, d);
                }
                /* query side: O, dnum, dden, G = Phi_Q^T [dnum | dden], dQ on requested rows */
                int64_t o = 0;
                for (int64_t i = 0; i < N; ++i) {
                    load_row(Q, elem, base + i * d, d, x);
                    features(x, d, Wh, L, P, beta, normalize, xhat, u, phi);
                    double den = sketch_read(S, phi, nfeat, d, num);
                    load_row(dO, elem, base + i * d, d, g);
                    double dOO = 0.0;
                    for (int64_t c = 0; c < d; ++c) dOO += g[c] * (num[c] / den);
                    for (int64_t c = 0; c < d; ++c) dnum[c] = g[c] / den;
                    double dden = -dOO / den;
                    for (int64_t j = 0; j < nfeat; ++j) {
                        double *row = G + j * (d + 1);
                        for (int64_t c = 0; c < d; ++c) row[c] += phi[j] * dnum[c];
                        row[d] += phi[j] * dden;
                    }
                    const int want = !rows || (o < nout && rows[o] == i);
                    if (!want && !wantg) continue;
                    for (int64_t j = 0; j < nfeat; ++j) {
                        const double *row = S + j * (d + 1);
                        double s = row[d] * dden;
                        for (int64_t c = 0; c < d; ++c) s += row[c] * dnum[c];
                        dphi[j] = s;
                    }
                    if (dbeta) dbeta[bh] += features_dbeta(u, phi, dphi, L, P, beta);
                    if (!want && !dW) continue;
                    features_backward(x, xhat, u, phi, dphi, d, Wh, L, P, beta, normalize, dxhat, dx, dz);
                    if (dW) add_dW(dW + bh * L * P * d, dz, xhat, d, L, P);
                    if (!want) continue;
                    memcpy(dQbh + o * d, dx, sizeof(double) * d);
                    ++o;
                }
                /* key side on requested rows (every key when dbeta is wanted) */
                int64_t o2 = 0;
                for (int64_t j0 = 0; j0 < N; ++j0) {
                    const int want = rows ? (o2 < nout && rows[o2] == j0) : 1;
                    if (!want && !wantg) {
                        if (!rows || o2 >= nout) break;
                        continue;
                    }
                    load_row(K, elem, base + j0 * d, d, x);
                    features(x, d, Wh, L, P, beta, normalize, xhat, u, phi);
                    load_row(V, elem, base + j0 * d, d, v);
                    if (want)
                        for (int64_t c = 0; c < d; ++c) dVbh[o2 * d + c] = 0.0;
                    for (int64_t j = 0; j < nfeat; ++j) {
                        const double *row = G + j * (d + 1);
                        double s = row[d];
                        for (int64_t c = 0; c < d; ++c) {
                            if (want) dVbh[o2 * d + c] += phi[j] * row[c];
                            s += row[c] * v[c];
                        }
                        dphi[j] = s;
                    }
                    if (dbeta) dbeta[bh] += features_dbeta(u, phi, dphi, L, P, beta);
                    if (!want && !dW) continue;
                    features_backward(x, xhat, u, phi, dphi, d, Wh, L, P, beta, normalize, dxhat, dx, dz);
                    if (dW) add_dW(dW + bh * L * P * d, dz, xhat, d, L, P);
                    if (!want) continue;
                    memcpy(dKbh + o2 * d, dx, sizeof(double) * d);
                    ++o2;
                }
            } else {
                /* forward order: prefix sketch S_t (Algorithm 2), den_t, dO_t . O_t, dQ */
                int64_t o = 0;
                for (int64_t t = 0; t < N; ++t) {
                    load_row(K, elem, base + t * d, d, x);
                    features(x, d, Wh, L, P, beta, normalize, xhat, u, phi);
                    load_row(V, elem, base + t * d, d, v);
                    sketch_add(S, phi, nfeat, v, d);
                    load_row(Q, elem, base + t * d, d, x);
                    features(x, d, Wh, L, P, beta, normalize, xhat, u, phi);
                    double den = sketch_read(S, phi, nfeat, d, num);
                    load_row(dO, elem, base + t * d, d, g);
                    double dOO = 0.0;
                    for (int64_t c = 0; c < d; ++c) dOO += g[c] * (num[c] / den);
                    den_all[t] = den;
                    dOO_all[t] = dOO;
                    const int want = !rows || (o < nout && rows[o] == t);
                    if (!want && !wantg) continue;
                    double dden = -dOO / den;
                    for (int64_t j = 0; j < nfeat; ++j) {
                        const double *row = S + j * (d + 1);
                        double s = row[d] * dden;
                        for (int64_t c = 0; c < d; ++c) s += row[c] * (g[c] / den);
                        dphi[j] = s;
                    }
                    if (dbeta) dbeta[bh] += features_dbeta(u, phi, dphi, L, P, beta);
                    if (!want && !dW) continue;
                    features_backward(x, xhat, u, phi, dphi, d, Wh, L, P, beta, normalize, dxhat, dx, dz);
                    if (dW) add_dW(dW + bh * L * P * d, dz, xhat, d, L, P);
                    if (!want) continue;
                    memcpy(dQbh + o * d, dx, sizeof(double) * d);
                    ++o;
                }
                /* reverse order: suffix sums G_j = sum_{t >= j} phi_Q(t) [dnum_t | dden_t], dK, dV */
                int64_t o2 = nout - 1;
                for (int64_t t = N - 1; t >= 0 && (o2 >= 0 || wantg); --t) {
                    load_row(Q, elem, base + t * d, d, x);
                    features(x, d, Wh, L, P, beta, normalize, xhat, u, phi);
                    load_row(dO, elem, base + t * d, d, g);
                    for (int64_t c = 0; c < d; ++c) dnum[c] = g[c] / den_all[t];
                    double dden = -dOO_all[t] / den_all[t];
                    for (int64_t j = 0; j < nfeat; ++j) {
                        double *row = G + j * (d + 1);
                        for (int64_t c = 0; c < d; ++c) row[c] += phi[j] * dnum[c];
                        row[d] += phi[j] * dden;
                    }
                    const int want = rows ? (o2 >= 0 && rows[o2] == t) : 1;
                    if (!want && !wantg) continue;
                    int64_t slot = rows ? o2 : t;
                    load_row(K, elem, base + t * d, d, x);
                    features(x, d, Wh, L, P, beta, normalize, xhat, u, phi);
                    load_row(V, elem, base + t * d, d, v);
                    if (want)
                        for (int64_t c = 0; c < d; ++c) dVbh[slot * d + c] = 0.0;
                    for (int64_t j = 0; j < nfeat; ++j) {
                        const double *row = G + j * (d + 1);
                        double s = row[d];
                        for (int64_t c = 0; c < d; ++c) {
                            if (want) dVbh[slot * d + c] += phi[j] * row[c];
                            s += row[c] * v[c];
                        }
                        dphi[j] = s;
                    }
                    if (dbeta) dbeta[bh] += features_dbeta(u, phi, dphi, L, P, beta);
                    if (!want && !dW) continue;
                    features_backward(x, xhat, u, phi, dphi, d, Wh, L, P, beta, normalize, dxhat, dx, dz);
                    if (dW) add_dW(dW + bh * L * P * d, dz, xhat, d, L, P);
                    if (!want) continue;
                    memcpy(dKbh + slot * d, dx, sizeof(double) * d);
                    --o2;
                }
            }
        }
        free(S); free(G); free(x); free(xhat); free(v); free(num); free(g); free(dnum);
        free(dxhat); free(dx); free(u); free(phi); free(dphi); free(dz); free(den_all); free(dOO_all);
    }
    return status;
}

/*
 * Angular attention, the target the soft hash estimates ("RACE Attention" slides, frame "Choose a
 * nonnegative kernel that can be sketched", paper Eqs. (3)-(4); reading notes 3.1): O(N^2) by its
 * definition,
 *
 *     O_i = sum_j S_ij V_j / sum_j S_ij,   S_ij = (1 - arccos(q_i . k_j / (|q_i| |k_j|)) / pi)^gamma,
 *
 * over j <= i when causal.  With gamma = P it is the kernel a P-bit hard hash collides with
 * (frame "A hash collision estimates a powered angular kernel").  Reading where the pages are
 * silent: a zero row has cosine 0 with every row (angle pi / 2, the value the soft features'
 * uniform buckets give); the cosine is clamped to [-1, 1] before arccos; 0^0 = 1.
 * Q, K, V: [B, H, N, d] of element type `elem`; O: [B, H, nout, d] float64 with `rows` as in
 * `race_oracle_forward`.  Returns 2 if a row's sum_j S_ij is zero (every key antipodal).
 */
int race_oracle_angular_forward(int64_t B, int64_t H, int64_t N, int64_t d, int elem,
                                const void *Q, const void *K, const void *V, double gamma,
                                int causal, const int64_t *rows, int64_t nrows, double *O,
                                int nthreads)
{
    if (check_args(B, H, N, d, elem, 1, 1, rows, nrows) || !(gamma >= 0.0)) return -1;
    const int64_t nout = rows ? nrows : N;
    const double pi = acos(-1.0);
    int status = 0;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t bh = 0; bh < B * H; ++bh) {
        double *q = malloc(sizeof(double) * d), *k = malloc(sizeof(double) * d);
        double *v = malloc(sizeof(double) * d), *num = malloc(sizeof(double) * d);
        if (!q || !k || !v || !num) {
#pragma omp atomic write
            status = -2;
        } else {
            const int64_t base = bh * N * d;
            for (int64_t o = 0; o < nout; ++o) {
                const int64_t i = rows ? rows[o] : o;
                load_row(Q, elem, base + i * d, d, q);
                double qq = 0.0;
                for (int64_t c = 0; c < d; ++c) qq += q[c] * q[c];
                for (int64_t c = 0; c < d; ++c) num[c] = 0.0;
                double den = 0.0;
                const int64_t jend = causal ? i + 1 : N;
                for (int64_t j = 0; j < jend; ++j) {
                    load_row(K, elem, base + j * d, d, k);
                    double kk = 0.0, qk = 0.0;
                    for (int64_t c = 0; c < d; ++c) { kk += k[c] * k[c]; qk += q[c] * k[c]; }
                    double cosang = (qq > 0.0 && kk > 0.0) ? qk / (sqrt(qq) * sqrt(kk)) : 0.0;
                    if (cosang > 1.0) cosang = 1.0;
                    if (cosang < -1.0) cosang = -1.0;
                    const double s = pow(1.0 - acos(cosang) / pi, gamma);
                    load_row(V, elem, base + j * d, d, v);
                    for (int64_t c = 0; c < d; ++c) num[c] += s * v[c];
                    den += s;
                }
                double *Oi = O + (bh * nout + o) * d;
                if (!(den > 0.0)) {
#pragma omp atomic write
                    status = 2;
                    for (int64_t c = 0; c < d; ++c) Oi[c] = NAN;
                } else {
                    for (int64_t c = 0; c < d; ++c) Oi[c] = num[c] / den;
                }
            }
        }
        free(q); free(k); free(v); free(num);
    }
    return status;
}
