// race_generic.cu -- CUDA-core kernels for every mode of RACE attention (float32 arithmetic,
// float32 or bfloat16 tensors).  They are the float32 path of the library and the baseline the
// tensor-core paths are checked against.
//
// Method: "RACE Attention" slides (arXiv:2510.04008v5), frames "Soft corner assignments make
// hashing differentiable" (Algorithm 1 features), "Each bucket stores mass and a weighted value
// sum" (sketches), "Normalize after combining the tables" (global ratio) and "Causality is a
// prefix update of the same statistics" (Algorithm 2).  The backward kernels apply the chain
// rule through those steps.
//
// Every CTA works on tiles of TT = 32 tokens held in shared memory as float32.  Bucket
// probabilities use the product form phi_r = prod_t sigmoid(2 beta u_t v_{r,t}), which equals
// the softmax over the 2^P hypercube corners (reading notes, section 2.4).
#include "race_common.cuh"
#include "race_launch.h"

namespace race {
namespace gen {

constexpr int NT = 256;   // threads per CTA
constexpr int TT = 32;    // tokens per tile (= warp size: lane <-> token in the featuriser)
constexpr int LRC = 64;   // sketch rows per CTA in the reduction kernels
constexpr int KACC = (LRC * (kMaxD + 1) + NT - 1) / NT;  // accumulators per thread, k_sketch
constexpr int KOUT = (TT * (kMaxD + 1) + NT - 1) / NT;   // outputs per thread, read-outs

// ------------------------------------------------------------------ shared-memory helpers

// Hyperplane rows of tables [l0, l1) into ws[(l - l0) * P + t][0..d) (row stride d + 1).
__device__ void load_w(const float *__restrict__ W, const Dims &D, int l0, int l1, float *ws)
{
    const int dp = D.d + 1;
    const int n = (l1 - l0) * D.P * D.d;
    const float *src = W + (int64_t)l0 * D.P * D.d;
    for (int i = threadIdx.x; i < n; i += NT) {
        int row = i / D.d, k = i - row * D.d;
        ws[row * dp + k] = src[i];
    }
}

// Rows [row0, row0 + cnt) of a [N, d] slice into xs[TT][d + 1]; rows past cnt are zero.
template <typename T>
__device__ void load_rows(const T *__restrict__ X, int64_t row0, int cnt, int d, float *xs)
{
    const int dp = d + 1;
    for (int i = threadIdx.x; i < TT * d; i += NT) {
        int t = i / d, k = i - t * d;
        xs[t * dp + k] = t < cnt ? ld_f(X, (row0 + t) * d + k) : 0.f;
    }
}

// Value rows with the mass column: vs[t][c] = V[t][c] for c < d, vs[t][d] = 1 (0 past cnt).
template <typename T>
__device__ void load_values(const T *__restrict__ V, int64_t row0, int cnt, int d, float *vs)
{
    const int dv = d + 1;
    for (int i = threadIdx.x; i < TT * dv; i += NT) {
        int t = i / dv, c = i - t * dv;
        float v = 0.f;
        if (t < cnt) v = c < d ? ld_f(V, (row0 + t) * d + c) : 1.f;
        vs[t * dv + c] = v;
    }
}

// Bucket probabilities of the TT rows in xs for feature columns [f0, f1) of the concatenated
// L*R vector.  inv_s[t] = 1/|x_t| (0 for a zero row, whose projections are then 0 and whose
// buckets are uniform).  u_s (optional) receives u = tanh(W xhat) as [TT][LP].  f_s receives
// phi as [TT][fst] at column (l*R + r - f0).  ws must start with table f0 / R.
__device__ void featurise(const float *xs, const Dims &D, const float *ws, int f0, int f1,
                          float *inv_s, float *u_s, float *f_s, int fst)
{
    const int dp = D.d + 1;
    for (int t = threadIdx.x; t < TT; t += NT) {
        float s = 0.f;
        for (int k = 0; k < D.d; ++k) s = fmaf(xs[t * dp + k], xs[t * dp + k], s);
        inv_s[t] = s > 0.f ? 1.0f / sqrtf(s) : 0.f;
    }
    __syncthreads();
    const int l0 = f0 / D.R, l1 = (f1 - 1) / D.R + 1, nl = l1 - l0;
    for (int pair = threadIdx.x; pair < TT * nl; pair += NT) {
        const int t = pair % TT, li = pair / TT, l = l0 + li;
        const float inv = inv_s[t];
        const float *x = xs + t * dp;
        float pp[kMaxP], pm[kMaxP];
#pragma unroll
        for (int p = 0; p < kMaxP; ++p) {
            pp[p] = pm[p] = 1.f;
            if (p < D.P) {
                const float *w = ws + (li * D.P + p) * dp;
                float z = 0.f;
                for (int k = 0; k < D.d; ++k) z = fmaf(w[k], x[k], z);
                const float u = tanhf(z * inv);
                if (u_s) u_s[t * D.LP + l * D.P + p] = u;
                const float a = 2.f * D.beta * u;
                pp[p] = 1.f / (1.f + expf(-a));  // corner coordinate +1
                pm[p] = 1.f / (1.f + expf(a));   // corner coordinate -1
            }
        }
        const int r0 = max(0, f0 - l * D.R), r1 = min(D.R, f1 - l * D.R);
        for (int r = r0; r < r1; ++r) {
            float prod = 1.f;
#pragma unroll
            for (int p = 0; p < kMaxP; ++p)
                if (p < D.P) prod *= ((r >> p) & 1) ? pp[p] : pm[p];
            f_s[t * fst + l * D.R + r - f0] = prod;
        }
    }
    __syncthreads();
}

// Chain rule back through `featurise` for all L tables.  Inputs: x rows (xs), inv_s, u_s,
// phi (f_s) and dphi (dphi_s) as [TT][fst]; ws must hold every table.  Output dx_s[TT][d+1].
// softmax: ds_r = phi_r (dphi_r - sum phi dphi); logits: du_t = beta sum_r ds_r v_{r,t};
// tanh: dz = du (1 - u^2); projection: dxhat = sum W^T dz; normalisation:
// dx = (dxhat - xhat (xhat . dxhat)) / |x|, and 0 for a zero row.
// Returns this thread's share of d(loss)/d(beta): the logits are beta (u . v_r), so each
// (token, table) adds sum_r ds_r (u . v_r) = sum_t u_t sum_r ds_r v_{r,t}.  Rows past a tile's
// count are zero, so their u = 0 and they add nothing.
__device__ float featurise_backward(const float *xs, const Dims &D, const float *ws,
                                    const float *inv_s, const float *u_s, const float *f_s,
                                    const float *dphi_s, int fst, float *dz_s, float *dx_s,
                                    float *red_s, float *dz_g = nullptr, int cnt = 0)
{
    float db = 0.f;
    const int dp = D.d + 1;
    for (int pair = threadIdx.x; pair < TT * D.L; pair += NT) {
        const int t = pair % TT, l = pair / TT;
        const float *ph = f_s + t * fst + l * D.R;
        const float *dph = dphi_s + t * fst + l * D.R;
        float c = 0.f;
        for (int r = 0; r < D.R; ++r) c = fmaf(ph[r], dph[r], c);
        float du[kMaxP];
#pragma unroll
        for (int p = 0; p < kMaxP; ++p) du[p] = 0.f;
        for (int r = 0; r < D.R; ++r) {
            const float ds = ph[r] * (dph[r] - c);
#pragma unroll
            for (int p = 0; p < kMaxP; ++p)
                if (p < D.P) du[p] += ((r >> p) & 1) ? ds : -ds;
        }
#pragma unroll
        for (int p = 0; p < kMaxP; ++p) {
            if (p < D.P) {
                const float u = u_s[t * D.LP + l * D.P + p];
                db = fmaf(u, du[p], db);
                dz_s[t * D.LP + l * D.P + p] = D.beta * du[p] * (1.f - u * u);
            }
        }
    }
    __syncthreads();
    if (dz_g)  // the tile's live rows of dz / |x| (d(loss)/d(W) is their product with the rows)
        for (int i = threadIdx.x; i < cnt * D.LP; i += NT) dz_g[(i / D.LP) * D.dzld + i % D.LP] = dz_s[i] * inv_s[i / D.LP];
    for (int i = threadIdx.x; i < TT * D.d; i += NT) {
        const int t = i / D.d, k = i - t * D.d;
        float s = 0.f;
        for (int j = 0; j < D.LP; ++j) s = fmaf(dz_s[t * D.LP + j], ws[j * dp + k], s);
        dx_s[t * dp + k] = s;
    }
    __syncthreads();
    for (int t = threadIdx.x; t < TT; t += NT) {
        float s = 0.f;
        for (int k = 0; k < D.d; ++k) s = fmaf(xs[t * dp + k], dx_s[t * dp + k], s);
        red_s[t] = s * inv_s[t] * inv_s[t];  // (xhat . dxhat) / |x|
    }
    __syncthreads();
    for (int i = threadIdx.x; i < TT * D.d; i += NT) {
        const int t = i / D.d, k = i - t * D.d;
        dx_s[t * dp + k] = inv_s[t] * (dx_s[t * dp + k] - xs[t * dp + k] * red_s[t]);
    }
    __syncthreads();
    return db;
}

// The CTA's d(loss)/d(beta) partial (one float per thread, summed in a fixed order) to
// dbpart[bh][blockIdx.x]; nothing when dbpart is null.  Every thread calls it.
__device__ void store_dbeta_partial(float db, float *scratch, float *dbpart, int64_t bh)
{
    if (!dbpart) return;
    const float s = block_sum_fixed(db, scratch);
    if (threadIdx.x == 0) dbpart[bh * gridDim.x + blockIdx.x] = s;
}

// ------------------------------------------------------------------ shared-memory layouts

struct SketchSmem {
    int ws, xs, ys, fs, inv;
    SmemLayout lay;
    __host__ __device__ SketchSmem(const Dims &D, int ntab)
    {
        const int dp = D.d + 1;
        ws = lay.take(ntab * D.P * dp);
        xs = lay.take(TT * dp);
        ys = lay.take(TT * dp);
        fs = lay.take(TT * (LRC + 1));
        inv = lay.take(TT);
    }
};

struct ReadoutSmem {
    int ws, xs, fs, inv, sch, outs;
    SmemLayout lay;
    __host__ __device__ explicit ReadoutSmem(const Dims &D)
    {
        const int dp = D.d + 1;
        ws = lay.take(D.LP * dp);
        xs = lay.take(TT * dp);
        fs = lay.take(TT * (D.LR + 1));
        inv = lay.take(TT);
        sch = lay.take(LRC * D.dv);
        outs = lay.take(TT * D.dv);
    }
};

struct QueryBwdSmem {
    int ws, xs, ys, fs, gs, us, inv, sch, sb, den, cc, dz, dx, red;
    SmemLayout lay;
    __host__ __device__ explicit QueryBwdSmem(const Dims &D)
    {
        const int dp = D.d + 1, fst = D.LR + 1;
        ws = lay.take(D.LP * dp);
        xs = lay.take(TT * dp);
        ys = lay.take(TT * dp);
        fs = lay.take(TT * fst);
        gs = lay.take(TT * fst);
        us = lay.take(TT * D.LP);
        inv = lay.take(TT);
        sch = lay.take(LRC * D.dv);
        sb = lay.take(D.LR);
        den = lay.take(TT);
        cc = lay.take(TT);
        dz = lay.take(TT * D.LP);
        dx = lay.take(TT * dp);
        red = lay.take(TT);
    }
};

struct KeyBwdSmem {
    int ws, xs, vs, fs, gs, us, inv, sch, dz, dx, red;
    SmemLayout lay;
    __host__ __device__ explicit KeyBwdSmem(const Dims &D)
    {
        const int dp = D.d + 1, fst = D.LR + 1;
        ws = lay.take(D.LP * dp);
        xs = lay.take(TT * dp);
        vs = lay.take(TT * dp);
        fs = lay.take(TT * fst);
        gs = lay.take(TT * fst);
        us = lay.take(TT * D.LP);
        inv = lay.take(TT);
        sch = lay.take(LRC * D.dv);
        dz = lay.take(TT * D.LP);
        dx = lay.take(TT * dp);
        red = lay.take(TT);
    }
};

struct CausalFwdSmem {
    int ws, S, xq, xk, vs, fq, fk, sc, inv, outs;
    SmemLayout lay;
    __host__ __device__ explicit CausalFwdSmem(const Dims &D)
    {
        const int dp = D.d + 1, fst = D.LR + 1;
        ws = lay.take(D.LP * dp);
        S = lay.take(D.LR * D.dv);
        xq = lay.take(TT * dp);
        xk = lay.take(TT * dp);
        vs = lay.take(TT * dp);
        fq = lay.take(TT * fst);
        fk = lay.take(TT * fst);
        sc = lay.take(TT * (TT + 1));
        inv = lay.take(TT);
        outs = lay.take(TT * D.dv);
    }
};

struct CausalBwdSmem {
    int ws, S, xq, xk, vs, ys, fq, fk, gs, us, sc, aux2, invq, invk, den, cc, dz, dx, red;
    SmemLayout lay;
    __host__ __device__ explicit CausalBwdSmem(const Dims &D)
    {
        const int dp = D.d + 1, fst = D.LR + 1;
        ws = lay.take(D.LP * dp);
        S = lay.take(D.LR * D.dv);
        xq = lay.take(TT * dp);
        xk = lay.take(TT * dp);
        vs = lay.take(TT * dp);
        ys = lay.take(TT * dp);
        fq = lay.take(TT * fst);
        fk = lay.take(TT * fst);
        gs = lay.take(TT * fst);
        us = lay.take(TT * D.LP);
        sc = lay.take(TT * (TT + 1));
        aux2 = lay.take(TT * (TT + 1));
        invq = lay.take(TT);
        invk = lay.take(TT);
        den = lay.take(TT);
        cc = lay.take(TT);
        dz = lay.take(TT * D.LP);
        dx = lay.take(TT * dp);
        red = lay.take(TT);
    }
};

// ------------------------------------------------------------------ kernels

// Partial weighted sketches over one token range and one block of LRC feature rows:
//   part[bh][s][f][c] = sum_{t in range s} phi_f(X_t) * y_t[c] * a_t   (c < d)
//   part[bh][s][f][d] = sum_{t in range s} phi_f(X_t) * b_t
// mode 0 (key sketch [A | B]):      X = K, y = V,  a = 1,          b = 1
// mode 1 (gradient sketch [dA|dB]): X = Q, y = dO, a = 1/den_t,    b = -(dO_t . O_t)/den_t
// (aux[t] = {1/den_t, dO_t . O_t}).  Grid (nsplit, ceil(LR / LRC), BH).
template <typename T>
__global__ void __launch_bounds__(NT) k_sketch(Dims D, const T *__restrict__ X,
                                               const T *__restrict__ Y,
                                               const float2 *__restrict__ aux,
                                               const float *__restrict__ W, int64_t seg_len,
                                               int nsplit, float *__restrict__ part, int mode)
{
    extern __shared__ float sm[];
    const int dp = D.d + 1;
    const int s = blockIdx.x;
    const int64_t bh = blockIdx.z;
    const int f0 = blockIdx.y * LRC, f1 = min(D.LR, f0 + LRC), nf = f1 - f0;
    const int l0 = f0 / D.R, l1 = (f1 - 1) / D.R + 1;
    const SketchSmem L(D, l1 - l0);
    float *ws = sm + L.ws, *xs = sm + L.xs, *ys = sm + L.ys, *fs = sm + L.fs, *inv = sm + L.inv;
    load_w(head_w(W, D, bh), D, l0, l1, ws);
    const T *Xb = X + bh * D.N * D.d;
    const T *Yb = Y + bh * D.N * D.d;
    const int64_t n_begin = (int64_t)s * seg_len;
    const int64_t n_end = min(D.N, n_begin + seg_len);
    const int nout = nf * D.dv;
    float acc[KACC];
#pragma unroll
    for (int k = 0; k < KACC; ++k) acc[k] = 0.f;
    for (int64_t n0 = n_begin; n0 < n_end; n0 += TT) {
        const int cnt = (int)min((int64_t)TT, n_end - n0);
        __syncthreads();
        load_rows(Xb, n0, cnt, D.d, xs);
        for (int i = threadIdx.x; i < TT * D.dv; i += NT) {
            const int t = i / D.dv, c = i - t * D.dv;
            float v = 0.f;
            if (t < cnt) {
                float a = 1.f, b = 1.f;
                if (mode == 1) {
                    const float2 q = aux[bh * D.N + n0 + t];
                    a = q.x;
                    b = -q.y * q.x;
                }
                v = c < D.d ? ld_f(Yb, (n0 + t) * D.d + c) * a : b;
            }
            ys[t * dp + c] = v;
        }
        __syncthreads();
        featurise(xs, D, ws, f0, f1, inv, nullptr, fs, LRC + 1);
#pragma unroll
        for (int k = 0; k < KACC; ++k) {
            const int o = threadIdx.x + k * NT;
            if (o < nout) {
                const int f = o / D.dv, c = o - f * D.dv;
                float a = acc[k];
                for (int t = 0; t < cnt; ++t) a = fmaf(fs[t * (LRC + 1) + f], ys[t * dp + c], a);
                acc[k] = a;
            }
        }
    }
    float *out = part + (((int64_t)bh * nsplit + s) * D.LR + f0) * D.dv;
#pragma unroll
    for (int k = 0; k < KACC; ++k) {
        const int o = threadIdx.x + k * NT;
        if (o < nout) out[o] = acc[k];
    }
}

// Fixed-order combination of the nsplit partial sketches of each (b, h):
// mode 0: out[bh][e] = sum_s part[bh][s][e]
// mode 1: out[bh][s][e] = sum_{s' < s} part[bh][s'][e]   (exclusive prefix over segments)
// mode 2: out[bh][s][e] = sum_{s' > s} part[bh][s'][e]   (exclusive suffix over segments)
// The partials are read in batches of 16 independent loads before they are added (in the same
// order as one at a time), so that the loads' latency overlaps.
__global__ void k_combine(const float *__restrict__ part, float *__restrict__ out, int64_t E,
                          int nsplit, int mode)
{
    constexpr int NB = 16;
    const int64_t bh = blockIdx.y;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < E;
         e += (int64_t)gridDim.x * blockDim.x) {
        const float *p = part + bh * nsplit * E + e;
        float s = 0.f;
        for (int i0 = 0; i0 < nsplit; i0 += NB) {
            float v[NB];
#pragma unroll
            for (int j = 0; j < NB; ++j) {
                const int i = mode == 2 ? nsplit - 1 - (i0 + j) : i0 + j;
                v[j] = i0 + j < nsplit ? p[(int64_t)i * E] : 0.f;
            }
#pragma unroll
            for (int j = 0; j < NB; ++j) {
                if (i0 + j < nsplit) {
                    const int i = mode == 2 ? nsplit - 1 - (i0 + j) : i0 + j;
                    if (mode != 0) out[(bh * nsplit + i) * E + e] = s;
                    s += v[j];
                }
            }
        }
        if (mode == 0) out[bh * E + e] = s;
    }
}

// d(loss)/d(beta) per (b, h) from the backward kernels' CTA partials: part holds two [BH][slots]
// arrays (query side, then key side), zero where no CTA wrote; out[bh] = their sum, taken in a
// fixed order (a strided share per thread, then the block in thread order).  Grid (BH), 256 threads.
__global__ void __launch_bounds__(256) k_dbeta_combine(const float *__restrict__ part, int slots, int64_t BH,
                                                        float *__restrict__ out)
{
    __shared__ float scratch[8];
    const int64_t bh = blockIdx.x;
    float s = 0.f;
    for (int side = 0; side < 2; ++side) {
        const float *p = part + ((int64_t)side * BH + bh) * slots;
        for (int i = threadIdx.x; i < slots; i += blockDim.x) s += p[i];
    }
    s = block_sum_fixed(s, scratch);
    if (threadIdx.x == 0) out[bh] = s;
}

// d(loss)/d(W) of problem bh, partial over the token range [blockIdx.x * span, + span): the
// projection z = W xhat has d(loss)/d(W) = sum over Q and K rows of dz xhat^T, and the backward
// kernels stored dz / |x| per row (stride dzld), so part[bh][blockIdx.x][lp][k] = sum over the
// range's rows n of dzq[n][lp] Q[n][k] + dzk[n][lp] K[n][k].  The rows go through shared memory in
// tiles of DW_ROWS, the Q rows then the K rows of each, copied with 16-byte loads that are issued
// one tile ahead (held in registers while the tile before is summed).  Thread (g, k) owns column k
// and LPB (>= dzld) accumulators over the rows of parity g, in order; half 1 adds half 0's sums
// last, so the summation order is fixed.  Grid (blocks, BH), NT threads, dw_smem_bytes of shared
// memory.
constexpr int DW_ROWS = 32;

__host__ __device__ inline size_t dw_smem_bytes(int d, int dzld, int lpb, size_t elem)
{
    const size_t tiles = (size_t)DW_ROWS * d * elem + (size_t)DW_ROWS * dzld * sizeof(float);
    const size_t red = (size_t)lpb * 128 * sizeof(float);
    return tiles > red ? tiles : red;
}

template <typename T, int LPB>
__global__ void __launch_bounds__(NT) k_dw_partial(Dims D, const T *__restrict__ Q, const T *__restrict__ K,
                                                    int64_t span, float *__restrict__ part)
{
    extern __shared__ __align__(16) unsigned char dwsm[];
    constexpr int XC = (DW_ROWS * kMaxD * (int)sizeof(T) / 16 + NT - 1) / NT;  // 16-byte pieces per thread
    constexpr int ZC = (DW_ROWS * 64 * 4 / 16 + NT - 1) / NT;
    const int d = D.d, LP = D.LP, ld = D.dzld;
    const T *xs = reinterpret_cast<const T *>(dwsm);
    const float *zs = reinterpret_cast<const float *>(dwsm + (size_t)DW_ROWS * d * sizeof(T));
    const int k = threadIdx.x & 127, g = threadIdx.x >> 7;
    const int64_t bh = blockIdx.y;
    const int64_t r0 = (int64_t)blockIdx.x * span, r1 = min(D.N, r0 + span);
    const int ntile = r1 > r0 ? (int)((r1 - r0 + DW_ROWS - 1) / DW_ROWS) : 0;
    float acc[LPB];
#pragma unroll
    for (int j = 0; j < LPB; ++j) acc[j] = 0.f;
    uint4 px[XC], pz[ZC];
    int nx = 0, nz = 0;  // pieces of the fetched tile
    auto fetch = [&](int it) {
        const int64_t n0 = r0 + (int64_t)(it >> 1) * DW_ROWS;
        const int cnt = (int)min((int64_t)DW_ROWS, r1 - n0);
        const uint4 *X = reinterpret_cast<const uint4 *>(((it & 1) ? K : Q) + (bh * D.N + n0) * d);
        const uint4 *Z = reinterpret_cast<const uint4 *>(((it & 1) ? D.dzk : D.dzq) + (bh * D.N + n0) * ld);
        nx = (int)((size_t)cnt * d * sizeof(T) / 16);
        nz = cnt * ld / 4;
#pragma unroll
        for (int c = 0; c < XC; ++c) {
            const int i = threadIdx.x + c * NT;
            if (i < nx) px[c] = X[i];
        }
#pragma unroll
        for (int c = 0; c < ZC; ++c) {
            const int i = threadIdx.x + c * NT;
            if (i < nz) pz[c] = Z[i];
        }
    };
    if (ntile > 0) fetch(0);
    for (int it = 0; it < 2 * ntile; ++it) {
        const int cnt = (int)min((int64_t)DW_ROWS, r1 - (r0 + (int64_t)(it >> 1) * DW_ROWS));
        __syncthreads();  // the previous tile is summed
#pragma unroll
        for (int c = 0; c < XC; ++c) {
            const int i = threadIdx.x + c * NT;
            if (i < nx) reinterpret_cast<uint4 *>(dwsm)[i] = px[c];
        }
#pragma unroll
        for (int c = 0; c < ZC; ++c) {
            const int i = threadIdx.x + c * NT;
            if (i < nz) reinterpret_cast<uint4 *>(const_cast<float *>(zs))[i] = pz[c];
        }
        __syncthreads();
        if (it + 1 < 2 * ntile) fetch(it + 1);  // in flight while this tile is summed
        if (k < d) {
            for (int r = g; r < cnt; r += 2) {
                const float x = ld_f(xs, (int64_t)r * d + k);
                const float4 *zr = reinterpret_cast<const float4 *>(zs + r * ld);
#pragma unroll
                for (int q = 0; q < LPB / 4; ++q) {
                    if (4 * q < ld) {
                        const float4 z4 = zr[q];
                        acc[4 * q] = fmaf(z4.x, x, acc[4 * q]);
                        acc[4 * q + 1] = fmaf(z4.y, x, acc[4 * q + 1]);
                        acc[4 * q + 2] = fmaf(z4.z, x, acc[4 * q + 2]);
                        acc[4 * q + 3] = fmaf(z4.w, x, acc[4 * q + 3]);
                    }
                }
            }
        }
    }
    __syncthreads();
    float *red = reinterpret_cast<float *>(dwsm);  // [LPB][128], over the tiles
    if (g == 0) {
#pragma unroll
        for (int j = 0; j < LPB; ++j) red[j * 128 + k] = acc[j];
    }
    __syncthreads();
    if (g == 1 && k < d) {
        float *out = part + ((int64_t)bh * gridDim.x + blockIdx.x) * (int64_t)LP * d;
#pragma unroll
        for (int j = 0; j < LPB; ++j)
            if (j < LP) out[(int64_t)j * d + k] = red[j * 128 + k] + acc[j];
    }
}

// Non-causal read-out: O_t = sum_f phi_f(Q_t) A[f] / sum_f phi_f(Q_t) B[f] with S = [A | B]
// ([BH][LR][dv]).  Grid (ceil(N / TT), BH).
template <typename T>
__global__ void __launch_bounds__(NT) k_readout(Dims D, const T *__restrict__ Q,
                                                const float *__restrict__ W,
                                                const float *__restrict__ S, T *__restrict__ O,
                                                unsigned *__restrict__ err)
{
    extern __shared__ float sm[];
    const ReadoutSmem L(D);
    float *ws = sm + L.ws, *xs = sm + L.xs, *fs = sm + L.fs, *inv = sm + L.inv;
    float *sch = sm + L.sch, *outs = sm + L.outs;
    const int64_t bh = blockIdx.y, n0 = (int64_t)blockIdx.x * TT;
    const int cnt = (int)min((int64_t)TT, D.N - n0);
    const int fst = D.LR + 1;
    load_w(head_w(W, D, bh), D, 0, D.L, ws);
    load_rows(Q + bh * D.N * D.d, n0, cnt, D.d, xs);
    __syncthreads();
    featurise(xs, D, ws, 0, D.LR, inv, nullptr, fs, fst);
    float acc[KOUT];
#pragma unroll
    for (int k = 0; k < KOUT; ++k) acc[k] = 0.f;
    const float *Sb = S + bh * D.LR * D.dv;
    for (int f0 = 0; f0 < D.LR; f0 += LRC) {
        const int nf = min(LRC, D.LR - f0);
        __syncthreads();
        for (int i = threadIdx.x; i < nf * D.dv; i += NT) sch[i] = Sb[f0 * D.dv + i];
        __syncthreads();
#pragma unroll
        for (int k = 0; k < KOUT; ++k) {
            const int o = threadIdx.x + k * NT;
            if (o < TT * D.dv) {
                const int t = o / D.dv, c = o - t * D.dv;
                float a = acc[k];
                for (int f = 0; f < nf; ++f) a = fmaf(fs[t * fst + f0 + f], sch[f * D.dv + c], a);
                acc[k] = a;
            }
        }
    }
#pragma unroll
    for (int k = 0; k < KOUT; ++k) {
        const int o = threadIdx.x + k * NT;
        if (o < TT * D.dv) outs[o] = acc[k];
    }
    __syncthreads();
    T *Ob = O + bh * D.N * D.d;
    for (int i = threadIdx.x; i < cnt * D.d; i += NT) {
        const int t = i / D.d, c = i - t * D.d;
        if (c == 0) flag_den(outs[t * D.dv + D.d], err);
        st_f(Ob, (n0 + t) * D.d + c, outs[t * D.dv + c] / outs[t * D.dv + D.d]);
    }
}

// Non-causal backward, query side.  With S = [A | B] and the recomputed phi = phi(Q_t):
//   den_t = phi . B,  g_t = A dO_t (LR numbers),  c_t = dO_t . O_t = phi . g_t / den_t,
//   dphi_t = (g_t - B c_t) / den_t,  dQ_t by the feature chain rule.
// Writes aux[t] = {1/den_t, c_t} for the gradient sketch.  Grid (ceil(N / TT), BH).
template <typename T>
__global__ void __launch_bounds__(NT) k_bwd_query(Dims D, const T *__restrict__ Q,
                                                  const T *__restrict__ dO,
                                                  const float *__restrict__ W,
                                                  const float *__restrict__ S, T *__restrict__ dQ,
                                                  float2 *__restrict__ aux, float *__restrict__ dbpart)
{
    extern __shared__ float sm[];
    const QueryBwdSmem L(D);
    float *ws = sm + L.ws, *xs = sm + L.xs, *ys = sm + L.ys, *fs = sm + L.fs, *gs = sm + L.gs;
    float *us = sm + L.us, *inv = sm + L.inv, *sch = sm + L.sch, *sb = sm + L.sb;
    float *den = sm + L.den, *cc = sm + L.cc, *dz = sm + L.dz, *dx = sm + L.dx, *red = sm + L.red;
    const int64_t bh = blockIdx.y, n0 = (int64_t)blockIdx.x * TT;
    const int cnt = (int)min((int64_t)TT, D.N - n0);
    const int dp = D.d + 1, fst = D.LR + 1;
    load_w(head_w(W, D, bh), D, 0, D.L, ws);
    load_rows(Q + bh * D.N * D.d, n0, cnt, D.d, xs);
    load_rows(dO + bh * D.N * D.d, n0, cnt, D.d, ys);
    __syncthreads();
    featurise(xs, D, ws, 0, D.LR, inv, us, fs, fst);
    const float *Sb = S + bh * D.LR * D.dv;
    for (int f0 = 0; f0 < D.LR; f0 += LRC) {
        const int nf = min(LRC, D.LR - f0);
        __syncthreads();
        for (int i = threadIdx.x; i < nf * D.dv; i += NT) sch[i] = Sb[f0 * D.dv + i];
        __syncthreads();
        for (int f = threadIdx.x; f < nf; f += NT) sb[f0 + f] = sch[f * D.dv + D.d];
        for (int o = threadIdx.x; o < TT * nf; o += NT) {
            const int t = o / nf, f = o - t * nf;
            float g = 0.f;
            for (int c = 0; c < D.d; ++c) g = fmaf(sch[f * D.dv + c], ys[t * dp + c], g);
            gs[t * fst + f0 + f] = g;
        }
    }
    __syncthreads();
    for (int t = threadIdx.x; t < TT; t += NT) {
        float dn = 0.f, pg = 0.f;
        for (int f = 0; f < D.LR; ++f) {
            dn = fmaf(fs[t * fst + f], sb[f], dn);
            pg = fmaf(fs[t * fst + f], gs[t * fst + f], pg);
        }
        den[t] = dn;
        cc[t] = pg / dn;
    }
    __syncthreads();
    for (int o = threadIdx.x; o < TT * D.LR; o += NT) {
        const int t = o / D.LR, f = o - t * D.LR;
        gs[t * fst + f] = (gs[t * fst + f] - sb[f] * cc[t]) / den[t];
    }
    __syncthreads();
    const float db = featurise_backward(xs, D, ws, inv, us, fs, gs, fst, dz, dx, red,
                                        D.dzq ? D.dzq + (bh * D.N + n0) * D.dzld : nullptr, cnt);
    T *dQb = dQ + bh * D.N * D.d;
    for (int i = threadIdx.x; i < cnt * D.d; i += NT) {
        const int t = i / D.d, c = i - t * D.d;
        st_f(dQb, (n0 + t) * D.d + c, dx[t * dp + c]);
    }
    for (int t = threadIdx.x; t < cnt; t += NT) aux[bh * D.N + n0 + t] = make_float2(1.f / den[t], cc[t]);
    store_dbeta_partial(db, red, dbpart, bh);
}

// Non-causal backward, key side.  With G = [dA | dB] = sum_t phi(Q_t) [dO_t/den_t | -c_t/den_t]:
//   dV_j = dA^T phi(K_j),  dphi_j = dA V_j + dB,  dK_j by the feature chain rule.
// Grid (ceil(N / TT), BH).
template <typename T>
__global__ void __launch_bounds__(NT) k_bwd_key(Dims D, const T *__restrict__ K,
                                                const T *__restrict__ V,
                                                const float *__restrict__ W,
                                                const float *__restrict__ G, T *__restrict__ dK,
                                                T *__restrict__ dV, float *__restrict__ dbpart)
{
    extern __shared__ float sm[];
    const KeyBwdSmem L(D);
    float *ws = sm + L.ws, *xs = sm + L.xs, *vs = sm + L.vs, *fs = sm + L.fs, *gs = sm + L.gs;
    float *us = sm + L.us, *inv = sm + L.inv, *sch = sm + L.sch, *dz = sm + L.dz, *dx = sm + L.dx;
    float *red = sm + L.red;
    const int64_t bh = blockIdx.y, n0 = (int64_t)blockIdx.x * TT;
    const int cnt = (int)min((int64_t)TT, D.N - n0);
    const int dp = D.d + 1, fst = D.LR + 1;
    load_w(head_w(W, D, bh), D, 0, D.L, ws);
    load_rows(K + bh * D.N * D.d, n0, cnt, D.d, xs);
    load_values(V + bh * D.N * D.d, n0, cnt, D.d, vs);
    __syncthreads();
    featurise(xs, D, ws, 0, D.LR, inv, us, fs, fst);
    float acc[KOUT];
#pragma unroll
    for (int k = 0; k < KOUT; ++k) acc[k] = 0.f;
    const float *Gb = G + bh * D.LR * D.dv;
    for (int f0 = 0; f0 < D.LR; f0 += LRC) {
        const int nf = min(LRC, D.LR - f0);
        __syncthreads();
        for (int i = threadIdx.x; i < nf * D.dv; i += NT) sch[i] = Gb[f0 * D.dv + i];
        __syncthreads();
#pragma unroll
        for (int k = 0; k < KOUT; ++k) {
            const int o = threadIdx.x + k * NT;
            if (o < TT * D.d) {
                const int t = o / D.d, c = o - t * D.d;
                float a = acc[k];
                for (int f = 0; f < nf; ++f) a = fmaf(fs[t * fst + f0 + f], sch[f * D.dv + c], a);
                acc[k] = a;
            }
        }
        for (int o = threadIdx.x; o < TT * nf; o += NT) {
            const int t = o / nf, f = o - t * nf;
            float g = 0.f;
            for (int c = 0; c <= D.d; ++c) g = fmaf(sch[f * D.dv + c], vs[t * dp + c], g);
            gs[t * fst + f0 + f] = g;
        }
    }
    __syncthreads();
    const float db = featurise_backward(xs, D, ws, inv, us, fs, gs, fst, dz, dx, red,
                                        D.dzk ? D.dzk + (bh * D.N + n0) * D.dzld : nullptr, cnt);
    T *dKb = dK + bh * D.N * D.d, *dVb = dV + bh * D.N * D.d;
#pragma unroll
    for (int k = 0; k < KOUT; ++k) {
        const int o = threadIdx.x + k * NT;
        if (o < TT * D.d) {
            const int t = o / D.d, c = o - t * D.d;
            if (t < cnt) st_f(dVb, (n0 + t) * D.d + c, acc[k]);
        }
    }
    for (int i = threadIdx.x; i < cnt * D.d; i += NT) {
        const int t = i / D.d, c = i - t * D.d;
        st_f(dKb, (n0 + t) * D.d + c, dx[t * dp + c]);
    }
    store_dbeta_partial(db, red, dbpart, bh);
}

// Causal forward over one segment (Algorithm 2 in tiles).  S starts as the sketch of all keys
// before the segment; for each tile: num_t = phi(Q_t) S + sum_{j <= t in tile}
// (phi(Q_t) . phi(K_j)) [V_j | 1], O_t = num_t[:d] / num_t[d]; then S += Phi_K^T [V | 1].
// Grid (nseg, BH).
template <typename T>
__global__ void __launch_bounds__(NT) k_causal_fwd(Dims D, const T *__restrict__ Q,
                                                   const T *__restrict__ K,
                                                   const T *__restrict__ V,
                                                   const float *__restrict__ W,
                                                   const float *__restrict__ S0, int64_t seg_len,
                                                   int nseg, T *__restrict__ O, unsigned *__restrict__ err)
{
    extern __shared__ float sm[];
    const CausalFwdSmem L(D);
    float *ws = sm + L.ws, *S = sm + L.S, *xq = sm + L.xq, *xk = sm + L.xk, *vs = sm + L.vs;
    float *fq = sm + L.fq, *fk = sm + L.fk, *sc = sm + L.sc, *inv = sm + L.inv, *outs = sm + L.outs;
    const int s = blockIdx.x;
    const int64_t bh = blockIdx.y;
    const int fst = D.LR + 1, dv = D.dv, E = D.LR * D.dv;
    load_w(head_w(W, D, bh), D, 0, D.L, ws);
    const float *S0b = S0 + ((int64_t)bh * nseg + s) * E;
    for (int i = threadIdx.x; i < E; i += NT) S[i] = S0b[i];
    const int64_t off = bh * D.N * D.d;
    const int64_t n_end = min(D.N, (int64_t)(s + 1) * seg_len);
    for (int64_t n0 = (int64_t)s * seg_len; n0 < n_end; n0 += TT) {
        const int cnt = (int)min((int64_t)TT, n_end - n0);
        __syncthreads();
        load_rows(Q + off, n0, cnt, D.d, xq);
        load_rows(K + off, n0, cnt, D.d, xk);
        load_values(V + off, n0, cnt, D.d, vs);
        __syncthreads();
        featurise(xq, D, ws, 0, D.LR, inv, nullptr, fq, fst);
        featurise(xk, D, ws, 0, D.LR, inv, nullptr, fk, fst);
        for (int o = threadIdx.x; o < TT * TT; o += NT) {
            const int t = o / TT, j = o - t * TT;
            float a = 0.f;
            if (j <= t && j < cnt)
                for (int f = 0; f < D.LR; ++f) a = fmaf(fq[t * fst + f], fk[j * fst + f], a);
            sc[t * (TT + 1) + j] = a;
        }
        __syncthreads();
        for (int o = threadIdx.x; o < TT * dv; o += NT) {
            const int t = o / dv, c = o - t * dv;
            float a = 0.f;
            for (int f = 0; f < D.LR; ++f) a = fmaf(fq[t * fst + f], S[f * dv + c], a);
            for (int j = 0; j <= t; ++j) a = fmaf(sc[t * (TT + 1) + j], vs[j * dv + c], a);
            outs[o] = a;
        }
        __syncthreads();
        for (int i = threadIdx.x; i < cnt * D.d; i += NT) {
            const int t = i / D.d, c = i - t * D.d;
            if (c == 0) flag_den(outs[t * dv + D.d], err);
            st_f(O + off, (n0 + t) * D.d + c, outs[t * dv + c] / outs[t * dv + D.d]);
        }
        for (int o = threadIdx.x; o < E; o += NT) {
            const int f = o / dv, c = o - f * dv;
            float a = S[o];
            for (int j = 0; j < cnt; ++j) a = fmaf(fk[j * fst + f], vs[j * dv + c], a);
            S[o] = a;
        }
    }
}

// Causal backward, forward-order pass over one segment: recomputes the prefix sketch S_t and
//   den_t = phi(Q_t) . S_t[:, d],  g_t = S_t[:, :d] dO_t,  c_t = phi(Q_t) . g_t / den_t,
//   dphi_Q(t) = (g_t - S_t[:, d] c_t) / den_t,  dQ_t by the feature chain rule,
// and writes aux[t] = {1/den_t, c_t}.  Grid (nseg, BH).
template <typename T>
__global__ void __launch_bounds__(NT) k_causal_bwd_q(Dims D, const T *__restrict__ Q,
                                                     const T *__restrict__ K,
                                                     const T *__restrict__ V,
                                                     const T *__restrict__ dO,
                                                     const float *__restrict__ W,
                                                     const float *__restrict__ S0, int64_t seg_len,
                                                     int nseg, T *__restrict__ dQ,
                                                     float2 *__restrict__ aux, float *__restrict__ dbpart)
{
    extern __shared__ float sm[];
    const CausalBwdSmem L(D);
    float *ws = sm + L.ws, *S = sm + L.S, *xq = sm + L.xq, *xk = sm + L.xk, *vs = sm + L.vs;
    float *ys = sm + L.ys, *fq = sm + L.fq, *fk = sm + L.fk, *gs = sm + L.gs, *us = sm + L.us;
    float *sc = sm + L.sc, *vdo = sm + L.aux2, *invq = sm + L.invq, *invk = sm + L.invk;
    float *den = sm + L.den, *cc = sm + L.cc, *dz = sm + L.dz, *dx = sm + L.dx, *red = sm + L.red;
    const int s = blockIdx.x;
    const int64_t bh = blockIdx.y;
    const int fst = D.LR + 1, dv = D.dv, dp = D.d + 1, E = D.LR * D.dv, TP = TT + 1;
    load_w(head_w(W, D, bh), D, 0, D.L, ws);
    const float *S0b = S0 + ((int64_t)bh * nseg + s) * E;
    for (int i = threadIdx.x; i < E; i += NT) S[i] = S0b[i];
    const int64_t off = bh * D.N * D.d;
    const int64_t n_end = min(D.N, (int64_t)(s + 1) * seg_len);
    float db = 0.f;
    for (int64_t n0 = (int64_t)s * seg_len; n0 < n_end; n0 += TT) {
        const int cnt = (int)min((int64_t)TT, n_end - n0);
        __syncthreads();
        load_rows(Q + off, n0, cnt, D.d, xq);
        load_rows(K + off, n0, cnt, D.d, xk);
        load_values(V + off, n0, cnt, D.d, vs);
        load_rows(dO + off, n0, cnt, D.d, ys);
        __syncthreads();
        featurise(xq, D, ws, 0, D.LR, invq, us, fq, fst);
        featurise(xk, D, ws, 0, D.LR, invk, nullptr, fk, fst);
        for (int o = threadIdx.x; o < TT * TT; o += NT) {
            const int t = o / TT, j = o - t * TT;
            float a = 0.f, b = 0.f;
            if (j <= t && j < cnt) {
                for (int f = 0; f < D.LR; ++f) a = fmaf(fq[t * fst + f], fk[j * fst + f], a);
                for (int c = 0; c < D.d; ++c) b = fmaf(vs[j * dv + c], ys[t * dp + c], b);
            }
            sc[t * TP + j] = a;
            vdo[t * TP + j] = b;
        }
        __syncthreads();
        for (int o = threadIdx.x; o < TT * D.LR; o += NT) {
            const int t = o / D.LR, f = o - t * D.LR;
            float g = 0.f;
            for (int c = 0; c < D.d; ++c) g = fmaf(S[f * dv + c], ys[t * dp + c], g);
            for (int j = 0; j <= t; ++j) g = fmaf(fk[j * fst + f], vdo[t * TP + j], g);
            gs[t * fst + f] = g;
        }
        __syncthreads();
        for (int t = threadIdx.x; t < TT; t += NT) {
            float dn = 0.f, pg = 0.f;
            for (int f = 0; f < D.LR; ++f) {
                dn = fmaf(fq[t * fst + f], S[f * dv + D.d], dn);
                pg = fmaf(fq[t * fst + f], gs[t * fst + f], pg);
            }
            for (int j = 0; j <= t; ++j) dn += sc[t * TP + j];
            den[t] = dn;
            cc[t] = pg / dn;
        }
        __syncthreads();
        for (int o = threadIdx.x; o < TT * D.LR; o += NT) {
            const int t = o / D.LR, f = o - t * D.LR;
            float sb = S[f * dv + D.d];
            for (int j = 0; j <= t && j < cnt; ++j) sb += fk[j * fst + f];
            gs[t * fst + f] = (gs[t * fst + f] - sb * cc[t]) / den[t];
        }
        __syncthreads();
        db += featurise_backward(xq, D, ws, invq, us, fq, gs, fst, dz, dx, red,
                                 D.dzq ? D.dzq + (bh * D.N + n0) * D.dzld : nullptr, cnt);
        for (int i = threadIdx.x; i < cnt * D.d; i += NT) {
            const int t = i / D.d, c = i - t * D.d;
            st_f(dQ + off, (n0 + t) * D.d + c, dx[t * dp + c]);
        }
        for (int t = threadIdx.x; t < cnt; t += NT) aux[bh * D.N + n0 + t] = make_float2(1.f / den[t], cc[t]);
        for (int o = threadIdx.x; o < E; o += NT) {
            const int f = o / dv, c = o - f * dv;
            float a = S[o];
            for (int j = 0; j < cnt; ++j) a = fmaf(fk[j * fst + f], vs[j * dv + c], a);
            S[o] = a;
        }
    }
    store_dbeta_partial(db, red, dbpart, bh);
}

// Causal backward, reverse-order pass over one segment.  G starts as the suffix gradient
// sketch of all queries after the segment; tiles are visited last to first.  With
// y_t = [dO_t / den_t | -c_t / den_t] and G_j = G + sum_{t >= j in tile} phi(Q_t) y_t:
//   dV_j = G_j[:, :d]^T phi(K_j),  dphi_K(j) = G_j [V_j | 1],  dK_j by the chain rule;
// then G += Phi_Q^T y.  Grid (nseg, BH).
template <typename T>
__global__ void __launch_bounds__(NT) k_causal_bwd_kv(Dims D, const T *__restrict__ Q,
                                                      const T *__restrict__ K,
                                                      const T *__restrict__ V,
                                                      const T *__restrict__ dO,
                                                      const float2 *__restrict__ aux,
                                                      const float *__restrict__ W,
                                                      const float *__restrict__ G0, int64_t seg_len,
                                                      int nseg, T *__restrict__ dK,
                                                      T *__restrict__ dV, float *__restrict__ dbpart)
{
    extern __shared__ float sm[];
    const CausalBwdSmem L(D);
    float *ws = sm + L.ws, *G = sm + L.S, *xq = sm + L.xq, *xk = sm + L.xk, *vs = sm + L.vs;
    float *ys = sm + L.ys, *fq = sm + L.fq, *fk = sm + L.fk, *gs = sm + L.gs, *us = sm + L.us;
    float *sc = sm + L.sc, *vy = sm + L.aux2, *invq = sm + L.invq, *invk = sm + L.invk;
    float *dz = sm + L.dz, *dx = sm + L.dx, *red = sm + L.red;
    const int s = blockIdx.x;
    const int64_t bh = blockIdx.y;
    const int fst = D.LR + 1, dv = D.dv, dp = D.d + 1, E = D.LR * D.dv, TP = TT + 1;
    load_w(head_w(W, D, bh), D, 0, D.L, ws);
    const float *G0b = G0 + ((int64_t)bh * nseg + s) * E;
    for (int i = threadIdx.x; i < E; i += NT) G[i] = G0b[i];
    const int64_t off = bh * D.N * D.d;
    const int64_t n_begin = (int64_t)s * seg_len;
    const int64_t n_end = min(D.N, n_begin + seg_len);
    if (n_begin >= n_end) return;
    const int64_t last = n_begin + ((n_end - 1 - n_begin) / TT) * TT;
    float db = 0.f;
    for (int64_t n0 = last; n0 >= n_begin; n0 -= TT) {
        const int cnt = (int)min((int64_t)TT, n_end - n0);
        __syncthreads();
        load_rows(Q + off, n0, cnt, D.d, xq);
        load_rows(K + off, n0, cnt, D.d, xk);
        load_values(V + off, n0, cnt, D.d, vs);
        for (int i = threadIdx.x; i < TT * dv; i += NT) {
            const int t = i / dv, c = i - t * dv;
            float v = 0.f;
            if (t < cnt) {
                const float2 q = aux[bh * D.N + n0 + t];
                v = c < D.d ? ld_f(dO + off, (n0 + t) * D.d + c) * q.x : -q.y * q.x;
            }
            ys[t * dp + c] = v;
        }
        __syncthreads();
        featurise(xq, D, ws, 0, D.LR, invq, nullptr, fq, fst);
        featurise(xk, D, ws, 0, D.LR, invk, us, fk, fst);
        for (int o = threadIdx.x; o < TT * TT; o += NT) {
            const int j = o / TT, t = o - j * TT;
            float a = 0.f, b = 0.f;
            if (t >= j && t < cnt) {
                for (int f = 0; f < D.LR; ++f) a = fmaf(fk[j * fst + f], fq[t * fst + f], a);
                for (int c = 0; c <= D.d; ++c) b = fmaf(vs[j * dv + c], ys[t * dp + c], b);
            }
            sc[j * TP + t] = a;
            vy[j * TP + t] = b;
        }
        __syncthreads();
        float acc[KOUT];
#pragma unroll
        for (int k = 0; k < KOUT; ++k) {
            acc[k] = 0.f;
            const int o = threadIdx.x + k * NT;
            if (o < TT * D.d) {
                const int j = o / D.d, c = o - j * D.d;
                float a = 0.f;
                for (int f = 0; f < D.LR; ++f) a = fmaf(fk[j * fst + f], G[f * dv + c], a);
                for (int t = j; t < TT; ++t) a = fmaf(sc[j * TP + t], ys[t * dp + c], a);
                acc[k] = a;
            }
        }
        for (int o = threadIdx.x; o < TT * D.LR; o += NT) {
            const int j = o / D.LR, f = o - j * D.LR;
            float g = 0.f;
            for (int c = 0; c <= D.d; ++c) g = fmaf(G[f * dv + c], vs[j * dv + c], g);
            for (int t = j; t < TT; ++t) g = fmaf(fq[t * fst + f], vy[j * TP + t], g);
            gs[j * fst + f] = g;
        }
        __syncthreads();
        db += featurise_backward(xk, D, ws, invk, us, fk, gs, fst, dz, dx, red,
                                 D.dzk ? D.dzk + (bh * D.N + n0) * D.dzld : nullptr, cnt);
#pragma unroll
        for (int k = 0; k < KOUT; ++k) {
            const int o = threadIdx.x + k * NT;
            if (o < TT * D.d) {
                const int j = o / D.d, c = o - j * D.d;
                if (j < cnt) st_f(dV + off, (n0 + j) * D.d + c, acc[k]);
            }
        }
        for (int i = threadIdx.x; i < cnt * D.d; i += NT) {
            const int t = i / D.d, c = i - t * D.d;
            st_f(dK + off, (n0 + t) * D.d + c, dx[t * dp + c]);
        }
        for (int o = threadIdx.x; o < E; o += NT) {
            const int f = o / dv, c = o - f * dv;
            float a = G[o];
            for (int t = 0; t < cnt; ++t) a = fmaf(fq[t * fst + f], ys[t * dp + c], a);
            G[o] = a;
        }
    }
    store_dbeta_partial(db, red, dbpart, bh);
}

}  // namespace gen

// ------------------------------------------------------------------ host launchers

namespace {

template <typename Kern>
cudaError_t prep(Kern k, size_t smem)
{
    if (smem > 48 * 1024) return cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    return cudaSuccess;
}

int lr_chunks(const Dims &D) { return (D.LR + gen::LRC - 1) / gen::LRC; }

}  // namespace

size_t generic_smem_bytes(const Dims &D, GenericKernel which)
{
    switch (which) {
        case GenericKernel::Sketch: return gen::SketchSmem(D, std::min(D.L, gen::LRC / D.R + 2)).lay.bytes();
        case GenericKernel::Readout: return gen::ReadoutSmem(D).lay.bytes();
        case GenericKernel::QueryBwd: return gen::QueryBwdSmem(D).lay.bytes();
        case GenericKernel::KeyBwd: return gen::KeyBwdSmem(D).lay.bytes();
        case GenericKernel::CausalFwd: return gen::CausalFwdSmem(D).lay.bytes();
        case GenericKernel::CausalBwd: return gen::CausalBwdSmem(D).lay.bytes();
    }
    return 0;
}

int generic_token_tile() { return gen::TT; }

template <typename T>
cudaError_t launch_sketch(const Dims &D, const T *X, const T *Y, const float2 *aux, const float *W,
                          int64_t seg_len, int nsplit, float *part, int mode, cudaStream_t st)
{
    const size_t smem = generic_smem_bytes(D, GenericKernel::Sketch);
    cudaError_t e = prep(gen::k_sketch<T>, smem);
    if (e != cudaSuccess) return e;
    dim3 grid(nsplit, lr_chunks(D), (unsigned)D.BH);
    return launch_kernel(mode == 0 ? "sketch_keys" : "sketch_grad", gen::k_sketch<T>, grid, dim3(gen::NT), smem, st,
                         D, X, Y, aux, W, seg_len, nsplit, part, mode);
}

cudaError_t launch_combine(const Dims &D, const float *part, float *out, int nsplit, int mode, cudaStream_t st)
{
    const int64_t E = (int64_t)D.LR * D.dv;
    dim3 grid((unsigned)std::min<int64_t>((E + 255) / 256, 64), (unsigned)D.BH);
    return launch_kernel("combine", gen::k_combine, grid, dim3(256), 0, st, part, out, E, nsplit, mode);
}

template <typename T>
cudaError_t launch_dw(const Dims &D, const T *Q, const T *K, int nblk, float *part, float *dW, cudaStream_t st)
{
    const int64_t span = (((D.N + nblk - 1) / nblk + gen::DW_ROWS - 1) / gen::DW_ROWS) * gen::DW_ROWS;
    const dim3 grid((unsigned)nblk, (unsigned)D.BH);
    const int lpb = D.dzld <= 4 ? 4 : D.dzld <= 8 ? 8 : D.dzld <= 16 ? 16 : D.dzld <= 32 ? 32 : 64;
    const size_t smem = gen::dw_smem_bytes(D.d, D.dzld, lpb, sizeof(T));
    cudaError_t e;
    switch (lpb) {
        case 4: e = launch_kernel("dw_partial", gen::k_dw_partial<T, 4>, grid, dim3(gen::NT), smem, st, D, Q, K, span, part); break;
        case 8: e = launch_kernel("dw_partial", gen::k_dw_partial<T, 8>, grid, dim3(gen::NT), smem, st, D, Q, K, span, part); break;
        case 16: e = launch_kernel("dw_partial", gen::k_dw_partial<T, 16>, grid, dim3(gen::NT), smem, st, D, Q, K, span, part); break;
        case 32: e = launch_kernel("dw_partial", gen::k_dw_partial<T, 32>, grid, dim3(gen::NT), smem, st, D, Q, K, span, part); break;
        default: e = launch_kernel("dw_partial", gen::k_dw_partial<T, 64>, grid, dim3(gen::NT), smem, st, D, Q, K, span, part); break;
    }
    if (e != cudaSuccess) return e;
    const int64_t E = (int64_t)D.LP * D.d;
    const dim3 cgrid((unsigned)std::min<int64_t>((E + 255) / 256, 64), (unsigned)D.BH);
    return launch_kernel("dw_combine", gen::k_combine, cgrid, dim3(256), 0, st, (const float *)part, dW, E, nblk, 0);
}

cudaError_t launch_dbeta_combine(const Dims &D, const float *part, int slots, float *dbeta, cudaStream_t st)
{
    return launch_kernel("dbeta_combine", gen::k_dbeta_combine, dim3((unsigned)D.BH), dim3(256), 0, st, part,
                         slots, D.BH, dbeta);
}

template <typename T>
cudaError_t launch_readout(const Dims &D, const T *Q, const float *W, const float *S, T *O, unsigned *err,
                           cudaStream_t st)
{
    const size_t smem = generic_smem_bytes(D, GenericKernel::Readout);
    cudaError_t e = prep(gen::k_readout<T>, smem);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)((D.N + gen::TT - 1) / gen::TT), (unsigned)D.BH);
    return launch_kernel("readout", gen::k_readout<T>, grid, dim3(gen::NT), smem, st, D, Q, W, S, O, err);
}

template <typename T>
cudaError_t launch_bwd_query(const Dims &D, const T *Q, const T *dO, const float *W, const float *S, T *dQ,
                             float2 *aux, float *dbpart, cudaStream_t st)
{
    const size_t smem = generic_smem_bytes(D, GenericKernel::QueryBwd);
    cudaError_t e = prep(gen::k_bwd_query<T>, smem);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)((D.N + gen::TT - 1) / gen::TT), (unsigned)D.BH);
    return launch_kernel("bwd_query", gen::k_bwd_query<T>, grid, dim3(gen::NT), smem, st, D, Q, dO, W, S, dQ, aux,
                         dbpart);
}

template <typename T>
cudaError_t launch_bwd_key(const Dims &D, const T *K, const T *V, const float *W, const float *G, T *dK, T *dV,
                           float *dbpart, cudaStream_t st)
{
    const size_t smem = generic_smem_bytes(D, GenericKernel::KeyBwd);
    cudaError_t e = prep(gen::k_bwd_key<T>, smem);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)((D.N + gen::TT - 1) / gen::TT), (unsigned)D.BH);
    return launch_kernel("bwd_key", gen::k_bwd_key<T>, grid, dim3(gen::NT), smem, st, D, K, V, W, G, dK, dV,
                         dbpart);
}

template <typename T>
cudaError_t launch_causal_fwd(const Dims &D, const T *Q, const T *K, const T *V, const float *W, const float *S0,
                              int64_t seg_len, int nseg, T *O, unsigned *err, cudaStream_t st)
{
    const size_t smem = generic_smem_bytes(D, GenericKernel::CausalFwd);
    cudaError_t e = prep(gen::k_causal_fwd<T>, smem);
    if (e != cudaSuccess) return e;
    dim3 grid(nseg, (unsigned)D.BH);
    return launch_kernel("causal_fwd", gen::k_causal_fwd<T>, grid, dim3(gen::NT), smem, st, D, Q, K, V, W, S0,
                         seg_len, nseg, O, err);
}

template <typename T>
cudaError_t launch_causal_bwd_q(const Dims &D, const T *Q, const T *K, const T *V, const T *dO, const float *W,
                                const float *S0, int64_t seg_len, int nseg, T *dQ, float2 *aux, float *dbpart,
                                cudaStream_t st)
{
    const size_t smem = generic_smem_bytes(D, GenericKernel::CausalBwd);
    cudaError_t e = prep(gen::k_causal_bwd_q<T>, smem);
    if (e != cudaSuccess) return e;
    dim3 grid(nseg, (unsigned)D.BH);
    return launch_kernel("causal_bwd_q", gen::k_causal_bwd_q<T>, grid, dim3(gen::NT), smem, st, D, Q, K, V, dO, W,
                         S0, seg_len, nseg, dQ, aux, dbpart);
}

template <typename T>
cudaError_t launch_causal_bwd_kv(const Dims &D, const T *Q, const T *K, const T *V, const T *dO,
                                 const float2 *aux, const float *W, const float *G0, int64_t seg_len, int nseg,
                                 T *dK, T *dV, float *dbpart, cudaStream_t st)
{
    const size_t smem = generic_smem_bytes(D, GenericKernel::CausalBwd);
    cudaError_t e = prep(gen::k_causal_bwd_kv<T>, smem);
    if (e != cudaSuccess) return e;
    dim3 grid(nseg, (unsigned)D.BH);
    return launch_kernel("causal_bwd_kv", gen::k_causal_bwd_kv<T>, grid, dim3(gen::NT), smem, st, D, Q, K, V, dO,
                         aux, W, G0, seg_len, nseg, dK, dV, dbpart);
}

#define RACE_INSTANTIATE(T)                                                                                    \
    template cudaError_t launch_sketch<T>(const Dims &, const T *, const T *, const float2 *, const float *,   \
                                          int64_t, int, float *, int, cudaStream_t);                           \
    template cudaError_t launch_readout<T>(const Dims &, const T *, const float *, const float *, T *,         \
                                           unsigned *, cudaStream_t);                                          \
    template cudaError_t launch_bwd_query<T>(const Dims &, const T *, const T *, const float *, const float *, \
                                             T *, float2 *, float *, cudaStream_t);                            \
    template cudaError_t launch_bwd_key<T>(const Dims &, const T *, const T *, const float *, const float *,   \
                                           T *, T *, float *, cudaStream_t);                                   \
    template cudaError_t launch_causal_fwd<T>(const Dims &, const T *, const T *, const T *, const float *,    \
                                              const float *, int64_t, int, T *, unsigned *, cudaStream_t);     \
    template cudaError_t launch_causal_bwd_q<T>(const Dims &, const T *, const T *, const T *, const T *,      \
                                                const float *, const float *, int64_t, int, T *, float2 *,     \
                                                float *, cudaStream_t);                                        \
    template cudaError_t launch_causal_bwd_kv<T>(const Dims &, const T *, const T *, const T *, const T *,     \
                                                 const float2 *, const float *, const float *, int64_t, int,   \
                                                 T *, T *, float *, cudaStream_t);                      \
    template cudaError_t launch_dw<T>(const Dims &, const T *, const T *, int, float *, float *, cudaStream_t);

RACE_INSTANTIATE(float)
RACE_INSTANTIATE(__nv_bfloat16)

}  // namespace race
