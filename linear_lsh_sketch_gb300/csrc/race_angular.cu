// race_angular.cu -- exact angular attention, O(N^2), CUDA cores.
//
// The kernel RACE's soft hash estimates ("RACE Attention" slides, frame "Choose a nonnegative
// kernel that can be sketched", paper Eqs. (3)-(4); with gamma = P it is the collision rate of a
// P-bit hard hash, frame "A hash collision estimates a powered angular kernel"):
//
//     O_i = sum_j S_ij V_j / sum_j S_ij,     S_ij = (1 - theta_ij / pi)^gamma,
//
// over j <= i when causal, theta_ij the angle between Q_i and K_j.  It is the exact reference
// for measuring the approximation error of the linear-time layer; it has no sketch.
//
// The angle is taken as theta = 2 atan2(|a - b|, |a + b|) for the unit rows a, b (|a - b| =
// 2 sin(theta / 2), |a + b| = 2 cos(theta / 2)), which keeps full relative accuracy at every
// angle, where arccos of a rounded cosine loses half the digits near 0 and pi.  A zero row is at
// angle pi / 2 to every row (the value uniform soft buckets give).
//
// One CTA per (tile of TQ queries, b, h): the queries stay in shared memory as unit rows; key
// tiles of TK unit rows and their values stream through; each thread forms TQ * TK / NT weights,
// then accumulates its outputs over the tile in a fixed order, so results are deterministic.
#include "race_launch.h"

namespace race {
namespace ang {

constexpr int NT = 256;
constexpr int TQ = 32, TK = 32;
constexpr int OPT = (TQ * (kMaxD + 1) + NT - 1) / NT;  // outputs per thread (d columns + the mass)

// Dynamic shared memory: query, key and value tiles with row stride d + 1 (floats), the tile's
// weights [TQ][TK + 1], and three per-row vectors.
__host__ __device__ inline size_t smem_floats(int d) { return (size_t)(TQ + 2 * TK) * (d + 1) + TQ * (TK + 1) + 3 * 32; }

// Unit copies of rows [row0, row0 + cnt) into xs[rows][d + 1] (zero rows stay zero, rows past
// cnt are zero) and nonzero-row flags into nz[].
template <typename T>
__device__ void load_unit_rows(const T *__restrict__ X, int64_t row0, int cnt, int rows, int d, float *xs,
                               float *nz, float *red)
{
    const int DP = d + 1;
    for (int i = threadIdx.x; i < rows * d; i += NT) {
        const int t = i / d, k = i - t * d;
        xs[t * DP + k] = t < cnt ? ld_f(X, (row0 + t) * d + k) : 0.f;
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int t = warp; t < rows; t += NT / 32) {  // one warp per row: sum of squares, fixed order
        float ss = 0.f;
        for (int k = lane; k < d; k += 32) ss = fmaf(xs[t * DP + k], xs[t * DP + k], ss);
#pragma unroll
        for (int m = 16; m > 0; m >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, m);
        if (lane == 0) red[t] = ss;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < rows * d; i += NT) {
        const int t = i / d, k = i - t * d;
        const float ss = red[t];
        xs[t * DP + k] = ss > 0.f ? xs[t * DP + k] / sqrtf(ss) : 0.f;
    }
    for (int t = threadIdx.x; t < rows; t += NT) nz[t] = red[t] > 0.f ? 1.f : 0.f;
    __syncthreads();
}

template <typename T>
__global__ void __launch_bounds__(NT) k_angular(Dims D, const T *__restrict__ Q, const T *__restrict__ K,
                                                const T *__restrict__ V, float gamma, int causal,
                                                T *__restrict__ O)
{
    extern __shared__ float sm[];
    const int d = D.d, DP = d + 1;
    float *qs = sm, *ks = qs + TQ * DP, *vs = ks + TK * DP, *w = vs + TK * DP;  // w: [TQ][TK + 1]
    float *qnz = w + TQ * (TK + 1), *knz = qnz + 32, *red = knz + 32;
    const int64_t bh = blockIdx.y, n0 = (int64_t)blockIdx.x * TQ;
    const int qcnt = (int)min((int64_t)TQ, D.N - n0);
    const int64_t off = bh * D.N * d;
    const float pi = 3.14159265358979f;
    load_unit_rows(Q + off, n0, qcnt, TQ, d, qs, qnz, red);

    float acc[OPT];
#pragma unroll
    for (int k = 0; k < OPT; ++k) acc[k] = 0.f;
    const int64_t kend = causal ? min(D.N, n0 + qcnt) : D.N;
    for (int64_t j0 = 0; j0 < kend; j0 += TK) {
        const int kcnt = (int)min((int64_t)TK, kend - j0);
        load_unit_rows(K + off, j0, kcnt, TK, d, ks, knz, red);
        for (int i = threadIdx.x; i < TK * d; i += NT) {
            const int t = i / d, c = i - t * d;
            vs[t * DP + c] = t < kcnt ? ld_f(V + off, (j0 + t) * d + c) : 0.f;
        }
        // weights of the tile's (query, key) pairs
        for (int pr = threadIdx.x; pr < TQ * TK; pr += NT) {
            const int tq = pr / TK, tk = pr - tq * TK;
            const int64_t i = n0 + tq, j = j0 + tk;
            float s = 0.f;
            if (tq < qcnt && tk < kcnt && (!causal || j <= i)) {
                float theta;
                if (qnz[tq] == 0.f || knz[tk] == 0.f) {
                    theta = 0.5f * pi;
                } else {
                    float dm = 0.f, dp = 0.f;
                    for (int c = 0; c < d; ++c) {
                        const float a = qs[tq * DP + c], b = ks[tk * DP + c];
                        dm = fmaf(a - b, a - b, dm);
                        dp = fmaf(a + b, a + b, dp);
                    }
                    theta = 2.f * atan2f(sqrtf(dm), sqrtf(dp));
                }
                s = powf(fmaxf(0.f, 1.f - theta / pi), gamma);
            }
            w[tq * (TK + 1) + tk] = s;
        }
        __syncthreads();
        // this thread's outputs: column c of query tq (c = d is the mass column)
#pragma unroll
        for (int k = 0; k < OPT; ++k) {
            const int o = threadIdx.x + k * NT;
            if (o < TQ * (d + 1)) {
                const int tq = o / (d + 1), c = o - tq * (d + 1);
                float a = acc[k];
                if (c < d) {
                    for (int tk = 0; tk < kcnt; ++tk) a = fmaf(w[tq * (TK + 1) + tk], vs[tk * DP + c], a);
                } else {
                    for (int tk = 0; tk < kcnt; ++tk) a += w[tq * (TK + 1) + tk];
                }
                acc[k] = a;
            }
        }
        __syncthreads();
    }
    // O = num / den: the mass column of each query goes through shared memory
    float *den = red;
#pragma unroll
    for (int k = 0; k < OPT; ++k) {
        const int o = threadIdx.x + k * NT;
        if (o < TQ * (d + 1)) {
            const int tq = o / (d + 1), c = o - tq * (d + 1);
            if (c == d) den[tq] = acc[k];
        }
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < OPT; ++k) {
        const int o = threadIdx.x + k * NT;
        if (o < TQ * (d + 1)) {
            const int tq = o / (d + 1), c = o - tq * (d + 1);
            if (c < d && tq < qcnt) st_f(O + off, (n0 + tq) * d + c, acc[k] / den[tq]);
        }
    }
}

}  // namespace ang

template <typename T>
cudaError_t launch_angular(const Dims &D, const T *Q, const T *K, const T *V, float gamma, int causal, T *O,
                           cudaStream_t st)
{
    const size_t smem = ang::smem_floats(D.d) * sizeof(float);
    cudaError_t e = cudaFuncSetAttribute(ang::k_angular<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)((D.N + ang::TQ - 1) / ang::TQ), (unsigned)D.BH);
    return launch_kernel("angular", ang::k_angular<T>, grid, dim3(ang::NT), smem, st, D, Q, K, V, gamma, causal, O);
}

template cudaError_t launch_angular<float>(const Dims &, const float *, const float *, const float *, float, int,
                                           float *, cudaStream_t);
template cudaError_t launch_angular<bf16_t>(const Dims &, const bf16_t *, const bf16_t *, const bf16_t *, float,
                                            int, bf16_t *, cudaStream_t);

}  // namespace race
