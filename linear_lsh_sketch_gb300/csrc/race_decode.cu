// race_decode.cu -- one causal decode step of RACE attention per (batch, head), CUDA cores.
//
// The recurrent form of Algorithm 2 ("RACE Attention" slides, frame "Causality is a prefix update
// of the same statistics"): the new key is added to the head's prefix sketch [A | B] (L R rows of
// d + 1 floats), then the new query reads it:
//
//     S += phi(k) [v | 1],        o = phi(q) . S[:, :d] / phi(q) . S[:, d]
//
// One CTA per (b, h).  The block normalises q and k, projects them (u = tanh(W xhat)) and forms
// their bucket probabilities in the product form phi_r = prod_t sigmoid(2 beta u_t v_{r,t}) (equal
// to the softmax over the 2^P corners); then the 8 warps split the sketch rows (lanes on
// consecutive columns), add the key, write the rows back and accumulate partial read-outs that a
// fixed-order shared-memory sum combines.  fp32 throughout; the work per step is one pass over
// the sketch, so a decode batch is bound by reading and writing it.
#include "race_launch.h"

namespace race {
namespace dec {

constexpr int NT = 256;
constexpr int MAXD = 128, MAXLP = 64, MAXLR = 256;

template <typename T>
__global__ void __launch_bounds__(NT) k_decode(const T *__restrict__ q, const T *__restrict__ k,
                                               const T *__restrict__ v, const float *__restrict__ W, Dims D,
                                               float *__restrict__ S, T *__restrict__ o)
{
    __shared__ float xs[2][MAXD];   // the q and k rows
    __shared__ float inv[2];        // 1 / |row| (0 for a zero row: its buckets are uniform)
    __shared__ float us[2][MAXLP];  // u = tanh(W xhat)
    __shared__ float ph[2][MAXLR];  // bucket probabilities of q and k
    __shared__ float den_s;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t bh = blockIdx.x;
    const int d = D.d, LP = D.LP, LR = D.LR, P = D.P, R = D.R;

    for (int i = tid; i < 2 * d; i += NT) {
        const int side = i >= d, c = i - side * d;
        xs[side][c] = ld_f(side ? k : q, bh * d + c);
    }
    __syncthreads();
    if (warp < 2) {  // warp 0: |q|^2, warp 1: |k|^2
        float ss = 0.f;
        for (int c = lane; c < d; c += 32) ss = fmaf(xs[warp][c], xs[warp][c], ss);
#pragma unroll
        for (int m = 16; m > 0; m >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, m);
        if (lane == 0) inv[warp] = ss > 0.f ? rsqrtf(ss) : 0.f;
    }
    __syncthreads();
    if (tid < 2 * MAXLP) {  // one projection per thread: side tid / MAXLP, row p = l P + t of W
        const int side = tid / MAXLP, p = tid - side * MAXLP;
        if (p < LP) {
            const float *w = head_w(W, D, bh) + (int64_t)p * d;
            float z = 0.f;
            for (int c = 0; c < d; ++c) z = fmaf(w[c], xs[side][c], z);
            us[side][p] = tanhf(z * inv[side]);
        }
    }
    __syncthreads();
    for (int i = tid; i < 2 * LR; i += NT) {  // phi_r of table l for each side
        const int side = i >= LR, j = i - side * LR, l = j / R, r = j - l * R;
        float pr = 1.f;
        for (int t = 0; t < P; ++t) {
            const float s = ((r >> t) & 1) ? 1.f : -1.f;
            pr *= 1.f / (1.f + __expf(-2.f * D.beta * us[side][l * P + t] * s));
        }
        ph[side][j] = pr;
    }
    __syncthreads();
    // warp w takes sketch rows w, w + 8, ...; lane l columns l, l + 32, ... (up to 5 of the d + 1):
    // all of a thread's loads are independent, and each warp's accesses to a row are contiguous
    constexpr int NW = NT / 32, CPL = (MAXD + 1 + 31) / 32;
    float acc[CPL], vc[CPL];
#pragma unroll
    for (int m = 0; m < CPL; ++m) {
        const int c = lane + 32 * m;
        acc[m] = 0.f;
        vc[m] = c < d ? ld_f(v, bh * d + c) : 1.f;
    }
    float *Sbh = S + bh * (int64_t)LR * (d + 1);
    for (int j = warp; j < LR; j += NW) {
        float *row = Sbh + (int64_t)j * (d + 1);
        const float pk = ph[1][j], pq = ph[0][j];
#pragma unroll
        for (int m = 0; m < CPL; ++m) {
            const int c = lane + 32 * m;
            if (c <= d) {
                const float sv = fmaf(pk, vc[m], row[c]);
                row[c] = sv;
                acc[m] = fmaf(pq, sv, acc[m]);
            }
        }
    }
    // per-warp partial read-outs -> column sums (fixed order over the warps)
    __shared__ float part[NW][CPL * 32];
#pragma unroll
    for (int m = 0; m < CPL; ++m) part[warp][lane + 32 * m] = acc[m];
    __syncthreads();
    if (tid <= d) {
        float sum = 0.f;
#pragma unroll
        for (int w = 0; w < NW; ++w) sum += part[w][tid];
        if (tid == d) den_s = sum;
        part[0][tid] = sum;
    }
    __syncthreads();
    if (tid < d) st_f(o, bh * d + tid, part[0][tid] / den_s);
}

}  // namespace dec

bool decode_supported(const Dims &D) { return D.d <= dec::MAXD && D.LP <= dec::MAXLP && D.LR <= dec::MAXLR; }

template <typename T>
cudaError_t launch_decode(const Dims &D, const T *q, const T *k, const T *v, const float *W, float *S, T *o,
                          cudaStream_t st)
{
    return launch_kernel("decode", dec::k_decode<T>, dim3((unsigned)D.BH), dim3(dec::NT), 0, st, q, k, v, W, D, S, o);
}

template cudaError_t launch_decode<float>(const Dims &, const float *, const float *, const float *, const float *,
                                          float *, float *, cudaStream_t);
template cudaError_t launch_decode<bf16_t>(const Dims &, const bf16_t *, const bf16_t *, const bf16_t *,
                                           const float *, float *, bf16_t *, cudaStream_t);

}  // namespace race
