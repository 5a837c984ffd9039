// race_decode.cu -- one causal decode step of RACE attention per (batch, head), CUDA cores.
//
// The recurrent form of Algorithm 2 ("RACE Attention" slides, frame "Causality is a prefix update
// of the same statistics"): the new key is added to the head's prefix sketch [A | B] (L R rows of
// d + 1 floats), then the new query reads it:
//
//     S += phi(k) [v | 1],        o = phi(q) . S[:, :d] / phi(q) . S[:, d]
//
// One CTA per (b, h).  Each warp first loads its first sketch rows into registers (they do not
// depend on the token), so that their latency overlaps the featurisation.  The warps then share
// the norms and the 2 L P projections z = w . x (lanes along d, butterfly sums), form
// u = tanh(z / |x|) and the bucket probabilities in the product form
// phi_r = prod_t sigmoid(2 beta u_t v_{r,t}) (equal to the softmax over the 2^P corners).  Last,
// the 8 warps split the sketch rows (lanes on consecutive columns), add the key, write the rows
// back and accumulate partial read-outs that a fixed-order shared-memory sum combines.  fp32
// throughout; the work per step is one pass over the sketch, so a decode batch is bound by
// reading and writing it.
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
    __shared__ float zs[2][MAXLP];  // z = W x (unnormalised projections)
    __shared__ float ph[2][MAXLR];  // bucket probabilities of q and k
    __shared__ float den_s;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t bh = blockIdx.x;
    const int d = D.d, LP = D.LP, LR = D.LR, P = D.P, R = D.R;
    constexpr int NW = NT / 32, CPL = (MAXD + 1 + 31) / 32;
    float *Sbh = S + bh * (int64_t)LR * (d + 1);

    // the warp's first NPF sketch rows (w, w + 8, ...), loaded before anything they wait for
    constexpr int NPF = 4;
    float pre[NPF][CPL];
#pragma unroll
    for (int f = 0; f < NPF; ++f) {
        const int j = warp + NW * f;
#pragma unroll
        for (int m = 0; m < CPL; ++m) {
            const int c = lane + 32 * m;
            pre[f][m] = (j < LR && c <= d) ? Sbh[(int64_t)j * (d + 1) + c] : 0.f;
        }
    }
    for (int i = tid; i < 2 * d; i += NT) {
        const int side = i >= d, c = i - side * d;
        xs[side][c] = ld_f(side ? k : q, bh * d + c);
    }
    __syncthreads();
    // warp-parallel: task 0 / 1 = |q|^2 / |k|^2, task 2 + 2 p + side = projection p of that side;
    // lanes take columns lane, lane + 32, ..., then a butterfly sum (same order on every run)
    const float *Wh = head_w(W, D, bh);
    for (int task = warp; task < 2 + 2 * LP; task += NW) {
        const int side = task < 2 ? task : (task - 2) & 1;
        const float *w = task < 2 ? xs[side] : Wh + (int64_t)((task - 2) >> 1) * d;
        float s = 0.f;
        for (int c = lane; c < d; c += 32) s = fmaf(w[c], xs[side][c], s);
#pragma unroll
        for (int m = 16; m > 0; m >>= 1) s += __shfl_xor_sync(0xffffffffu, s, m);
        if (lane == 0) {
            if (task < 2)
                inv[side] = s > 0.f ? rsqrtf(s) : 0.f;
            else
                zs[side][(task - 2) >> 1] = s;
        }
    }
    __syncthreads();
    for (int i = tid; i < 2 * LR; i += NT) {  // phi_r of table l for each side, u = tanh(z / |x|)
        const int side = i >= LR, j = i - side * LR, l = j / R, r = j - l * R;
        float pr = 1.f;
        for (int t = 0; t < P; ++t) {
            const float s = ((r >> t) & 1) ? 1.f : -1.f;
            const float u = tanhf(zs[side][l * P + t] * inv[side]);
            pr *= 1.f / (1.f + __expf(-2.f * D.beta * u * s));
        }
        ph[side][j] = pr;
    }
    float acc[CPL], vc[CPL];
#pragma unroll
    for (int m = 0; m < CPL; ++m) {
        const int c = lane + 32 * m;
        acc[m] = 0.f;
        vc[m] = c < d ? ld_f(v, bh * d + c) : 1.f;
    }
    __syncthreads();
    // warp w takes sketch rows w, w + 8, ...; lane l columns l, l + 32, ... (up to 5 of the d + 1):
    // all of a thread's loads are independent, and each warp's accesses to a row are contiguous.
    // The first NPF rows come from the registers loaded at the start.
    auto update_row = [&](int j, const float (&cur)[CPL]) {
        float *row = Sbh + (int64_t)j * (d + 1);
        const float pk = ph[1][j], pq = ph[0][j];
#pragma unroll
        for (int m = 0; m < CPL; ++m) {
            const int c = lane + 32 * m;
            if (c <= d) {
                const float sv = fmaf(pk, vc[m], cur[m]);
                row[c] = sv;
                acc[m] = fmaf(pq, sv, acc[m]);
            }
        }
    };
#pragma unroll
    for (int f = 0; f < NPF; ++f)
        if (warp + NW * f < LR) update_row(warp + NW * f, pre[f]);
    for (int j = warp + NW * NPF; j < LR; j += NW) {
        const float *row = Sbh + (int64_t)j * (d + 1);
        float cur[CPL];
#pragma unroll
        for (int m = 0; m < CPL; ++m) {
            const int c = lane + 32 * m;
            cur[m] = c <= d ? row[c] : 0.f;
        }
        update_row(j, cur);
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
