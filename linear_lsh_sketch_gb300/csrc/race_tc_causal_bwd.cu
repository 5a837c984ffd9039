// race_tc_causal_bwd.cu -- tensor-core (mma.sync bf16 -> fp32) causal RACE attention backward.
//
// The chain rule through Algorithm 2 ("RACE Attention" slides, frame "Causality is a prefix
// update of the same statistics"), in 64-token chunks.  With S_t the inclusive prefix sketch
// [A | B], den_t = phi(Q_t) . B_t, g_t = A_t dO_t and c_t = dO_t . O_t = phi(Q_t) . g_t / den_t:
//
//   query side (forward order):  dphi_Q(t) = (g_t - B_t c_t) / den_t
//   key side (reverse order):    G_j = sum_{t >= j} phi_Q(t) [dO_t | -c_t] / den_t
//                                dV_j = G_j,A^T phi_K(j),   dphi_K(j) = G_j,A V_j + G_j,B
//
// followed by the softmax / tanh / projection / normalisation Jacobians.  Inside a chunk:
//   g_t    = S_prev,A dO_t + sum_{j <= t} phi_K(j) (V_j . dO_t)
//   B_t    = S_prev,B + sum_{j <= t} phi_K(j)             (lower-triangular ones x F_K)
//   dV_j   = F_K G_next,A + sum_{t >= j} (phi_K(j) . phi_Q(t)) / den_t dO_t
//   dphi_K = V G_next,A^T + G_next,B + sum_{t >= j} phi_Q(t) (V_j . dO_t - c_t) / den_t
// Every product is a 16x8x16 bf16 tensor-core tile with fp32 accumulation; the carried sketches
// stay fp32 in registers and are read through double-buffered bf16 hi + lo copies.
//
// Pass 1 (k_causal_bwd_q_tc) also sums each segment's G contribution; an exclusive suffix scan
// over segments gives pass 2 (k_causal_bwd_kv_tc) the G that follows its segment.  In both
// passes warp (rb, h) owns token rows 16 rb .. 16 rb + 15; h = 0 featurises the Q rows and
// h = 1 the K rows, and the two warps of a row block split the remaining work between them.
#include "race_common.cuh"
#include "race_launch.h"
#include "race_tc_common.cuh"

namespace race {
namespace tc {

template <int D, int P, int LRP>
struct BwdCfg {
    static constexpr int R = 1 << P;
    static constexpr int XS = D + 8, FS = LRP + 8, SS = D + 8, US = LPP + 1;
    static constexpr int NTO = D / 8 + 1, NC = D / 16, KQ = D / 16, KF = LRP / 16, MT = LRP / 16;
    static constexpr int SNT = (NTO + 7) / 8;
    static constexpr int NL = LRP / 8;      // feature n-tiles
    static constexpr int VS = C + 8;        // stride of the chunk x chunk bf16 staging tile
    static constexpr int DPS = LRP + 1;     // stride of dphi rows (fp32)
    static constexpr int ZS = LPP + 8;      // stride of dz rows (bf16)
    static constexpr int X_BYTES = C * XS * 2;
    static constexpr int S_BYTES = LRP * SS * 2;
    static constexpr int OFF_X = 0;                              // [buf][q, k, v, do]
    static constexpr int OFF_FQ = OFF_X + 8 * X_BYTES;
    static constexpr int OFF_FK = OFF_FQ + C * FS * 2;
    static constexpr int OFF_FQS = OFF_FK + C * FS * 2;
    static constexpr int OFF_S = OFF_FQS + C * FS * 2;           // [buf][hi, lo]
    static constexpr int OFF_W = OFF_S + 4 * S_BYTES;
    static constexpr int OFF_CC = OFF_W + 2 * LPP * XS * 2;      // chunk x chunk staging
    static constexpr int OFF_DPHI = OFF_CC + C * VS * 2;
    static constexpr int OFF_DZ = OFF_DPHI + C * DPS * 4;
    static constexpr int OFF_U = OFF_DZ + C * ZS * 2;            // [warp][16][US]
    static constexpr int OFF_TOK = OFF_U + 8 * 16 * US * 4;      // 6 per-token fp32 vectors
    static constexpr int OFF_BAR = OFF_TOK + 6 * C * 4;
    static constexpr int BYTES = OFF_BAR + 16;
};

__device__ __forceinline__ void mma_a(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    mma16816(c, a[0], a[1], a[2], a[3], b0, b1);
}

// A fragment (16 x 16) of a row-major [m][k] tile at base (u32 shared address of element
// (m0, k0) for lane 0's pattern is added by the caller's precomputed lane offset).
__device__ __forceinline__ uint32_t a_lane_offset(int stride, int lane)
{
    return 2u * (((lane & 7) + 8 * ((lane >> 3) & 1)) * stride + 8 * (lane >> 4));
}
// B fragments of two n-tiles from an [n][k] tile (non-transposing x4 load).
__device__ __forceinline__ uint32_t bnk_lane_offset(int stride, int lane)
{
    return 2u * (((lane & 7) + 8 * (lane >> 4)) * stride + 8 * ((lane >> 3) & 1));
}
// B fragments of two n-tiles from a [k][n] tile (transposing x4 load).
__device__ __forceinline__ uint32_t bkn_lane_offset(int stride, int lane)
{
    return 2u * (((lane & 7) + 8 * ((lane >> 3) & 1)) * stride + 8 * (lane >> 4));
}
// A fragment of M^T from a [k][m] tile (transposing x4 load).
__device__ __forceinline__ uint32_t akm_lane_offset(int stride, int lane)
{
    return 2u * (((lane & 7) + 8 * (lane >> 4)) * stride + 8 * ((lane >> 3) & 1));
}
// One B fragment (x2) from an [n][k] tile.
__device__ __forceinline__ uint32_t bnk2_lane_offset(int stride, int lane)
{
    return 2u * ((lane & 7) * stride + 8 * ((lane >> 3) & 1));
}
// One B fragment (x2, transposing) from a [k][n] tile.
__device__ __forceinline__ uint32_t bkn2_lane_offset(int stride, int lane)
{
    return 2u * (((lane & 7) + 8 * ((lane >> 3) & 1)) * stride);
}

// Loads a carried sketch ([LR][D+1] float32 block) into the fp32 fragments warp w owns and
// into the bf16 hi/lo copy.
template <int D, int P, int LRP>
__device__ __forceinline__ void load_sketch(const Dims &Dm, const float *__restrict__ src, int warp, int lane,
                                            float (&st)[BwdCfg<D, P, LRP>::SNT][BwdCfg<D, P, LRP>::MT][4],
                                            bf16 *hi, bf16 *lo)
{
    using B = BwdCfg<D, P, LRP>;
    const int g = lane >> 2, q = lane & 3;
#pragma unroll
    for (int j = 0; j < B::SNT; ++j) {
        const int nt = warp + 8 * j;
#pragma unroll
        for (int mt = 0; mt < B::MT; ++mt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int lr = 16 * mt + g + 8 * (e >> 1), c = 8 * nt + 2 * q + (e & 1);
                st[j][mt][e] = (nt < B::NTO && lr < Dm.LR && c <= D) ? src[lr * (D + 1) + c] : 0.f;
            }
    }
    for (int i = threadIdx.x; i < LRP * (D + 8); i += NTH) {
        const int lr = i / (D + 8), c = i - lr * (D + 8);
        const float v = (lr < Dm.LR && c <= D) ? src[lr * (D + 1) + c] : 0.f;
        bf16 h16, l16;
        split_bf16(v, h16, l16);
        hi[lr * B::SS + c] = h16;
        lo[lr * B::SS + c] = l16;
    }
}

template <int D, int P, int LRP>
__device__ __forceinline__ void refresh_sketch(const float (&st)[BwdCfg<D, P, LRP>::SNT][BwdCfg<D, P, LRP>::MT][4],
                                               int warp, int lane, bf16 *hi, bf16 *lo)
{
    using B = BwdCfg<D, P, LRP>;
    const int g = lane >> 2, q = lane & 3;
#pragma unroll
    for (int j = 0; j < B::SNT; ++j) {
        const int nt = warp + 8 * j;
        if (nt < B::NTO) {
#pragma unroll
            for (int mt = 0; mt < B::MT; ++mt)
#pragma unroll
                for (int e2 = 0; e2 < 2; ++e2) {
                    const int lr = 16 * mt + g + 8 * e2, c = 8 * nt + 2 * q;
                    bf16 h0, l0, h1, l1;
                    split_bf16(st[j][mt][2 * e2], h0, l0);
                    split_bf16(st[j][mt][2 * e2 + 1], h1, l1);
                    __nv_bfloat162 hh, ll;
                    hh.x = h0;
                    hh.y = h1;
                    ll.x = l0;
                    ll.y = l1;
                    *reinterpret_cast<__nv_bfloat162 *>(hi + lr * B::SS + c) = hh;
                    *reinterpret_cast<__nv_bfloat162 *>(lo + lr * B::SS + c) = ll;
                }
        }
    }
}

// st[owned n-tiles][m-tiles] += feat^T y over the chunk: feat = [C][FS] features (rows = tokens),
// y = [C][XS] token tile.  The mass n-tile reads column d of y when MASSCOL, else a ones column.
template <int D, int P, int LRP, bool MASSCOL>
__device__ __forceinline__ void sketch_update(float (&st)[BwdCfg<D, P, LRP>::SNT][BwdCfg<D, P, LRP>::MT][4],
                                              const bf16 *feat, const bf16 *y, int warp, int lane)
{
    using B = BwdCfg<D, P, LRP>;
    const uint32_t fbase = smem_u32(feat) + akm_lane_offset(B::FS, lane);
    const uint32_t ybase = smem_u32(y) + bkn2_lane_offset(B::XS, lane);
#pragma unroll
    for (int kb = 0; kb < 4; ++kb) {
        uint32_t af[B::MT][4];
#pragma unroll
        for (int mt = 0; mt < B::MT; ++mt)
            ldsm_x4_t(fbase + 2 * (16 * kb * B::FS + 16 * mt), af[mt][0], af[mt][1], af[mt][2], af[mt][3]);
#pragma unroll
        for (int j = 0; j < B::SNT; ++j) {
            const int nt = warp + 8 * j;
            if (nt < B::NTO) {
                uint32_t b0, b1;
                if (nt < D / 8 || MASSCOL)
                    ldsm_x2_t(ybase + 2 * (16 * kb * B::XS + 8 * nt), b0, b1);
                else
                    mass_fragment(lane, b0, b1);
#pragma unroll
                for (int mt = 0; mt < B::MT; ++mt) mma_a(st[j][mt], af[mt], b0, b1);
            }
        }
    }
}

template <int D, int P, int LRP>
__device__ __forceinline__ void store_sketch(const Dims &Dm,
                                             const float (&st)[BwdCfg<D, P, LRP>::SNT][BwdCfg<D, P, LRP>::MT][4],
                                             float *__restrict__ out, int warp, int lane)
{
    using B = BwdCfg<D, P, LRP>;
    const int g = lane >> 2, q = lane & 3;
#pragma unroll
    for (int j = 0; j < B::SNT; ++j) {
        const int nt = warp + 8 * j;
        if (nt < B::NTO) {
#pragma unroll
            for (int mt = 0; mt < B::MT; ++mt)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int lr = 16 * mt + g + 8 * (e >> 1), c = 8 * nt + 2 * q + (e & 1);
                    if (lr < Dm.LR && c <= D) out[lr * (D + 1) + c] = st[j][mt][e];
                }
        }
    }
}

// dxhat = dz (W_hi + W_lo) for rows 16 rb .., column half h, plus the row partials of x . dxhat
// written to red_half[row].
template <int D, int XS, int ZS>
__device__ __forceinline__ void back_project(const bf16 *dzs, const bf16 *wc, const bf16 *xs, int rb, int h, int lane,
                                             float (&acc)[D / 16][4], float *red_half)
{
    constexpr int NC = D / 16;
    const int g = lane >> 2, q = lane & 3;
#pragma unroll
    for (int i = 0; i < NC; ++i)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[i][e] = 0.f;
    uint32_t a[4];
    ldsm_x4(smem_u32(dzs + 16 * rb * ZS) + a_lane_offset(ZS, lane), a[0], a[1], a[2], a[3]);
    const uint32_t whi = smem_u32(wc + 8 * h * NC) + bkn_lane_offset(XS, lane);
    const uint32_t wlo = whi + 2 * LPP * XS;
#pragma unroll
    for (int i = 0; i < NC; i += 2) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(whi + 16 * i, b0, b1, b2, b3);
        mma_a(acc[i], a, b0, b1);
        mma_a(acc[i + 1], a, b2, b3);
        ldsm_x4_t(wlo + 16 * i, b0, b1, b2, b3);
        mma_a(acc[i], a, b0, b1);
        mma_a(acc[i + 1], a, b2, b3);
    }
    float p0 = 0.f, p1 = 0.f;
    const int t0 = 16 * rb + g;
#pragma unroll
    for (int i = 0; i < NC; ++i) {
        const int c = 8 * (h * NC + i) + 2 * q;
        const float2 x0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(xs + t0 * XS + c));
        const float2 x1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(xs + (t0 + 8) * XS + c));
        p0 = fmaf(x0.x, acc[i][0], fmaf(x0.y, acc[i][1], p0));
        p1 = fmaf(x1.x, acc[i][2], fmaf(x1.y, acc[i][3], p1));
    }
    p0 += __shfl_xor_sync(0xffffffffu, p0, 1);
    p0 += __shfl_xor_sync(0xffffffffu, p0, 2);
    p1 += __shfl_xor_sync(0xffffffffu, p1, 1);
    p1 += __shfl_xor_sync(0xffffffffu, p1, 2);
    if (q == 0) {
        red_half[t0] = p0;
        red_half[t0 + 8] = p1;
    }
}

// dx = inv (dxhat - x inv^2 (x . dxhat)) staged as bf16; x . dxhat = red[t] + red[C + t].
template <int D, int XS>
__device__ __forceinline__ void stage_dx(const float (&acc)[D / 16][4], const bf16 *xs, const float *inv,
                                         const float *red, int rb, int h, int lane, bf16 *stage)
{
    constexpr int NC = D / 16;
    const int g = lane >> 2, q = lane & 3;
    const int t0 = 16 * rb + g, t1 = t0 + 8;
    const float i0 = inv[t0], i1 = inv[t1];
    const float k0 = i0 * i0 * (red[t0] + red[C + t0]);
    const float k1 = i1 * i1 * (red[t1] + red[C + t1]);
#pragma unroll
    for (int i = 0; i < NC; ++i) {
        const int c = 8 * (h * NC + i) + 2 * q;
        const float2 x0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(xs + t0 * XS + c));
        const float2 x1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(xs + t1 * XS + c));
        *reinterpret_cast<uint32_t *>(stage + t0 * XS + c) =
            pack_bf16(i0 * (acc[i][0] - x0.x * k0), i0 * (acc[i][1] - x0.y * k0));
        *reinterpret_cast<uint32_t *>(stage + t1 * XS + c) =
            pack_bf16(i1 * (acc[i][2] - x1.x * k1), i1 * (acc[i][3] - x1.y * k1));
    }
}

// Stores 16 staged rows (row block rb), column half h, to global rows n0 + t (t < cnt).
template <int D, int XS>
__device__ __forceinline__ void store_rows(const bf16 *stage, bf16 *__restrict__ dst, int64_t n0, int cnt, int rb,
                                           int h, int lane)
{
    constexpr int CHR = D / 16;
#pragma unroll
    for (int i = lane; i < 16 * CHR; i += 32) {
        const int rr = i / CHR, cc = i - rr * CHR;
        const int t = 16 * rb + rr;
        if (t < cnt) {
            const int c = h * (D / 2) + 8 * cc;
            *reinterpret_cast<uint4 *>(dst + (n0 + t) * D + c) = *reinterpret_cast<const uint4 *>(stage + t * XS + c);
        }
    }
}

// Common set-up: zero the token tiles and feature tiles (stale rows stay finite), split W,
// zero dz beyond L * P, and initialise the two load mbarriers.
template <int D, int P, int LRP>
__device__ __forceinline__ void bwd_setup(const Dims &Dm, const float *__restrict__ W, unsigned char *smem)
{
    using B = BwdCfg<D, P, LRP>;
    zero_smem(smem, B::OFF_S);
    zero_smem(smem + B::OFF_DZ, C * B::ZS * 2);
    __syncthreads();
    load_w_split<D, B::XS>(W, Dm.LP, reinterpret_cast<bf16 *>(smem + B::OFF_W));
    if (threadIdx.x == 0) {
        const uint32_t bar = smem_u32(smem + B::OFF_BAR);
        mbar_init(bar, 1);
        mbar_init(bar + 8, 1);
        fence_mbar_init();
    }
    fence_proxy_async();
}

// ------------------------------------------------------------------ pass 1: dQ, aux, G totals

template <int D, int P, int LRP>
__global__ void __launch_bounds__(NTH, 1)
    k_causal_bwd_q_tc(Dims Dm, const bf16 *__restrict__ Q, const bf16 *__restrict__ K, const bf16 *__restrict__ V,
                      const bf16 *__restrict__ dO, const float *__restrict__ W, const float *__restrict__ S0,
                      int64_t seg_len, int nseg, bf16 *__restrict__ dQ, float2 *__restrict__ aux,
                      float *__restrict__ Gseg, unsigned *__restrict__ err, float *__restrict__ dbpart)
{
    using B = BwdCfg<D, P, LRP>;
    constexpr int NC = B::NC;
    extern __shared__ __align__(128) unsigned char smem[];
    auto xt = [&](int buf, int tile) { return reinterpret_cast<bf16 *>(smem + B::OFF_X + (4 * buf + tile) * B::X_BYTES); };
    auto sh = [&](int buf, int lohi) { return reinterpret_cast<bf16 *>(smem + B::OFF_S + (2 * buf + lohi) * B::S_BYTES); };
    bf16 *fq = reinterpret_cast<bf16 *>(smem + B::OFF_FQ);
    bf16 *fk = reinterpret_cast<bf16 *>(smem + B::OFF_FK);
    bf16 *fqs = reinterpret_cast<bf16 *>(smem + B::OFF_FQS);
    bf16 *wc = reinterpret_cast<bf16 *>(smem + B::OFF_W);
    bf16 *vds = reinterpret_cast<bf16 *>(smem + B::OFF_CC);
    float *dphi = reinterpret_cast<float *>(smem + B::OFF_DPHI);
    bf16 *dzs = reinterpret_cast<bf16 *>(smem + B::OFF_DZ);
    float *tok = reinterpret_cast<float *>(smem + B::OFF_TOK);
    float *invq = tok, *red = tok + C;  // red: [2][C]
    const uint32_t bar0 = smem_u32(smem + B::OFF_BAR);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, q = lane & 3;
    const int rb = warp & 3, h = warp >> 2;
    float *ust = reinterpret_cast<float *>(smem + B::OFF_U) + warp * 16 * B::US;
    const int s = blockIdx.x;
    const int64_t bh = blockIdx.y;
    const int64_t off = bh * Dm.N * D;
    const int64_t n_begin = (int64_t)s * seg_len;
    const int64_t n_end = min(Dm.N, n_begin + seg_len);
    float db = 0.f;  // this thread's d(loss)/d(beta) share (dbpart only)
    const int t0 = 16 * rb + g, t1 = t0 + 8;

    bwd_setup<D, P, LRP>(Dm, head_w(W, Dm, bh), smem);
    float st[B::SNT][B::MT][4], gacc[B::SNT][B::MT][4];
    load_sketch<D, P, LRP>(Dm, S0 + ((int64_t)bh * nseg + s) * Dm.LR * (D + 1), warp, lane, st, sh(0, 0), sh(0, 1));
#pragma unroll
    for (int j = 0; j < B::SNT; ++j)
#pragma unroll
        for (int mt = 0; mt < B::MT; ++mt)
#pragma unroll
            for (int e = 0; e < 4; ++e) gacc[j][mt][e] = 0.f;
    __syncthreads();
    if (n_begin < n_end) {
        const int cnt0 = (int)min((int64_t)C, n_end - n_begin);
        if (tid == 0) mbar_arrive_expect_tx(bar0, 4 * cnt0 * D * 2);
        __syncthreads();
        issue_rows<D, B::XS>(xt(0, 0), xt(0, 1), xt(0, 2), xt(0, 3), Q + off, K + off, V + off, dO + off, 4, n_begin,
                             cnt0, bar0);
    }

    uint32_t phase[2] = {0u, 0u};
    int buf = 0;
    for (int64_t n0 = n_begin; n0 < n_end; n0 += C, buf ^= 1) {
        const int cnt = (int)min((int64_t)C, n_end - n0);
        const bool landed = mbar_wait(bar0 + 8 * buf, phase[buf]);
        phase[buf] ^= 1u;
        const int64_t n1 = n0 + C;
        const int cnt1 = n1 < n_end ? (int)min((int64_t)C, n_end - n1) : 0;
        fence_proxy_async();
        if (tid == 0 && cnt1 > 0) mbar_arrive_expect_tx(bar0 + 8 * (buf ^ 1), 4 * cnt1 * D * 2);
        if (__syncthreads_or(!landed)) {
            if (tid == 0) atomicOr(err, kErrWaitTimeout);
            mbar_wait(bar0 + 8 * buf, phase[buf] ^ 1u);
            return;
        }
        if (cnt1 > 0) {
            issue_rows<D, B::XS>(xt(buf ^ 1, 0), xt(buf ^ 1, 1), xt(buf ^ 1, 2), xt(buf ^ 1, 3), Q + off, K + off,
                                 V + off, dO + off, 4, n1, cnt1, bar0 + 8 * (buf ^ 1));
        }
        bf16 *xqb = xt(buf, 0), *xkb = xt(buf, 1), *xvb = xt(buf, 2), *xdob = xt(buf, 3);
        const bf16 *shi = sh(buf, 0), *slo = sh(buf, 1);

        // P1: h = 0 featurises Q rows (keeps u for the Jacobian), h = 1 featurises K rows
        {
            float u[LPP / 8][4], inv0, inv1;
            project16<D, B::XS>((h ? xkb : xqb) + 16 * rb * B::XS, wc, lane, u, inv0, inv1);
            stage_u<B::US>(u, ust, lane);
            if (h == 0 && q == 0) {
                invq[t0] = inv0;
                invq[t1] = inv1;
            }
            __syncwarp();
            features16<P, B::US, B::FS>(ust, Dm.L, Dm.beta, 16 * rb, cnt, (h ? fk : fq) + 16 * rb * B::FS, lane);
        }
        __syncthreads();

        // P2: h = 1 stages (V_j . dO_t) for j <= t and updates S; h = 0 computes scores, den, g1
        float gq[B::NL][4], den0 = 0.f, den1 = 0.f;
        if (h == 1) {
            const uint32_t dobase = smem_u32(xdob + 16 * rb * B::XS) + a_lane_offset(B::XS, lane);
            const uint32_t vbase = smem_u32(xvb) + bnk2_lane_offset(B::XS, lane);
            uint32_t ado[B::KQ][4];
#pragma unroll
            for (int ks = 0; ks < B::KQ; ++ks) ldsm_x4(dobase + 32 * ks, ado[ks][0], ado[ks][1], ado[ks][2], ado[ks][3]);
#pragma unroll
            for (int jt = 0; jt < 8; ++jt) {
                if (jt <= 2 * rb + 1) {
                    float va[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int ks = 0; ks < B::KQ; ++ks) {
                        uint32_t b0, b1;
                        ldsm_x2(vbase + 2 * (8 * jt * B::XS + 16 * ks), b0, b1);
                        mma_a(va, ado[ks], b0, b1);
                    }
                    const int j = 8 * jt + 2 * q;
                    *reinterpret_cast<uint32_t *>(vds + t0 * B::VS + j) =
                        pack_bf16(j <= t0 ? va[0] : 0.f, j + 1 <= t0 ? va[1] : 0.f);
                    *reinterpret_cast<uint32_t *>(vds + t1 * B::VS + j) =
                        pack_bf16(j <= t1 ? va[2] : 0.f, j + 1 <= t1 ? va[3] : 0.f);
                }
            }
        } else {
            uint32_t aq[B::KF][4];
            const uint32_t qbase = smem_u32(fq + 16 * rb * B::FS) + a_lane_offset(B::FS, lane);
#pragma unroll
            for (int kf = 0; kf < B::KF; ++kf) ldsm_x4(qbase + 32 * kf, aq[kf][0], aq[kf][1], aq[kf][2], aq[kf][3]);
            {
                // den = (masked scores) . 1 + phi_Q . S_prev,B
                const uint32_t kbase = smem_u32(fk) + bnk2_lane_offset(B::FS, lane);
                float om[4] = {0.f, 0.f, 0.f, 0.f};
                uint32_t m0, m1;
                mass_fragment(lane, m0, m1);
#pragma unroll
                for (int kb = 0; kb < 4; ++kb) {
                    if (kb <= rb) {
                        float sc[2][4];
#pragma unroll
                        for (int jj = 0; jj < 2; ++jj) {
                            const int jt = 2 * kb + jj;
#pragma unroll
                            for (int e = 0; e < 4; ++e) sc[jj][e] = 0.f;
#pragma unroll
                            for (int kf = 0; kf < B::KF; ++kf) {
                                uint32_t b0, b1;
                                ldsm_x2(kbase + 2 * (8 * jt * B::FS + 16 * kf), b0, b1);
                                mma_a(sc[jj], aq[kf], b0, b1);
                            }
                            if (kb == rb) {
#pragma unroll
                                for (int e = 0; e < 4; ++e)
                                    if (8 * jt + 2 * q + (e & 1) > 16 * rb + g + 8 * (e >> 1)) sc[jj][e] = 0.f;
                            }
                        }
                        const uint32_t sa[4] = {pack_bf16(sc[0][0], sc[0][1]), pack_bf16(sc[0][2], sc[0][3]),
                                                pack_bf16(sc[1][0], sc[1][1]), pack_bf16(sc[1][2], sc[1][3])};
                        mma_a(om, sa, m0, m1);
                    }
                }
                const uint32_t mh = smem_u32(shi + D) + bkn2_lane_offset(B::SS, lane);
                const uint32_t ml = smem_u32(slo + D) + bkn2_lane_offset(B::SS, lane);
#pragma unroll
                for (int kf = 0; kf < B::KF; ++kf) {
                    uint32_t b0, b1;
                    ldsm_x2_t(mh + 32 * kf * B::SS, b0, b1);
                    mma_a(om, aq[kf], b0, b1);
                    ldsm_x2_t(ml + 32 * kf * B::SS, b0, b1);
                    mma_a(om, aq[kf], b0, b1);
                }
                den0 = __shfl_sync(0xffffffffu, om[0], lane & ~3);
                den1 = __shfl_sync(0xffffffffu, om[2], lane & ~3);
            }
            // g1 = S_prev,A dO over all feature columns
            const uint32_t dobase = smem_u32(xdob + 16 * rb * B::XS) + a_lane_offset(B::XS, lane);
            const uint32_t hb = smem_u32(shi) + bnk_lane_offset(B::SS, lane);
            const uint32_t lb = smem_u32(slo) + bnk_lane_offset(B::SS, lane);
#pragma unroll
            for (int i = 0; i < B::NL; ++i)
#pragma unroll
                for (int e = 0; e < 4; ++e) gq[i][e] = 0.f;
#pragma unroll
            for (int ks = 0; ks < B::KQ; ++ks) {
                uint32_t a[4];
                ldsm_x4(dobase + 32 * ks, a[0], a[1], a[2], a[3]);
#pragma unroll
                for (int i = 0; i < B::NL; i += 2) {
                    const uint32_t o = 2 * (8 * i * B::SS + 16 * ks);
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4(hb + o, b0, b1, b2, b3);
                    mma_a(gq[i], a, b0, b1);
                    mma_a(gq[i + 1], a, b2, b3);
                    ldsm_x4(lb + o, b0, b1, b2, b3);
                    mma_a(gq[i], a, b0, b1);
                    mma_a(gq[i + 1], a, b2, b3);
                }
            }
        }
        __syncthreads();

        // P3: h = 0 finishes dphi_Q and the feature Jacobian; h = 1 updates S and its next copy
        if (h == 0) {
            float sb[B::NL][4];
#pragma unroll
            for (int i = 0; i < B::NL; ++i)
#pragma unroll
                for (int e = 0; e < 4; ++e) sb[i][e] = 0.f;
            const uint32_t vdbase = smem_u32(vds + 16 * rb * B::VS) + a_lane_offset(B::VS, lane);
            const uint32_t fkb = smem_u32(fk) + bkn_lane_offset(B::FS, lane);
#pragma unroll
            for (int kb = 0; kb < 4; ++kb) {
                if (kb <= rb) {
                    uint32_t av[4], al[4];
                    ldsm_x4(vdbase + 32 * kb, av[0], av[1], av[2], av[3]);
                    tril_ones_fragment(16 * rb, 16 * kb, lane, al);
#pragma unroll
                    for (int i = 0; i < B::NL; i += 2) {
                        uint32_t b0, b1, b2, b3;
                        ldsm_x4_t(fkb + 2 * (16 * kb * B::FS + 8 * i), b0, b1, b2, b3);
                        mma_a(gq[i], av, b0, b1);
                        mma_a(gq[i + 1], av, b2, b3);
                        mma_a(sb[i], al, b0, b1);
                        mma_a(sb[i + 1], al, b2, b3);
                    }
                }
            }
            // c = phi_Q . g / den, then dphi = (g - B_t c) / den
            float p0 = 0.f, p1 = 0.f;
#pragma unroll
            for (int i = 0; i < B::NL; ++i) {
                const int lr = 8 * i + 2 * q;
                const float2 f0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(fq + t0 * B::FS + lr));
                const float2 f1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(fq + t1 * B::FS + lr));
                p0 = fmaf(f0.x, gq[i][0], fmaf(f0.y, gq[i][1], p0));
                p1 = fmaf(f1.x, gq[i][2], fmaf(f1.y, gq[i][3], p1));
            }
            p0 += __shfl_xor_sync(0xffffffffu, p0, 1);
            p0 += __shfl_xor_sync(0xffffffffu, p0, 2);
            p1 += __shfl_xor_sync(0xffffffffu, p1, 1);
            p1 += __shfl_xor_sync(0xffffffffu, p1, 2);
            const bool l0 = t0 < cnt, l1 = t1 < cnt;
            const float rd0 = l0 ? __frcp_rn(den0) : 0.f, rd1 = l1 ? __frcp_rn(den1) : 0.f;
            const float c0 = p0 * rd0, c1 = p1 * rd1;
#pragma unroll
            for (int i = 0; i < B::NL; ++i) {
                const int lr = 8 * i + 2 * q;
                const float sb0 = __bfloat162float(shi[lr * B::SS + D]) + __bfloat162float(slo[lr * B::SS + D]);
                const float sb1 =
                    __bfloat162float(shi[(lr + 1) * B::SS + D]) + __bfloat162float(slo[(lr + 1) * B::SS + D]);
                dphi[t0 * B::DPS + lr] = (gq[i][0] - (sb[i][0] + sb0) * c0) * rd0;
                dphi[t0 * B::DPS + lr + 1] = (gq[i][1] - (sb[i][1] + sb1) * c0) * rd0;
                dphi[t1 * B::DPS + lr] = (gq[i][2] - (sb[i][2] + sb0) * c1) * rd1;
                dphi[t1 * B::DPS + lr + 1] = (gq[i][3] - (sb[i][3] + sb1) * c1) * rd1;
            }
            if (q == 0) {
                xdob[t0 * B::XS + D] = __float2bfloat16_rn(-c0);
                xdob[t1 * B::XS + D] = __float2bfloat16_rn(-c1);
                if (l0) aux[bh * Dm.N + n0 + t0] = make_float2(rd0, c0);
                if (l1) aux[bh * Dm.N + n0 + t1] = make_float2(rd1, c1);
            }
            // phi_Q / den for the gradient sketch (row t scaled by rd of its thread pair)
#pragma unroll
            for (int i = 0; i < B::NL; ++i) {
                const int lr = 8 * i + 2 * q;
                const float2 f0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(fq + t0 * B::FS + lr));
                const float2 f1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(fq + t1 * B::FS + lr));
                *reinterpret_cast<uint32_t *>(fqs + t0 * B::FS + lr) = pack_bf16(f0.x * rd0, f0.y * rd0);
                *reinterpret_cast<uint32_t *>(fqs + t1 * B::FS + lr) = pack_bf16(f1.x * rd1, f1.y * rd1);
            }
            __syncwarp();
            features_backward16<P, B::US, B::DPS, B::ZS>(ust, dphi + 16 * rb * B::DPS, Dm.L, Dm.beta,
                                                         dzs + 16 * rb * B::ZS, lane, dbpart ? &db : nullptr,
                                                         16 * rb, cnt);
        }
        sketch_update<D, P, LRP, false>(st, fk, xvb, warp, lane);
        refresh_sketch<D, P, LRP>(st, warp, lane, sh(buf ^ 1, 0), sh(buf ^ 1, 1));
        __syncthreads();

        // P4: dxhat halves, gradient-sketch totals
        float dx[NC][4];
        back_project<D, B::XS, B::ZS>(dzs, wc, xqb, rb, h, lane, dx, red + h * C);
        sketch_update<D, P, LRP, true>(gacc, fqs, xdob, warp, lane);
        __syncthreads();

        // P5: dQ = normalisation backward, staged in the consumed K tile
        stage_dx<D, B::XS>(dx, xqb, invq, red, rb, h, lane, xkb);
        __syncwarp();
        store_rows<D, B::XS>(xkb, dQ + off, n0, cnt, rb, h, lane);
    }
    store_sketch<D, P, LRP>(Dm, gacc, Gseg + ((int64_t)bh * nseg + s) * Dm.LR * (D + 1), warp, lane);
    if (dbpart) {  // this CTA's query-side d(loss)/d(beta) partial, summed in a fixed order
        const float sdb = block_sum_fixed(db, red);
        if (tid == 0) dbpart[bh * gridDim.x + blockIdx.x] = sdb;
    }
}

// ------------------------------------------------------------------ pass 2: dK, dV

template <int D, int P, int LRP>
__global__ void __launch_bounds__(NTH, 1)
    k_causal_bwd_kv_tc(Dims Dm, const bf16 *__restrict__ Q, const bf16 *__restrict__ K, const bf16 *__restrict__ V,
                       const bf16 *__restrict__ dO, const float2 *__restrict__ aux, const float *__restrict__ W,
                       const float *__restrict__ G0, int64_t seg_len, int nseg, bf16 *__restrict__ dK,
                       bf16 *__restrict__ dV, unsigned *__restrict__ err, float *__restrict__ dbpart)
{
    using B = BwdCfg<D, P, LRP>;
    constexpr int NC = B::NC;
    extern __shared__ __align__(128) unsigned char smem[];
    auto xt = [&](int buf, int tile) { return reinterpret_cast<bf16 *>(smem + B::OFF_X + (4 * buf + tile) * B::X_BYTES); };
    auto gh = [&](int buf, int lohi) { return reinterpret_cast<bf16 *>(smem + B::OFF_S + (2 * buf + lohi) * B::S_BYTES); };
    bf16 *fq = reinterpret_cast<bf16 *>(smem + B::OFF_FQ);
    bf16 *fk = reinterpret_cast<bf16 *>(smem + B::OFF_FK);
    bf16 *fqs = reinterpret_cast<bf16 *>(smem + B::OFF_FQS);
    bf16 *wc = reinterpret_cast<bf16 *>(smem + B::OFF_W);
    bf16 *wst = reinterpret_cast<bf16 *>(smem + B::OFF_CC);
    float *dphi = reinterpret_cast<float *>(smem + B::OFF_DPHI);
    bf16 *dzs = reinterpret_cast<bf16 *>(smem + B::OFF_DZ);
    float *tok = reinterpret_cast<float *>(smem + B::OFF_TOK);
    float *invk = tok, *rden = tok + C, *ccs = tok + 2 * C, *red = tok + 3 * C;  // red: [2][C]
    const uint32_t bar0 = smem_u32(smem + B::OFF_BAR);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, q = lane & 3;
    const int rb = warp & 3, h = warp >> 2;
    float *ust = reinterpret_cast<float *>(smem + B::OFF_U) + warp * 16 * B::US;
    const int s = blockIdx.x;
    const int64_t bh = blockIdx.y;
    const int64_t off = bh * Dm.N * D;
    const int64_t n_begin = (int64_t)s * seg_len;
    const int64_t n_end = min(Dm.N, n_begin + seg_len);
    float db = 0.f;  // this thread's d(loss)/d(beta) share (dbpart only)
    const int j0 = 16 * rb + g, j1 = j0 + 8;  // key rows of this warp's row block

    bwd_setup<D, P, LRP>(Dm, head_w(W, Dm, bh), smem);
    float gst[B::SNT][B::MT][4];
    load_sketch<D, P, LRP>(Dm, G0 + ((int64_t)bh * nseg + s) * Dm.LR * (D + 1), warp, lane, gst, gh(0, 0), gh(0, 1));
    __syncthreads();
    if (n_begin >= n_end) return;
    const int64_t last = n_begin + ((n_end - 1 - n_begin) / C) * C;
    {
        const int cnt0 = (int)min((int64_t)C, n_end - last);
        if (tid == 0) mbar_arrive_expect_tx(bar0, 4 * cnt0 * D * 2);
        __syncthreads();
        issue_rows<D, B::XS>(xt(0, 0), xt(0, 1), xt(0, 2), xt(0, 3), Q + off, K + off, V + off, dO + off, 4, last,
                             cnt0, bar0);
    }

    uint32_t phase[2] = {0u, 0u};
    int buf = 0;
    for (int64_t n0 = last; n0 >= n_begin; n0 -= C, buf ^= 1) {
        const int cnt = (int)min((int64_t)C, n_end - n0);
        const bool landed = mbar_wait(bar0 + 8 * buf, phase[buf]);
        phase[buf] ^= 1u;
        const int64_t n1 = n0 - C;
        const bool more = n1 >= n_begin;
        fence_proxy_async();
        if (tid == 0 && more) mbar_arrive_expect_tx(bar0 + 8 * (buf ^ 1), 4 * C * D * 2);
        for (int t = tid; t < C; t += NTH) {
            float2 a = make_float2(0.f, 0.f);
            if (t < cnt) a = aux[bh * Dm.N + n0 + t];
            rden[t] = a.x;
            ccs[t] = a.y;
        }
        if (__syncthreads_or(!landed)) {
            if (tid == 0) atomicOr(err, kErrWaitTimeout);
            mbar_wait(bar0 + 8 * buf, phase[buf] ^ 1u);
            return;
        }
        if (more) {
            issue_rows<D, B::XS>(xt(buf ^ 1, 0), xt(buf ^ 1, 1), xt(buf ^ 1, 2), xt(buf ^ 1, 3), Q + off, K + off,
                                 V + off, dO + off, 4, n1, C, bar0 + 8 * (buf ^ 1));
        }
        bf16 *xqb = xt(buf, 0), *xkb = xt(buf, 1), *xvb = xt(buf, 2), *xdob = xt(buf, 3);
        const bf16 *ghi = gh(buf, 0), *glo = gh(buf, 1);

        // P1: h = 0 featurises Q rows (phi_Q and phi_Q / den) and writes -c into the dO tile's
        // mass column; h = 1 featurises K rows (keeps u for the Jacobian)
        {
            float u[LPP / 8][4], inv0, inv1;
            project16<D, B::XS>((h ? xkb : xqb) + 16 * rb * B::XS, wc, lane, u, inv0, inv1);
            stage_u<B::US>(u, ust, lane);
            if (h == 1 && q == 0) {
                invk[j0] = inv0;
                invk[j1] = inv1;
            }
            __syncwarp();
            if (h == 0) {
                features16<P, B::US, B::FS>(ust, Dm.L, Dm.beta, 16 * rb, cnt, fq + 16 * rb * B::FS, lane, rden,
                                            fqs + 16 * rb * B::FS);
                if (lane < 16) xdob[(16 * rb + lane) * B::XS + D] = __float2bfloat16_rn(-ccs[16 * rb + lane]);
            } else {
                features16<P, B::US, B::FS>(ust, Dm.L, Dm.beta, 16 * rb, cnt, fk + 16 * rb * B::FS, lane);
            }
        }
        __syncthreads();

        // P2: h = 1: dV (all columns) from (phi_K . phi_Q)/den and G_next; h = 0: the staged block
        // (V_j . dO_t - c_t)/den_t for t >= j, and dphi_K's G_next part (with G_next,B)
        if (h == 1) {
            uint32_t ak[B::KF][4];
            const uint32_t kbase = smem_u32(fk + 16 * rb * B::FS) + a_lane_offset(B::FS, lane);
#pragma unroll
            for (int kf = 0; kf < B::KF; ++kf) ldsm_x4(kbase + 32 * kf, ak[kf][0], ak[kf][1], ak[kf][2], ak[kf][3]);
            float dva[2 * NC][4];
#pragma unroll
            for (int i = 0; i < 2 * NC; ++i)
#pragma unroll
                for (int e = 0; e < 4; ++e) dva[i][e] = 0.f;
            const uint32_t qb = smem_u32(fq) + bnk2_lane_offset(B::FS, lane);
            const uint32_t dob = smem_u32(xdob) + bkn_lane_offset(B::XS, lane);
#pragma unroll
            for (int kb = 0; kb < 4; ++kb) {
                if (kb >= rb) {
                    float pt[2][4];
#pragma unroll
                    for (int jj = 0; jj < 2; ++jj) {
                        const int tt = 2 * kb + jj;
#pragma unroll
                        for (int e = 0; e < 4; ++e) pt[jj][e] = 0.f;
#pragma unroll
                        for (int kf = 0; kf < B::KF; ++kf) {
                            uint32_t b0, b1;
                            ldsm_x2(qb + 2 * (8 * tt * B::FS + 16 * kf), b0, b1);
                            mma_a(pt[jj], ak[kf], b0, b1);
                        }
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int t = 8 * tt + 2 * q + (e & 1), j = 16 * rb + g + 8 * (e >> 1);
                            pt[jj][e] = t >= j ? pt[jj][e] * rden[t] : 0.f;
                        }
                    }
                    const uint32_t pa[4] = {pack_bf16(pt[0][0], pt[0][1]), pack_bf16(pt[0][2], pt[0][3]),
                                            pack_bf16(pt[1][0], pt[1][1]), pack_bf16(pt[1][2], pt[1][3])};
#pragma unroll
                    for (int i = 0; i < 2 * NC; i += 2) {
                        uint32_t b0, b1, b2, b3;
                        ldsm_x4_t(dob + 2 * (16 * kb * B::XS + 8 * i), b0, b1, b2, b3);
                        mma_a(dva[i], pa, b0, b1);
                        mma_a(dva[i + 1], pa, b2, b3);
                    }
                }
            }
            const uint32_t hb = smem_u32(ghi) + bkn_lane_offset(B::SS, lane);
            const uint32_t lb = smem_u32(glo) + bkn_lane_offset(B::SS, lane);
#pragma unroll
            for (int kf = 0; kf < B::KF; ++kf) {
#pragma unroll
                for (int i = 0; i < 2 * NC; i += 2) {
                    const uint32_t o = 2 * (16 * kf * B::SS + 8 * i);
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4_t(hb + o, b0, b1, b2, b3);
                    mma_a(dva[i], ak[kf], b0, b1);
                    mma_a(dva[i + 1], ak[kf], b2, b3);
                    ldsm_x4_t(lb + o, b0, b1, b2, b3);
                    mma_a(dva[i], ak[kf], b0, b1);
                    mma_a(dva[i + 1], ak[kf], b2, b3);
                }
            }
            // dV staged in the consumed Q tile (its only use was the projection)
#pragma unroll
            for (int i = 0; i < 2 * NC; ++i) {
                const int c = 8 * i + 2 * q;
                *reinterpret_cast<uint32_t *>(xqb + j0 * B::XS + c) = pack_bf16(dva[i][0], dva[i][1]);
                *reinterpret_cast<uint32_t *>(xqb + j1 * B::XS + c) = pack_bf16(dva[i][2], dva[i][3]);
            }
            __syncwarp();
            store_rows<D, B::XS>(xqb, dV + off, n0, cnt, rb, 0, lane);
            store_rows<D, B::XS>(xqb, dV + off, n0, cnt, rb, 1, lane);
        } else {
            const uint32_t vbase = smem_u32(xvb + 16 * rb * B::XS) + a_lane_offset(B::XS, lane);
            uint32_t av[B::KQ][4];
#pragma unroll
            for (int ks = 0; ks < B::KQ; ++ks) ldsm_x4(vbase + 32 * ks, av[ks][0], av[ks][1], av[ks][2], av[ks][3]);
            const uint32_t dob = smem_u32(xdob) + bnk2_lane_offset(B::XS, lane);
#pragma unroll
            for (int tt = 0; tt < 8; ++tt) {
                if (tt >= 2 * rb) {
                    float va[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int ks = 0; ks < B::KQ; ++ks) {
                        uint32_t b0, b1;
                        ldsm_x2(dob + 2 * (8 * tt * B::XS + 16 * ks), b0, b1);
                        mma_a(va, av[ks], b0, b1);
                    }
                    const int t = 8 * tt + 2 * q;
                    const float r0 = rden[t], r1 = rden[t + 1], c0 = ccs[t], c1 = ccs[t + 1];
                    *reinterpret_cast<uint32_t *>(wst + j0 * B::VS + t) =
                        pack_bf16(t >= j0 ? (va[0] - c0) * r0 : 0.f, t + 1 >= j0 ? (va[1] - c1) * r1 : 0.f);
                    *reinterpret_cast<uint32_t *>(wst + j1 * B::VS + t) =
                        pack_bf16(t >= j1 ? (va[2] - c0) * r0 : 0.f, t + 1 >= j1 ? (va[3] - c1) * r1 : 0.f);
                }
            }
            float dpk[B::NL][4];
#pragma unroll
            for (int i = 0; i < B::NL; ++i)
#pragma unroll
                for (int e = 0; e < 4; ++e) dpk[i][e] = 0.f;
            const uint32_t hb = smem_u32(ghi) + bnk_lane_offset(B::SS, lane);
            const uint32_t lb = smem_u32(glo) + bnk_lane_offset(B::SS, lane);
#pragma unroll
            for (int ks = 0; ks < B::KQ; ++ks) {
#pragma unroll
                for (int i = 0; i < B::NL; i += 2) {
                    const uint32_t o = 2 * (8 * i * B::SS + 16 * ks);
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4(hb + o, b0, b1, b2, b3);
                    mma_a(dpk[i], av[ks], b0, b1);
                    mma_a(dpk[i + 1], av[ks], b2, b3);
                    ldsm_x4(lb + o, b0, b1, b2, b3);
                    mma_a(dpk[i], av[ks], b0, b1);
                    mma_a(dpk[i + 1], av[ks], b2, b3);
                }
            }
#pragma unroll
            for (int i = 0; i < B::NL; ++i) {
                const int lr = 8 * i + 2 * q;
                const float gb0 = __bfloat162float(ghi[lr * B::SS + D]) + __bfloat162float(glo[lr * B::SS + D]);
                const float gb1 =
                    __bfloat162float(ghi[(lr + 1) * B::SS + D]) + __bfloat162float(glo[(lr + 1) * B::SS + D]);
                dphi[j0 * B::DPS + lr] = dpk[i][0] + gb0;
                dphi[j0 * B::DPS + lr + 1] = dpk[i][1] + gb1;
                dphi[j1 * B::DPS + lr] = dpk[i][2] + gb0;
                dphi[j1 * B::DPS + lr + 1] = dpk[i][3] + gb1;
            }
        }
        // G += phi_Q^T [dO | -c] / den on the owned n-tiles and its copy for the next chunk
        sketch_update<D, P, LRP, true>(gst, fqs, xdob, warp, lane);
        refresh_sketch<D, P, LRP>(gst, warp, lane, gh(buf ^ 1, 0), gh(buf ^ 1, 1));
        __syncthreads();

        // P3: h = 1 adds dphi_K's intra-chunk part and runs the feature Jacobian of its K rows
        if (h == 1) {
            float dpk[B::NL][4];
#pragma unroll
            for (int i = 0; i < B::NL; ++i)
#pragma unroll
                for (int e = 0; e < 4; ++e) dpk[i][e] = 0.f;
            const uint32_t wbase = smem_u32(wst + 16 * rb * B::VS) + a_lane_offset(B::VS, lane);
            const uint32_t qkb = smem_u32(fq) + bkn_lane_offset(B::FS, lane);
#pragma unroll
            for (int kb = 0; kb < 4; ++kb) {
                if (kb >= rb) {
                    uint32_t aw[4];
                    ldsm_x4(wbase + 32 * kb, aw[0], aw[1], aw[2], aw[3]);
#pragma unroll
                    for (int i = 0; i < B::NL; i += 2) {
                        uint32_t b0, b1, b2, b3;
                        ldsm_x4_t(qkb + 2 * (16 * kb * B::FS + 8 * i), b0, b1, b2, b3);
                        mma_a(dpk[i], aw, b0, b1);
                        mma_a(dpk[i + 1], aw, b2, b3);
                    }
                }
            }
#pragma unroll
            for (int i = 0; i < B::NL; ++i) {
                const int lr = 8 * i + 2 * q;
                dphi[j0 * B::DPS + lr] += dpk[i][0];
                dphi[j0 * B::DPS + lr + 1] += dpk[i][1];
                dphi[j1 * B::DPS + lr] += dpk[i][2];
                dphi[j1 * B::DPS + lr + 1] += dpk[i][3];
            }
            __syncwarp();
            features_backward16<P, B::US, B::DPS, B::ZS>(ust, dphi + 16 * rb * B::DPS, Dm.L, Dm.beta,
                                                         dzs + 16 * rb * B::ZS, lane, dbpart ? &db : nullptr,
                                                         16 * rb, cnt);
        }
        __syncthreads();

        // P4: dxhat halves of the K rows
        float dx[NC][4];
        back_project<D, B::XS, B::ZS>(dzs, wc, xkb, rb, h, lane, dx, red + h * C);
        __syncthreads();

        // P5: dK staged in the consumed V tile
        stage_dx<D, B::XS>(dx, xkb, invk, red, rb, h, lane, xvb);
        __syncwarp();
        store_rows<D, B::XS>(xvb, dK + off, n0, cnt, rb, h, lane);
    }
    if (dbpart) {  // this CTA's key-side d(loss)/d(beta) partial, summed in a fixed order
        const float sdb = block_sum_fixed(db, red);
        if (tid == 0) dbpart[bh * gridDim.x + blockIdx.x] = sdb;
    }
}

}  // namespace tc

// ------------------------------------------------------------------ host side

namespace {

constexpr size_t kSmemLimit = 227 * 1024;

template <int D, int P, int LRP>
constexpr bool bwd_fits()
{
    return tc::BwdCfg<D, P, LRP>::BYTES <= kSmemLimit;
}

template <int D, int P, int LRP>
cudaError_t launch_bwd_q_inst(const Dims &Dm, const bf16_t *Q, const bf16_t *K, const bf16_t *V, const bf16_t *dO,
                              const float *W, const float *S0, int64_t seg_len, int nseg, bf16_t *dQ, float2 *aux,
                              float *Gseg, unsigned *err, float *dbpart, cudaStream_t st)
{
    using B = tc::BwdCfg<D, P, LRP>;
    if constexpr (!bwd_fits<D, P, LRP>()) {
        return cudaErrorInvalidValue;
    } else {
        auto kern = tc::k_causal_bwd_q_tc<D, P, LRP>;
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, B::BYTES);
        if (e != cudaSuccess) return e;
        return launch_kernel("tc_causal_bwd_q", kern, dim3(nseg, (unsigned)Dm.BH), dim3(tc::NTH), (size_t)B::BYTES,
                             st, Dm, Q, K, V, dO, W, S0, seg_len, nseg, dQ, aux, Gseg, err, dbpart);
    }
}

template <int D, int P, int LRP>
cudaError_t launch_bwd_kv_inst(const Dims &Dm, const bf16_t *Q, const bf16_t *K, const bf16_t *V, const bf16_t *dO,
                               const float2 *aux, const float *W, const float *G0, int64_t seg_len, int nseg,
                               bf16_t *dK, bf16_t *dV, unsigned *err, float *dbpart, cudaStream_t st)
{
    using B = tc::BwdCfg<D, P, LRP>;
    if constexpr (!bwd_fits<D, P, LRP>()) {
        return cudaErrorInvalidValue;
    } else {
        auto kern = tc::k_causal_bwd_kv_tc<D, P, LRP>;
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, B::BYTES);
        if (e != cudaSuccess) return e;
        return launch_kernel("tc_causal_bwd_kv", kern, dim3(nseg, (unsigned)Dm.BH), dim3(tc::NTH), (size_t)B::BYTES,
                             st, Dm, Q, K, V, dO, aux, W, G0, seg_len, nseg, dK, dV, err, dbpart);
    }
}

}  // namespace

#define RACE_TC_BWD_CASES(X) \
    X(128, 2, 32) X(128, 2, 64) X(128, 3, 32) X(128, 3, 64) X(128, 4, 32) X(128, 4, 64) \
    X(64, 2, 32) X(64, 2, 64) X(64, 3, 32) X(64, 3, 64) X(64, 4, 32) X(64, 4, 64)

bool causal_tc_bwd_supported(const Dims &Dm)
{
    if (!causal_tc_supported(Dm)) return false;
#define RACE_FITS(DD, PP, LRPP) \
    if (Dm.d == DD && Dm.P == PP && Dm.LR <= LRPP) return bwd_fits<DD, PP, LRPP>();
    RACE_TC_BWD_CASES(RACE_FITS)
#undef RACE_FITS
    return false;
}

cudaError_t launch_causal_tc_bwd_q(const Dims &Dm, const bf16_t *Q, const bf16_t *K, const bf16_t *V,
                                   const bf16_t *dO, const float *W, const float *S0, int64_t seg_len, int nseg,
                                   bf16_t *dQ, float2 *aux, float *Gseg, unsigned *err, float *dbpart,
                                   cudaStream_t st)
{
#define RACE_CASE(DD, PP, LRPP)                               \
    if (Dm.d == DD && Dm.P == PP && Dm.LR <= LRPP)            \
        return launch_bwd_q_inst<DD, PP, LRPP>(Dm, Q, K, V, dO, W, S0, seg_len, nseg, dQ, aux, Gseg, err, dbpart, st);
    RACE_TC_BWD_CASES(RACE_CASE)
#undef RACE_CASE
    return cudaErrorInvalidValue;
}

cudaError_t launch_causal_tc_bwd_kv(const Dims &Dm, const bf16_t *Q, const bf16_t *K, const bf16_t *V,
                                    const bf16_t *dO, const float2 *aux, const float *W, const float *G0,
                                    int64_t seg_len, int nseg, bf16_t *dK, bf16_t *dV, unsigned *err,
                                    float *dbpart, cudaStream_t st)
{
#define RACE_CASE(DD, PP, LRPP)                               \
    if (Dm.d == DD && Dm.P == PP && Dm.LR <= LRPP)            \
        return launch_bwd_kv_inst<DD, PP, LRPP>(Dm, Q, K, V, dO, aux, W, G0, seg_len, nseg, dK, dV, err, dbpart, st);
    RACE_TC_BWD_CASES(RACE_CASE)
#undef RACE_CASE
    return cudaErrorInvalidValue;
}

}  // namespace race
