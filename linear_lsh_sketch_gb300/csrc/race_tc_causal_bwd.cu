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
// stay fp32 in registers and are read through bf16 hi + lo copies.
//
// Pass 1 (k_causal_bwd_q_tc) also sums each segment's G contribution; an exclusive suffix scan
// over segments gives pass 2 (k_causal_bwd_kv_tc) the G that follows its segment.
#include "race_common.cuh"
#include "race_launch.h"
#include "race_mma.cuh"
#include "race_tc_common.cuh"

namespace race {
namespace tc {

template <int D, int LRP, int LPP>
struct BwdCfg {
    using Cf = CausalCfg<D, LRP, LPP>;
    static constexpr int XS = Cf::XS, FS = Cf::FS, SS = Cf::SS, US = Cf::US, NWP = Cf::NWP;
    static constexpr int NTO = Cf::NTO, KQ = Cf::KQ, KF = Cf::KF, MT = Cf::MT, SNT = Cf::SNT;
    static constexpr int VS = C + 8;     // stride of the chunk x chunk bf16 staging tile
    static constexpr int DPS = LRP + 1;  // stride of dphi (fp32)
    static constexpr int ZS = LPP + 8;   // stride of dz (bf16)
    static constexpr int NLH = LRP / 16; // feature n-tiles per column half
    static constexpr int X_BYTES = C * XS * 2;
    static constexpr int OFF_XQ = 0;
    static constexpr int OFF_XK = OFF_XQ + 2 * X_BYTES;
    static constexpr int OFF_XV = OFF_XK + 2 * X_BYTES;
    static constexpr int OFF_XDO = OFF_XV + 2 * X_BYTES;
    static constexpr int OFF_FQ = OFF_XDO + 2 * X_BYTES;
    static constexpr int OFF_FK = OFF_FQ + C * FS * 2;
    static constexpr int OFF_FQS = OFF_FK + C * FS * 2;
    static constexpr int OFF_SHI = OFF_FQS + C * FS * 2;
    static constexpr int OFF_SLO = OFF_SHI + LRP * SS * 2;
    static constexpr int OFF_W = OFF_SLO + LRP * SS * 2;
    static constexpr int OFF_U = OFF_W + NWP * XS * 2;
    static constexpr int OFF_CC = OFF_U + 2 * C * US * 4;   // chunk x chunk staging
    static constexpr int OFF_DPHI = OFF_CC + C * VS * 2;
    static constexpr int OFF_DZ = OFF_DPHI + C * DPS * 4;
    static constexpr int OFF_TOK = OFF_DZ + C * ZS * 2;     // 6 per-token fp32 vectors
    static constexpr int BYTES = OFF_TOK + 6 * C * 4;
};

// Loads a (hi, lo) pair of B fragments for two adjacent n-tiles from a [n][k] layout.
__device__ __forceinline__ void ldsm_b_nk_x4(const bf16 *base, int stride, int n0, int k0, int lane, uint32_t &b0,
                                             uint32_t &b1, uint32_t &b2, uint32_t &b3)
{
    ldsm_x4(smem_u32(base + (n0 + (lane & 7) + 8 * (lane >> 4)) * stride + k0 + 8 * ((lane >> 3) & 1)), b0, b1, b2,
            b3);
}

// Two adjacent n-tiles of B from a [k][n] layout (transposing load).
__device__ __forceinline__ void ldsm_b_kn_x4(const bf16 *base, int stride, int k0, int n0, int lane, uint32_t &b0,
                                             uint32_t &b1, uint32_t &b2, uint32_t &b3)
{
    ldsm_x4_t(smem_u32(base + (k0 + (lane & 7) + 8 * ((lane >> 3) & 1)) * stride + n0 + 8 * (lane >> 4)), b0, b1, b2,
              b3);
}

// A fragment (16 x 16) from a row-major [m][k] layout.
__device__ __forceinline__ void ldsm_a(const bf16 *base, int stride, int m0, int k0, int lane, uint32_t (&a)[4])
{
    ldsm_x4(smem_u32(base + (m0 + (lane & 7) + 8 * ((lane >> 3) & 1)) * stride + k0 + 8 * (lane >> 4)), a[0], a[1],
            a[2], a[3]);
}

// A fragment of M^T from a [k][m] layout (transposing load).
__device__ __forceinline__ void ldsm_a_km(const bf16 *base, int stride, int k0, int m0, int lane, uint32_t (&a)[4])
{
    ldsm_x4_t(smem_u32(base + (k0 + (lane & 7) + 8 * (lane >> 4)) * stride + m0 + 8 * ((lane >> 3) & 1)), a[0], a[1],
              a[2], a[3]);
}

__device__ __forceinline__ void mma_a(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    mma16816(c, a[0], a[1], a[2], a[3], b0, b1);
}

// Shared set-up of both passes: hyperplanes (hi/lo), zero padding of the feature tiles, of dz
// beyond LP, and of the columns d+1 .. d+7 of the dO tiles (column d carries -c per chunk).
template <int D, int LRP, int LPP>
__device__ __forceinline__ void bwd_setup(const Dims &Dm, const float *__restrict__ W, bf16 *wc, bf16 *fq, bf16 *fk,
                                          bf16 *fqs, bf16 *dzs, bf16 *xdo)
{
    using B = BwdCfg<D, LRP, LPP>;
    const int tid = threadIdx.x;
    for (int i = tid; i < LPP * D; i += NTH) {
        const int row = i / D, k = i - row * D;
        const float w = row < Dm.LP ? W[row * D + k] : 0.f;
        bf16 hi, lo;
        split_bf16(w, hi, lo);
        wc[row * B::XS + k] = hi;
        wc[(LPP + row) * B::XS + k] = lo;
    }
    const bf16 zero = __float2bfloat16_rn(0.f);
    for (int i = tid; i < C * LRP; i += NTH) {
        const int t = i / LRP, c = i - t * LRP;
        if (c >= Dm.LR) fq[t * B::FS + c] = fk[t * B::FS + c] = fqs[t * B::FS + c] = zero;
    }
    for (int i = tid; i < C * LPP; i += NTH) {
        const int t = i / LPP, c = i - t * LPP;
        if (c >= Dm.LP) dzs[t * B::ZS + c] = zero;
    }
    for (int i = tid; i < 2 * C * 8; i += NTH) {
        const int t = i / 8, c = D + (i & 7);
        xdo[t * B::XS + c] = zero;
    }
}

// fp32 fragments of a carried sketch (the n-tiles warp w owns) and its bf16 hi/lo copy from a
// [LR][D+1] float32 block.
template <int D, int LRP, int LPP>
__device__ __forceinline__ void load_sketch(const Dims &Dm, const float *__restrict__ src, int warp, int lane,
                                            float (&st)[BwdCfg<D, LRP, LPP>::SNT][BwdCfg<D, LRP, LPP>::MT][4],
                                            bf16 *hi, bf16 *lo)
{
    using B = BwdCfg<D, LRP, LPP>;
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

template <int D, int LRP, int LPP>
__device__ __forceinline__ void refresh_sketch(const float (&st)[BwdCfg<D, LRP, LPP>::SNT][BwdCfg<D, LRP, LPP>::MT][4],
                                               int warp, int lane, bf16 *hi, bf16 *lo)
{
    using B = BwdCfg<D, LRP, LPP>;
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

// acc[owned n-tiles][m-tiles] += A^T Y over the chunk: A = [C][FS] features (rows = tokens),
// Y = [C][XS] token tile (its column d is the mass column of the last n-tile when MASSCOL,
// otherwise the mass tile multiplies a ones column).
template <int D, int LRP, int LPP, bool MASSCOL>
__device__ __forceinline__ void sketch_update(float (&st)[BwdCfg<D, LRP, LPP>::SNT][BwdCfg<D, LRP, LPP>::MT][4],
                                              const bf16 *feat, const bf16 *y, int warp, int lane)
{
    using B = BwdCfg<D, LRP, LPP>;
#pragma unroll
    for (int kb = 0; kb < 4; ++kb) {
        uint32_t af[B::MT][4];
#pragma unroll
        for (int mt = 0; mt < B::MT; ++mt) ldsm_a_km(feat, B::FS, 16 * kb, 16 * mt, lane, af[mt]);
#pragma unroll
        for (int j = 0; j < B::SNT; ++j) {
            const int nt = warp + 8 * j;
            if (nt < B::NTO) {
                uint32_t b0, b1;
                if (nt < D / 8 || MASSCOL)
                    ldsm_x2_t(smem_u32(y + (16 * kb + (lane & 7) + 8 * ((lane >> 3) & 1)) * B::XS + 8 * nt), b0, b1);
                else
                    mass_fragment(lane, b0, b1);
#pragma unroll
                for (int mt = 0; mt < B::MT; ++mt) mma_a(st[j][mt], af[mt], b0, b1);
            }
        }
    }
}

template <int D, int LRP, int LPP>
__device__ __forceinline__ void store_sketch(const Dims &Dm,
                                             const float (&st)[BwdCfg<D, LRP, LPP>::SNT][BwdCfg<D, LRP, LPP>::MT][4],
                                             float *__restrict__ out, int warp, int lane)
{
    using B = BwdCfg<D, LRP, LPP>;
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

// ------------------------------------------------------------------ pass 1: dQ, aux, G totals

template <int D, int LRP, int LPP>
__global__ void __launch_bounds__(NTH, 1)
    k_causal_bwd_q_tc(Dims Dm, const bf16 *__restrict__ Q, const bf16 *__restrict__ K, const bf16 *__restrict__ V,
                      const bf16 *__restrict__ dO, const float *__restrict__ W, const float *__restrict__ S0,
                      int64_t seg_len, int nseg, bf16 *__restrict__ dQ, float2 *__restrict__ aux,
                      float *__restrict__ Gseg)
{
    using B = BwdCfg<D, LRP, LPP>;
    extern __shared__ __align__(128) unsigned char smem[];
    bf16 *xq = reinterpret_cast<bf16 *>(smem + B::OFF_XQ);
    bf16 *xk = reinterpret_cast<bf16 *>(smem + B::OFF_XK);
    bf16 *xv = reinterpret_cast<bf16 *>(smem + B::OFF_XV);
    bf16 *xdo = reinterpret_cast<bf16 *>(smem + B::OFF_XDO);
    bf16 *fq = reinterpret_cast<bf16 *>(smem + B::OFF_FQ);
    bf16 *fk = reinterpret_cast<bf16 *>(smem + B::OFF_FK);
    bf16 *fqs = reinterpret_cast<bf16 *>(smem + B::OFF_FQS);
    bf16 *shi = reinterpret_cast<bf16 *>(smem + B::OFF_SHI);
    bf16 *slo = reinterpret_cast<bf16 *>(smem + B::OFF_SLO);
    bf16 *wc = reinterpret_cast<bf16 *>(smem + B::OFF_W);
    float *ust = reinterpret_cast<float *>(smem + B::OFF_U);
    bf16 *vds = reinterpret_cast<bf16 *>(smem + B::OFF_CC);
    float *dphi = reinterpret_cast<float *>(smem + B::OFF_DPHI);
    bf16 *dzs = reinterpret_cast<bf16 *>(smem + B::OFF_DZ);
    float *tok = reinterpret_cast<float *>(smem + B::OFF_TOK);
    float *invq = tok, *den = tok + C, *rden = tok + 2 * C, *ccs = tok + 3 * C, *red = tok + 4 * C;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, q = lane & 3;
    const int rb = warp & 3, h = warp >> 2;
    const int s = blockIdx.x;
    const int64_t bh = blockIdx.y;
    const int64_t off = bh * Dm.N * D;
    const int64_t n_begin = (int64_t)s * seg_len;
    const int64_t n_end = min(Dm.N, n_begin + seg_len);
    const int t0 = 16 * rb + g, t1 = t0 + 8;

    bwd_setup<D, LRP, LPP>(Dm, W, wc, fq, fk, fqs, dzs, xdo);
    float st[B::SNT][B::MT][4], gacc[B::SNT][B::MT][4];
    load_sketch<D, LRP, LPP>(Dm, S0 + ((int64_t)bh * nseg + s) * Dm.LR * (D + 1), warp, lane, st, shi, slo);
#pragma unroll
    for (int j = 0; j < B::SNT; ++j)
#pragma unroll
        for (int mt = 0; mt < B::MT; ++mt)
#pragma unroll
            for (int e = 0; e < 4; ++e) gacc[j][mt][e] = 0.f;

    if (n_begin < n_end) {
        const int cnt0 = (int)min((int64_t)C, n_end - n_begin);
        load_tile_async<D, B::XS>(xq, Q + off, n_begin, cnt0);
        load_tile_async<D, B::XS>(xk, K + off, n_begin, cnt0);
        load_tile_async<D, B::XS>(xv, V + off, n_begin, cnt0);
        load_tile_async<D, B::XS>(xdo, dO + off, n_begin, cnt0);
    }
    cp_async_commit();

    int buf = 0;
    for (int64_t n0 = n_begin; n0 < n_end; n0 += C, buf ^= 1) {
        const int cnt = (int)min((int64_t)C, n_end - n0);
        cp_async_wait<0>();
        __syncthreads();
        {
            const int64_t n1 = n0 + C;
            if (n1 < n_end) {
                const int cnt1 = (int)min((int64_t)C, n_end - n1);
                const int o = (buf ^ 1) * C * B::XS;
                load_tile_async<D, B::XS>(xq + o, Q + off, n1, cnt1);
                load_tile_async<D, B::XS>(xk + o, K + off, n1, cnt1);
                load_tile_async<D, B::XS>(xv + o, V + off, n1, cnt1);
                load_tile_async<D, B::XS>(xdo + o, dO + off, n1, cnt1);
            }
            cp_async_commit();
        }
        bf16 *xqb = xq + buf * C * B::XS, *xkb = xk + buf * C * B::XS;
        bf16 *xvb = xv + buf * C * B::XS, *xdob = xdo + buf * C * B::XS;

        // P1: projections
        project_rows<D, LRP, LPP>(xqb, wc, ust, rb, h, lane, invq);
        project_rows<D, LRP, LPP>(xkb, wc, ust + C * B::US, rb, h, lane);
        __syncthreads();
        // P2: features
        featurise_tiles<D, LRP, LPP>(Dm, ust, fq, fk, 2, cnt);
        __syncthreads();

        // P3: scores, den, V.dO block, g (sketch part)
        uint32_t aq[B::KF][4];
#pragma unroll
        for (int kf = 0; kf < B::KF; ++kf) ldsm_a(fq, B::FS, 16 * rb, 16 * kf, lane, aq[kf]);
        float gq[B::NLH][4];
        float den0, den1;
        {
            uint32_t sa[4][4];
            {
                float sc[8][4];
#pragma unroll
                for (int jt = 0; jt < 8; ++jt) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) sc[jt][e] = 0.f;
                    if (jt <= 2 * rb + 1) {
#pragma unroll
                        for (int kf = 0; kf < B::KF; ++kf) {
                            uint32_t b0, b1;
                            ldsm_x2(smem_u32(fk + (8 * jt + (lane & 7)) * B::FS + 16 * kf + 8 * ((lane >> 3) & 1)),
                                    b0, b1);
                            mma_a(sc[jt], aq[kf], b0, b1);
                        }
                        if (jt >= 2 * rb) {
#pragma unroll
                            for (int e = 0; e < 4; ++e)
                                if (8 * jt + 2 * q + (e & 1) > 16 * rb + g + 8 * (e >> 1)) sc[jt][e] = 0.f;
                        }
                    }
                }
#pragma unroll
                for (int kb = 0; kb < 4; ++kb) {
                    sa[kb][0] = pack_bf16(sc[2 * kb][0], sc[2 * kb][1]);
                    sa[kb][1] = pack_bf16(sc[2 * kb][2], sc[2 * kb][3]);
                    sa[kb][2] = pack_bf16(sc[2 * kb + 1][0], sc[2 * kb + 1][1]);
                    sa[kb][3] = pack_bf16(sc[2 * kb + 1][2], sc[2 * kb + 1][3]);
                }
            }
            float om[4] = {0.f, 0.f, 0.f, 0.f};
            uint32_t m0, m1;
            mass_fragment(lane, m0, m1);
#pragma unroll
            for (int kb = 0; kb < 4; ++kb)
                if (kb <= rb) mma_a(om, sa[kb], m0, m1);
#pragma unroll
            for (int kf = 0; kf < B::KF; ++kf) {
                const int addr = (16 * kf + (lane & 7) + 8 * ((lane >> 3) & 1)) * B::SS + D;
                uint32_t b0, b1;
                ldsm_x2_t(smem_u32(shi + addr), b0, b1);
                mma_a(om, aq[kf], b0, b1);
                ldsm_x2_t(smem_u32(slo + addr), b0, b1);
                mma_a(om, aq[kf], b0, b1);
            }
            den0 = __shfl_sync(0xffffffffu, om[0], lane & ~3);
            den1 = __shfl_sync(0xffffffffu, om[2], lane & ~3);
        }
        {
            uint32_t ado[B::KQ][4];
#pragma unroll
            for (int ks = 0; ks < B::KQ; ++ks) ldsm_a(xdob, B::XS, 16 * rb, 16 * ks, lane, ado[ks]);
            // (V_j . dO_t) for j <= t, key tiles split between the two column-half warps
#pragma unroll
            for (int jt = 0; jt < 8; ++jt) {
                if (jt <= 2 * rb + 1 && (jt & 1) == h) {
                    float va[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int ks = 0; ks < B::KQ; ++ks) {
                        uint32_t b0, b1;
                        ldsm_x2(smem_u32(xvb + (8 * jt + (lane & 7)) * B::XS + 16 * ks + 8 * ((lane >> 3) & 1)), b0,
                                b1);
                        mma_a(va, ado[ks], b0, b1);
                    }
                    const int j = 8 * jt + 2 * q;
                    *reinterpret_cast<uint32_t *>(vds + t0 * B::VS + j) =
                        pack_bf16(j <= t0 ? va[0] : 0.f, j + 1 <= t0 ? va[1] : 0.f);
                    *reinterpret_cast<uint32_t *>(vds + t1 * B::VS + j) =
                        pack_bf16(j <= t1 ? va[2] : 0.f, j + 1 <= t1 ? va[3] : 0.f);
                }
            }
            // g = S_prev,A dO for this warp's feature half
#pragma unroll
            for (int i = 0; i < B::NLH; ++i)
#pragma unroll
                for (int e = 0; e < 4; ++e) gq[i][e] = 0.f;
#pragma unroll
            for (int ks = 0; ks < B::KQ; ++ks) {
#pragma unroll
                for (int i = 0; i < B::NLH; i += 2) {
                    const int nt = h * B::NLH + i;
                    uint32_t b0, b1, b2, b3;
                    ldsm_b_nk_x4(shi, B::SS, 8 * nt, 16 * ks, lane, b0, b1, b2, b3);
                    mma_a(gq[i], ado[ks], b0, b1);
                    mma_a(gq[i + 1], ado[ks], b2, b3);
                    ldsm_b_nk_x4(slo, B::SS, 8 * nt, 16 * ks, lane, b0, b1, b2, b3);
                    mma_a(gq[i], ado[ks], b0, b1);
                    mma_a(gq[i + 1], ado[ks], b2, b3);
                }
            }
        }
        if (h == 0 && q == 0) {
            den[t0] = den0;
            den[t1] = den1;
        }
        __syncthreads();

        // P4: g (intra part), prefix mass B_t, partial phi_Q . g
        float sb[B::NLH][4];
        {
#pragma unroll
            for (int i = 0; i < B::NLH; ++i)
#pragma unroll
                for (int e = 0; e < 4; ++e) sb[i][e] = 0.f;
#pragma unroll
            for (int kb = 0; kb < 4; ++kb) {
                if (kb <= rb) {
                    uint32_t av[4], al[4];
                    ldsm_a(vds, B::VS, 16 * rb, 16 * kb, lane, av);
                    tril_ones_fragment(16 * rb, 16 * kb, lane, al);
#pragma unroll
                    for (int i = 0; i < B::NLH; i += 2) {
                        const int nt = h * B::NLH + i;
                        uint32_t b0, b1, b2, b3;
                        ldsm_b_kn_x4(fk, B::FS, 16 * kb, 8 * nt, lane, b0, b1, b2, b3);
                        mma_a(gq[i], av, b0, b1);
                        mma_a(gq[i + 1], av, b2, b3);
                        mma_a(sb[i], al, b0, b1);
                        mma_a(sb[i + 1], al, b2, b3);
                    }
                }
            }
            float p0 = 0.f, p1 = 0.f;
#pragma unroll
            for (int i = 0; i < B::NLH; ++i) {
                const int lr = 8 * (h * B::NLH + i) + 2 * q;
                const float2 f0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(fq + t0 * B::FS + lr));
                const float2 f1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(fq + t1 * B::FS + lr));
                p0 = fmaf(f0.x, gq[i][0], fmaf(f0.y, gq[i][1], p0));
                p1 = fmaf(f1.x, gq[i][2], fmaf(f1.y, gq[i][3], p1));
                const float sb0 = __bfloat162float(shi[lr * B::SS + D]) + __bfloat162float(slo[lr * B::SS + D]);
                const float sb1 =
                    __bfloat162float(shi[(lr + 1) * B::SS + D]) + __bfloat162float(slo[(lr + 1) * B::SS + D]);
                sb[i][0] += sb0;
                sb[i][1] += sb1;
                sb[i][2] += sb0;
                sb[i][3] += sb1;
            }
            p0 += __shfl_xor_sync(0xffffffffu, p0, 1);
            p0 += __shfl_xor_sync(0xffffffffu, p0, 2);
            p1 += __shfl_xor_sync(0xffffffffu, p1, 1);
            p1 += __shfl_xor_sync(0xffffffffu, p1, 2);
            if (q == 0) {
                red[h * C + t0] = p0;
                red[h * C + t1] = p1;
            }
        }
        __syncthreads();

        // P5: c_t = dO_t . O_t, dphi_Q = (g - B_t c) / den
        {
            const bool l0 = t0 < cnt, l1 = t1 < cnt;
            const float rd0 = l0 ? 1.f / den[t0] : 0.f, rd1 = l1 ? 1.f / den[t1] : 0.f;
            const float c0 = (red[t0] + red[C + t0]) * rd0, c1 = (red[t1] + red[C + t1]) * rd1;
#pragma unroll
            for (int i = 0; i < B::NLH; ++i) {
                const int lr = 8 * (h * B::NLH + i) + 2 * q;
                dphi[t0 * B::DPS + lr] = (gq[i][0] - sb[i][0] * c0) * rd0;
                dphi[t0 * B::DPS + lr + 1] = (gq[i][1] - sb[i][1] * c0) * rd0;
                dphi[t1 * B::DPS + lr] = (gq[i][2] - sb[i][2] * c1) * rd1;
                dphi[t1 * B::DPS + lr + 1] = (gq[i][3] - sb[i][3] * c1) * rd1;
            }
            if (h == 0 && q == 0) {
                rden[t0] = rd0;
                rden[t1] = rd1;
                ccs[t0] = c0;
                ccs[t1] = c1;
                xdob[t0 * B::XS + D] = __float2bfloat16_rn(-c0);
                xdob[t1 * B::XS + D] = __float2bfloat16_rn(-c1);
                if (l0) aux[bh * Dm.N + n0 + t0] = make_float2(rd0, c0);
                if (l1) aux[bh * Dm.N + n0 + t1] = make_float2(rd1, c1);
            }
        }
        __syncthreads();

        // P6: feature Jacobian (Q side) and phi_Q / den for the gradient sketch
        featurise_backward_tiles<B::US, B::DPS, B::ZS>(Dm, ust, dphi, dzs);
        for (int i = tid; i < C * Dm.LR; i += NTH) {
            const int t = i / Dm.LR, c = i - t * Dm.LR;
            fqs[t * B::FS + c] = __float2bfloat16_rn(__bfloat162float(fq[t * B::FS + c]) * rden[t]);
        }
        __syncthreads();

        // P7: dQ projection back, gradient-sketch totals, prefix sketch update
        float dx[D / 16][4];
        back_project<D, LPP, B::XS, B::ZS>(dzs, wc, xqb, rb, h, lane, dx, red + h * C);
        sketch_update<D, LRP, LPP, true>(gacc, fqs, xdob, warp, lane);
        sketch_update<D, LRP, LPP, false>(st, fk, xvb, warp, lane);
        __syncthreads();

        // P8: dQ = normalisation backward, staged in the consumed K tile; refresh S copies
        stage_dx<D, B::XS>(dx, xqb, invq, red, rb, h, lane, xkb);
        __syncwarp();
        store_rows<D, B::XS>(xkb, dQ + off, n0, cnt, rb, h, lane);
        refresh_sketch<D, LRP, LPP>(st, warp, lane, shi, slo);
    }
    cp_async_wait<0>();
    store_sketch<D, LRP, LPP>(Dm, gacc, Gseg + ((int64_t)bh * nseg + s) * Dm.LR * (D + 1), warp, lane);
}

// ------------------------------------------------------------------ pass 2: dK, dV

template <int D, int LRP, int LPP>
__global__ void __launch_bounds__(NTH, 1)
    k_causal_bwd_kv_tc(Dims Dm, const bf16 *__restrict__ Q, const bf16 *__restrict__ K, const bf16 *__restrict__ V,
                       const bf16 *__restrict__ dO, const float2 *__restrict__ aux, const float *__restrict__ W,
                       const float *__restrict__ G0, int64_t seg_len, int nseg, bf16 *__restrict__ dK,
                       bf16 *__restrict__ dV)
{
    using B = BwdCfg<D, LRP, LPP>;
    extern __shared__ __align__(128) unsigned char smem[];
    bf16 *xq = reinterpret_cast<bf16 *>(smem + B::OFF_XQ);
    bf16 *xk = reinterpret_cast<bf16 *>(smem + B::OFF_XK);
    bf16 *xv = reinterpret_cast<bf16 *>(smem + B::OFF_XV);
    bf16 *xdo = reinterpret_cast<bf16 *>(smem + B::OFF_XDO);
    bf16 *fq = reinterpret_cast<bf16 *>(smem + B::OFF_FQ);
    bf16 *fk = reinterpret_cast<bf16 *>(smem + B::OFF_FK);
    bf16 *fqs = reinterpret_cast<bf16 *>(smem + B::OFF_FQS);
    bf16 *ghi = reinterpret_cast<bf16 *>(smem + B::OFF_SHI);
    bf16 *glo = reinterpret_cast<bf16 *>(smem + B::OFF_SLO);
    bf16 *wc = reinterpret_cast<bf16 *>(smem + B::OFF_W);
    float *ust = reinterpret_cast<float *>(smem + B::OFF_U);
    bf16 *wst = reinterpret_cast<bf16 *>(smem + B::OFF_CC);
    float *dphi = reinterpret_cast<float *>(smem + B::OFF_DPHI);
    bf16 *dzs = reinterpret_cast<bf16 *>(smem + B::OFF_DZ);
    float *tok = reinterpret_cast<float *>(smem + B::OFF_TOK);
    float *invk = tok, *rden = tok + C, *ccs = tok + 2 * C, *red = tok + 3 * C;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, q = lane & 3;
    const int rb = warp & 3, h = warp >> 2;
    const int s = blockIdx.x;
    const int64_t bh = blockIdx.y;
    const int64_t off = bh * Dm.N * D;
    const int64_t n_begin = (int64_t)s * seg_len;
    const int64_t n_end = min(Dm.N, n_begin + seg_len);
    const int j0 = 16 * rb + g, j1 = j0 + 8;  // key rows of this warp

    bwd_setup<D, LRP, LPP>(Dm, W, wc, fq, fk, fqs, dzs, xdo);
    float gst[B::SNT][B::MT][4];
    load_sketch<D, LRP, LPP>(Dm, G0 + ((int64_t)bh * nseg + s) * Dm.LR * (D + 1), warp, lane, gst, ghi, glo);
    if (n_begin >= n_end) return;

    const int64_t last = n_begin + ((n_end - 1 - n_begin) / C) * C;
    {
        const int cnt0 = (int)min((int64_t)C, n_end - last);
        load_tile_async<D, B::XS>(xq, Q + off, last, cnt0);
        load_tile_async<D, B::XS>(xk, K + off, last, cnt0);
        load_tile_async<D, B::XS>(xv, V + off, last, cnt0);
        load_tile_async<D, B::XS>(xdo, dO + off, last, cnt0);
    }
    cp_async_commit();

    int buf = 0;
    for (int64_t n0 = last; n0 >= n_begin; n0 -= C, buf ^= 1) {
        const int cnt = (int)min((int64_t)C, n_end - n0);
        cp_async_wait<0>();
        __syncthreads();
        {
            const int64_t n1 = n0 - C;
            if (n1 >= n_begin) {
                const int o = (buf ^ 1) * C * B::XS;
                load_tile_async<D, B::XS>(xq + o, Q + off, n1, C);
                load_tile_async<D, B::XS>(xk + o, K + off, n1, C);
                load_tile_async<D, B::XS>(xv + o, V + off, n1, C);
                load_tile_async<D, B::XS>(xdo + o, dO + off, n1, C);
            }
            cp_async_commit();
        }
        bf16 *xqb = xq + buf * C * B::XS, *xkb = xk + buf * C * B::XS;
        bf16 *xvb = xv + buf * C * B::XS, *xdob = xdo + buf * C * B::XS;
        for (int t = tid; t < C; t += NTH) {
            float2 a = make_float2(0.f, 0.f);
            if (t < cnt) a = aux[bh * Dm.N + n0 + t];
            rden[t] = a.x;
            ccs[t] = a.y;
        }

        // P1: projections
        project_rows<D, LRP, LPP>(xqb, wc, ust, rb, h, lane);
        project_rows<D, LRP, LPP>(xkb, wc, ust + C * B::US, rb, h, lane, invk);
        __syncthreads();
        // P2: features (phi_Q, phi_Q / den, phi_K); -c_t into the dO tile's mass column
        featurise_tiles<D, LRP, LPP>(Dm, ust, fq, fk, 2, cnt, rden, fqs);
        for (int t = tid; t < C; t += NTH) xdob[t * B::XS + D] = __float2bfloat16_rn(-ccs[t]);
        __syncthreads();

        // P3: dV, the staged (V_j . dO_t - c_t) / den_t block, dphi_K (G_next part)
        constexpr int NC = D / 16;
        float dpk[B::NLH][4];
        {
            uint32_t ak[B::KF][4];
#pragma unroll
            for (int kf = 0; kf < B::KF; ++kf) ldsm_a(fk, B::FS, 16 * rb, 16 * kf, lane, ak[kf]);
            float dva[NC][4];
#pragma unroll
            for (int i = 0; i < NC; ++i)
#pragma unroll
                for (int e = 0; e < 4; ++e) dva[i][e] = 0.f;
            {
                // (phi_K(j) . phi_Q(t)) / den_t for t >= j, as A fragments over query blocks
                uint32_t pa[4][4];
                {
                    float pt[8][4];
#pragma unroll
                    for (int tt = 0; tt < 8; ++tt) {
#pragma unroll
                        for (int e = 0; e < 4; ++e) pt[tt][e] = 0.f;
                        if (tt >= 2 * rb) {
#pragma unroll
                            for (int kf = 0; kf < B::KF; ++kf) {
                                uint32_t b0, b1;
                                ldsm_x2(smem_u32(fq + (8 * tt + (lane & 7)) * B::FS + 16 * kf + 8 * ((lane >> 3) & 1)),
                                        b0, b1);
                                mma_a(pt[tt], ak[kf], b0, b1);
                            }
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const int t = 8 * tt + 2 * q + (e & 1), j = 16 * rb + g + 8 * (e >> 1);
                                pt[tt][e] = t >= j ? pt[tt][e] * rden[t] : 0.f;
                            }
                        }
                    }
#pragma unroll
                    for (int kb = 0; kb < 4; ++kb) {
                        pa[kb][0] = pack_bf16(pt[2 * kb][0], pt[2 * kb][1]);
                        pa[kb][1] = pack_bf16(pt[2 * kb][2], pt[2 * kb][3]);
                        pa[kb][2] = pack_bf16(pt[2 * kb + 1][0], pt[2 * kb + 1][1]);
                        pa[kb][3] = pack_bf16(pt[2 * kb + 1][2], pt[2 * kb + 1][3]);
                    }
                }
#pragma unroll
                for (int kb = 0; kb < 4; ++kb) {
                    if (kb >= rb) {
#pragma unroll
                        for (int i = 0; i < NC; i += 2) {
                            uint32_t b0, b1, b2, b3;
                            ldsm_b_kn_x4(xdob, B::XS, 16 * kb, 8 * (h * NC + i), lane, b0, b1, b2, b3);
                            mma_a(dva[i], pa[kb], b0, b1);
                            mma_a(dva[i + 1], pa[kb], b2, b3);
                        }
                    }
                }
            }
#pragma unroll
            for (int kf = 0; kf < B::KF; ++kf) {
#pragma unroll
                for (int i = 0; i < NC; i += 2) {
                    uint32_t b0, b1, b2, b3;
                    ldsm_b_kn_x4(ghi, B::SS, 16 * kf, 8 * (h * NC + i), lane, b0, b1, b2, b3);
                    mma_a(dva[i], ak[kf], b0, b1);
                    mma_a(dva[i + 1], ak[kf], b2, b3);
                    ldsm_b_kn_x4(glo, B::SS, 16 * kf, 8 * (h * NC + i), lane, b0, b1, b2, b3);
                    mma_a(dva[i], ak[kf], b0, b1);
                    mma_a(dva[i + 1], ak[kf], b2, b3);
                }
            }
            // dV staged in the consumed Q tile (its only use was the projection)
#pragma unroll
            for (int i = 0; i < NC; ++i) {
                const int c = 8 * (h * NC + i) + 2 * q;
                *reinterpret_cast<uint32_t *>(xqb + j0 * B::XS + c) = pack_bf16(dva[i][0], dva[i][1]);
                *reinterpret_cast<uint32_t *>(xqb + j1 * B::XS + c) = pack_bf16(dva[i][2], dva[i][3]);
            }
        }
        {
            uint32_t av[B::KQ][4];
#pragma unroll
            for (int ks = 0; ks < B::KQ; ++ks) ldsm_a(xvb, B::XS, 16 * rb, 16 * ks, lane, av[ks]);
#pragma unroll
            for (int tt = 0; tt < 8; ++tt) {
                if (tt >= 2 * rb && (tt & 1) == h) {
                    float va[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int ks = 0; ks < B::KQ; ++ks) {
                        uint32_t b0, b1;
                        ldsm_x2(smem_u32(xdob + (8 * tt + (lane & 7)) * B::XS + 16 * ks + 8 * ((lane >> 3) & 1)), b0,
                                b1);
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
#pragma unroll
            for (int i = 0; i < B::NLH; ++i)
#pragma unroll
                for (int e = 0; e < 4; ++e) dpk[i][e] = 0.f;
#pragma unroll
            for (int ks = 0; ks < B::KQ; ++ks) {
#pragma unroll
                for (int i = 0; i < B::NLH; i += 2) {
                    const int nt = h * B::NLH + i;
                    uint32_t b0, b1, b2, b3;
                    ldsm_b_nk_x4(ghi, B::SS, 8 * nt, 16 * ks, lane, b0, b1, b2, b3);
                    mma_a(dpk[i], av[ks], b0, b1);
                    mma_a(dpk[i + 1], av[ks], b2, b3);
                    ldsm_b_nk_x4(glo, B::SS, 8 * nt, 16 * ks, lane, b0, b1, b2, b3);
                    mma_a(dpk[i], av[ks], b0, b1);
                    mma_a(dpk[i + 1], av[ks], b2, b3);
                }
            }
        }
        __syncwarp();
        store_rows<D, B::XS>(xqb, dV + off, n0, cnt, rb, h, lane);
        __syncthreads();

        // P4: dphi_K intra part and the mass term
        {
#pragma unroll
            for (int kb = 0; kb < 4; ++kb) {
                if (kb >= rb) {
                    uint32_t aw[4];
                    ldsm_a(wst, B::VS, 16 * rb, 16 * kb, lane, aw);
#pragma unroll
                    for (int i = 0; i < B::NLH; i += 2) {
                        const int nt = h * B::NLH + i;
                        uint32_t b0, b1, b2, b3;
                        ldsm_b_kn_x4(fq, B::FS, 16 * kb, 8 * nt, lane, b0, b1, b2, b3);
                        mma_a(dpk[i], aw, b0, b1);
                        mma_a(dpk[i + 1], aw, b2, b3);
                    }
                }
            }
#pragma unroll
            for (int i = 0; i < B::NLH; ++i) {
                const int lr = 8 * (h * B::NLH + i) + 2 * q;
                const float gb0 = __bfloat162float(ghi[lr * B::SS + D]) + __bfloat162float(glo[lr * B::SS + D]);
                const float gb1 =
                    __bfloat162float(ghi[(lr + 1) * B::SS + D]) + __bfloat162float(glo[(lr + 1) * B::SS + D]);
                dphi[j0 * B::DPS + lr] = dpk[i][0] + gb0;
                dphi[j0 * B::DPS + lr + 1] = dpk[i][1] + gb1;
                dphi[j1 * B::DPS + lr] = dpk[i][2] + gb0;
                dphi[j1 * B::DPS + lr + 1] = dpk[i][3] + gb1;
            }
        }
        __syncthreads();

        // P5: feature Jacobian (K side)
        featurise_backward_tiles<B::US, B::DPS, B::ZS>(Dm, ust + C * B::US, dphi, dzs);
        __syncthreads();

        // P6: dK projection back; G += phi_Q^T [dO | -c] / den
        float dx[D / 16][4];
        back_project<D, LPP, B::XS, B::ZS>(dzs, wc, xkb, rb, h, lane, dx, red + h * C);
        sketch_update<D, LRP, LPP, true>(gst, fqs, xdob, warp, lane);
        __syncthreads();

        // P7: dK staged in the consumed V tile; refresh G copies
        stage_dx<D, B::XS>(dx, xkb, invk, red, rb, h, lane, xvb);
        __syncwarp();
        store_rows<D, B::XS>(xvb, dK + off, n0, cnt, rb, h, lane);
        refresh_sketch<D, LRP, LPP>(gst, warp, lane, ghi, glo);
    }
    cp_async_wait<0>();
}

}  // namespace tc

// ------------------------------------------------------------------ host side

namespace {

constexpr size_t kSmemLimit = 227 * 1024;

template <int D, int LRP, int LPP>
cudaError_t launch_bwd_q_inst(const Dims &Dm, const bf16_t *Q, const bf16_t *K, const bf16_t *V, const bf16_t *dO,
                              const float *W, const float *S0, int64_t seg_len, int nseg, bf16_t *dQ, float2 *aux,
                              float *Gseg, cudaStream_t st)
{
    using B = tc::BwdCfg<D, LRP, LPP>;
    if constexpr (B::BYTES > kSmemLimit) {
        return cudaErrorInvalidValue;
    } else {
        auto kern = tc::k_causal_bwd_q_tc<D, LRP, LPP>;
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, B::BYTES);
        if (e != cudaSuccess) return e;
        return launch_kernel("tc_causal_bwd_q", kern, dim3(nseg, (unsigned)Dm.BH), dim3(tc::NTH), (size_t)B::BYTES,
                             st, Dm, Q, K, V, dO, W, S0, seg_len, nseg, dQ, aux, Gseg);
    }
}

template <int D, int LRP, int LPP>
cudaError_t launch_bwd_kv_inst(const Dims &Dm, const bf16_t *Q, const bf16_t *K, const bf16_t *V, const bf16_t *dO,
                               const float2 *aux, const float *W, const float *G0, int64_t seg_len, int nseg,
                               bf16_t *dK, bf16_t *dV, cudaStream_t st)
{
    using B = tc::BwdCfg<D, LRP, LPP>;
    if constexpr (B::BYTES > kSmemLimit) {
        return cudaErrorInvalidValue;
    } else {
        auto kern = tc::k_causal_bwd_kv_tc<D, LRP, LPP>;
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, B::BYTES);
        if (e != cudaSuccess) return e;
        return launch_kernel("tc_causal_bwd_kv", kern, dim3(nseg, (unsigned)Dm.BH), dim3(tc::NTH), (size_t)B::BYTES,
                             st, Dm, Q, K, V, dO, aux, W, G0, seg_len, nseg, dK, dV);
    }
}

template <int D, int LRP, int LPP>
constexpr bool bwd_fits()
{
    return tc::BwdCfg<D, LRP, LPP>::BYTES <= kSmemLimit;
}

}  // namespace

bool causal_tc_bwd_supported(const Dims &Dm)
{
    if (!causal_tc_supported(Dm)) return false;
    const bool lr32 = Dm.LR <= 32, lp16 = Dm.LP <= 16;
    if (Dm.d == 128) return lr32 ? (lp16 ? bwd_fits<128, 32, 16>() : bwd_fits<128, 32, 32>())
                                 : (lp16 ? bwd_fits<128, 64, 16>() : bwd_fits<128, 64, 32>());
    return lr32 ? (lp16 ? bwd_fits<64, 32, 16>() : bwd_fits<64, 32, 32>())
                : (lp16 ? bwd_fits<64, 64, 16>() : bwd_fits<64, 64, 32>());
}

#define RACE_TC_BWD_DISPATCH(FN, ...)                                                   \
    const bool lr32 = Dm.LR <= 32, lp16 = Dm.LP <= 16;                                  \
    if (Dm.d == 128) {                                                                  \
        if (lr32 && lp16) return FN<128, 32, 16>(__VA_ARGS__);                          \
        if (lr32) return FN<128, 32, 32>(__VA_ARGS__);                                  \
        if (lp16) return FN<128, 64, 16>(__VA_ARGS__);                                  \
        return FN<128, 64, 32>(__VA_ARGS__);                                            \
    }                                                                                   \
    if (lr32 && lp16) return FN<64, 32, 16>(__VA_ARGS__);                               \
    if (lr32) return FN<64, 32, 32>(__VA_ARGS__);                                       \
    if (lp16) return FN<64, 64, 16>(__VA_ARGS__);                                       \
    return FN<64, 64, 32>(__VA_ARGS__);

cudaError_t launch_causal_tc_bwd_q(const Dims &Dm, const bf16_t *Q, const bf16_t *K, const bf16_t *V,
                                   const bf16_t *dO, const float *W, const float *S0, int64_t seg_len, int nseg,
                                   bf16_t *dQ, float2 *aux, float *Gseg, cudaStream_t st)
{
    RACE_TC_BWD_DISPATCH(launch_bwd_q_inst, Dm, Q, K, V, dO, W, S0, seg_len, nseg, dQ, aux, Gseg, st)
}

cudaError_t launch_causal_tc_bwd_kv(const Dims &Dm, const bf16_t *Q, const bf16_t *K, const bf16_t *V,
                                    const bf16_t *dO, const float2 *aux, const float *W, const float *G0,
                                    int64_t seg_len, int nseg, bf16_t *dK, bf16_t *dV, cudaStream_t st)
{
    RACE_TC_BWD_DISPATCH(launch_bwd_kv_inst, Dm, Q, K, V, dO, aux, W, G0, seg_len, nseg, dK, dV, st)
}

}  // namespace race
