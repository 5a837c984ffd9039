// race_tc_common.cuh -- pieces shared by the tensor-core causal kernels: chunk geometry,
// asynchronous tile loads, the tensor-core projection z = X (W_hi + W_lo)^T with tanh, the bucket
// featuriser, and constant fragments.
#pragma once

#include "race_common.cuh"
#include "race_mma.cuh"

namespace race {
namespace tc {

using bf16 = __nv_bfloat16;
using namespace race::mma;

constexpr int C = 64;     // tokens per chunk
constexpr int NTH = 256;  // 8 warps

template <int D, int LRP, int LPP>
struct CausalCfg {
    static constexpr int XS = D + 8;        // row stride (elements) of token tiles
    static constexpr int FS = LRP + 8;      // row stride of feature tiles
    static constexpr int SS = D + 8;        // row stride of the bf16 state copies (d, mass, 7 zeros)
    static constexpr int NWP = 2 * LPP;     // hyperplane rows: LPP hi rows then LPP lo rows
    static constexpr int US = LPP + 1;      // row stride of the staged tanh projections (fp32)
    static constexpr int NTO = D / 8 + 1;   // output / state n-tiles including the mass tile
    static constexpr int KQ = D / 16;       // k-steps over d
    static constexpr int KF = LRP / 16;     // k-steps over features
    static constexpr int MT = LRP / 16;     // state m-tiles
    static constexpr int SNT = (NTO + 7) / 8;  // state n-tiles per warp (warp w owns w, w+8, ...)
    static constexpr int NLT = LPP / 16;    // lp tiles (of 8) per projection warp
    static constexpr int X_BYTES = C * XS * 2;
    static constexpr int OFF_XQ = 0;
    static constexpr int OFF_XK = OFF_XQ + 2 * X_BYTES;
    static constexpr int OFF_XV = OFF_XK + 2 * X_BYTES;
    static constexpr int OFF_FQ = OFF_XV + 2 * X_BYTES;
    static constexpr int OFF_FK = OFF_FQ + C * FS * 2;
    static constexpr int OFF_SHI = OFF_FK + C * FS * 2;
    static constexpr int OFF_SLO = OFF_SHI + LRP * SS * 2;
    static constexpr int OFF_W = OFF_SLO + LRP * SS * 2;
    static constexpr int OFF_U = OFF_W + NWP * XS * 2;
    static constexpr int BYTES = OFF_U + 2 * C * US * 4;
};

// cp.async a [C, D] bf16 tile (rows n0 .. n0 + cnt of a [N, D] slice) into a padded smem tile;
// rows past cnt are zero filled.
template <int D, int XS>
__device__ __forceinline__ void load_tile_async(bf16 *dst, const bf16 *__restrict__ src, int64_t n0, int cnt)
{
    constexpr int CH = D / 8;
    for (int i = threadIdx.x; i < C * CH; i += NTH) {
        const int r = i / CH, cc = i - r * CH;
        const bf16 *s = src + (n0 + (r < cnt ? r : 0)) * D + cc * 8;
        cp_async16(smem_u32(dst + r * XS + cc * 8), s, r < cnt ? 16 : 0);
    }
}

// z = X W^T for 16 rows (warp row block rb) and this warp's lp tiles (half h), normalised by
// 1/|x| and passed through tanh; the results go to ust[row][lp] (fp32).
template <int D, int LRP, int LPP>
__device__ __forceinline__ void project_rows(const bf16 *xs, const bf16 *wc, float *ust, int rb, int h, int lane,
                                             float *inv_out = nullptr)
{
    using Cf = CausalCfg<D, LRP, LPP>;
    float zh[Cf::NLT][4], zl[Cf::NLT][4];
#pragma unroll
    for (int i = 0; i < Cf::NLT; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) zh[i][j] = zl[i][j] = 0.f;
    float ss0 = 0.f, ss1 = 0.f;
    const int arow = 16 * rb + (lane & 7) + 8 * ((lane >> 3) & 1);
#pragma unroll
    for (int ks = 0; ks < Cf::KQ; ++ks) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4(smem_u32(xs + arow * Cf::XS + 16 * ks + 8 * (lane >> 4)), a0, a1, a2, a3);
        {
            float2 f0 = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162 *>(&a0));
            float2 f1 = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162 *>(&a1));
            float2 f2 = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162 *>(&a2));
            float2 f3 = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162 *>(&a3));
            ss0 = fmaf(f0.x, f0.x, fmaf(f0.y, f0.y, fmaf(f2.x, f2.x, fmaf(f2.y, f2.y, ss0))));
            ss1 = fmaf(f1.x, f1.x, fmaf(f1.y, f1.y, fmaf(f3.x, f3.x, fmaf(f3.y, f3.y, ss1))));
        }
#pragma unroll
        for (int lt = 0; lt < Cf::NLT; ++lt) {
            const int hirow = 8 * (h * Cf::NLT + lt);
            const int wrow = ((lane >> 4) ? LPP + hirow : hirow) + (lane & 7);
            uint32_t bh0, bh1, bl0, bl1;
            ldsm_x4(smem_u32(wc + wrow * Cf::XS + 16 * ks + 8 * ((lane >> 3) & 1)), bh0, bh1, bl0, bl1);
            mma16816(zh[lt], a0, a1, a2, a3, bh0, bh1);
            mma16816(zl[lt], a0, a1, a2, a3, bl0, bl1);
        }
    }
    ss0 += __shfl_xor_sync(0xffffffffu, ss0, 1);
    ss0 += __shfl_xor_sync(0xffffffffu, ss0, 2);
    ss1 += __shfl_xor_sync(0xffffffffu, ss1, 1);
    ss1 += __shfl_xor_sync(0xffffffffu, ss1, 2);
    const float inv0 = ss0 > 0.f ? 1.0f / sqrtf(ss0) : 0.f;
    const float inv1 = ss1 > 0.f ? 1.0f / sqrtf(ss1) : 0.f;
    const int g = lane >> 2, q = lane & 3;
    const int r0 = 16 * rb + g, r1 = r0 + 8;
    if (inv_out && h == 0 && q == 0) {
        inv_out[r0] = inv0;
        inv_out[r1] = inv1;
    }
#pragma unroll
    for (int lt = 0; lt < Cf::NLT; ++lt) {
        const int col = 8 * (h * Cf::NLT + lt) + 2 * q;
        ust[r0 * Cf::US + col] = tanhf((zh[lt][0] + zl[lt][0]) * inv0);
        ust[r0 * Cf::US + col + 1] = tanhf((zh[lt][1] + zl[lt][1]) * inv0);
        ust[r1 * Cf::US + col] = tanhf((zh[lt][2] + zl[lt][2]) * inv1);
        ust[r1 * Cf::US + col + 1] = tanhf((zh[lt][3] + zl[lt][3]) * inv1);
    }
}

// Bucket features of the staged tanh projections: F[t][l*R + r] = prod_p sigmoid(+-2 beta u);
// rows t >= cnt are zero.  Work items (side, table, token), lanes over tokens.
template <int D, int LRP, int LPP>
__device__ __forceinline__ void featurise_tiles(const Dims &Dm, const float *ust, bf16 *f0, bf16 *f1,
                                                int nsides, int cnt, const float *scale0 = nullptr,
                                                bf16 *f0s = nullptr)
{
    using Cf = CausalCfg<D, LRP, LPP>;
    const int total = nsides * Dm.L * C;
    for (int it = threadIdx.x; it < total; it += NTH) {
        const int t = it % C;
        const int l = (it / C) % Dm.L;
        const int side = it / (C * Dm.L);
        const float *u = ust + side * C * Cf::US + t * Cf::US + l * Dm.P;
        bf16 *F = (side == 0 ? f0 : f1) + t * Cf::FS + l * Dm.R;
        float pp[kMaxP], pm[kMaxP];
#pragma unroll
        for (int p = 0; p < kMaxP; ++p) {
            pp[p] = pm[p] = 1.f;
            if (p < Dm.P) {
                const float a = 2.f * Dm.beta * u[p];
                pp[p] = 1.f / (1.f + expf(-a));
                pm[p] = 1.f / (1.f + expf(a));
            }
        }
        const bool live = t < cnt;
        const bool scaled = side == 0 && f0s != nullptr;
        const float sc = scaled && live ? scale0[t] : 0.f;
        bf16 *Fs = scaled ? f0s + t * Cf::FS + l * Dm.R : nullptr;
        for (int r = 0; r < Dm.R; ++r) {
            float prod = 1.f;
#pragma unroll
            for (int p = 0; p < kMaxP; ++p)
                if (p < Dm.P) prod *= ((r >> p) & 1) ? pp[p] : pm[p];
            F[r] = __float2bfloat16_rn(live ? prod : 0.f);
            if (scaled) Fs[r] = __float2bfloat16_rn(prod * sc);
        }
    }
}

// B fragment of the mass column: n = 0 holds ones, other columns zero.
__device__ __forceinline__ void mass_fragment(int lane, uint32_t &b0, uint32_t &b1)
{
    const uint32_t one2 = 0x3F803F80u;  // two bf16 ones
    b0 = b1 = (lane >> 2) == 0 ? one2 : 0u;
}

// Chain rule back through the featuriser for the tokens of one tile, in float32.  u comes from
// ust ([C][US], tanh projections), dphi from dphi_s ([C][DPS], fp32).  phi is recomputed from u.
// Writes dz = beta * (sum_r phi_r (dphi_r - phi . dphi) v_{r,p}) * (1 - u_p^2) as bf16 into
// dz_s[t][l * P + p] (row stride ZS).
template <int US, int DPS, int ZS>
__device__ __forceinline__ void featurise_backward_tiles(const Dims &Dm, const float *ust, const float *dphi_s,
                                                         bf16 *dz_s)
{
    const int total = Dm.L * C;
    for (int it = threadIdx.x; it < total; it += NTH) {
        const int t = it % C, l = it / C;
        const float *u = ust + t * US + l * Dm.P;
        const float *dph = dphi_s + t * DPS + l * Dm.R;
        float pp[kMaxP], pm[kMaxP];
#pragma unroll
        for (int p = 0; p < kMaxP; ++p) {
            pp[p] = pm[p] = 1.f;
            if (p < Dm.P) {
                const float a = 2.f * Dm.beta * u[p];
                pp[p] = 1.f / (1.f + expf(-a));
                pm[p] = 1.f / (1.f + expf(a));
            }
        }
        float c = 0.f;
        for (int r = 0; r < Dm.R; ++r) {
            float prod = 1.f;
#pragma unroll
            for (int p = 0; p < kMaxP; ++p)
                if (p < Dm.P) prod *= ((r >> p) & 1) ? pp[p] : pm[p];
            c = fmaf(prod, dph[r], c);
        }
        float du[kMaxP];
#pragma unroll
        for (int p = 0; p < kMaxP; ++p) du[p] = 0.f;
        for (int r = 0; r < Dm.R; ++r) {
            float prod = 1.f;
#pragma unroll
            for (int p = 0; p < kMaxP; ++p)
                if (p < Dm.P) prod *= ((r >> p) & 1) ? pp[p] : pm[p];
            const float ds = prod * (dph[r] - c);
#pragma unroll
            for (int p = 0; p < kMaxP; ++p)
                if (p < Dm.P) du[p] += ((r >> p) & 1) ? ds : -ds;
        }
#pragma unroll
        for (int p = 0; p < kMaxP; ++p)
            if (p < Dm.P) dz_s[t * ZS + l * Dm.P + p] = __float2bfloat16_rn(Dm.beta * du[p] * (1.f - u[p] * u[p]));
    }
}

// dxhat for 16 rows (row block rb) and this warp's column half h: dxhat = dz (W_hi + W_lo), with
// dz [C][ZS] bf16 and W rows in wc ([2 LPP][XS]: hi rows then lo rows).  Returns the fragments
// acc[D/16][4] (n-tile i covers columns 8 (h D/16 + i) ..), and adds the row partials of
// x . dxhat over those columns into red[row] via shared-memory atomics-free quad reduction:
// the caller passes red_half = red + h * C.
template <int D, int LPP, int XS, int ZS>
__device__ __forceinline__ void back_project(const bf16 *dz_s, const bf16 *wc, const bf16 *xs, int rb, int h,
                                             int lane, float (&acc)[D / 16][4], float *red_half)
{
    constexpr int NC = D / 16;
    const int g = lane >> 2, q = lane & 3;
#pragma unroll
    for (int i = 0; i < NC; ++i)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[i][e] = 0.f;
    const int arow = 16 * rb + (lane & 7) + 8 * ((lane >> 3) & 1);
    const int vrow = (lane & 7) + 8 * ((lane >> 3) & 1);
#pragma unroll
    for (int kz = 0; kz < LPP / 16; ++kz) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4(smem_u32(dz_s + arow * ZS + 16 * kz + 8 * (lane >> 4)), a0, a1, a2, a3);
#pragma unroll
        for (int i = 0; i < NC; i += 2) {
            const int col = 8 * (h * NC + i) + 8 * (lane >> 4);
            uint32_t b0, b1, b2, b3;
            ldsm_x4_t(smem_u32(wc + (16 * kz + vrow) * XS + col), b0, b1, b2, b3);
            mma16816(acc[i], a0, a1, a2, a3, b0, b1);
            mma16816(acc[i + 1], a0, a1, a2, a3, b2, b3);
            ldsm_x4_t(smem_u32(wc + (LPP + 16 * kz + vrow) * XS + col), b0, b1, b2, b3);
            mma16816(acc[i], a0, a1, a2, a3, b0, b1);
            mma16816(acc[i + 1], a0, a1, a2, a3, b2, b3);
        }
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

// Finish the normalisation backward for the fragments of back_project and stage dx as bf16:
// dx = inv (dxhat - x inv^2 (x . dxhat)), x . dxhat = red[t] + red[C + t].
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

// Store 16 staged rows (row block rb), column half h, of a [C][XS] bf16 stage to global rows
// n0 + t (t < cnt) of a [N, D] slice.
template <int D, int XS>
__device__ __forceinline__ void store_rows(const bf16 *stage, bf16 *__restrict__ dst, int64_t n0, int cnt, int rb,
                                           int h, int lane)
{
    constexpr int CHR = D / 16;
    for (int i = lane; i < 16 * CHR; i += 32) {
        const int rr = i / CHR, cc = i - rr * CHR;
        const int t = 16 * rb + rr;
        if (t < cnt) {
            const int c = h * (D / 2) + 8 * cc;
            *reinterpret_cast<uint4 *>(dst + (n0 + t) * D + c) = *reinterpret_cast<const uint4 *>(stage + t * XS + c);
        }
    }
}

// Lower-triangular ones as an A fragment: element (row t, col j) = 1 if j <= t, for the 16x16
// block whose rows start at row0 and columns at col0.
__device__ __forceinline__ void tril_ones_fragment(int row0, int col0, int lane, uint32_t (&a)[4])
{
    const int g = lane >> 2, q = lane & 3;
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const int t = row0 + g + 8 * (r & 1);
        const int j = col0 + 2 * q + 8 * (r >> 1);
        a[r] = pack_bf16(j <= t ? 1.f : 0.f, j + 1 <= t ? 1.f : 0.f);
    }
}

}  // namespace tc
}  // namespace race
