// race_tc_causal.cu -- tensor-core (mma.sync bf16 -> fp32) causal RACE attention forward.
//
// Algorithm 2 of the paper ("RACE Attention" slides, frame "Causality is a prefix update of the
// same statistics"; reading notes section 2.6) evaluated in chunks of C = 64 tokens.  With
// F = [phi^(1) | ... | phi^(L)] the concatenated bucket features (L*R columns, zero padded to
// LRP) and S the running sketch [A | B] (LRP x (d + 8): d content columns, the mass column, zeros):
//
//   O_chunk = ((F_Q F_K^T) masked to j <= t) [V | 1]  +  F_Q S_prev,    O = num / den
//   S      += F_K^T [V | 1]
//
// Every product is a 16x8x16 bf16 tensor-core tile with fp32 accumulation.  S is kept as fp32
// fragments in registers across chunks (warp w owns n-tiles w, w + 8, ...); the read-out uses a
// double-buffered bf16 hi + lo copy (about 16 mantissa bits).  Bucket features are recomputed:
// z = X (W_hi + W_lo)^T on tensor cores, u = tanh(z / |x|), phi by products of sigmoids on CUDA
// cores (the product form of the softmax over hypercube corners, reading notes section 2.4).
//
// One CTA (8 warps) walks one segment of a (batch, head) sequence; its starting sketch comes
// from a first pass (TOTALS: per-segment sums of F_K^T [V | 1]) and an exclusive scan over
// segments.  Token tiles arrive by bulk (TMA) row copies into double buffers, completing on
// mbarriers.  Per chunk: warp (rb, h) projects and featurises rows 16 rb .. of Q (h = 0) or K
// (h = 1); after one CTA barrier it computes outputs for rows 16 rb .., column half h, and
// updates the state n-tiles it owns.
#include "race_common.cuh"
#include "race_launch.h"
#include "race_tc_common.cuh"

namespace race {
namespace tc {

template <int D, int P, int LRP>
struct FwdCfg {
    static constexpr int R = 1 << P;
    static constexpr int XS = D + 8;        // row stride (elements) of token tiles and W
    static constexpr int FS = LRP + 8;      // row stride of feature tiles
    static constexpr int SS = D + 8;        // row stride of the bf16 state copies (d, mass, 7 zeros)
    static constexpr int US = LPP + 1;      // row stride of the per-warp tanh stage (fp32)
    static constexpr int NTO = D / 8 + 1;   // state n-tiles including the mass tile
    static constexpr int NC = D / 16;       // content n-tiles per column half
    static constexpr int KF = LRP / 16;     // k-steps over features
    static constexpr int MT = LRP / 16;     // state m-tiles
    static constexpr int SNT = (NTO + 7) / 8;
    static constexpr int X_BYTES = C * XS * 2;
    static constexpr int S_BYTES = LRP * SS * 2;
    static constexpr int OFF_X = 0;                              // [buf][tile q, k, v]
    static constexpr int OFF_FQ = OFF_X + 6 * X_BYTES;
    static constexpr int OFF_FK = OFF_FQ + C * FS * 2;
    static constexpr int OFF_S = OFF_FK + C * FS * 2;            // [buf][hi, lo]
    static constexpr int OFF_W = OFF_S + 4 * S_BYTES;
    static constexpr int OFF_U = OFF_W + 2 * LPP * XS * 2;        // [warp][16][US]
    static constexpr int OFF_BAR = OFF_U + 8 * 16 * US * 4;
    static constexpr int BYTES = OFF_BAR + 16;
};

template <int D, int P, int LRP, bool TOTALS>
__global__ void __launch_bounds__(NTH, 1)
    k_causal_tc(Dims Dm, const bf16 *__restrict__ Q, const bf16 *__restrict__ K, const bf16 *__restrict__ V,
                const float *__restrict__ W, const float *__restrict__ S0, int64_t seg_len, int nseg,
                bf16 *__restrict__ O, float *__restrict__ Sout, unsigned *__restrict__ err)
{
    using Cf = FwdCfg<D, P, LRP>;
    extern __shared__ __align__(128) unsigned char smem[];
    auto xt = [&](int buf, int tile) { return reinterpret_cast<bf16 *>(smem + Cf::OFF_X + (3 * buf + tile) * Cf::X_BYTES); };
    bf16 *fq = reinterpret_cast<bf16 *>(smem + Cf::OFF_FQ);
    bf16 *fk = reinterpret_cast<bf16 *>(smem + Cf::OFF_FK);
    auto sh = [&](int buf, int lohi) { return reinterpret_cast<bf16 *>(smem + Cf::OFF_S + (2 * buf + lohi) * Cf::S_BYTES); };
    bf16 *wc = reinterpret_cast<bf16 *>(smem + Cf::OFF_W);
    const uint32_t bar0 = smem_u32(smem + Cf::OFF_BAR);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, q = lane & 3;
    const int rb = warp & 3, h = warp >> 2;
    float *ust = reinterpret_cast<float *>(smem + Cf::OFF_U) + warp * 16 * Cf::US;
    const int s = blockIdx.x;
    const int64_t bh = blockIdx.y;
    const int64_t off = bh * Dm.N * D;
    const int64_t n_begin = (int64_t)s * seg_len;
    const int64_t n_end = min(Dm.N, n_begin + seg_len);
    const int ntiles = TOTALS ? 2 : 3;  // tiles per chunk: (q,) k, v
    // tiles per chunk in slot order: fwd (q, k, v), totals (k, v)
    const bf16 *src0 = TOTALS ? K + off : Q + off, *src1 = TOTALS ? V + off : K + off, *src2 = V + off;
    const int t_first = TOTALS ? 1 : 0;  // first tile slot used

    // ---- set-up: zero tiles (stale rows past the sequence end stay finite), W split, state
    zero_smem(smem, Cf::OFF_W);
    __syncthreads();
    load_w_split<D, Cf::XS>(head_w(W, Dm, bh), Dm.LP, wc);
    float st[Cf::SNT][Cf::MT][4];
    const float *S0b = TOTALS ? nullptr : S0 + ((int64_t)bh * nseg + s) * Dm.LR * (D + 1);
#pragma unroll
    for (int j = 0; j < Cf::SNT; ++j) {
        const int nt = warp + 8 * j;
#pragma unroll
        for (int mt = 0; mt < Cf::MT; ++mt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int lr = 16 * mt + g + 8 * (e >> 1), c = 8 * nt + 2 * q + (e & 1);
                st[j][mt][e] = (!TOTALS && nt < Cf::NTO && lr < Dm.LR && c <= D) ? S0b[lr * (D + 1) + c] : 0.f;
            }
    }
    if (!TOTALS) {
        for (int i = tid; i < LRP * (D + 8); i += NTH) {
            const int lr = i / (D + 8), c = i - lr * (D + 8);
            const float v = (lr < Dm.LR && c <= D) ? S0b[lr * (D + 1) + c] : 0.f;
            bf16 hi, lo;
            split_bf16(v, hi, lo);
            sh(0, 0)[lr * Cf::SS + c] = hi;
            sh(0, 1)[lr * Cf::SS + c] = lo;
        }
    }
    if (tid == 0) {
        mbar_init(bar0, 1);
        mbar_init(bar0 + 8, 1);
        fence_mbar_init();
    }
    fence_proxy_async();
    __syncthreads();
    if (n_begin < n_end) {
        const int cnt0 = (int)min((int64_t)C, n_end - n_begin);
        if (tid == 0) mbar_arrive_expect_tx(bar0, ntiles * cnt0 * D * 2);
        __syncthreads();
        issue_rows<D, Cf::XS>(xt(0, t_first), xt(0, t_first + 1), xt(0, 2), nullptr, src0, src1, src2, nullptr,
                              ntiles, n_begin, cnt0, bar0);
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
        if (tid == 0 && cnt1 > 0) mbar_arrive_expect_tx(bar0 + 8 * (buf ^ 1), ntiles * cnt1 * D * 2);
        if (__syncthreads_or(!landed)) {  // a copy never arrived: report, give it one more bounded wait, stop
            if (tid == 0) atomicOr(err, kErrWaitTimeout);
            mbar_wait(bar0 + 8 * buf, phase[buf] ^ 1u);
            return;
        }
        if (cnt1 > 0) {
            issue_rows<D, Cf::XS>(xt(buf ^ 1, t_first), xt(buf ^ 1, t_first + 1), xt(buf ^ 1, 2), nullptr, src0, src1,
                                  src2, nullptr, ntiles, n1, cnt1, bar0 + 8 * (buf ^ 1));
        }
        bf16 *xqb = xt(buf, 0), *xkb = xt(buf, 1), *xvb = xt(buf, 2);

        // P1: projection and features of rows 16 rb .. of Q (h = 0) or K (h = 1)
        if (!TOTALS || h == 1) {
            float u[LPP / 8][4], inv0, inv1;
            project16<D, Cf::XS>((h ? xkb : xqb) + 16 * rb * Cf::XS, wc, lane, u, inv0, inv1);
            stage_u<Cf::US>(u, ust, lane);
            __syncwarp();
            features16<P, Cf::US, Cf::FS>(ust, Dm.L, Dm.beta, 16 * rb, cnt, (h ? fk : fq) + 16 * rb * Cf::FS, lane);
        }
        __syncthreads();

        const int cur = buf;  // state copy holding S before this chunk
        if (!TOTALS) {
            // P2a: outputs of rows 16 rb .. 16 rb + 15, column half h
            const uint32_t qbase =
                smem_u32(fq + (16 * rb + (lane & 7) + 8 * ((lane >> 3) & 1)) * Cf::FS + 8 * (lane >> 4));
            uint32_t aq[Cf::KF][4];
#pragma unroll
            for (int kf = 0; kf < Cf::KF; ++kf) ldsm_x4(qbase + 32 * kf, aq[kf][0], aq[kf][1], aq[kf][2], aq[kf][3]);
            uint32_t sa[4][4];
            {
                const uint32_t kbase = smem_u32(fk + (lane & 7) * Cf::FS + 8 * ((lane >> 3) & 1));
                float sc[8][4];
#pragma unroll
                for (int jt = 0; jt < 8; ++jt) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) sc[jt][e] = 0.f;
                    if (jt <= 2 * rb + 1) {
#pragma unroll
                        for (int kf = 0; kf < Cf::KF; ++kf) {
                            uint32_t b0, b1;
                            ldsm_x2(kbase + 2 * (8 * jt * Cf::FS + 16 * kf), b0, b1);
                            mma16816(sc[jt], aq[kf][0], aq[kf][1], aq[kf][2], aq[kf][3], b0, b1);
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
            constexpr int NC = Cf::NC;
            float oc[NC + 1][4];
#pragma unroll
            for (int i = 0; i <= NC; ++i)
#pragma unroll
                for (int e = 0; e < 4; ++e) oc[i][e] = 0.f;
            const int vrow = (lane & 7) + 8 * ((lane >> 3) & 1);
            const uint32_t vbase = smem_u32(xvb + vrow * Cf::XS + 8 * h * NC + 8 * (lane >> 4));
            uint32_t m0, m1;
            mass_fragment(lane, m0, m1);
#pragma unroll
            for (int kb = 0; kb < 4; ++kb) {
                if (kb <= rb) {
#pragma unroll
                    for (int i = 0; i < NC; i += 2) {
                        uint32_t b0, b1, b2, b3;
                        ldsm_x4_t(vbase + 2 * (16 * kb * Cf::XS + 8 * i), b0, b1, b2, b3);
                        mma16816(oc[i], sa[kb][0], sa[kb][1], sa[kb][2], sa[kb][3], b0, b1);
                        mma16816(oc[i + 1], sa[kb][0], sa[kb][1], sa[kb][2], sa[kb][3], b2, b3);
                    }
                    mma16816(oc[NC], sa[kb][0], sa[kb][1], sa[kb][2], sa[kb][3], m0, m1);
                }
            }
            const uint32_t hbase = smem_u32(sh(cur, 0) + vrow * Cf::SS + 8 * h * NC + 8 * (lane >> 4));
            const uint32_t lbase = smem_u32(sh(cur, 1) + vrow * Cf::SS + 8 * h * NC + 8 * (lane >> 4));
            const uint32_t hmass = smem_u32(sh(cur, 0) + vrow * Cf::SS + D);
            const uint32_t lmass = smem_u32(sh(cur, 1) + vrow * Cf::SS + D);
#pragma unroll
            for (int kf = 0; kf < Cf::KF; ++kf) {
#pragma unroll
                for (int i = 0; i < NC; i += 2) {
                    const uint32_t o = 2 * (16 * kf * Cf::SS + 8 * i);
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4_t(hbase + o, b0, b1, b2, b3);
                    mma16816(oc[i], aq[kf][0], aq[kf][1], aq[kf][2], aq[kf][3], b0, b1);
                    mma16816(oc[i + 1], aq[kf][0], aq[kf][1], aq[kf][2], aq[kf][3], b2, b3);
                    ldsm_x4_t(lbase + o, b0, b1, b2, b3);
                    mma16816(oc[i], aq[kf][0], aq[kf][1], aq[kf][2], aq[kf][3], b0, b1);
                    mma16816(oc[i + 1], aq[kf][0], aq[kf][1], aq[kf][2], aq[kf][3], b2, b3);
                }
                uint32_t b0, b1;
                ldsm_x2_t(hmass + 32 * kf * Cf::SS, b0, b1);
                mma16816(oc[NC], aq[kf][0], aq[kf][1], aq[kf][2], aq[kf][3], b0, b1);
                ldsm_x2_t(lmass + 32 * kf * Cf::SS, b0, b1);
                mma16816(oc[NC], aq[kf][0], aq[kf][1], aq[kf][2], aq[kf][3], b0, b1);
            }
            // O = num / den, staged as bf16 in the consumed Q tile, then stored row by row
            const float r0 = __frcp_rn(__shfl_sync(0xffffffffu, oc[NC][0], lane & ~3));
            const float r1 = __frcp_rn(__shfl_sync(0xffffffffu, oc[NC][2], lane & ~3));
            const int t0 = 16 * rb + g;
#pragma unroll
            for (int i = 0; i < NC; ++i) {
                const int c = 8 * (h * NC + i) + 2 * q;
                *reinterpret_cast<uint32_t *>(xqb + t0 * Cf::XS + c) = pack_bf16(oc[i][0] * r0, oc[i][1] * r0);
                *reinterpret_cast<uint32_t *>(xqb + (t0 + 8) * Cf::XS + c) = pack_bf16(oc[i][2] * r1, oc[i][3] * r1);
            }
            __syncwarp();
            constexpr int CHR = D / 16;  // 16-byte chunks per half row
#pragma unroll
            for (int i = lane; i < 16 * CHR; i += 32) {
                const int rr = i / CHR, cc = i - rr * CHR;
                const int t = 16 * rb + rr;
                if (t < cnt) {
                    const int c = h * (D / 2) + 8 * cc;
                    *reinterpret_cast<uint4 *>(O + off + (n0 + t) * D + c) =
                        *reinterpret_cast<const uint4 *>(xqb + t * Cf::XS + c);
                }
            }
        }

        // P2b: S += F_K^T [V | 1] on the owned n-tiles; refresh their bf16 copy for the next chunk
        {
            const uint32_t fkbase = smem_u32(fk + ((lane & 7) + 8 * (lane >> 4)) * Cf::FS + 8 * ((lane >> 3) & 1));
            const uint32_t vb = smem_u32(xvb + ((lane & 7) + 8 * ((lane >> 3) & 1)) * Cf::XS);
#pragma unroll
            for (int kb = 0; kb < 4; ++kb) {
                uint32_t af[Cf::MT][4];
#pragma unroll
                for (int mt = 0; mt < Cf::MT; ++mt)
                    ldsm_x4_t(fkbase + 2 * (16 * kb * Cf::FS + 16 * mt), af[mt][0], af[mt][1], af[mt][2], af[mt][3]);
#pragma unroll
                for (int j = 0; j < Cf::SNT; ++j) {
                    const int nt = warp + 8 * j;
                    if (nt < Cf::NTO) {
                        uint32_t b0, b1;
                        if (nt < D / 8)
                            ldsm_x2_t(vb + 2 * (16 * kb * Cf::XS + 8 * nt), b0, b1);
                        else
                            mass_fragment(lane, b0, b1);
#pragma unroll
                        for (int mt = 0; mt < Cf::MT; ++mt)
                            mma16816(st[j][mt], af[mt][0], af[mt][1], af[mt][2], af[mt][3], b0, b1);
                    }
                }
            }
            if (!TOTALS) {
                bf16 *nhi = sh(cur ^ 1, 0), *nlo = sh(cur ^ 1, 1);
#pragma unroll
                for (int j = 0; j < Cf::SNT; ++j) {
                    const int nt = warp + 8 * j;
                    if (nt < Cf::NTO) {
#pragma unroll
                        for (int mt = 0; mt < Cf::MT; ++mt)
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
                                *reinterpret_cast<__nv_bfloat162 *>(nhi + lr * Cf::SS + c) = hh;
                                *reinterpret_cast<__nv_bfloat162 *>(nlo + lr * Cf::SS + c) = ll;
                            }
                    }
                }
            }
        }
    }

    if (TOTALS) {
        float *out = Sout + ((int64_t)bh * nseg + s) * Dm.LR * (D + 1);
#pragma unroll
        for (int j = 0; j < Cf::SNT; ++j) {
            const int nt = warp + 8 * j;
            if (nt < Cf::NTO) {
#pragma unroll
                for (int mt = 0; mt < Cf::MT; ++mt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int lr = 16 * mt + g + 8 * (e >> 1), c = 8 * nt + 2 * q + (e & 1);
                        if (lr < Dm.LR && c <= D) out[lr * (D + 1) + c] = st[j][mt][e];
                    }
            }
        }
    }
}

}  // namespace tc

// ------------------------------------------------------------------ host side

namespace {

template <int D, int P, int LRP, bool TOTALS>
cudaError_t launch_causal_tc_inst(const Dims &Dm, const bf16_t *Q, const bf16_t *K, const bf16_t *V, const float *W,
                                  const float *S0, int64_t seg_len, int nseg, bf16_t *O, float *Sout, unsigned *err,
                                  cudaStream_t st)
{
    using Cf = tc::FwdCfg<D, P, LRP>;
    auto kern = tc::k_causal_tc<D, P, LRP, TOTALS>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cf::BYTES);
    if (e != cudaSuccess) return e;
    dim3 grid(nseg, (unsigned)Dm.BH);
    return launch_kernel(TOTALS ? "tc_causal_totals" : "tc_causal_fwd", kern, grid, dim3(tc::NTH), (size_t)Cf::BYTES,
                         st, Dm, Q, K, V, W, S0, seg_len, nseg, O, Sout, err);
}

template <bool TOTALS>
cudaError_t dispatch_causal_tc(const Dims &Dm, const bf16_t *Q, const bf16_t *K, const bf16_t *V, const float *W,
                               const float *S0, int64_t seg_len, int nseg, bf16_t *O, float *Sout, unsigned *err,
                               cudaStream_t st)
{
#define RACE_TC_CASE(DD, PP, LRPP)                                                                            \
    if (Dm.d == DD && Dm.P == PP && Dm.LR <= LRPP)                                                            \
        return launch_causal_tc_inst<DD, PP, LRPP, TOTALS>(Dm, Q, K, V, W, S0, seg_len, nseg, O, Sout, err, st);
    RACE_TC_CASE(128, 2, 32)
    RACE_TC_CASE(128, 2, 64)
    RACE_TC_CASE(128, 3, 32)
    RACE_TC_CASE(128, 3, 64)
    RACE_TC_CASE(128, 4, 32)
    RACE_TC_CASE(128, 4, 64)
    RACE_TC_CASE(64, 2, 32)
    RACE_TC_CASE(64, 2, 64)
    RACE_TC_CASE(64, 3, 32)
    RACE_TC_CASE(64, 3, 64)
    RACE_TC_CASE(64, 4, 32)
    RACE_TC_CASE(64, 4, 64)
#undef RACE_TC_CASE
    return cudaErrorInvalidValue;
}

}  // namespace

bool causal_tc_supported(const Dims &Dm)
{
    return (Dm.d == 64 || Dm.d == 128) && Dm.P >= 2 && Dm.P <= 4 && Dm.LR <= 64 && Dm.LP <= tc::LPP;
}

int causal_tc_chunk() { return tc::C; }

cudaError_t launch_causal_tc_totals(const Dims &Dm, const bf16_t *K, const bf16_t *V, const float *W,
                                    int64_t seg_len, int nseg, float *Sout, unsigned *err, cudaStream_t st)
{
    return dispatch_causal_tc<true>(Dm, K, K, V, W, nullptr, seg_len, nseg, nullptr, Sout, err, st);
}

cudaError_t launch_causal_tc_fwd(const Dims &Dm, const bf16_t *Q, const bf16_t *K, const bf16_t *V, const float *W,
                                 const float *S0, int64_t seg_len, int nseg, bf16_t *O, unsigned *err,
                                 cudaStream_t st)
{
    return dispatch_causal_tc<false>(Dm, Q, K, V, W, S0, seg_len, nseg, O, nullptr, err, st);
}

}  // namespace race
