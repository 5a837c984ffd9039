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
// The chunk sizes are chosen so every product is a 16x8x16 bf16 tensor-core tile.  S is kept as
// fp32 accumulators in registers across chunks (each warp owns a column block); the read-out
// uses its bf16 hi + lo split (about 16 mantissa bits).  Bucket features are recomputed from
// the projections: z = X (W_hi + W_lo)^T on tensor cores (X bf16 exact, W split in two bf16
// parts), u = tanh(z / |x|), phi_r = prod_t sigmoid(2 beta u_t v_{r,t}) on CUDA cores.
//
// One CTA (8 warps) walks one segment of a (batch, head) sequence; the segment's starting sketch
// comes from a first pass (TOTALS = true: per-segment sums of F_K^T [V | 1]) and an exclusive
// scan over segments.  Tiles are double buffered with cp.async.
#include "race_common.cuh"
#include "race_launch.h"
#include "race_mma.cuh"
#include "race_tc_common.cuh"

namespace race {
namespace tc {

using bf16 = __nv_bfloat16;
using namespace race::mma;


template <int D, int LRP, int LPP, bool TOTALS>
__global__ void __launch_bounds__(NTH, 1)
    k_causal_tc(Dims Dm, const bf16 *__restrict__ Q, const bf16 *__restrict__ K, const bf16 *__restrict__ V,
                const float *__restrict__ W, const float *__restrict__ S0, int64_t seg_len, int nseg,
                bf16 *__restrict__ O, float *__restrict__ Sout)
{
    using Cf = CausalCfg<D, LRP, LPP>;
    extern __shared__ __align__(128) unsigned char smem[];
    bf16 *xq = reinterpret_cast<bf16 *>(smem + Cf::OFF_XQ);
    bf16 *xk = reinterpret_cast<bf16 *>(smem + Cf::OFF_XK);
    bf16 *xv = reinterpret_cast<bf16 *>(smem + Cf::OFF_XV);
    bf16 *fq = reinterpret_cast<bf16 *>(smem + Cf::OFF_FQ);
    bf16 *fk = reinterpret_cast<bf16 *>(smem + Cf::OFF_FK);
    bf16 *shi = reinterpret_cast<bf16 *>(smem + Cf::OFF_SHI);
    bf16 *slo = reinterpret_cast<bf16 *>(smem + Cf::OFF_SLO);
    bf16 *wc = reinterpret_cast<bf16 *>(smem + Cf::OFF_W);
    float *ust = reinterpret_cast<float *>(smem + Cf::OFF_U);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, q = lane & 3;
    const int rb = warp & 3, h = warp >> 2;
    const int s = blockIdx.x;
    const int64_t bh = blockIdx.y;
    const int64_t off = bh * Dm.N * D;
    const int64_t n_begin = (int64_t)s * seg_len;
    const int64_t n_end = min(Dm.N, n_begin + seg_len);

    // hyperplanes as bf16 hi / lo rows; zero feature padding
    for (int i = tid; i < LPP * D; i += NTH) {
        const int row = i / D, k = i - row * D;
        const float w = row < Dm.LP ? W[row * D + k] : 0.f;
        bf16 hi, lo;
        split_bf16(w, hi, lo);
        wc[row * Cf::XS + k] = hi;
        wc[(LPP + row) * Cf::XS + k] = lo;
    }
    for (int i = tid; i < C * LRP; i += NTH) {
        const int t = i / LRP, c = i - t * LRP;
        if (c >= Dm.LR) {
            fq[t * Cf::FS + c] = __float2bfloat16_rn(0.f);
            fk[t * Cf::FS + c] = __float2bfloat16_rn(0.f);
        }
    }

    // running sketch: fp32 fragments of the n-tiles this warp owns, plus the bf16 hi/lo copy
    float st[Cf::SNT][Cf::MT][4];
#pragma unroll
    for (int j = 0; j < Cf::SNT; ++j) {
        const int nt = warp + 8 * j;
#pragma unroll
        for (int mt = 0; mt < Cf::MT; ++mt) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int lr = 16 * mt + g + 8 * (e >> 1), c = 8 * nt + 2 * q + (e & 1);
                float v = 0.f;
                if (!TOTALS && nt < Cf::NTO && lr < Dm.LR && c <= D)
                    v = S0[(((int64_t)bh * nseg + s) * Dm.LR + lr) * (D + 1) + c];
                st[j][mt][e] = v;
            }
        }
    }
    if (!TOTALS) {
        for (int i = tid; i < LRP * (D + 8); i += NTH) {
            const int lr = i / (D + 8), c = i - lr * (D + 8);
            float v = 0.f;
            if (lr < Dm.LR && c <= D) v = S0[(((int64_t)bh * nseg + s) * Dm.LR + lr) * (D + 1) + c];
            bf16 hi, lo;
            split_bf16(v, hi, lo);
            shi[lr * Cf::SS + c] = hi;
            slo[lr * Cf::SS + c] = lo;
        }
    }

    if (n_begin < n_end) {
        const int cnt0 = (int)min((int64_t)C, n_end - n_begin);
        if (!TOTALS) load_tile_async<D, Cf::XS>(xq, Q + off, n_begin, cnt0);
        load_tile_async<D, Cf::XS>(xk, K + off, n_begin, cnt0);
        load_tile_async<D, Cf::XS>(xv, V + off, n_begin, cnt0);
    }
    cp_async_commit();

    int buf = 0;
    for (int64_t n0 = n_begin; n0 < n_end; n0 += C, buf ^= 1) {
        const int cnt = (int)min((int64_t)C, n_end - n0);
        cp_async_wait<0>();
        __syncthreads();
        // prefetch the next chunk into the other buffer
        {
            const int64_t n1 = n0 + C;
            if (n1 < n_end) {
                const int cnt1 = (int)min((int64_t)C, n_end - n1);
                if (!TOTALS) load_tile_async<D, Cf::XS>(xq + (buf ^ 1) * C * Cf::XS, Q + off, n1, cnt1);
                load_tile_async<D, Cf::XS>(xk + (buf ^ 1) * C * Cf::XS, K + off, n1, cnt1);
                load_tile_async<D, Cf::XS>(xv + (buf ^ 1) * C * Cf::XS, V + off, n1, cnt1);
            }
            cp_async_commit();
        }
        const bf16 *xqb = xq + buf * C * Cf::XS;
        const bf16 *xkb = xk + buf * C * Cf::XS;
        const bf16 *xvb = xv + buf * C * Cf::XS;

        // 1. projections -> tanh, staged per side
        if (!TOTALS) project_rows<D, LRP, LPP>(xqb, wc, ust, rb, h, lane);
        project_rows<D, LRP, LPP>(xkb, wc, ust + C * Cf::US, rb, h, lane);
        __syncthreads();
        // 2. bucket features
        if (TOTALS)
            featurise_tiles<D, LRP, LPP>(Dm, ust + C * Cf::US, fk, fk, 1, cnt);
        else
            featurise_tiles<D, LRP, LPP>(Dm, ust, fq, fk, 2, cnt);
        __syncthreads();

        if (!TOTALS) {
            // 3. outputs of rows 16 rb .. 16 rb + 15, column half h
            uint32_t aq[Cf::KF][4];
            const int arow = 16 * rb + (lane & 7) + 8 * ((lane >> 3) & 1);
#pragma unroll
            for (int kf = 0; kf < Cf::KF; ++kf)
                ldsm_x4(smem_u32(fq + arow * Cf::FS + 16 * kf + 8 * (lane >> 4)), aq[kf][0], aq[kf][1], aq[kf][2],
                        aq[kf][3]);
            float sc[8][4];
#pragma unroll
            for (int jt = 0; jt < 8; ++jt) {
#pragma unroll
                for (int e = 0; e < 4; ++e) sc[jt][e] = 0.f;
                if (jt <= 2 * rb + 1) {
#pragma unroll
                    for (int kf = 0; kf < Cf::KF; ++kf) {
                        uint32_t b0, b1;
                        ldsm_x2(smem_u32(fk + (8 * jt + (lane & 7)) * Cf::FS + 16 * kf + 8 * ((lane >> 3) & 1)), b0,
                                b1);
                        mma16816(sc[jt], aq[kf][0], aq[kf][1], aq[kf][2], aq[kf][3], b0, b1);
                    }
                    if (jt >= 2 * rb) {  // diagonal block: keep keys j <= query t
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int j = 8 * jt + 2 * q + (e & 1);
                            const int t = 16 * rb + g + 8 * (e >> 1);
                            if (j > t) sc[jt][e] = 0.f;
                        }
                    }
                }
            }
            uint32_t sa[4][4];
#pragma unroll
            for (int kb = 0; kb < 4; ++kb) {
                sa[kb][0] = pack_bf16(sc[2 * kb][0], sc[2 * kb][1]);
                sa[kb][1] = pack_bf16(sc[2 * kb][2], sc[2 * kb][3]);
                sa[kb][2] = pack_bf16(sc[2 * kb + 1][0], sc[2 * kb + 1][1]);
                sa[kb][3] = pack_bf16(sc[2 * kb + 1][2], sc[2 * kb + 1][3]);
            }
            constexpr int NC = D / 16;  // content n-tiles per column half
            float oc[NC + 1][4];
#pragma unroll
            for (int i = 0; i <= NC; ++i)
#pragma unroll
                for (int e = 0; e < 4; ++e) oc[i][e] = 0.f;
            const int vrow = (lane & 7) + 8 * ((lane >> 3) & 1);
            // intra-chunk: (masked scores) x [V | 1]
#pragma unroll
            for (int kb = 0; kb < 4; ++kb) {
                if (kb <= rb) {
#pragma unroll
                    for (int i = 0; i < NC; i += 2) {
                        const int nt = h * NC + i;
                        uint32_t b0, b1, b2, b3;
                        ldsm_x4_t(smem_u32(xvb + (16 * kb + vrow) * Cf::XS + 8 * nt + 8 * (lane >> 4)), b0, b1, b2, b3);
                        mma16816(oc[i], sa[kb][0], sa[kb][1], sa[kb][2], sa[kb][3], b0, b1);
                        mma16816(oc[i + 1], sa[kb][0], sa[kb][1], sa[kb][2], sa[kb][3], b2, b3);
                    }
                    uint32_t m0, m1;
                    mass_fragment(lane, m0, m1);
                    mma16816(oc[NC], sa[kb][0], sa[kb][1], sa[kb][2], sa[kb][3], m0, m1);
                }
            }
            // inter-chunk: F_Q x (S_hi + S_lo)
#pragma unroll
            for (int kf = 0; kf < Cf::KF; ++kf) {
#pragma unroll
                for (int i = 0; i < NC; i += 2) {
                    const int nt = h * NC + i;
                    const int addr = (16 * kf + vrow) * Cf::SS + 8 * nt + 8 * (lane >> 4);
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4_t(smem_u32(shi + addr), b0, b1, b2, b3);
                    mma16816(oc[i], aq[kf][0], aq[kf][1], aq[kf][2], aq[kf][3], b0, b1);
                    mma16816(oc[i + 1], aq[kf][0], aq[kf][1], aq[kf][2], aq[kf][3], b2, b3);
                    ldsm_x4_t(smem_u32(slo + addr), b0, b1, b2, b3);
                    mma16816(oc[i], aq[kf][0], aq[kf][1], aq[kf][2], aq[kf][3], b0, b1);
                    mma16816(oc[i + 1], aq[kf][0], aq[kf][1], aq[kf][2], aq[kf][3], b2, b3);
                }
                const int maddr = (16 * kf + vrow) * Cf::SS + D;
                uint32_t b0, b1;
                ldsm_x2_t(smem_u32(shi + maddr), b0, b1);
                mma16816(oc[NC], aq[kf][0], aq[kf][1], aq[kf][2], aq[kf][3], b0, b1);
                ldsm_x2_t(smem_u32(slo + maddr), b0, b1);
                mma16816(oc[NC], aq[kf][0], aq[kf][1], aq[kf][2], aq[kf][3], b0, b1);
            }
            // O = num / den, staged as bf16 in the consumed Q tile, then stored row by row
            const float den0 = __shfl_sync(0xffffffffu, oc[NC][0], lane & ~3);
            const float den1 = __shfl_sync(0xffffffffu, oc[NC][2], lane & ~3);
            const float r0 = 1.f / den0, r1 = 1.f / den1;
            bf16 *ost = const_cast<bf16 *>(xqb);
            const int t0 = 16 * rb + g;
#pragma unroll
            for (int i = 0; i < NC; ++i) {
                const int c = 8 * (h * NC + i) + 2 * q;
                *reinterpret_cast<uint32_t *>(ost + t0 * Cf::XS + c) = pack_bf16(oc[i][0] * r0, oc[i][1] * r0);
                *reinterpret_cast<uint32_t *>(ost + (t0 + 8) * Cf::XS + c) = pack_bf16(oc[i][2] * r1, oc[i][3] * r1);
            }
            __syncwarp();
            constexpr int CHR = D / 16;  // 16-byte chunks per half row
            for (int i = lane; i < 16 * CHR; i += 32) {
                const int rr = i / CHR, cc = i - rr * CHR;
                const int t = 16 * rb + rr;
                if (t < cnt) {
                    const int c = h * (D / 2) + 8 * cc;
                    *reinterpret_cast<uint4 *>(O + off + (n0 + t) * D + c) =
                        *reinterpret_cast<const uint4 *>(ost + t * Cf::XS + c);
                }
            }
            __syncthreads();  // every warp has read S_hi / S_lo of this chunk
        }

        // 4. S += F_K^T [V | 1] on the n-tiles this warp owns
#pragma unroll
        for (int kb = 0; kb < 4; ++kb) {
            uint32_t af[Cf::MT][4];
#pragma unroll
            for (int mt = 0; mt < Cf::MT; ++mt) {
                const int k = 16 * kb + (lane & 7) + 8 * (lane >> 4);
                const int m = 16 * mt + 8 * ((lane >> 3) & 1);
                ldsm_x4_t(smem_u32(fk + k * Cf::FS + m), af[mt][0], af[mt][1], af[mt][2], af[mt][3]);
            }
#pragma unroll
            for (int j = 0; j < Cf::SNT; ++j) {
                const int nt = warp + 8 * j;
                if (nt < Cf::NTO) {
                    uint32_t b0, b1;
                    if (nt < D / 8)
                        ldsm_x2_t(smem_u32(xvb + (16 * kb + (lane & 7) + 8 * ((lane >> 3) & 1)) * Cf::XS + 8 * nt), b0,
                                  b1);
                    else
                        mass_fragment(lane, b0, b1);
#pragma unroll
                    for (int mt = 0; mt < Cf::MT; ++mt)
                        mma16816(st[j][mt], af[mt][0], af[mt][1], af[mt][2], af[mt][3], b0, b1);
                }
            }
        }
        if (!TOTALS) {
#pragma unroll
            for (int j = 0; j < Cf::SNT; ++j) {
                const int nt = warp + 8 * j;
                if (nt < Cf::NTO) {
#pragma unroll
                    for (int mt = 0; mt < Cf::MT; ++mt) {
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
                            *reinterpret_cast<__nv_bfloat162 *>(shi + lr * Cf::SS + c) = hh;
                            *reinterpret_cast<__nv_bfloat162 *>(slo + lr * Cf::SS + c) = ll;
                        }
                    }
                }
            }
        }
        __syncthreads();
    }
    cp_async_wait<0>();

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

template <int D, int LRP, int LPP, bool TOTALS>
cudaError_t launch_causal_tc_inst(const Dims &Dm, const bf16_t *Q, const bf16_t *K, const bf16_t *V, const float *W,
                                  const float *S0, int64_t seg_len, int nseg, bf16_t *O, float *Sout, cudaStream_t st)
{
    using Cf = tc::CausalCfg<D, LRP, LPP>;
    auto kern = tc::k_causal_tc<D, LRP, LPP, TOTALS>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cf::BYTES);
    if (e != cudaSuccess) return e;
    dim3 grid(nseg, (unsigned)Dm.BH);
    return launch_kernel(TOTALS ? "tc_causal_totals" : "tc_causal_fwd", kern, grid, dim3(tc::NTH), (size_t)Cf::BYTES,
                         st, Dm, Q, K, V, W, S0, seg_len, nseg, O, Sout);
}

template <bool TOTALS>
cudaError_t dispatch_causal_tc(const Dims &Dm, const bf16_t *Q, const bf16_t *K, const bf16_t *V, const float *W,
                               const float *S0, int64_t seg_len, int nseg, bf16_t *O, float *Sout, cudaStream_t st)
{
    const bool lr32 = Dm.LR <= 32, lp16 = Dm.LP <= 16;
#define RACE_TC_CASE(DD, LRPP, LPPP)                                                                             \
    if (Dm.d == DD && (LRPP == 32) == lr32 && (LPPP == 16) == lp16)                                              \
        return launch_causal_tc_inst<DD, LRPP, LPPP, TOTALS>(Dm, Q, K, V, W, S0, seg_len, nseg, O, Sout, st);
    RACE_TC_CASE(128, 32, 16)
    RACE_TC_CASE(128, 32, 32)
    RACE_TC_CASE(128, 64, 16)
    RACE_TC_CASE(128, 64, 32)
    RACE_TC_CASE(64, 32, 16)
    RACE_TC_CASE(64, 32, 32)
    RACE_TC_CASE(64, 64, 16)
    RACE_TC_CASE(64, 64, 32)
#undef RACE_TC_CASE
    return cudaErrorInvalidValue;
}

}  // namespace

bool causal_tc_supported(const Dims &Dm) { return (Dm.d == 64 || Dm.d == 128) && Dm.LR <= 64 && Dm.LP <= 32; }

int causal_tc_chunk() { return tc::C; }

cudaError_t launch_causal_tc_totals(const Dims &Dm, const bf16_t *K, const bf16_t *V, const float *W,
                                    int64_t seg_len, int nseg, float *Sout, cudaStream_t st)
{
    return dispatch_causal_tc<true>(Dm, K, K, V, W, nullptr, seg_len, nseg, nullptr, Sout, st);
}

cudaError_t launch_causal_tc_fwd(const Dims &Dm, const bf16_t *Q, const bf16_t *K, const bf16_t *V, const float *W,
                                 const float *S0, int64_t seg_len, int nseg, bf16_t *O, cudaStream_t st)
{
    return dispatch_causal_tc<false>(Dm, Q, K, V, W, S0, seg_len, nseg, O, nullptr, st);
}

}  // namespace race
