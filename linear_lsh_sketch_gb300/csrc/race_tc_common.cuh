// race_tc_common.cuh -- pieces shared by the tensor-core causal kernels: chunk geometry, bulk
// (TMA) row copies completing on mbarriers with bounded waits, the tensor-core projection
// z = X (W_hi + W_lo)^T, the bucket featuriser, and constant fragments.
#pragma once

#include "race_common.cuh"
#include "race_mma.cuh"

namespace race {
namespace tc {

using bf16 = __nv_bfloat16;
using namespace race::mma;

constexpr int C = 64;      // tokens per chunk
constexpr int NTH = 256;   // 8 warps
constexpr int LPP = 16;    // projection columns (L * P <= 16), hi rows then lo rows in the W tile

// Error bits written to the workspace status word.
constexpr unsigned kErrWaitTimeout = 1u;

// ------------------------------------------------------------------ mbarriers and bulk copies

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
}

// Orders this thread's earlier generic-proxy shared-memory accesses before later async-proxy
// (bulk copy) writes to the same memory.
__device__ __forceinline__ void fence_proxy_async()
{
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(bar), "r"(bytes) : "memory");
}

// Bulk (TMA) copy of `bytes` (multiple of 16, both addresses 16-byte aligned) from global to
// this CTA's shared memory, completing on the mbarrier at `bar`.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

// Nanoseconds of the GPU's global timer.
__device__ __forceinline__ uint64_t globaltimer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;\n" : "=l"(t));
    return t;
}

// Every wait on an asynchronous copy or a peer warp gives up after this many nanoseconds (or
// 2^22 polls, whichever comes first): a healthy wait ends within microseconds, and a stalled one
// must end the kernel rather than hold the GPU.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

// One poll of the mbarrier phase with parity `phase` (may suspend the thread briefly).
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t phase)
{
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(phase)
        : "memory");
    return ok != 0;
}

// Waits for the mbarrier phase with parity `phase`; gives up after the bounds above and returns
// false.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t phase)
{
    if (mbar_try(bar, phase)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (int i = 1; i < (1 << 22); ++i) {
        if (mbar_try(bar, phase)) return true;
        if ((i & 15) == 0 && globaltimer_ns() - t0 > kWaitLimitNs) break;
    }
    return false;
}

// Issues the bulk row copies of up to 4 token tiles ([C][XS] bf16, rows n0 .. n0 + cnt of
// [N, D] slices; tile i goes from src_i to dst_i).  Warp w copies rows 8 w .. 8 w + 7; lane l
// handles tile l / 8.  The caller has registered ntiles * cnt * D * 2 expected bytes on `bar`.
template <int D, int XS>
__device__ __forceinline__ void issue_rows(bf16 *d0, bf16 *d1, bf16 *d2, bf16 *d3, const bf16 *s0, const bf16 *s1,
                                           const bf16 *s2, const bf16 *s3, int ntiles, int64_t n0, int cnt,
                                           uint32_t bar)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int tile = lane >> 3, row = 8 * warp + (lane & 7);
    if (tile < ntiles && row < cnt) {
        bf16 *dst = tile == 0 ? d0 : tile == 1 ? d1 : tile == 2 ? d2 : d3;
        const bf16 *src = tile == 0 ? s0 : tile == 1 ? s1 : tile == 2 ? s2 : s3;
        bulk_g2s(smem_u32(dst + row * XS), src + (n0 + row) * D, D * 2, bar);
    }
}

// ------------------------------------------------------------------ nonlinearities

// Reciprocal from the hardware approximation (about 1 ulp; denormal results flush to zero, which
// only the saturated ends of tanh and sigmoid reach, where the exact value rounds to 0 as well).
__device__ __forceinline__ float rcp_fast(float x)
{
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

// tanh with about 1e-7 absolute error (all that the bucket probabilities are sensitive to).
__device__ __forceinline__ float tanh_abs(float x)
{
    return 1.f - 2.f * rcp_fast(1.f + __expf(2.f * x));
}

// sigmoid(a) and sigmoid(-a) without overflow for any finite a.
__device__ __forceinline__ void sigmoid_pair(float a, float &sp, float &sm)
{
    const float e = __expf(-fabsf(a));
    const float big = rcp_fast(1.f + e), small = e * big;
    sp = a >= 0.f ? big : small;
    sm = a >= 0.f ? small : big;
}

// The 2^P bucket probabilities of one table from its P tanh projections:
// phi_r = prod_t sigmoid(2 beta u_t v_{r,t}), v_{r,t} = +1 iff bit t of r is set.
template <int P>
__device__ __forceinline__ void bucket_probs(const float *u, float beta, float (&ph)[1 << P])
{
    ph[0] = 1.f;
#pragma unroll
    for (int p = 0; p < P; ++p) {
        float sp, sm;
        sigmoid_pair(2.f * beta * u[p], sp, sm);
#pragma unroll
        for (int r = 0; r < (1 << p); ++r) {
            ph[r + (1 << p)] = ph[r] * sp;
            ph[r] *= sm;
        }
    }
}

// ------------------------------------------------------------------ projection and features

// z = X (W_hi + W_lo)^T for the 16 rows at xs (row stride XS) and all LPP projection columns;
// returns u = tanh(z / |x|) as fragments (tile lt: rows g, g+8; columns 8 lt + 2q, +1) and the
// inverse row norms (0 for a zero row).
template <int D, int XS>
__device__ __forceinline__ void project16(const bf16 *xs, const bf16 *wc, int lane, float (&u)[LPP / 8][4],
                                          float &inv0, float &inv1)
{
    float zh[LPP / 8][4], zl[LPP / 8][4];
#pragma unroll
    for (int i = 0; i < LPP / 8; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) zh[i][j] = zl[i][j] = 0.f;
    float ss0 = 0.f, ss1 = 0.f;
    const uint32_t abase = smem_u32(xs + ((lane & 7) + 8 * ((lane >> 3) & 1)) * XS + 8 * (lane >> 4));
    // W rows: lanes 0-15 address hi rows, 16-31 lo rows (x4: hi k0-7, hi k8-15, lo k0-7, lo k8-15)
    const uint32_t wbase = smem_u32(wc + (((lane >> 4) ? LPP : 0) + (lane & 7)) * XS + 8 * ((lane >> 3) & 1));
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4(abase + 32 * ks, a0, a1, a2, a3);
        const float2 f0 = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162 *>(&a0));
        const float2 f1 = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162 *>(&a1));
        const float2 f2 = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162 *>(&a2));
        const float2 f3 = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162 *>(&a3));
        ss0 = fmaf(f0.x, f0.x, fmaf(f0.y, f0.y, fmaf(f2.x, f2.x, fmaf(f2.y, f2.y, ss0))));
        ss1 = fmaf(f1.x, f1.x, fmaf(f1.y, f1.y, fmaf(f3.x, f3.x, fmaf(f3.y, f3.y, ss1))));
#pragma unroll
        for (int lt = 0; lt < LPP / 8; ++lt) {
            uint32_t bh0, bh1, bl0, bl1;
            ldsm_x4(wbase + 2 * (8 * lt * XS + 16 * ks), bh0, bh1, bl0, bl1);
            mma16816(zh[lt], a0, a1, a2, a3, bh0, bh1);
            mma16816(zl[lt], a0, a1, a2, a3, bl0, bl1);
        }
    }
    ss0 += __shfl_xor_sync(0xffffffffu, ss0, 1);
    ss0 += __shfl_xor_sync(0xffffffffu, ss0, 2);
    ss1 += __shfl_xor_sync(0xffffffffu, ss1, 1);
    ss1 += __shfl_xor_sync(0xffffffffu, ss1, 2);
    inv0 = ss0 > 0.f ? rsqrtf(ss0) : 0.f;
    inv1 = ss1 > 0.f ? rsqrtf(ss1) : 0.f;
#pragma unroll
    for (int lt = 0; lt < LPP / 8; ++lt) {
        u[lt][0] = tanh_abs((zh[lt][0] + zl[lt][0]) * inv0);
        u[lt][1] = tanh_abs((zh[lt][1] + zl[lt][1]) * inv0);
        u[lt][2] = tanh_abs((zh[lt][2] + zl[lt][2]) * inv1);
        u[lt][3] = tanh_abs((zh[lt][3] + zl[lt][3]) * inv1);
    }
}

// Writes the u fragments of 16 rows to a warp-private [16][US] fp32 stage.
template <int US>
__device__ __forceinline__ void stage_u(const float (&u)[LPP / 8][4], float *ust, int lane)
{
    const int g = lane >> 2, q = lane & 3;
#pragma unroll
    for (int lt = 0; lt < LPP / 8; ++lt) {
        const int c = 8 * lt + 2 * q;
        ust[g * US + c] = u[lt][0];
        ust[g * US + c + 1] = u[lt][1];
        ust[(g + 8) * US + c] = u[lt][2];
        ust[(g + 8) * US + c + 1] = u[lt][3];
    }
}

// Bucket features of 16 staged rows: F[row][l R + r] = phi^(l)_r (bf16), zero for rows with
// t0 + row >= cnt; optionally also Fs = phi * scale[row] (bf16).  Items (row, table) over lanes.
template <int P, int US, int FS>
__device__ __forceinline__ void features16(const float *ust, int L, float beta, int t0, int cnt, bf16 *F, int lane,
                                           const float *scale = nullptr, bf16 *Fs = nullptr)
{
    constexpr int R = 1 << P;
    for (int it = lane; it < 16 * L; it += 32) {
        const int row = it & 15, l = it >> 4;
        float ph[R];
        bucket_probs<P>(ust + row * US + l * P, beta, ph);
        const float live = (t0 + row < cnt) ? 1.f : 0.f;
        uint32_t *dst = reinterpret_cast<uint32_t *>(F + row * FS + l * R);
#pragma unroll
        for (int r = 0; r < R; r += 2) dst[r / 2] = pack_bf16(ph[r] * live, ph[r + 1] * live);
        if (Fs) {
            const float sc = live * scale[t0 + row];
            uint32_t *dss = reinterpret_cast<uint32_t *>(Fs + row * FS + l * R);
#pragma unroll
            for (int r = 0; r < R; r += 2) dss[r / 2] = pack_bf16(ph[r] * sc, ph[r + 1] * sc);
        }
    }
}

// Chain rule back through the featuriser for 16 rows: u from the warp's stage ([16][US]),
// dphi rows ([16][DPS], fp32).  phi is recomputed; writes
// dz_p = beta * sum_r phi_r (dphi_r - phi . dphi) v_{r,p} * (1 - u_p^2) as bf16 to dz ([16][ZS]).
// db (optional): adds the d(loss)/d(beta) share sum_p u_p sum_r ds_r v_{r,p} of the rows
// t0 + row < cnt (the logits are beta (u . v_r)); stale rows past cnt add nothing.
template <int P, int US, int DPS, int ZS>
__device__ __forceinline__ void features_backward16(const float *ust, const float *dphi, int L, float beta,
                                                    bf16 *dz, int lane, float *db = nullptr, int t0 = 0,
                                                    int cnt = 0)
{
    constexpr int R = 1 << P;
    for (int it = lane; it < 16 * L; it += 32) {
        const int row = it & 15, l = it >> 4;
        const float *u = ust + row * US + l * P;
        float ph[R];
        bucket_probs<P>(u, beta, ph);
        const float *dph = dphi + row * DPS + l * R;
        float c = 0.f;
#pragma unroll
        for (int r = 0; r < R; ++r) c = fmaf(ph[r], dph[r], c);
        float du[P];
#pragma unroll
        for (int p = 0; p < P; ++p) du[p] = 0.f;
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const float ds = ph[r] * (dph[r] - c);
#pragma unroll
            for (int p = 0; p < P; ++p) du[p] += ((r >> p) & 1) ? ds : -ds;
        }
        if (db && t0 + row < cnt) {
            float a = *db;
#pragma unroll
            for (int p = 0; p < P; ++p) a = fmaf(u[p], du[p], a);
            *db = a;
        }
#pragma unroll
        for (int p = 0; p < P; ++p) dz[row * ZS + l * P + p] = __float2bfloat16_rn(beta * du[p] * (1.f - u[p] * u[p]));
    }
}

// B fragment of the mass column: n = 0 holds ones, other columns zero.
__device__ __forceinline__ void mass_fragment(int lane, uint32_t &b0, uint32_t &b1)
{
    const uint32_t one2 = 0x3F803F80u;  // two bf16 ones
    b0 = b1 = (lane >> 2) == 0 ? one2 : 0u;
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

// Hyperplanes as bf16 hi rows [0, LPP) and lo rows [LPP, 2 LPP) of a [2 LPP][XS] tile; rows
// past L * P are zero.
template <int D, int XS>
__device__ __forceinline__ void load_w_split(const float *__restrict__ W, int LP, bf16 *wc)
{
    for (int i = threadIdx.x; i < LPP * D; i += NTH) {
        const int row = i / D, k = i - row * D;
        const float w = row < LP ? W[row * D + k] : 0.f;
        bf16 hi, lo;
        split_bf16(w, hi, lo);
        wc[row * XS + k] = hi;
        wc[(LPP + row) * XS + k] = lo;
    }
}

// Zero-fills n bytes (multiple of 16) of shared memory.
__device__ __forceinline__ void zero_smem(void *p, int nbytes)
{
    uint4 *q = reinterpret_cast<uint4 *>(p);
    for (int i = threadIdx.x; i < nbytes / 16; i += NTH) q[i] = make_uint4(0, 0, 0, 0);
}

}  // namespace tc
}  // namespace race
