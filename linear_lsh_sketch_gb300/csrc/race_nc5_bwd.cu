// race_nc5_bwd.cu -- tcgen05 (TMEM accumulator) backward kernels of non-causal RACE attention,
// bf16 tensors.
//
// The pages print no backward pass; these kernels apply the chain rule to the forward of the
// "RACE Attention" slides (frames "Soft corner assignments make hashing differentiable",
// "Each bucket stores mass and a weighted value sum", "Normalize after combining the tables").
// With S = [A | B] the combined key sketch, den_t = phi(Q_t) . B and c_t = dO_t . O_t:
//
//   query side:  g_t = A dO_t (one number per sketch row),  c_t = phi(Q_t) . g_t / den_t,
//                dphi_Q(t) = (g_t - B c_t) / den_t
//   key side:    with G = [G_A | G_B] = sum_t phi(Q_t) [dO_t | -c_t] / den_t (the gradient sketch,
//                built by the sketch kernel in its second mode):
//                dV_j = G_A^T phi(K_j),  dphi_K(j) = G_A V_j + G_B
//
// and, for both sides, the Jacobians of the softmax over corners (ds_r = phi_r (dphi_r - phi .
// dphi)), of the corner logits (du_p = beta sum_r ds_r v_{r,p}), of tanh (dz = du (1 - u^2)), of
// the projection (dxhat = dz (W_hi + W_lo)) and of the row normalisation
// (dx = (dxhat - xhat (xhat . dxhat)) / |x|).
//
// Tensor-core products (M = 128 tokens, fp32 in TMEM): z = X W^T; g = dO A^T (query) or
// dphi = V G_A^T (key) with the sketch in shared memory as bf16 (hi, plus lo when it fits);
// dV = Phi_K G_A with Phi_K written by the featurising threads into TMEM (tcgen05.st) and used
// as the A operand; dxhat = dz W with dz also in TMEM.  Tables are handled in pairs (two tables
// give 2P projection columns, a whole number of packed bf16 words), pairs alternating between
// the two warps that share a token row.
#include "race_launch.h"
#include "race_nc5_common.cuh"

namespace race {
namespace nc5 {

// Rows lr < LR of a [LR][d + 1] fp32 sketch as bf16 SW128 tiles [d / 64][lrp rows][64] (hi, and
// lo = rest if `lo` is set) and its column d as fp32 `mass[lrp]`; rows LR .. lrp - 1 are zero.
template <int D>
__device__ __forceinline__ void load_sketch_rows(const float *__restrict__ S, int LR, int lrp, uint32_t hi,
                                                 uint32_t lo, bool split, float *mass)
{
    const uint32_t blk = (uint32_t)lrp * 128;
    for (int i = threadIdx.x; i < lrp * (D / 8); i += NTH) {
        const int lr = i / (D / 8), c = i - lr * (D / 8);
        uint32_t hw[4], lw[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            float v0 = 0.f, v1 = 0.f;
            if (lr < LR) {
                v0 = S[(int64_t)lr * (D + 1) + 8 * c + 2 * j];
                v1 = S[(int64_t)lr * (D + 1) + 8 * c + 2 * j + 1];
            }
            const bf16 h0 = __float2bfloat16_rn(v0), h1 = __float2bfloat16_rn(v1);
            hw[j] = bfp::pack_bf16(__bfloat162float(h0), __bfloat162float(h1));
            lw[j] = bfp::pack_bf16(v0 - __bfloat162float(h0), v1 - __bfloat162float(h1));
        }
        const uint32_t off = (c >> 3) * blk + sw_chunk(lr, c & 7);
        st_shared_v4(hi + off, hw[0], hw[1], hw[2], hw[3]);
        if (split) st_shared_v4(lo + off, lw[0], lw[1], lw[2], lw[3]);
    }
    for (int i = threadIdx.x; i < lrp; i += NTH) mass[i] = i < LR ? S[(int64_t)i * (D + 1) + D] : 0.f;
}

// Packs n fp32 values (n even) as bf16 pairs into n / 2 TMEM columns of this thread's lane.
template <int N>
__device__ __forceinline__ void st_bf16_cols(uint32_t taddr, const float (&v)[N])
{
    static_assert(N % 2 == 0, "pairs");
    constexpr int W = N / 2;
    if constexpr (W <= 8 && (W & (W - 1)) == 0) {
        uint32_t r[W];
#pragma unroll
        for (int j = 0; j < W; ++j) r[j] = bfp::pack_bf16(v[2 * j], v[2 * j + 1]);
        stn<W>(taddr, r);
    } else if constexpr (W % 8 == 0) {
#pragma unroll
        for (int b = 0; b < W / 8; ++b) {
            uint32_t r[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) r[j] = bfp::pack_bf16(v[16 * b + 2 * j], v[16 * b + 2 * j + 1]);
            stn<8>(taddr + 8 * b, r);
        }
    } else {
#pragma unroll
        for (int j = 0; j < W; ++j) {
            const uint32_t r[1] = {bfp::pack_bf16(v[2 * j], v[2 * j + 1])};
            stn<1>(taddr + j, r);
        }
    }
}

__host__ __device__ inline int round16(int x) { return (x + 15) & ~15; }
__host__ __device__ inline uint32_t round32u(uint32_t x) { return (x + 31) & ~31u; }
__host__ __device__ inline uint32_t pow2_cols(uint32_t need) { return need <= 128 ? 128 : need <= 256 ? 256 : 512; }

struct BwdLayout {
    uint32_t stg, x, shi, slo, mass, whi, wlo, red, bar, slot, bytes, sblk;
    int lrp;
    bool split;
    __host__ __device__ BwdLayout(int D, int LR, bool want_split)
    {
        const uint32_t KB = D / 64;
        lrp = round16(LR);
        sblk = (uint32_t)lrp * 128;
        stg = 2 * KB * BLK;
        x = 0;
        shi = 2 * stg;
        split = want_split;
        slo = shi + KB * sblk;
        mass = slo + (split ? KB * sblk : 0);
        whi = mass + (((uint32_t)lrp * 4 + 1023) & ~1023u);
        wlo = whi + KB * WBLK;
        red = wlo + KB * WBLK;
        bar = red + 8 * C * 4;
        slot = bar + 32;
        bytes = slot + 16;
    }
};

// TMEM columns.  Query side: g / dxhat at 0, z at zc, dz (bf16 pairs) at zc + 32.
// Key side: dphi / dV at 0, dxhat at d, z at zc, Phi_K (bf16 pairs) at zc + 32, dz after it.
__host__ __device__ inline uint32_t bwdq_zc(int D, int lrp) { return round32u((uint32_t)(lrp > D ? lrp : D)); }
__host__ __device__ inline uint32_t bwdq_cols(int D, int lrp) { return pow2_cols(bwdq_zc(D, lrp) + 48); }
__host__ __device__ inline uint32_t bwdk_zc(int D, int lrp) { return round32u((uint32_t)(lrp > 2 * D ? lrp : 2 * D)); }
__host__ __device__ inline uint32_t bwdk_cols(int D, int lrp) { return pow2_cols(bwdk_zc(D, lrp) + 32 + lrp / 2 + 16); }

// ------------------------------------------------------------------ query side

// dQ and aux[t] = {1 / den_t, c_t} for the CTA's tiles.  S: combined key sketch [BH][LR][d + 1].
// DB: also the CTA's query-side d(loss)/d(beta) partial to dbpart[bh][blockIdx.x].
template <int D, int P, int LT, bool DB>
__global__ void __launch_bounds__(NTH, 1)
    k_bwdq5(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmdO,
            const __grid_constant__ CUtensorMap tmdQ, Dims Dm, const float *__restrict__ W,
            const float *__restrict__ S, float2 *__restrict__ aux, int64_t seg_len, int split_s,
            unsigned *__restrict__ err, float *__restrict__ dbpart)
{
    constexpr int KB = D / 64;
    constexpr int R = 1 << P;
    constexpr int LMAX = LPP / P;
    constexpr int NPAIR = (LMAX + 1) / 2;
    // with 32 or more buckets per table the per-table code is long: one copy of it, looped over
    // the tables at run time (unrolled copies overflowed the instruction cache)
    constexpr bool ROLL = R >= 32;
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023) & ~1023u;
    unsigned char *sm = smem_raw + (base - raw);
    const BwdLayout Ly(D, Dm.LR, split_s != 0);
    float *red = reinterpret_cast<float *>(sm + Ly.red);
    const float *mass = reinterpret_cast<const float *>(sm + Ly.mass);
    const uint32_t bar_load = base + Ly.bar, bar_a = bar_load + 16, bar_b = bar_load + 24;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, q4 = warp & 3, h = warp >> 2;
    const int t = 32 * q4 + lane;
    const int64_t bh = blockIdx.y;
    const int64_t n_begin = (int64_t)blockIdx.x * seg_len;
    const int64_t n_end = min(Dm.N, n_begin + seg_len);
    const int ntile = n_end > n_begin ? (int)((n_end - n_begin + C - 1) / C) : 0;
    const int lrp = Ly.lrp;
    const uint32_t zc = bwdq_zc(D, lrp), dzc = zc + 32, ncols = bwdq_cols(D, lrp);
    const float beta = Dm.beta;
    const int L = LT > 0 ? LT : Dm.L;  // LT > 0: per-table loops unroll without guards

    if (warp == 0) tmem_alloc(base + Ly.slot, ncols);
    load_w_tiles<D>(head_w(W, Dm, bh), Dm.LP, sm + Ly.whi, sm + Ly.wlo);
    load_sketch_rows<D>(S + bh * Dm.LR * (D + 1), Dm.LR, lrp, base + Ly.shi, base + Ly.slo, Ly.split,
                        reinterpret_cast<float *>(sm + Ly.mass));
    if (tid == 0) {
        mbar_init(bar_load, 1);
        mbar_init(bar_load + 8, 1);
        mbar_init(bar_a, 1);
        mbar_init(bar_b, 1);
        tc::fence_mbar_init();
        prefetch_tmap(&tmQ);
        prefetch_tmap(&tmdO);
        prefetch_tmap(&tmdQ);
    }
    tc::fence_proxy_async();
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(sm + Ly.slot);
    const uint32_t tlane = tmem + ((uint32_t)(32 * q4) << 16);
    if (h == 0) {  // dz columns of tables >= L stay zero (they meet zero hyperplane rows)
        const uint32_t zr[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        stn<8>(tlane + dzc, zr);
        stn<8>(tlane + dzc + 8, zr);
        wait_st();
    }
    fence_before();
    __syncthreads();
    fence_after();

    auto issue_load = [&](int i) {
        const int s = i & 1;
        const uint32_t xs = base + Ly.x + s * Ly.stg, ys = xs + KB * BLK;
        const int y = (int)(n_begin + (int64_t)i * C);
        mbar_arrive_expect_tx(bar_load + 8 * s, 2 * KB * BLK);
#pragma unroll
        for (int kb = 0; kb < KB; ++kb) {
            tma_load(xs + kb * BLK, &tmQ, 64 * kb, y, (int)bh, bar_load + 8 * s);
            tma_load(ys + kb * BLK, &tmdO, 64 * kb, y, (int)bh, bar_load + 8 * s);
        }
    };
    if (tid == 0) {
        if (ntile > 0) issue_load(0);
        if (ntile > 1) issue_load(1);
    }

    bool failed = false;
    float db = 0.f;  // this thread's d(loss)/d(beta) share (DB only)
    int i = 0;
    for (; i < ntile; ++i) {
        const int s = i & 1;
        const int64_t n0 = n_begin + (int64_t)i * C;
        const int cnt = (int)min((int64_t)C, n_end - n0);
        const uint32_t xs = base + Ly.x + s * Ly.stg, ys = xs + KB * BLK;
        if (wait_all(bar_load + 8 * s, (i >> 1) & 1)) {
            failed = true;
            break;
        }
        if (tid == 0) {
            fence_after();
            issue_projection<D>(tmem + zc, xs, base + Ly.whi, base + Ly.wlo);
            const uint32_t id_g = idesc_bf16(128, lrp, 0, 0);
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
                const uint32_t ko = (ks >> 2) * BLK + (ks & 3) * 32, so = (ks >> 2) * Ly.sblk + (ks & 3) * 32;
                umma(tmem, desc_k(ys + ko), desc_k(base + Ly.shi + so), id_g, ks > 0);
                if (Ly.split) umma(tmem, desc_k(ys + ko), desc_k(base + Ly.slo + so), id_g, true);
            }
            commit(bar_a);
        }
        red[h * C + t] = half_sumsq<D>(xs, t, h);
        if (wait_all(bar_a, i & 1)) {
            failed = true;
            break;
        }
        fence_after();
        if (tid == 0 && i >= 1 && i + 1 < ntile) {
            bulk_wait_read0();  // tile i - 1's dQ store read the other stage
            issue_load(i + 1);
        }
        float z[LPP];
        {
            float a[32];
            ld32(tlane + zc, a);
#pragma unroll
            for (int k = 0; k < LPP; ++k) z[k] = a[k];
        }
        const float ssq = red[t] + red[C + t];
        const float inv = ssq > 0.f ? rsqrtf(ssq) : 0.f;
        const bool live = t < cnt;

        // phase A: den and phi . g over this half's tables
        float den_p = 0.f, pg_p = 0.f;
        auto den_table = [&](int l) {
            float u[P], ph[R], g[R], zl[P];
            table_z<P>(z, l, zl);
#pragma unroll
            for (int p = 0; p < P; ++p) u[p] = tc::tanh_abs(zl[p] * inv);
            tc::bucket_probs<P>(u, beta, ph);
            ld_cols<R>(tlane + l * R, g);
#pragma unroll
            for (int r = 0; r < R; ++r) {
                den_p = fmaf(ph[r], mass[l * R + r], den_p);
                pg_p = fmaf(ph[r], g[r], pg_p);
            }
        };
        if constexpr (ROLL) {
#pragma unroll 1
            for (int l = 2 * h; l < L; l += (l & 1) ? 3 : 1) den_table(l);  // pairs h, h + 2, ...
        } else {
#pragma unroll
            for (int pr = 0; pr < NPAIR; ++pr) {
                if ((pr & 1) != h || 2 * pr >= L) continue;
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    const int l = 2 * pr + k;
                    if (l >= LMAX || l >= L) continue;
                    den_table(l);
                }
            }
        }
        red[(2 + h) * C + t] = den_p;
        red[(4 + h) * C + t] = pg_p;
        __syncthreads();
        const float den = red[2 * C + t] + red[3 * C + t];
        const float rd = live ? __frcp_rn(den) : 0.f;
        const float cc = (red[4 * C + t] + red[5 * C + t]) * rd;
        if (h == 0 && live) aux[bh * Dm.N + n0 + t] = make_float2(rd, cc);

        // phase B: dphi = (g - B c) / den, then the feature Jacobian -> dz (bf16 pairs in TMEM);
        // x . dxhat = z . dz (dxhat = W^T dz with dz as the product sees it, z = W x), this half's share
        float zdz = 0.f;
        auto jac_table = [&](int l, float (&dzl)[P]) {
            float u[P], ph[R], g[R], zl[P];
            table_z<P>(z, l, zl);
#pragma unroll
            for (int p = 0; p < P; ++p) u[p] = tc::tanh_abs(zl[p] * inv);
            tc::bucket_probs<P>(u, beta, ph);
            ld_cols<R>(tlane + l * R, g);
#pragma unroll
            for (int r = 0; r < R; ++r) g[r] = (g[r] - mass[l * R + r] * cc) * rd;
            table_backward<P, DB>(u, ph, g, beta, dzl, &db);
#pragma unroll
            for (int p = 0; p < P; ++p) zdz = fmaf(__bfloat162float(__float2bfloat16_rn(dzl[p])), zl[p], zdz);
        };
        // d(loss)/d(W): table pair pr's dz / |q| of this Q row (DB instances only: the API takes
        // them whenever d(loss)/d(W) is asked for, and the others stay free of the code)
        auto store_dz = [&](int pr, const float (&dz)[2 * P]) {
            if (DB && Dm.dzq != nullptr && live) {
                float *o = Dm.dzq + (bh * Dm.N + n0 + t) * Dm.dzld + 2 * pr * P;
#pragma unroll
                for (int j = 0; j < 2 * P; ++j)
                    if (2 * pr * P + j < Dm.LP) o[j] = dz[j] * inv;
            }
        };
        if constexpr (ROLL) {
#pragma unroll 1
            for (int pr = h; 2 * pr < L; pr += 2) {
                float dz[2 * P];
#pragma unroll 1
                for (int k = 0; k < 2; ++k) {
                    const int l = 2 * pr + k;
                    float dzl[P];
                    if (l < L) {
                        jac_table(l, dzl);
                    } else {
#pragma unroll
                        for (int p = 0; p < P; ++p) dzl[p] = 0.f;
                    }
#pragma unroll
                    for (int p = 0; p < P; ++p) {  // static indices: dz stays in registers
                        if (k == 0) dz[p] = dzl[p];
                        else dz[P + p] = dzl[p];
                    }
                }
                store_dz(pr, dz);
                st_bf16_cols<2 * P>(tlane + dzc + pr * P, dz);
            }
        } else {
#pragma unroll
            for (int pr = 0; pr < NPAIR; ++pr) {
                if ((pr & 1) != h || 2 * pr >= L) continue;
                float dz[2 * P];
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    const int l = 2 * pr + k;
                    if (l >= LMAX || l >= L) {
#pragma unroll
                        for (int p = 0; p < P; ++p) dz[k * P + p] = 0.f;
                        continue;
                    }
                    float dzl[P];
                    jac_table(l, dzl);
#pragma unroll
                    for (int p = 0; p < P; ++p) dz[k * P + p] = dzl[p];
                }
                store_dz(pr, dz);
                st_bf16_cols<2 * P>(tlane + dzc + pr * P, dz);
            }
        }
        red[(6 + h) * C + t] = zdz;
        wait_st();
        fence_before();
        __syncthreads();
        if (tid == 0) {
            fence_after();
            constexpr uint32_t id_x = idesc_bf16(128, D, 0, 1);
#pragma unroll
            for (int ks = 0; ks < LPP / 16; ++ks) {
                umma_ts(tmem, tmem + dzc + 8 * ks, desc_mn(base + Ly.whi + ks * 2048, WBLK), id_x, ks > 0);
                umma_ts(tmem, tmem + dzc + 8 * ks, desc_mn(base + Ly.wlo + ks * 2048, WBLK), id_x, true);
            }
            commit(bar_b);
        }
        if (wait_all(bar_b, i & 1)) {
            failed = true;
            break;
        }
        fence_after();

        // epilogue: dQ = inv (dxhat - x inv^2 (x . dxhat)), this half's columns
        float dx[D / 2];
        uint4 xw[D / 16];
#pragma unroll
        for (int j = 0; j < D / 16; ++j) {
            const int c = h * (D / 16) + j;
            xw[j] = ld_shared_v4(xs + (c >> 3) * BLK + sw_chunk(t, c & 7));
        }
#pragma unroll
        for (int cc16 = 0; cc16 < D / 32; ++cc16) {
            float v[16];
            ld16(tlane + h * (D / 2) + 16 * cc16, v);
#pragma unroll
            for (int k = 0; k < 16; ++k) dx[16 * cc16 + k] = v[k];
        }
        const float kk = inv * inv * (red[6 * C + t] + red[7 * C + t]);
#pragma unroll
        for (int j = 0; j < D / 16; ++j) {
            const int c = h * (D / 16) + j;
            const uint32_t w4[4] = {xw[j].x, xw[j].y, xw[j].z, xw[j].w};
            uint32_t o[4];
#pragma unroll
            for (int k = 0; k < 4; ++k)
                o[k] = bfp::pack_bf16(inv * (dx[8 * j + 2 * k] - bf_lo(w4[k]) * kk),
                                      inv * (dx[8 * j + 2 * k + 1] - bf_hi(w4[k]) * kk));
            st_shared_v4(ys + (c >> 3) * BLK + sw_chunk(t, c & 7), o[0], o[1], o[2], o[3]);
        }
        tc::fence_proxy_async();
        fence_before();
        __syncthreads();
        if (tid == 0) {
#pragma unroll
            for (int kb = 0; kb < KB; ++kb) tma_store(&tmdQ, 64 * kb, (int)n0, (int)bh, ys + kb * BLK);
            bulk_commit();
        }
    }
    if (failed) {
        if (tid == 0) atomicOr(err, kErrTimeout);
        if (i < ntile) mbar_wait(bar_load + 8 * (i & 1), (i >> 1) & 1);
        if (i + 1 < ntile) mbar_wait(bar_load + 8 * ((i + 1) & 1), ((i + 1) >> 1) & 1);
    }
    if constexpr (DB) {
        const float sdb = block_sum_fixed(db, red);
        if (tid == 0) dbpart[bh * gridDim.x + blockIdx.x] = sdb;
    }
    if (tid == 0) bulk_wait0();
    fence_before();
    __syncthreads();
    if (warp == 0) {
        fence_after();
        tmem_dealloc(tmem, ncols);
    }
}

// ------------------------------------------------------------------ key side

// dK and dV for the CTA's tiles.  G: combined gradient sketch [BH][LR][d + 1].
// DB: also the CTA's key-side d(loss)/d(beta) partial to dbpart[bh][blockIdx.x].
template <int D, int P, int LT, bool DB>
__global__ void __launch_bounds__(NTH, 1)
    k_bwdk5(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
            const __grid_constant__ CUtensorMap tmdK, const __grid_constant__ CUtensorMap tmdV, Dims Dm,
            const float *__restrict__ W, const float *__restrict__ G, int64_t seg_len, int split_s,
            unsigned *__restrict__ err, float *__restrict__ dbpart)
{
    constexpr int KB = D / 64;
    constexpr int R = 1 << P;
    constexpr int LMAX = LPP / P;
    constexpr int NPAIR = (LMAX + 1) / 2;
    // with 32 or more buckets per table the per-table code is long: one copy of it, looped over
    // the tables at run time (unrolled copies overflowed the instruction cache)
    constexpr bool ROLL = R >= 32;
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023) & ~1023u;
    unsigned char *sm = smem_raw + (base - raw);
    const BwdLayout Ly(D, Dm.LR, split_s != 0);
    float *red = reinterpret_cast<float *>(sm + Ly.red);
    const float *gmass = reinterpret_cast<const float *>(sm + Ly.mass);
    const uint32_t bar_load = base + Ly.bar, bar_a = bar_load + 16, bar_b = bar_load + 24;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, q4 = warp & 3, h = warp >> 2;
    const int t = 32 * q4 + lane;
    const int64_t bh = blockIdx.y;
    const int64_t n_begin = (int64_t)blockIdx.x * seg_len;
    const int64_t n_end = min(Dm.N, n_begin + seg_len);
    const int ntile = n_end > n_begin ? (int)((n_end - n_begin + C - 1) / C) : 0;
    const int lrp = Ly.lrp;
    const uint32_t zc = bwdk_zc(D, lrp), fkc = zc + 32, dzc = fkc + lrp / 2, ncols = bwdk_cols(D, lrp);
    const float beta = Dm.beta;
    const int L = LT > 0 ? LT : Dm.L;  // LT > 0: per-table loops unroll without guards

    if (warp == 0) tmem_alloc(base + Ly.slot, ncols);
    load_w_tiles<D>(head_w(W, Dm, bh), Dm.LP, sm + Ly.whi, sm + Ly.wlo);
    load_sketch_rows<D>(G + bh * Dm.LR * (D + 1), Dm.LR, lrp, base + Ly.shi, base + Ly.slo, Ly.split,
                        reinterpret_cast<float *>(sm + Ly.mass));
    if (tid == 0) {
        mbar_init(bar_load, 1);
        mbar_init(bar_load + 8, 1);
        mbar_init(bar_a, 1);
        mbar_init(bar_b, 1);
        tc::fence_mbar_init();
        prefetch_tmap(&tmK);
        prefetch_tmap(&tmV);
        prefetch_tmap(&tmdK);
        prefetch_tmap(&tmdV);
    }
    tc::fence_proxy_async();
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(sm + Ly.slot);
    const uint32_t tlane = tmem + ((uint32_t)(32 * q4) << 16);
    {  // feature columns past L R and dz columns past L P stay zero (K padding of the products)
        const uint32_t zr[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        const uint32_t nz = lrp / 2 + 16;
        for (uint32_t c0 = 8 * h; c0 < nz; c0 += 16) stn<8>(tlane + fkc + c0, zr);
        wait_st();
    }
    fence_before();
    __syncthreads();
    fence_after();

    auto issue_load = [&](int i) {
        const int s = i & 1;
        const uint32_t xs = base + Ly.x + s * Ly.stg, ys = xs + KB * BLK;
        const int y = (int)(n_begin + (int64_t)i * C);
        mbar_arrive_expect_tx(bar_load + 8 * s, 2 * KB * BLK);
#pragma unroll
        for (int kb = 0; kb < KB; ++kb) {
            tma_load(xs + kb * BLK, &tmK, 64 * kb, y, (int)bh, bar_load + 8 * s);
            tma_load(ys + kb * BLK, &tmV, 64 * kb, y, (int)bh, bar_load + 8 * s);
        }
    };
    if (tid == 0) {
        if (ntile > 0) issue_load(0);
        if (ntile > 1) issue_load(1);
    }

    bool failed = false;
    float db = 0.f;  // this thread's d(loss)/d(beta) share (DB only)
    int i = 0;
    for (; i < ntile; ++i) {
        const int s = i & 1;
        const int64_t n0 = n_begin + (int64_t)i * C;
        const int cnt = (int)min((int64_t)C, n_end - n0);
        const uint32_t xs = base + Ly.x + s * Ly.stg, ys = xs + KB * BLK;
        if (wait_all(bar_load + 8 * s, (i >> 1) & 1)) {
            failed = true;
            break;
        }
        if (tid == 0) {
            fence_after();
            issue_projection<D>(tmem + zc, xs, base + Ly.whi, base + Ly.wlo);
            const uint32_t id_p = idesc_bf16(128, lrp, 0, 0);
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
                const uint32_t ko = (ks >> 2) * BLK + (ks & 3) * 32, so = (ks >> 2) * Ly.sblk + (ks & 3) * 32;
                umma(tmem, desc_k(ys + ko), desc_k(base + Ly.shi + so), id_p, ks > 0);
                if (Ly.split) umma(tmem, desc_k(ys + ko), desc_k(base + Ly.slo + so), id_p, true);
            }
            commit(bar_a);
        }
        red[h * C + t] = half_sumsq<D>(xs, t, h);
        if (wait_all(bar_a, i & 1)) {
            failed = true;
            break;
        }
        fence_after();
        if (tid == 0 && i >= 1 && i + 1 < ntile) {
            bulk_wait_read0();  // tile i - 1's dK / dV stores read the other stage
            issue_load(i + 1);
        }
        float z[LPP];
        {
            float a[32];
            ld32(tlane + zc, a);
#pragma unroll
            for (int k = 0; k < LPP; ++k) z[k] = a[k];
        }
        const float ssq = red[t] + red[C + t];
        const float inv = ssq > 0.f ? rsqrtf(ssq) : 0.f;

        // features -> TMEM (A operand of dV); dphi = V G_A^T + G_B -> feature Jacobian -> dz;
        // x . dxhat = z . dz (dxhat = W^T dz with dz as the product sees it, z = W x), this half's share
        float zdz = 0.f;
        auto key_table = [&](int l, float (&dzl)[P]) {
            float u[P], ph[R], dph[R], zl[P];
            table_z<P>(z, l, zl);
#pragma unroll
            for (int p = 0; p < P; ++p) u[p] = tc::tanh_abs(zl[p] * inv);
            tc::bucket_probs<P>(u, beta, ph);
            st_bf16_cols<R>(tlane + fkc + l * (R / 2), ph);
            ld_cols<R>(tlane + l * R, dph);
#pragma unroll
            for (int r = 0; r < R; ++r) dph[r] += gmass[l * R + r];
            table_backward<P, DB>(u, ph, dph, beta, dzl, &db);
#pragma unroll
            for (int p = 0; p < P; ++p) zdz = fmaf(__bfloat162float(__float2bfloat16_rn(dzl[p])), zl[p], zdz);
        };
        // d(loss)/d(W): table pair pr's dz / |k| of this K row (DB instances only)
        auto store_dz = [&](int pr, const float (&dz)[2 * P]) {
            if (DB && Dm.dzk != nullptr && t < cnt) {
                float *o = Dm.dzk + (bh * Dm.N + n0 + t) * Dm.dzld + 2 * pr * P;
#pragma unroll
                for (int j = 0; j < 2 * P; ++j)
                    if (2 * pr * P + j < Dm.LP) o[j] = dz[j] * inv;
            }
        };
        if constexpr (ROLL) {
#pragma unroll 1
            for (int pr = h; 2 * pr < L; pr += 2) {
                float dz[2 * P];
#pragma unroll 1
                for (int k = 0; k < 2; ++k) {
                    const int l = 2 * pr + k;
                    float dzl[P];
                    if (l < L) {
                        key_table(l, dzl);
                    } else {
#pragma unroll
                        for (int p = 0; p < P; ++p) dzl[p] = 0.f;
                    }
#pragma unroll
                    for (int p = 0; p < P; ++p) {  // static indices: dz stays in registers
                        if (k == 0) dz[p] = dzl[p];
                        else dz[P + p] = dzl[p];
                    }
                }
                store_dz(pr, dz);
                st_bf16_cols<2 * P>(tlane + dzc + pr * P, dz);
            }
        } else {
#pragma unroll
            for (int pr = 0; pr < NPAIR; ++pr) {
                if ((pr & 1) != h || 2 * pr >= L) continue;
                float dz[2 * P];
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    const int l = 2 * pr + k;
                    if (l >= LMAX || l >= L) {
#pragma unroll
                        for (int p = 0; p < P; ++p) dz[k * P + p] = 0.f;
                        continue;
                    }
                    float dzl[P];
                    key_table(l, dzl);
#pragma unroll
                    for (int p = 0; p < P; ++p) dz[k * P + p] = dzl[p];
                }
                store_dz(pr, dz);
                st_bf16_cols<2 * P>(tlane + dzc + pr * P, dz);
            }
        }
        red[(6 + h) * C + t] = zdz;
        wait_st();
        fence_before();
        __syncthreads();
        if (warp == 0) {  // the run-time K loop issues from the converged warp (one elected lane)
            fence_after();
            constexpr uint32_t id_x = idesc_bf16(128, D, 0, 1);
            for (int ks = 0; ks < lrp / 16; ++ks) {
                umma_ts_w(tmem, tmem + fkc + 8 * ks, desc_mn(base + Ly.shi + ks * 2048, Ly.sblk), id_x, ks > 0);
                if (Ly.split)
                    umma_ts_w(tmem, tmem + fkc + 8 * ks, desc_mn(base + Ly.slo + ks * 2048, Ly.sblk), id_x, true);
            }
#pragma unroll
            for (int ks = 0; ks < LPP / 16; ++ks) {
                umma_ts_w(tmem + D, tmem + dzc + 8 * ks, desc_mn(base + Ly.whi + ks * 2048, WBLK), id_x, ks > 0);
                umma_ts_w(tmem + D, tmem + dzc + 8 * ks, desc_mn(base + Ly.wlo + ks * 2048, WBLK), id_x, true);
            }
            commit_w(bar_b);
        }
        if (wait_all(bar_b, i & 1)) {
            failed = true;
            break;
        }
        fence_after();

        // epilogue: dK (normalisation backward) staged in the V tile, dV staged in the K tile
        float dx[D / 2];
        uint4 xw[D / 16];
#pragma unroll
        for (int j = 0; j < D / 16; ++j) {
            const int c = h * (D / 16) + j;
            xw[j] = ld_shared_v4(xs + (c >> 3) * BLK + sw_chunk(t, c & 7));
        }
#pragma unroll
        for (int cc16 = 0; cc16 < D / 32; ++cc16) {
            float v[16];
            ld16(tlane + D + h * (D / 2) + 16 * cc16, v);
#pragma unroll
            for (int k = 0; k < 16; ++k) dx[16 * cc16 + k] = v[k];
        }
        // each thread overwrites only the K-row half it has just read (its dV half)
        const float kk = inv * inv * (red[6 * C + t] + red[7 * C + t]);
#pragma unroll
        for (int j = 0; j < D / 16; ++j) {
            const int c = h * (D / 16) + j;
            const uint32_t w4[4] = {xw[j].x, xw[j].y, xw[j].z, xw[j].w};
            uint32_t o[4];
#pragma unroll
            for (int k = 0; k < 4; ++k)
                o[k] = bfp::pack_bf16(inv * (dx[8 * j + 2 * k] - bf_lo(w4[k]) * kk),
                                      inv * (dx[8 * j + 2 * k + 1] - bf_hi(w4[k]) * kk));
            st_shared_v4(ys + (c >> 3) * BLK + sw_chunk(t, c & 7), o[0], o[1], o[2], o[3]);
        }
#pragma unroll
        for (int cc16 = 0; cc16 < D / 32; ++cc16) {
            float v[16];
            ld16(tlane + h * (D / 2) + 16 * cc16, v);
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int c = h * (D / 16) + 2 * cc16 + j;
                st_shared_v4(xs + (c >> 3) * BLK + sw_chunk(t, c & 7), bfp::pack_bf16(v[8 * j], v[8 * j + 1]),
                             bfp::pack_bf16(v[8 * j + 2], v[8 * j + 3]), bfp::pack_bf16(v[8 * j + 4], v[8 * j + 5]),
                             bfp::pack_bf16(v[8 * j + 6], v[8 * j + 7]));
            }
        }
        tc::fence_proxy_async();
        fence_before();
        __syncthreads();
        if (tid == 0) {
#pragma unroll
            for (int kb = 0; kb < KB; ++kb) {
                tma_store(&tmdK, 64 * kb, (int)n0, (int)bh, ys + kb * BLK);
                tma_store(&tmdV, 64 * kb, (int)n0, (int)bh, xs + kb * BLK);
            }
            bulk_commit();
        }
    }
    if (failed) {
        if (tid == 0) atomicOr(err, kErrTimeout);
        if (i < ntile) mbar_wait(bar_load + 8 * (i & 1), (i >> 1) & 1);
        if (i + 1 < ntile) mbar_wait(bar_load + 8 * ((i + 1) & 1), ((i + 1) >> 1) & 1);
    }
    if constexpr (DB) {
        const float sdb = block_sum_fixed(db, red);
        if (tid == 0) dbpart[bh * gridDim.x + blockIdx.x] = sdb;
    }
    if (tid == 0) bulk_wait0();
    fence_before();
    __syncthreads();
    if (warp == 0) {
        fence_after();
        tmem_dealloc(tmem, ncols);
    }
}

}  // namespace nc5

// ------------------------------------------------------------------ host side

cudaError_t make_token_map(CUtensorMap *map, const void *base, const Dims &D);

namespace {

constexpr size_t kSmemMax = 227 * 1024;

template <typename K>
cudaError_t prep_bwd(K kern, size_t bytes)
{
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

// Persistent split of the token tiles: about (SMs x CTAs per SM) CTAs over all (b, h).
int64_t bwd_seg(const Dims &Dm, size_t smem)
{
    const int per_sm = std::max<int>(1, std::min<int>(2, (int)(kSmemMax / smem)));
    const int64_t ntiles = (Dm.N + nc5::C - 1) / nc5::C;
    int64_t want = std::max<int64_t>(1, ((int64_t)Dm.sms * per_sm + Dm.BH - 1) / Dm.BH);
    want = std::min(want, ntiles);
    return ((ntiles + want - 1) / want) * nc5::C;
}

nc5::BwdLayout bwd_layout(const Dims &Dm)
{
    const nc5::BwdLayout with_lo(Dm.d, Dm.LR, true);
    return nc5::BwdLayout(Dm.d, Dm.LR, with_lo.bytes + 1024 <= kSmemMax);
}

template <int D, int P, int LT>
cudaError_t bwdq_launch(const Dims &Dm, const CUtensorMap &mq, const CUtensorMap &mdo, const CUtensorMap &mdq,
                        const float *W, const float *S, float2 *aux, unsigned *err, float *dbpart, cudaStream_t st)
{
    const nc5::BwdLayout Ly = bwd_layout(Dm);
    const size_t smem = Ly.bytes + 1024;
    auto kern = dbpart ? nc5::k_bwdq5<D, P, LT, true> : nc5::k_bwdq5<D, P, LT, false>;
    cudaError_t e = prep_bwd(kern, smem);
    if (e != cudaSuccess) return e;
    const int64_t seg = bwd_seg(Dm, smem);
    const int64_t nseg = (Dm.N + seg - 1) / seg;
    return launch_kernel("tc5_bwd_query", kern, dim3((unsigned)nseg, (unsigned)Dm.BH), dim3(nc5::NTH), smem, st, mq,
                         mdo, mdq, Dm, W, S, aux, seg, (int)Ly.split, err, dbpart);
}

// The named non-causal workloads' shapes run with L compiled in: (d, P, L) = (64, 3, 3), (128, 6, 4).
template <int D, int P>
cudaError_t bwdq_inst(const Dims &Dm, const CUtensorMap &mq, const CUtensorMap &mdo, const CUtensorMap &mdq,
                      const float *W, const float *S, float2 *aux, unsigned *err, float *dbpart, cudaStream_t st)
{
    if constexpr (D == 64 && P == 3)
        if (Dm.L == 3) return bwdq_launch<D, P, 3>(Dm, mq, mdo, mdq, W, S, aux, err, dbpart, st);
    if constexpr (D == 128 && P == 6)
        if (Dm.L == 4) return bwdq_launch<D, P, 4>(Dm, mq, mdo, mdq, W, S, aux, err, dbpart, st);
    return bwdq_launch<D, P, 0>(Dm, mq, mdo, mdq, W, S, aux, err, dbpart, st);
}

template <int D, int P, int LT>
cudaError_t bwdk_launch(const Dims &Dm, const CUtensorMap &mk, const CUtensorMap &mv, const CUtensorMap &mdk,
                        const CUtensorMap &mdv, const float *W, const float *G, unsigned *err, float *dbpart,
                        cudaStream_t st)
{
    const nc5::BwdLayout Ly = bwd_layout(Dm);
    const size_t smem = Ly.bytes + 1024;
    auto kern = dbpart ? nc5::k_bwdk5<D, P, LT, true> : nc5::k_bwdk5<D, P, LT, false>;
    cudaError_t e = prep_bwd(kern, smem);
    if (e != cudaSuccess) return e;
    const int64_t seg = bwd_seg(Dm, smem);
    const int64_t nseg = (Dm.N + seg - 1) / seg;
    return launch_kernel("tc5_bwd_key", kern, dim3((unsigned)nseg, (unsigned)Dm.BH), dim3(nc5::NTH), smem, st, mk,
                         mv, mdk, mdv, Dm, W, G, seg, (int)Ly.split, err, dbpart);
}

// The named non-causal workloads' shapes run with L compiled in: (d, P, L) = (64, 3, 3), (128, 6, 4).
template <int D, int P>
cudaError_t bwdk_inst(const Dims &Dm, const CUtensorMap &mk, const CUtensorMap &mv, const CUtensorMap &mdk,
                      const CUtensorMap &mdv, const float *W, const float *G, unsigned *err, float *dbpart,
                      cudaStream_t st)
{
    if constexpr (D == 64 && P == 3)
        if (Dm.L == 3) return bwdk_launch<D, P, 3>(Dm, mk, mv, mdk, mdv, W, G, err, dbpart, st);
    if constexpr (D == 128 && P == 6)
        if (Dm.L == 4) return bwdk_launch<D, P, 4>(Dm, mk, mv, mdk, mdv, W, G, err, dbpart, st);
    return bwdk_launch<D, P, 0>(Dm, mk, mv, mdk, mdv, W, G, err, dbpart, st);
}

#define RACE_NC5B_DISPATCH(FN, ...)                        \
    switch (Dm.d * 16 + Dm.P) {                            \
        case 64 * 16 + 1: return FN<64, 1>(__VA_ARGS__);   \
        case 64 * 16 + 2: return FN<64, 2>(__VA_ARGS__);   \
        case 64 * 16 + 3: return FN<64, 3>(__VA_ARGS__);   \
        case 64 * 16 + 4: return FN<64, 4>(__VA_ARGS__);   \
        case 64 * 16 + 5: return FN<64, 5>(__VA_ARGS__);   \
        case 64 * 16 + 6: return FN<64, 6>(__VA_ARGS__);   \
        case 128 * 16 + 1: return FN<128, 1>(__VA_ARGS__); \
        case 128 * 16 + 2: return FN<128, 2>(__VA_ARGS__); \
        case 128 * 16 + 3: return FN<128, 3>(__VA_ARGS__); \
        case 128 * 16 + 4: return FN<128, 4>(__VA_ARGS__); \
        case 128 * 16 + 5: return FN<128, 5>(__VA_ARGS__); \
        case 128 * 16 + 6: return FN<128, 6>(__VA_ARGS__); \
        default: return cudaErrorInvalidValue;             \
    }

}  // namespace

int nc5_bwd_nseg(const Dims &Dm)
{
    const int64_t seg = bwd_seg(Dm, bwd_layout(Dm).bytes + 1024);
    return (int)((Dm.N + seg - 1) / seg);
}

cudaError_t launch_nc5_bwd_query(const Dims &Dm, const bf16_t *Q, const bf16_t *dO, const float *W, const float *S,
                                 bf16_t *dQ, float2 *aux, unsigned *err, float *dbpart, cudaStream_t st)
{
    CUtensorMap mq, mdo, mdq;
    cudaError_t e = make_token_map(&mq, Q, Dm);
    if (e == cudaSuccess) e = make_token_map(&mdo, dO, Dm);
    if (e == cudaSuccess) e = make_token_map(&mdq, dQ, Dm);
    if (e != cudaSuccess) return e;
    RACE_NC5B_DISPATCH(bwdq_inst, Dm, mq, mdo, mdq, W, S, aux, err, dbpart, st)
}

cudaError_t launch_nc5_bwd_key(const Dims &Dm, const bf16_t *K, const bf16_t *V, const float *W, const float *G,
                               bf16_t *dK, bf16_t *dV, unsigned *err, float *dbpart, cudaStream_t st)
{
    CUtensorMap mk, mv, mdk, mdv;
    cudaError_t e = make_token_map(&mk, K, Dm);
    if (e == cudaSuccess) e = make_token_map(&mv, V, Dm);
    if (e == cudaSuccess) e = make_token_map(&mdk, dK, Dm);
    if (e == cudaSuccess) e = make_token_map(&mdv, dV, Dm);
    if (e != cudaSuccess) return e;
    RACE_NC5B_DISPATCH(bwdk_inst, Dm, mk, mv, mdk, mdv, W, G, err, dbpart, st)
}

}  // namespace race
