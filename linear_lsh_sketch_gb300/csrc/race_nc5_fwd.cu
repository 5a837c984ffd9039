// race_nc5_fwd.cu -- tcgen05 (TMEM accumulator) kernels of non-causal RACE attention, bf16
// tensors: the split-N sketch reduction and the query read-out.
//
// "RACE Attention" slides (arXiv:2510.04008v5): frame "Soft corner assignments make hashing
// differentiable" (Algorithm 1 bucket features), "Each bucket stores mass and a weighted value
// sum" (the per-table sketches A = Phi_K^T V and B = Phi_K^T 1) and "Normalize after combining
// the tables" (O = sum_l Phi_Q A / sum_l Phi_Q B); reading notes sections 2.4-2.5.
//
// Both kernels walk 128-token tiles brought in by TMA (two stages; three for the sketch's X tiles
// when L R <= 64).  Per tile one thread issues
// the projection z = X (W_hi + W_lo)^T on the tensor cores into TMEM; every thread turns its
// token row of z into bucket probabilities (tanh, products of sigmoids) and writes them, bf16,
// into a 128-byte-swizzled feature tile Phi (token rows, L * R columns).  Then:
//   sketch:   [A | B] (+)= Phi^T [Y | m]   (M = 128 sketch rows per block, N = d + 16, K = 128
//             tokens; Y = V and m = 1 for the keys, or Y = dO and m = -c with Phi scaled by
//             1 / den for the gradient sketch of the backward pass), accumulated in TMEM over
//             the CTA's token range and written out as one fp32 partial per CTA;
//   read-out: [num | den] = Phi_Q [A | B]  (M = 128 tokens, N = d + 16, K = L R) with the
//             combined sketch held in shared memory as bf16 (hi, and lo = rest when it fits);
//             O = num / den is staged in the consumed Q tile and stored by TMA.
#include "race_launch.h"
#include "race_nc5_common.cuh"

namespace race {
namespace nc5 {

// ------------------------------------------------------------------ sketch reduction

constexpr int NTHW = NTH + 32;  // 8 compute warps + 1 control warp (TMA and MMA issue)

struct SketchLayout {
    uint32_t stg, x, y, f, fbytes, whi, wlo, mass, red, bar, slot, bytes;
    int nmb, nf, nx;
    __host__ __device__ SketchLayout(int D, int LR)
    {
        const uint32_t KB = D / 64;
        nmb = (LR + 127) / 128;
        // one feature buffer: M = 128 sketch rows per block, as two 64-column blocks; with L R <= 64
        // the second block of each M = 128 operand is padding (its accumulator lanes are never
        // read), so the buffer keeps only the first and the operand's second block points at the
        // next 16 KB of shared memory (the other buffer, or the W tiles after it)
        const bool half_f = LR <= 64;
        fbytes = half_f ? BLK : 2 * nmb * BLK;
        const uint32_t fixed = 2 * 2 * KB * BLK + 2 * KB * WBLK + 2 * 4096 + 2 * 2 * C * 4 + 256;
        nf = (fixed + 2 * fbytes + 1024 <= 227 * 1024) ? 2 : 1;  // double-buffer the features if they fit
        // a third X stage when it fits: the X tile of tile i + 3 is requested once tile i's
        // features are in, which keeps enough bytes in flight to cover the load latency
        nx = (half_f && fixed + KB * BLK + nf * fbytes + 1024 <= 227 * 1024) ? 3 : 2;
        stg = KB * BLK;
        x = 0;                  // X stages [nx][KB blocks]
        y = x + nx * stg;       // Y stages [2][KB blocks]
        f = y + 2 * stg;        // feature buffers [nf]
        whi = f + nf * fbytes;
        wlo = whi + KB * WBLK;
        mass = wlo + KB * WBLK;  // mass operand [2] (4 KB each)
        red = mass + 2 * 4096;   // row-norm halves [2 parities][2][C]
        bar = red + 2 * 2 * C * 4;
        slot = bar + 128;
        bytes = slot + 16;
    }
};

__host__ __device__ inline uint32_t sketch_zcol(int D, int nmb) { return nmb == 1 ? ((D + 16 + 31) & ~31) : 448; }
__host__ __device__ inline uint32_t sketch_tmem_cols(int D, int nmb)
{
    const uint32_t need = sketch_zcol(D, nmb) + 2 * LPP;  // two projection buffers
    return need <= 128 ? 128 : need <= 256 ? 256 : 512;
}

// The features of tile i + 1 can be ready before the issuing warp has observed those of tile i
// (its projection is issued early), so "features ready" has one barrier per tile parity.
enum : uint32_t { SB_X0, SB_X1, SB_X2, SB_Y0, SB_Y1, SB_P0, SB_P1, SB_S0, SB_S1, SB_F0, SB_F1, SB_CS, SB_DONE,
                  SB_COUNT };

// mode 0: X = K, Y = V, m = 1.  mode 1: X = Q, Y = dO, Phi scaled by aux.x = 1/den, m = -aux.y
// (= -c, split into bf16 hi and lo rows).  part: [BH][nsplit][LR][d + 1] fp32.  frows (may be
// null): every token's feature row, bf16 [BH][N][feature_row_stride(LR)], and its 1 / |x|, fp32
// [BH][N] (invrows), for later passes.
// Warp 8 issues the TMA copies and MMAs; the projection of tile i + 1 is issued ahead of the
// sketch product of tile i, so the compute warps featurise tile i + 1 while it runs.
template <int D, int P, int LT>
__global__ void __launch_bounds__(NTHW, 1)
    k_sketch5(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmY, Dims Dm,
              const float *__restrict__ W, const float2 *__restrict__ aux, int64_t seg_len, int nsplit,
              float *__restrict__ part, bf16 *__restrict__ frows, float *__restrict__ invrows,
              unsigned *__restrict__ err, int mode)
{
    constexpr int KB = D / 64;
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023) & ~1023u;
    unsigned char *sm = smem_raw + (base - raw);
    const SketchLayout Ly(D, Dm.LR);
    const int nmb = Ly.nmb, nf = Ly.nf, nx = Ly.nx;
    float *red = reinterpret_cast<float *>(sm + Ly.red);
    auto bar = [&](uint32_t i) { return base + Ly.bar + 8 * i; };
    volatile int *abort = reinterpret_cast<volatile int *>(sm + Ly.slot + 8);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, q4 = warp & 3, h = (warp >> 2) & 1;
    const bool compute = warp < 8;
    const int t = 32 * q4 + lane;
    const int split = blockIdx.x;
    const int64_t bh = blockIdx.y;
    const int64_t n_begin = (int64_t)split * seg_len;
    const int64_t n_end = min(Dm.N, n_begin + seg_len);
    const int ntile = n_end > n_begin ? (int)((n_end - n_begin + C - 1) / C) : 0;
    const uint32_t zcol = sketch_zcol(D, nmb), ncols = sketch_tmem_cols(D, nmb);

    // ---- set-up
    if (warp == 0) tmem_alloc(base + Ly.slot, ncols);
    if (compute) {
        zero_region(sm + Ly.f, nf * Ly.fbytes);
        init_mass_tile(sm + Ly.mass, mode == 0);  // mode 1 writes rows 0 and 1 per tile
        init_mass_tile(sm + Ly.mass + 4096, mode == 0);
        load_w_tiles<D>(head_w(W, Dm, bh), Dm.LP, sm + Ly.whi, sm + Ly.wlo);
    }
    if (tid == NTH) {
        for (uint32_t i = 0; i < SB_COUNT; ++i) mbar_init(bar(i), (i == SB_F0 || i == SB_F1) ? 8 : i == SB_CS ? NTH : 1);
        *abort = 0;
        tc::fence_mbar_init();
        prefetch_tmap(&tmX);
        prefetch_tmap(&tmY);
    }
    tc::fence_proxy_async();
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(sm + Ly.slot);
    const uint32_t tlane = tmem + ((uint32_t)(32 * q4) << 16);

    if (!compute) {
        // ---------------------------------------------------------------- control warp
        {  // the whole control warp, converged: one elected lane issues each copy and product
            auto load = [&](int i, bool is_y) {
                const int s = is_y ? i & 1 : i % nx;
                const uint32_t b = bar((is_y ? SB_Y0 : SB_X0) + s);
                const uint32_t dst = base + (is_y ? Ly.y : Ly.x) + s * Ly.stg;
                expect_tx_w(b, KB * BLK);
#pragma unroll
                for (int kb = 0; kb < KB; ++kb)
                    tma_load_w(dst + kb * BLK, is_y ? &tmY : &tmX, 64 * kb, (int)(n_begin + (int64_t)i * C), (int)bh, b);
            };
            Counts<5> issued, done;  // X0, X1, X2, Y0, Y1
            for (int i = 0; i < nx && i < ntile; ++i) {
                load(i, false);
                issued.inc(i);
            }
            for (int i = 0; i < 2 && i < ntile; ++i) {
                load(i, true);
                issued.inc(3 + i);
            }
            constexpr uint32_t id_v = idesc_bf16(128, D, 1, 1);
            constexpr uint32_t id_m = idesc_bf16(128, 16, 1, 0);
            auto proj = [&](int i) {
                const int s = i & 1, sx = i % nx;
                if (!wait_phase_w(bar(SB_X0 + sx), (i / nx) & 1, abort)) return false;
                done.inc(sx);
                fence_after();
                issue_projection_w<D>(tmem + zcol + LPP * s, base + Ly.x + sx * Ly.stg, base + Ly.whi, base + Ly.wlo);
                commit_w(bar(SB_P0 + s));
                return true;
            };
            bool ok = ntile == 0 || proj(0);
            for (int i = 0; i < ntile && ok; ++i) {
                const int s = i & 1;
                if (i + 1 < ntile && !(ok = proj(i + 1))) break;
                if (!(ok = wait_phase_w(bar(SB_F0 + s), (i >> 1) & 1, abort))) break;
                if (!(ok = wait_phase_w(bar(SB_Y0 + s), (i >> 1) & 1, abort))) break;
                done.inc(3 + s);
                fence_after();
                const uint32_t fbuf = base + Ly.f + (i % nf) * Ly.fbytes;
                const uint32_t mbuf = base + Ly.mass + (mode ? (i & 1) * 4096 : 0);
                const uint32_t ys = base + Ly.y + s * Ly.stg;
                for (int m = 0; m < nmb; ++m) {
                    const uint32_t acc = tmem + m * 256;
#pragma unroll
                    for (int ks = 0; ks < C / 16; ++ks) {
                        const uint64_t a = desc_mn(fbuf + 2 * m * BLK + ks * 2048, BLK);  // rows 64+: next 16 KB
                        const bool accum = i > 0 || ks > 0;
                        umma_w(acc, a, desc_mn(ys + ks * 2048, BLK), id_v, accum);
                        umma_w(acc + D, a, desc_k(mbuf + (ks >> 2) * 2048 + (ks & 3) * 32), id_m, accum);
                    }
                }
                commit_w(bar(SB_S0 + s));
                // X stage of tile i: read by its projection and norms (both done: features are in)
                if (i + nx < ntile) {
                    load(i + nx, false);
                    issued.inc(i % nx);
                }
                // Y stage s ^ 1: read by the sketch product of tile i - 1
                if (i >= 1 && i + 1 < ntile) {
                    if (!(ok = wait_phase_w(bar(SB_S0 + (s ^ 1)), ((i - 1) >> 1) & 1, abort))) break;
                    load(i + 1, true);
                    issued.inc(3 + (s ^ 1));
                }
            }
            if (ok) commit_w(bar(SB_DONE));
            if (!ok) {
                if (lane == 0) atomicOr(err, kErrTimeout);
                *abort = 1;
#pragma unroll
                for (int b = 0; b < 5; ++b)
                    if (issued.v[b] > done.v[b]) mbar_wait(bar(SB_X0 + b), done.v[b] & 1);
            }
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------------------- compute warps
        bool ok = true;
        for (int i = 0; i < ntile && ok; ++i) {
            const int s = i & 1;
            const int64_t n0 = n_begin + (int64_t)i * C;
            const int cnt = (int)min((int64_t)C, n_end - n0);
            if (!(ok = wait_phase(bar(SB_X0 + i % nx), (i / nx) & 1, abort))) break;
            float *rd_ = red + (i & 1) * 2 * C;
            rd_[h * C + t] = half_sumsq<D>(base + Ly.x + (i % nx) * Ly.stg, t, h);
            if (!(ok = group_sync(bar(SB_CS), i & 1, abort))) break;
            const float ssq = rd_[t] + rd_[C + t];
            const float inv = ssq > 0.f ? rsqrtf(ssq) : 0.f;
            if (!(ok = wait_phase(bar(SB_P0 + s), (i >> 1) & 1, abort))) break;
            fence_after();
            float z[LPP];
            {
                uint32_t a[32];
                ld32_nw(tlane + zcol + LPP * s, a);
                wait_ld();
                reg_fence(a);
#pragma unroll
                for (int k = 0; k < LPP; ++k) z[k] = uf(a[k]);
            }
            // the feature buffer (and mass operand) of this tile were last read by an earlier product
            if (nf == 2 && i >= 2) {
                if (!(ok = wait_phase(bar(SB_S0 + s), ((i - 2) >> 1) & 1, abort))) break;
            } else if (nf == 1 && i >= 1) {
                if (!(ok = wait_phase(bar(SB_S0 + (s ^ 1)), ((i - 1) >> 1) & 1, abort))) break;
            }
            if (mode == 1 && nf == 1 && i >= 2) {  // mass buffer s was read by the product of tile i - 2
                if (!(ok = wait_phase(bar(SB_S0 + s), ((i - 2) >> 1) & 1, abort))) break;
            }
            const bool live = t < cnt;
            float scale = live ? 1.f : 0.f;
            if (mode == 1) {
                float2 a = make_float2(0.f, 0.f);
                if (live) a = aux[bh * Dm.N + n0 + t];
                scale *= a.x;
                if (h == 0) {
                    const float mcv = -a.y;
                    const bf16 mhi = __float2bfloat16_rn(mcv);
                    const bf16 mlo = __float2bfloat16_rn(mcv - __bfloat162float(mhi));
                    unsigned char *mt = sm + Ly.mass + (i & 1) * 4096 + (t >> 6) * 2048;
                    *reinterpret_cast<bf16 *>(mt + sw_elem(0, t & 63)) = mhi;
                    *reinterpret_cast<bf16 *>(mt + sw_elem(1, t & 63)) = mlo;
                }
            }
            bf16 *grow = (frows != nullptr && live) ? frows + (bh * Dm.N + n0 + t) * feature_row_stride(Dm.LR) : nullptr;
            if (grow != nullptr && h == 0) invrows[bh * Dm.N + n0 + t] = inv;
            write_features<P>(z, inv, Dm.beta, LT > 0 ? LT : Dm.L, h, scale, t, base + Ly.f + (i % nf) * Ly.fbytes,
                              grow);
            warp_signal(bar(SB_F0 + s));
        }
        if (ok && ntile > 0) ok = wait_phase(bar(SB_DONE), 0, abort);
        float *out = part + ((int64_t)bh * nsplit + split) * Dm.LR * (D + 1);
        if (ok) {
            fence_after();
            // epilogue: sketch row lr = 128 m + t of block m; the two halves split the columns
            for (int m = 0; m < (ntile > 0 ? nmb : 0); ++m) {
                const int lr = 128 * m + t;
                const uint32_t acc = tlane + m * 256;
#pragma unroll
                for (int cc = 0; cc < D / 64; ++cc) {
                    const int c0 = h * (D / 2) + 32 * cc;
                    uint32_t v[32];
                    ld32_nw(acc + c0, v);
                    wait_ld();
                    reg_fence(v);
                    if (lr < Dm.LR) {
#pragma unroll
                        for (int k = 0; k < 32; ++k) out[(int64_t)lr * (D + 1) + c0 + k] = uf(v[k]);
                    }
                }
                if (h == 1) {
                    uint32_t m0, m1;
                    ld1_nw(acc + D, m0);
                    ld1_nw(acc + D + 1, m1);
                    wait_ld();
                    reg_fence1(m0);
                    reg_fence1(m1);
                    if (lr < Dm.LR) out[(int64_t)lr * (D + 1) + D] = mode == 1 ? uf(m0) + uf(m1) : uf(m0);
                }
            }
            if (ntile == 0)  // an empty range contributes a zero partial (its accumulator was never written)
                for (int e = tid; e < Dm.LR * (D + 1); e += NTH) out[e] = 0.f;
        }
    }
    fence_before();
    __syncthreads();
    if (warp == 0) {
        fence_after();
        tmem_dealloc(tmem, ncols);
    }
}

// ------------------------------------------------------------------ read-out

struct ReadoutLayout {
    uint32_t stg, x, f, shi, slo, whi, wlo, red, bar, slot, bytes, sblk;
    int fb;
    bool split;
    __host__ __device__ ReadoutLayout(int D, int LR, bool want_split)
    {
        const uint32_t KB = D / 64;
        fb = (LR + 63) / 64;
        sblk = (uint32_t)(D + 16) * 128;
        stg = KB * BLK;
        x = 0;
        f = 2 * stg;
        shi = f + fb * BLK;
        split = want_split;
        slo = shi + fb * sblk;
        whi = slo + (split ? fb * sblk : 0);
        wlo = whi + KB * WBLK;
        red = wlo + KB * WBLK;
        bar = red + 2 * C * 4;
        slot = bar + 32;
        bytes = slot + 16;
    }
};

__host__ __device__ inline uint32_t readout_zcol(int D) { return (D + 16 + 31) & ~31; }
__host__ __device__ inline uint32_t readout_tmem_cols(int D) { return readout_zcol(D) + LPP <= 128 ? 128 : 256; }

// O = Phi_Q [A | B] content / mass for the CTA's tiles.  S: combined sketch [BH][LR][d + 1].
template <int D, int P, int LT>
__global__ void __launch_bounds__(NTH, 1)
    k_readout5(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmO, Dims Dm,
               const float *__restrict__ W, const float *__restrict__ S, int64_t seg_len, int split_s,
               unsigned *__restrict__ err)
{
    constexpr int KB = D / 64;
    constexpr int NS = D + 16;  // sketch operand rows: d content rows, the mass row, zero rows
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023) & ~1023u;
    unsigned char *sm = smem_raw + (base - raw);
    const ReadoutLayout Ly(D, Dm.LR, split_s != 0);
    float *red = reinterpret_cast<float *>(sm + Ly.red);
    const uint32_t bar_load = base + Ly.bar, bar_proj = bar_load + 16, bar_o = bar_load + 24;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, q4 = warp & 3, h = warp >> 2;
    const int t = 32 * q4 + lane;
    const int64_t bh = blockIdx.y;
    const int64_t n_begin = (int64_t)blockIdx.x * seg_len;
    const int64_t n_end = min(Dm.N, n_begin + seg_len);
    const int ntile = n_end > n_begin ? (int)((n_end - n_begin + C - 1) / C) : 0;
    const uint32_t zcol = readout_zcol(D), ncols = readout_tmem_cols(D);
    const int ksteps = (Dm.LR + 15) / 16;

    // ---- set-up: sketch operand (K-major B: row n = output column, 64-column blocks of lr)
    if (warp == 0) tmem_alloc(base + Ly.slot, ncols);
    zero_region(sm + Ly.f, Ly.fb * BLK);
    load_w_tiles<D>(head_w(W, Dm, bh), Dm.LP, sm + Ly.whi, sm + Ly.wlo);
    {
        const float *Sb = S + bh * Dm.LR * (D + 1);
        const int nchunk = Ly.fb * 8;  // 8-lr chunks per operand row
        for (int i = tid; i < NS * nchunk; i += NTH) {
            const int c = i / NS, n = i - c * NS;  // consecutive threads: consecutive rows n
            uint32_t hw[4], lw[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                float v[2];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int k = 8 * c + 2 * j + e;
                    v[e] = (n <= D && k < Dm.LR) ? Sb[(int64_t)k * (D + 1) + n] : 0.f;
                }
                const bf16 h0 = __float2bfloat16_rn(v[0]), h1 = __float2bfloat16_rn(v[1]);
                hw[j] = bfp::pack_bf16(__bfloat162float(h0), __bfloat162float(h1));
                lw[j] = bfp::pack_bf16(v[0] - __bfloat162float(h0), v[1] - __bfloat162float(h1));
            }
            const uint32_t off = (c >> 3) * Ly.sblk + sw_chunk(n, c & 7);
            st_shared_v4(base + Ly.shi + off, hw[0], hw[1], hw[2], hw[3]);
            if (Ly.split) st_shared_v4(base + Ly.slo + off, lw[0], lw[1], lw[2], lw[3]);
        }
    }
    if (tid == 0) {
        mbar_init(bar_load, 1);
        mbar_init(bar_load + 8, 1);
        mbar_init(bar_proj, 1);
        mbar_init(bar_o, 1);
        tc::fence_mbar_init();
        prefetch_tmap(&tmQ);
        prefetch_tmap(&tmO);
    }
    tc::fence_proxy_async();
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(sm + Ly.slot);
    const uint32_t tlane = tmem + ((uint32_t)(32 * q4) << 16);

    auto issue_load = [&](int i) {
        const int s = i & 1;
        const uint32_t xs = base + Ly.x + s * Ly.stg;
        mbar_arrive_expect_tx(bar_load + 8 * s, KB * BLK);
#pragma unroll
        for (int kb = 0; kb < KB; ++kb)
            tma_load(xs + kb * BLK, &tmQ, 64 * kb, (int)(n_begin + (int64_t)i * C), (int)bh, bar_load + 8 * s);
    };
    if (tid == 0) {
        if (ntile > 0) issue_load(0);
        if (ntile > 1) issue_load(1);
    }

    bool failed = false;
    int i = 0;
    for (; i < ntile; ++i) {
        const int s = i & 1;
        const int64_t n0 = n_begin + (int64_t)i * C;
        const int cnt = (int)min((int64_t)C, n_end - n0);
        const uint32_t xs = base + Ly.x + s * Ly.stg;
        if (wait_all(bar_load + 8 * s, (i >> 1) & 1)) {
            failed = true;
            break;
        }
        if (tid == 0) {
            fence_after();
            issue_projection<D>(tmem + zcol, xs, base + Ly.whi, base + Ly.wlo);
            commit(bar_proj);
        }
        red[h * C + t] = half_sumsq<D>(xs, t, h);
        if (wait_all(bar_proj, i & 1)) {
            failed = true;
            break;
        }
        fence_after();
        float z[LPP];
        {
            float a[32];
            ld32(tlane + zcol, a);
#pragma unroll
            for (int k = 0; k < LPP; ++k) z[k] = a[k];
        }
        const float ssq = red[t] + red[C + t];
        const float inv = ssq > 0.f ? rsqrtf(ssq) : 0.f;
        write_features<P>(z, inv, Dm.beta, LT > 0 ? LT : Dm.L, h, t < cnt ? 1.f : 0.f, t, base + Ly.f);
        tc::fence_proxy_async();
        fence_before();
        __syncthreads();
        if (warp == 0) {  // the run-time K loop issues from the converged warp (one elected lane)
            fence_after();
            constexpr uint32_t id_o = idesc_bf16(128, NS, 0, 0);
            for (int ks = 0; ks < ksteps; ++ks) {
                const uint32_t fo = (ks >> 2) * BLK + (ks & 3) * 32, so = (ks >> 2) * Ly.sblk + (ks & 3) * 32;
                umma_w(tmem, desc_k(base + Ly.f + fo), desc_k(base + Ly.shi + so), id_o, ks > 0);
                if (Ly.split) umma_w(tmem, desc_k(base + Ly.f + fo), desc_k(base + Ly.slo + so), id_o, true);
            }
            commit_w(bar_o);
            // the other stage was last read by tile i - 1's output store: let that finish, then refill
            if (lane == 0 && i >= 1 && i + 1 < ntile) {
                bulk_wait_read0();
                issue_load(i + 1);
            }
            __syncwarp();
        }
        if (wait_all(bar_o, i & 1)) {
            failed = true;
            break;
        }
        fence_after();
        // epilogue: O row t = num / den, bf16, staged in this tile's (consumed) Q stage
        {
            float v[16];
            ld16(tlane + D, v);
            const float rd = __frcp_rn(v[0]);
            if (h == 0 && t < cnt) flag_den(v[0], err);
#pragma unroll
            for (int cc = 0; cc < D / 32; ++cc) {
                const int c0 = h * (D / 2) + 16 * cc;
                ld16(tlane + c0, v);
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const int ch = (c0 >> 3) + j;
                    st_shared_v4(xs + (ch >> 3) * BLK + sw_chunk(t, ch & 7),
                                 bfp::pack_bf16(v[8 * j] * rd, v[8 * j + 1] * rd),
                                 bfp::pack_bf16(v[8 * j + 2] * rd, v[8 * j + 3] * rd),
                                 bfp::pack_bf16(v[8 * j + 4] * rd, v[8 * j + 5] * rd),
                                 bfp::pack_bf16(v[8 * j + 6] * rd, v[8 * j + 7] * rd));
                }
            }
        }
        tc::fence_proxy_async();
        fence_before();
        __syncthreads();
        if (tid == 0) {
#pragma unroll
            for (int kb = 0; kb < KB; ++kb) tma_store(&tmO, 64 * kb, (int)n0, (int)bh, xs + kb * BLK);
            bulk_commit();
        }
    }
    if (failed) {
        if (tid == 0) atomicOr(err, kErrTimeout);
        if (i < ntile) mbar_wait(bar_load + 8 * (i & 1), (i >> 1) & 1);
        if (i + 1 < ntile) mbar_wait(bar_load + 8 * ((i + 1) & 1), ((i + 1) >> 1) & 1);
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

namespace {

using EncodeTiled = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                 const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled encoder()
{
    static EncodeTiled fn = [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            p = nullptr;
        return reinterpret_cast<EncodeTiled>(p);
    }();
    return fn;
}

}  // namespace

// [BH][N][d] bf16 token tensor as a 3-D TMA map with 64 x 128 boxes and 128-byte swizzle; rows
// past N read as zero and are dropped on store.
cudaError_t make_token_map(CUtensorMap *map, const void *base, const Dims &D)
{
    EncodeTiled enc = encoder();
    if (!enc) return cudaErrorNotSupported;
    const cuuint64_t dims[3] = {(cuuint64_t)D.d, (cuuint64_t)D.N, (cuuint64_t)D.BH};
    const cuuint64_t strides[2] = {(cuuint64_t)D.d * 2, (cuuint64_t)D.N * D.d * 2};
    const cuuint32_t box[3] = {64, (cuuint32_t)nc5::C, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box,
                           estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

bool nc5_supported(const Dims &D)
{
    return (D.d == 64 || D.d == 128) && D.P >= 1 && D.P <= 6 && D.LP <= nc5::LPP && D.LR <= 256 &&
           D.N <= 0x7FFFFFFF && D.BH <= 0x7FFFFFFF;
}

int nc5_tile() { return nc5::C; }

int nc5_sketch_ctas_per_sm(const Dims &D)
{
    const nc5::SketchLayout Ly(D.d, D.LR);
    const int by_smem = (int)((228 * 1024) / (Ly.bytes + 1024 + 1024));
    const int by_tmem = 512 / (int)nc5::sketch_tmem_cols(D.d, Ly.nmb);
    return std::max(1, std::min(2, std::min(by_smem, by_tmem)));
}

namespace {

template <typename K>
cudaError_t prep_smem(K kern, size_t bytes)
{
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

template <int D, int P, int LT>
cudaError_t sketch_launch(const Dims &Dm, const CUtensorMap &mx, const CUtensorMap &my, const float *W,
                          const float2 *aux, int64_t seg_len, int nsplit, float *part, bf16_t *frows, float *invrows,
                          unsigned *err, int mode, cudaStream_t st)
{
    const nc5::SketchLayout Ly(D, Dm.LR);
    const size_t smem = Ly.bytes + 1024;
    auto kern = nc5::k_sketch5<D, P, LT>;
    cudaError_t e = prep_smem(kern, smem);
    if (e != cudaSuccess) return e;
    return launch_kernel(mode ? "tc5_sketch_grad" : "tc5_sketch_keys", kern, dim3(nsplit, (unsigned)Dm.BH),
                         dim3(nc5::NTHW), smem, st, mx, my, Dm, W, aux, seg_len, nsplit, part, frows, invrows, err,
                         mode);
}

// The named workloads' shapes run with L compiled in: (d, P, L) = (128, 3, 3), (64, 3, 3), (128, 6, 4).
template <int D, int P>
cudaError_t sketch_inst(const Dims &Dm, const CUtensorMap &mx, const CUtensorMap &my, const float *W,
                        const float2 *aux, int64_t seg_len, int nsplit, float *part, bf16_t *frows, float *invrows,
                        unsigned *err, int mode, cudaStream_t st)
{
    if constexpr (P == 3)
        if (Dm.L == 3)
            return sketch_launch<D, P, 3>(Dm, mx, my, W, aux, seg_len, nsplit, part, frows, invrows, err, mode, st);
    if constexpr (D == 128 && P == 6)
        if (Dm.L == 4)
            return sketch_launch<D, P, 4>(Dm, mx, my, W, aux, seg_len, nsplit, part, frows, invrows, err, mode, st);
    return sketch_launch<D, P, 0>(Dm, mx, my, W, aux, seg_len, nsplit, part, frows, invrows, err, mode, st);
}

template <int D, int P, int LT>
cudaError_t readout_launch(const Dims &Dm, const CUtensorMap &mq, const CUtensorMap &mo, const float *W,
                           const float *S, unsigned *err, cudaStream_t st)
{
    const nc5::ReadoutLayout with_lo(D, Dm.LR, true);
    const bool split = with_lo.bytes + 1024 <= 227 * 1024;
    const nc5::ReadoutLayout Ly(D, Dm.LR, split);
    const size_t smem = Ly.bytes + 1024;
    auto kern = nc5::k_readout5<D, P, LT>;
    cudaError_t e = prep_smem(kern, smem);
    if (e != cudaSuccess) return e;
    const int per_sm = std::max<int>(1, std::min<int>(2, (int)((227 * 1024) / smem)));
    const int64_t ntiles = (Dm.N + nc5::C - 1) / nc5::C;
    int64_t want = std::max<int64_t>(1, ((int64_t)Dm.sms * per_sm + Dm.BH - 1) / Dm.BH);
    want = std::min(want, ntiles);
    const int64_t seg = ((ntiles + want - 1) / want) * nc5::C;
    const int64_t nseg = (Dm.N + seg - 1) / seg;
    return launch_kernel("tc5_readout", kern, dim3((unsigned)nseg, (unsigned)Dm.BH), dim3(nc5::NTH), smem, st, mq,
                         mo, Dm, W, S, seg, (int)split, err);
}

// The named non-causal workloads' shapes run with L compiled in: (d, P, L) = (64, 3, 3), (128, 6, 4).
template <int D, int P>
cudaError_t readout_inst(const Dims &Dm, const CUtensorMap &mq, const CUtensorMap &mo, const float *W,
                         const float *S, unsigned *err, cudaStream_t st)
{
    if constexpr (D == 64 && P == 3)
        if (Dm.L == 3) return readout_launch<D, P, 3>(Dm, mq, mo, W, S, err, st);
    if constexpr (D == 128 && P == 6)
        if (Dm.L == 4) return readout_launch<D, P, 4>(Dm, mq, mo, W, S, err, st);
    return readout_launch<D, P, 0>(Dm, mq, mo, W, S, err, st);
}

#define RACE_NC5_DISPATCH(FN, ...)                               \
    switch (Dm.d * 16 + Dm.P) {                                  \
        case 64 * 16 + 1: return FN<64, 1>(__VA_ARGS__);         \
        case 64 * 16 + 2: return FN<64, 2>(__VA_ARGS__);         \
        case 64 * 16 + 3: return FN<64, 3>(__VA_ARGS__);         \
        case 64 * 16 + 4: return FN<64, 4>(__VA_ARGS__);         \
        case 64 * 16 + 5: return FN<64, 5>(__VA_ARGS__);         \
        case 64 * 16 + 6: return FN<64, 6>(__VA_ARGS__);         \
        case 128 * 16 + 1: return FN<128, 1>(__VA_ARGS__);       \
        case 128 * 16 + 2: return FN<128, 2>(__VA_ARGS__);       \
        case 128 * 16 + 3: return FN<128, 3>(__VA_ARGS__);       \
        case 128 * 16 + 4: return FN<128, 4>(__VA_ARGS__);       \
        case 128 * 16 + 5: return FN<128, 5>(__VA_ARGS__);       \
        case 128 * 16 + 6: return FN<128, 6>(__VA_ARGS__);       \
        default: return cudaErrorInvalidValue;                   \
    }

}  // namespace

cudaError_t launch_nc5_sketch(const Dims &Dm, const bf16_t *X, const bf16_t *Y, const float2 *aux, const float *W,
                              int64_t seg_len, int nsplit, float *part, unsigned *err, cudaStream_t st,
                              bf16_t *frows, float *invrows)
{
    CUtensorMap mx, my;
    cudaError_t e = make_token_map(&mx, X, Dm);
    if (e == cudaSuccess) e = make_token_map(&my, Y, Dm);
    if (e != cudaSuccess) return e;
    const int mode = aux ? 1 : 0;
    if ((frows == nullptr) != (invrows == nullptr)) return cudaErrorInvalidValue;
    RACE_NC5_DISPATCH(sketch_inst, Dm, mx, my, W, aux, seg_len, nsplit, part, frows, invrows, err, mode, st)
}

cudaError_t launch_nc5_readout(const Dims &Dm, const bf16_t *Q, const float *W, const float *S, bf16_t *O,
                               unsigned *err, cudaStream_t st)
{
    CUtensorMap mq, mo;
    cudaError_t e = make_token_map(&mq, Q, Dm);
    if (e == cudaSuccess) e = make_token_map(&mo, O, Dm);
    if (e != cudaSuccess) return e;
    RACE_NC5_DISPATCH(readout_inst, Dm, mq, mo, W, S, err, st)
}

}  // namespace race
