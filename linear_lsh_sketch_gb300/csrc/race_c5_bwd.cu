// race_c5_bwd.cu -- tcgen05 (TMEM accumulator) causal RACE attention backward, key side, bf16.
//
// The chain rule through Algorithm 2 ("RACE Attention" slides, frame "Causality is a prefix
// update of the same statistics"; the pages print no backward).  With den_t, c_t = dO_t . O_t
// (from the query-side pass) and F'_Q = phi(Q_t) / den_t, the gradient sketch of every token at
// or after j is G_j = [G_A | G_B] = sum_{t >= j} F'_Q(t)^T [dO_t | -c_t].  Then
//
//   dV_j        = G_j,A^T phi(K_j)
//   dphi_K(j)   = G_j,A V_j + G_j,B
//
// In chunks of C = 128 tokens walked in reverse, with G_next the sketch of every later token:
//   dV      = F_K G_next,A  +  mask_{t >= j}(F_K F'_Q^T) dO
//   dphi_K  = V G_next,A^T + G_next,B  +  mask_{t >= j}(V dO^T - 1 c^T) F'_Q
//   G_next += F'_Q^T [dO | -c]
// followed by the key-side feature Jacobian (softmax over corners, tanh, projection, row
// normalisation).  All products run on tcgen05 with fp32 accumulators in TMEM; F_K and both
// masked matrices are written to TMEM by the CUDA cores and used as A operands; F'_Q stays in one
// swizzled shared tile that serves as B operand (K- and MN-major) and as A operand; the carried
// G_next is converted each chunk to a bf16 hi + lo shared operand.
//
// Nothing of the features is recomputed here: the query-side pass writes F'_Q (L R bf16 per
// token), and the forward's segment-sum pass stored phi(K) and 1 / |k| for every key; this pass
// reads those rows.  K is still read, for its projection (the Jacobian's u = tanh(W k / |k|)) and
// for dK.  The gradient-sketch update of a chunk is issued right after its first product group,
// so it runs, and its bf16 operand copy is made, while the masks are applied.
// Roles: warp 8 issues every TMA copy and MMA; warps 0-3 copy the F'_Q and phi(K) rows into
// their tile and TMEM, write dV and convert G; warps 4-7 take u from the projection, run the
// Jacobian and write dK.  Hand-offs use mbarriers; dK and dV rows go straight from registers to
// global memory.
#include "race_launch.h"
#include "race_nc5_common.cuh"

namespace race {
namespace c5b {

using namespace race::nc5;

constexpr int NTHW = NTH + 32;

// TMEM columns (512 allocated) for sketch widths L R <= LRM (32, or 64 when d = 64).
// With L R <= 32 (PACK) the G operand's hi and lo halves share one shared-memory block, V G^T is
// one N = 64 product per K step (dphi_K's hi part, plus M2 F'_Q^T, in columns 0..31 of DP, its
// lo part in 32..63), and dz takes DP's first 16 columns once the Jacobian has read them.
template <int D, int LRM>
struct KvCols {
    static constexpr bool PACK = LRM == 32;
    static constexpr uint32_t SC = 0;          // F_K F'_Q^T, then P2 as bf16 pairs (in place, per half)
    static constexpr uint32_t DV = 128;        // V dO^T, then M2 as bf16 pairs (in place), then dxhat
    static constexpr uint32_t DVV = 256;       // dV (d columns)
    static constexpr uint32_t ZK = 288;        // K-row projections, 32 columns (dead before dV is written)
    static constexpr uint32_t DP = DVV + D;    // dphi_K (LRM columns; 64 with PACK)
    static constexpr uint32_t FK = DP + (PACK ? 64 : LRM);  // F_K as bf16 pairs (A operand), LRM / 2 columns
    static constexpr uint32_t DZ = PACK ? DP : FK + LRM / 2;  // dz as bf16 pairs (A operand), 16 columns
    static constexpr uint32_t GT = PACK ? FK + LRM / 2 : DZ + 16;  // G^T (lanes = d), LRM columns
    static constexpr uint32_t GB = GT + LRM;   // G_B (lanes = sketch row), 16 columns (0 and 1 used)
    static_assert(GB + 16 <= 512 && ZK + 32 <= DVV + D, "key-side TMEM budget");
};
constexpr uint32_t T_COLS = 512;

enum : uint32_t { B_Q, B_K, B_V, B_DO, B_PROJ, B_A, B_B, B_C, B_FEAT, B_MASK, B_JAC, B_GOP, B_DVR, B_CS1, B_CS2, B_G,
                  B_COUNT };

// Staging of one chunk's rows, copied in a chunk ahead: F'_Q and phi(K) (2 LRM-byte slots), c
// and 1 / |k| (4 bytes each); z of the K rows keeps LP <= LPZ rows (L P <= 16 whenever L R <= 32).
template <int LRM>
struct KvStage {
    static constexpr uint32_t SLOT = 2 * LRM;
    static constexpr uint32_t FQ = 0, FK = C * SLOT, CV = 2 * C * SLOT, KI = CV + C * 4, BYTES = KI + C * 4;
    static constexpr int LPZ = LRM == 64 ? 32 : 16;
};

struct BwdLayout {
    uint32_t stage, k, v, dO, fq, ghi, glo, whi, wlo, ncm, gb, cvec, zk, bar, slot, bytes, kbb;
    __host__ __device__ BwdLayout(int D, int LRM)
    {
        const uint32_t stg = (uint32_t)C * (4 * LRM + 8);
        const uint32_t lpz = LRM == 64 ? 32 : 16;
        kbb = (uint32_t)(D / 64) * BLK;
        stage = 0;  // two staging buffers
        k = stage + 2 * stg;
        v = k + kbb;
        dO = v + kbb;
        fq = dO + kbb;  // F'_Q [t][lr], one 64-column block
        ghi = fq + BLK;
        glo = ghi + BLK;  // G operand [d rows][lr], hi and lo blocks (L R <= 32: lo in ghi's columns 32..63)
        whi = glo + BLK;  // W in pair layout (hi and lo blocks interleaved); wlo = its first lo block
        wlo = whi + WBLK;
        ncm = whi + 2 * (uint32_t)(D / 64) * WBLK;  // -c as a K-major N = 16 operand (rows 0, 1 = hi, lo)
        gb = ncm + 4096;                         // G_B fp32 [2 parities][LRM]
        cvec = gb + 8 * LRM;                     // c_t fp32 [C]
        zk = cvec + 4 * C;   // z = W x of the K rows, fp32 [lpz][C]
        bar = zk + 4 * lpz * C;
        slot = bar + 128;
        bytes = slot + 16;
    }
};

// DB: also the CTA's key-side d(loss)/d(beta) partial to dbpart[bh][blockIdx.x].  LRM: the
// widest L R the instance supports (32, or 64 when d = 64).
template <int D, int P, int LT, int LRM, bool DB>
__global__ void __launch_bounds__(NTHW, 1)
    k_causal_bwdkv5(const bf16 *__restrict__ fq_in, const bf16 *__restrict__ fk_in, const float *__restrict__ kinv_in,
                    const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO, Dims Dm,
                    const float *__restrict__ W, const float2 *__restrict__ aux, const float *__restrict__ G0,
                    int64_t seg_len, int nseg, bf16 *__restrict__ dK, bf16 *__restrict__ dV,
                    unsigned *__restrict__ err, float *__restrict__ dbpart)
{
    constexpr int KB = D / 64;
    constexpr int R = 1 << P;
    constexpr int LMAX = LPP / P;
    constexpr int LRMAX = LRM;  // sketch rows this instance supports
    using Cols = KvCols<D, LRM>;
    // the K projection as one N = 64 product (hi and lo parts side by side, inside dV's columns)
    constexpr bool MERGE_PROJ = D == 128 && LRM == 32;
    static_assert(!MERGE_PROJ || KvCols<D, LRM>::ZK + 2 * LPP <= KvCols<D, LRM>::DVV + D, "projection inside dV");
    constexpr uint32_t T_SC = Cols::SC, T_DV = Cols::DV, T_DVV = Cols::DVV, T_ZK = Cols::ZK, T_DP = Cols::DP;
    constexpr uint32_t T_FK = Cols::FK, T_DZ = Cols::DZ, T_GT = Cols::GT, T_GB = Cols::GB;
    using Stg = KvStage<LRM>;
    constexpr uint32_t STG_FQ = Stg::FQ, STG_FK = Stg::FK, STG_C = Stg::CV, STG_KI = Stg::KI, STG = Stg::BYTES;
    constexpr uint32_t SLOT = Stg::SLOT;
    constexpr int LPZ = Stg::LPZ;
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023) & ~1023u;
    unsigned char *sm = smem_raw + (base - raw);
    const BwdLayout Ly(D, LRM);
    auto bar = [&](uint32_t i) { return base + Ly.bar + 8 * i; };
    volatile int *abort = reinterpret_cast<volatile int *>(sm + Ly.slot + 8);
    float *gb = reinterpret_cast<float *>(sm + Ly.gb);
    float *cvec = reinterpret_cast<float *>(sm + Ly.cvec);
    float *zk_s = reinterpret_cast<float *>(sm + Ly.zk);
    const bool wide = ((reinterpret_cast<uintptr_t>(dK) | reinterpret_cast<uintptr_t>(dV)) & 31) == 0;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, q4 = warp & 3, h = (warp >> 2) & 1;
    const bool compute = warp < 8;
    const int t = 32 * q4 + lane;
    const int s = blockIdx.x;
    const int64_t bh = blockIdx.y;
    const int64_t n_begin = (int64_t)s * seg_len;
    const int64_t n_end = min(Dm.N, n_begin + seg_len);
    const int nchunk = n_end > n_begin ? (int)((n_end - n_begin + C - 1) / C) : 0;
    // LT > 0: the table count is a compile-time constant, so the per-table loops unroll without
    // run-time guards and the tables' independent chains interleave
    const int L = LT > 0 ? LT : Dm.L;
    const int LR = LT > 0 ? LT * (1 << P) : Dm.LR;
    const int LP = L * P;
    const float beta = Dm.beta;
    const int64_t off = bh * Dm.N * D;

    // ---- set-up
    if (warp == 0) tmem_alloc(base + Ly.slot, T_COLS);
    if (compute) {
        zero_region(sm + Ly.fq, BLK);
        zero_region(sm + Ly.ghi, 2 * BLK);
        init_mass_tile(sm + Ly.ncm, false);
        load_w_pair<D>(head_w(W, Dm, bh), Dm.LP, sm + Ly.whi);
    }
    if (tid == NTH) {
        for (uint32_t i = 0; i < B_COUNT; ++i) {
            uint32_t cnt = 1;
            if (i == B_FEAT || i == B_MASK) cnt = 8;
            if (i == B_JAC || i == B_GOP || i == B_DVR) cnt = 4;
            if (i == B_CS1 || i == B_CS2) cnt = NTH;
            mbar_init(bar(i), cnt);
        }
        *abort = 0;
        tc::fence_mbar_init();
        prefetch_tmap(&tmK);
        prefetch_tmap(&tmV);
        prefetch_tmap(&tmdO);
    }
    tc::fence_proxy_async();
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(sm + Ly.slot);
    const uint32_t tlane = tmem + ((uint32_t)(32 * q4) << 16);

    // gradient sketch of every token after the segment -> TMEM (G^T lanes = d, G_B lanes = row);
    // the F_K and dz operand columns past L R and L P stay zero
    if (compute) {
        const float *Gb = G0 + ((int64_t)bh * nseg + s) * LR * (D + 1);
        if (h == 0) {
            if (t < D) {
                for (int c0 = 0; c0 < LRMAX; c0 += 8) {
                    uint32_t r[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j) r[j] = __float_as_uint(c0 + j < LR ? Gb[(c0 + j) * (D + 1) + t] : 0.f);
                    stn<8>(tlane + T_GT + c0, r);
                }
            }
            const uint32_t m[2] = {__float_as_uint(t < LR ? Gb[t * (D + 1) + D] : 0.f), 0u};
            stn<2>(tlane + T_GB, m);
        } else {
            const uint32_t zr[8] = {0, 0, 0, 0, 0, 0, 0, 0};
            // T_FK (and T_DZ after it when it has columns of its own)
            for (int c0 = 0; c0 < LRMAX / 2 + (Cols::PACK ? 0 : 16); c0 += 8) stn<8>(tlane + T_FK + c0, zr);
        }
        wait_st();
    }
    fence_before();
    __syncthreads();
    fence_after();

    // G (TMEM) -> bf16 hi / lo operand rows d (columns = sketch rows, 32 at a time) and fp32 G_B
    // (buffer par_out, read by the Jacobian of the chunk that uses this G); warps 0-3
    auto convert_g = [&](int par_out) {
        if constexpr (LRMAX == 32) {
            uint32_t ar[32], gb0 = 0, gb1 = 0;
            if (t < D) ld32_nw(tlane + T_GT, ar);
            if (q4 == 0) {
                ld1_nw(tlane + T_GB, gb0);
                ld1_nw(tlane + T_GB + 1, gb1);
            }
            wait_ld();
            reg_fence(ar);
            reg_fence1(gb0);
            reg_fence1(gb1);
            if (t < D) {
                float a[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) a[j] = uf(ar[j]);
                uint32_t hw[16], lw[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const float x0 = 2 * j < LR ? a[2 * j] : 0.f, x1 = 2 * j + 1 < LR ? a[2 * j + 1] : 0.f;
                    const bf16 h0 = __float2bfloat16_rn(x0), h1 = __float2bfloat16_rn(x1);
                    hw[j] = bfp::pack_bf16(__bfloat162float(h0), __bfloat162float(h1));
                    lw[j] = bfp::pack_bf16(x0 - __bfloat162float(h0), x1 - __bfloat162float(h1));
                }
#pragma unroll
                for (int c = 0; c < 4; ++c) {  // hi in columns 0..31, lo in 32..63 of one block
                    st_shared_v4(base + Ly.ghi + sw_chunk(t, c), hw[4 * c], hw[4 * c + 1], hw[4 * c + 2], hw[4 * c + 3]);
                    st_shared_v4(base + Ly.ghi + sw_chunk(t, 4 + c), lw[4 * c], lw[4 * c + 1], lw[4 * c + 2], lw[4 * c + 3]);
                }
            }
            if (q4 == 0) gb[32 * par_out + lane] = lane < LR ? uf(gb0) + uf(gb1) : 0.f;  // -sum F'_Q c, c as hi + lo
        } else {
#pragma unroll
            for (int half = 0; half < LRMAX / 32; ++half) {
                uint32_t ar[32];
                if (t < D) ld32_nw(tlane + T_GT + 32 * half, ar);
                wait_ld();
                reg_fence(ar);
                if (t < D) {
                    uint32_t hw[16], lw[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int c0 = 32 * half + 2 * j;
                        const float x0 = c0 < LR ? uf(ar[2 * j]) : 0.f, x1 = c0 + 1 < LR ? uf(ar[2 * j + 1]) : 0.f;
                        const bf16 h0 = __float2bfloat16_rn(x0), h1 = __float2bfloat16_rn(x1);
                        hw[j] = bfp::pack_bf16(__bfloat162float(h0), __bfloat162float(h1));
                        lw[j] = bfp::pack_bf16(x0 - __bfloat162float(h0), x1 - __bfloat162float(h1));
                    }
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const int ch = 4 * half + c;
                        st_shared_v4(base + Ly.ghi + sw_chunk(t, ch), hw[4 * c], hw[4 * c + 1], hw[4 * c + 2], hw[4 * c + 3]);
                        st_shared_v4(base + Ly.glo + sw_chunk(t, ch), lw[4 * c], lw[4 * c + 1], lw[4 * c + 2], lw[4 * c + 3]);
                    }
                }
            }
            if (32 * q4 < LRMAX) {  // lane = sketch row: -sum F'_Q c, c as bf16 hi + lo
                uint32_t gb0 = 0, gb1 = 0;
                ld1_nw(tlane + T_GB, gb0);
                ld1_nw(tlane + T_GB + 1, gb1);
                wait_ld();
                reg_fence1(gb0);
                reg_fence1(gb1);
                gb[LRMAX * par_out + t] = t < LR ? uf(gb0) + uf(gb1) : 0.f;
            }
        }
    };

    float db = 0.f;  // this thread's d(loss)/d(beta) share (DB only)
    if (!compute) {
        // ---------------------------------------------------------------- control warp
        if (lane == 0) {
            auto load_tiles = [&](int k, uint32_t which) {  // which: 2 = V  4 = dO  8 = K
                const int c = nchunk - 1 - k;
                const int y = (int)(n_begin + (int64_t)c * C);
                if (which & 8) {
                    mbar_arrive_expect_tx(bar(B_K), KB * BLK);
#pragma unroll
                    for (int kb = 0; kb < KB; ++kb) tma_load(base + Ly.k + kb * BLK, &tmK, 64 * kb, y, (int)bh, bar(B_K));
                }
                if (which & 2) {
                    mbar_arrive_expect_tx(bar(B_V), KB * BLK);
#pragma unroll
                    for (int kb = 0; kb < KB; ++kb) tma_load(base + Ly.v + kb * BLK, &tmV, 64 * kb, y, (int)bh, bar(B_V));
                }
                if (which & 4) {
                    mbar_arrive_expect_tx(bar(B_DO), KB * BLK);
#pragma unroll
                    for (int kb = 0; kb < KB; ++kb)
                        tma_load(base + Ly.dO + kb * BLK, &tmdO, 64 * kb, y, (int)bh, bar(B_DO));
                }
            };
            int issued[4] = {0, 0, 0, 0}, done[4] = {0, 0, 0, 0};  // -, V, dO, K loads issued / waited for
            if (nchunk > 0) {
                load_tiles(0, 14);
                issued[1] = issued[2] = issued[3] = 1;
            }
            constexpr uint32_t id_sc = idesc_bf16(128, 128, 0, 0);
            constexpr uint32_t id_dvo = idesc_bf16(128, 128, 0, 0);
            constexpr uint32_t id_dp = idesc_bf16(128, LRMAX, 0, 1);
            constexpr uint32_t id_dp64 = idesc_bf16(128, 64, 0, 1);
            constexpr uint32_t id_dv = idesc_bf16(128, D, 0, 0);
            constexpr uint32_t id_pdo = idesc_bf16(128, D, 0, 1);
            constexpr uint32_t id_mf = idesc_bf16(128, LRMAX, 0, 1);
            constexpr uint32_t id_x = idesc_bf16(128, D, 0, 1);
            constexpr uint32_t id_gt = idesc_bf16(128, LRMAX, 1, 1);
            constexpr uint32_t id_gb = idesc_bf16(128, 16, 1, 0);
            // MN-major A operands with M = 128 read a second 64-column block at start + LBO: for
            // F'_Q (sketch rows 64..127) and for dO^T at d = 64 (rows d 64..127) that block only feeds
            // accumulator lanes nobody reads, so it points at the next whole 16 KB tile
            const uint64_t d_fq_k = desc_k(base + Ly.fq), d_fq_mn = desc_mn(base + Ly.fq, BLK);
            // PACK: the lo half of G starts 64 bytes into the rows of the hi half's block
            const uint64_t d_ghi_k = desc_k(base + Ly.ghi),
                           d_glo_k = Cols::PACK ? desc_k(base + Ly.ghi) + (64 >> 4) : desc_k(base + Ly.glo);
            const uint64_t d_ghi_mn = desc_mn(base + Ly.ghi, BLK), d_glo_mn = desc_mn(base + Ly.glo, BLK);
            const uint64_t d_v_k = desc_k(base + Ly.v), d_do_k = desc_k(base + Ly.dO);
            const uint64_t d_do_mn = desc_mn(base + Ly.dO, BLK);
            const uint64_t d_do_mt = desc_mn(base + Ly.dO, BLK);
            const uint64_t d_ncm = desc_k(base + Ly.ncm);
            const uint64_t d_whi = desc_mn(base + Ly.whi, 2 * WBLK), d_wlo = desc_mn(base + Ly.wlo, 2 * WBLK);
            bool ok = true;
            for (int k = 0; k < nchunk && ok; ++k) {
                const uint32_t par = k & 1;
                if (!(ok = wait_phase(bar(B_K), par, abort))) break;
                ++done[3];
                // the projection reuses TMEM columns of the previous chunk's dV
                if (k >= 1 && !(ok = wait_phase(bar(B_DVR), (k - 1) & 1, abort))) break;
                fence_after();
                issue_projection_pair<D, MERGE_PROJ>(tmem + T_ZK, base + Ly.k, base + Ly.whi);
                commit(bar(B_PROJ));
                // group A once the features and the previous chunk's G operand are in
                if (!(ok = wait_phase(bar(B_FEAT), par, abort))) break;
                if (!(ok = wait_phase(bar(B_GOP), par, abort))) break;
                if (!(ok = wait_phase(bar(B_V), par, abort))) break;
                ++done[1];
                if (!(ok = wait_phase(bar(B_DO), par, abort))) break;
                ++done[2];
                fence_after();
                for (int ks = 0; ks < LRMAX / 16; ++ks)
                    umma_ts(tmem + T_SC, tmem + T_FK + 8 * ks, d_fq_k + (uint64_t)(2 * ks), id_sc, ks > 0);
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint64_t ko = (uint64_t)((ks >> 2) * BLK + (ks & 3) * 32) >> 4;
                    umma(tmem + T_DV, d_v_k + ko, d_do_k + ko, id_dvo, ks > 0);
                    if constexpr (Cols::PACK) {  // G hi and lo as one N = 64 operand
                        umma(tmem + T_DP, d_v_k + ko, d_ghi_mn + (uint64_t)(ks * 128), id_dp64, ks > 0);
                    } else {
                        umma(tmem + T_DP, d_v_k + ko, d_ghi_mn + (uint64_t)(ks * 128), id_dp, ks > 0);
                        umma(tmem + T_DP, d_v_k + ko, d_glo_mn + (uint64_t)(ks * 128), id_dp, true);
                    }
                }
                for (int ks = 0; ks < LRMAX / 16; ++ks) {
                    umma_ts(tmem + T_DVV, tmem + T_FK + 8 * ks, d_ghi_k + (uint64_t)(2 * ks), id_dv, ks > 0);
                    umma_ts(tmem + T_DVV, tmem + T_FK + 8 * ks, d_glo_k + (uint64_t)(2 * ks), id_dv, true);
                }
                commit(bar(B_A));
                // the gradient sketch G += F'_Q^T [dO | -c] of this chunk (under its own commit: the G
                // conversion waits for it while the masks are applied)
#pragma unroll
                for (int ks = 0; ks < C / 16; ++ks) {
                    const uint64_t ko = (uint64_t)(ks * 2048) >> 4, kk = (uint64_t)((ks >> 2) * 2048 + (ks & 3) * 32) >> 4;
                    umma(tmem + T_GT, d_do_mt + ko, d_fq_mn + ko, id_gt, true);
                    umma(tmem + T_GB, d_fq_mn + ko, d_ncm + kk, id_gb, true);
                }
                commit(bar(B_G));
                // group B: masked products
                if (!(ok = wait_phase(bar(B_MASK), par, abort))) break;
                fence_after();
#pragma unroll
                for (int ks = 0; ks < C / 16; ++ks) {
                    const uint32_t ac = (ks < 4 ? 8 * ks : 64 + 8 * (ks - 4));  // in-place bf16 columns
                    umma_ts(tmem + T_DVV, tmem + T_SC + ac, d_do_mn + (uint64_t)(ks * 128), id_pdo, true);
                    umma_ts(tmem + T_DP, tmem + T_DV + ac, d_fq_mn + (uint64_t)(ks * 128), id_mf, true);
                }
                commit(bar(B_B));
                if (k + 1 < nchunk) {  // group A (the only reader of V) completed before the mask
                    load_tiles(k + 1, 2);
                    ++issued[1];
                    // dO is last read by group B
                    if (!(ok = wait_phase(bar(B_B), par, abort))) break;
                    load_tiles(k + 1, 4);
                    ++issued[2];
                }
                // group C: dxhat, for the dK epilogue
                if (!(ok = wait_phase(bar(B_JAC), par, abort))) break;
                fence_after();
                if (k + 1 < nchunk) {  // the K rows are parked in TMEM by now
                    load_tiles(k + 1, 8);
                    ++issued[3];
                }
                for (int ks = 0; ks < LPP / 16; ++ks) {
                    umma_ts(tmem + T_DV, tmem + T_DZ + 8 * ks, d_whi + (uint64_t)(ks * 128), id_x, ks > 0);
                    umma_ts(tmem + T_DV, tmem + T_DZ + 8 * ks, d_wlo + (uint64_t)(ks * 128), id_x, true);
                }
                commit(bar(B_C));
            }
            if (!ok) {
                atomicOr(err, kErrTimeout);
                *abort = 1;
                const uint32_t bars[4] = {0u, bar(B_V), bar(B_DO), bar(B_K)};
#pragma unroll
                for (int b = 1; b < 4; ++b)
                    if (issued[b] > done[b]) mbar_wait(bars[b], done[b] & 1);
            }
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------------------- compute warps
        if (h == 0) {
            convert_g(0);
            warp_signal(bar(B_GOP));
        }
        // Row data of chunk kk (in reverse order), copied into staging buffer kk & 1 a chunk ahead by
        // the thread that consumes it: F'_Q, phi(K) and c of row t (warps 0-3), 1 / |k| (warps 4-7).
        // Chunks run backwards and only the last one can be partial.
        const int lrs = feature_row_stride(LR);
        const bf16 *fq_bh = fq_in + bh * Dm.N * lrs;
        const bf16 *fk_bh = fk_in + bh * Dm.N * lrs;
        const float *c_bh = reinterpret_cast<const float *>(aux + bh * Dm.N) + 1;  // .y of each {1/den, c}
        const float *kinv_bh = kinv_in + bh * Dm.N;
        auto stage_rows = [&](int kk) {
            const int64_t row = n_begin + (int64_t)(nchunk - 1 - kk) * C + t;
            const uint32_t buf = base + Ly.stage + (uint32_t)(kk & 1) * STG;
            if (row < n_end) {
                if (h == 0) {
#pragma unroll
                    for (int ch = 0; ch < LRMAX / 8; ++ch) {
                        if (8 * ch < lrs) {
                            cp_async16(buf + STG_FQ + t * SLOT + 16 * ch, fq_bh + row * lrs + 8 * ch);
                            cp_async16(buf + STG_FK + t * SLOT + 16 * ch, fk_bh + row * lrs + 8 * ch);
                        }
                    }
                    cp_async4(buf + STG_C + t * 4, c_bh + 2 * row);
                } else {
                    cp_async4(buf + STG_KI + t * 4, kinv_bh + row);
                }
            }
            cp_async_commit();
        };
        if (nchunk > 0) stage_rows(0);
        for (int k = 0; k < nchunk; ++k) {
            const uint32_t par = k & 1;
            const int c = nchunk - 1 - k;
            const int64_t n0 = n_begin + (int64_t)c * C;
            const int cnt = (int)min((int64_t)C, n_end - n0);
            const bool live = t < cnt;
            const uint32_t buf = base + Ly.stage + par * STG;
            float inv = 0.f;  // 1 / |K row| (warps 4-7)
            // K rows keep z in shared memory; with L compiled in they also keep u = tanh(z inv) in
            // registers (L P of them), otherwise the Jacobian recomputes it from z
            float uk[LT > 0 ? LPZ : 1];
            cp_async_wait_all();
            if (h == 0) {
                // F'_Q row t -> shared tile row t and phi(K) row t -> TMEM (zero past the end);
                // -c_t -> rows 0 / 1 of the mass operand; then the next chunk's rows
                if constexpr (LRMAX == 32) {
                    uint32_t fk0[8], fk1[8];  // phi(K) row t as bf16 pairs
#pragma unroll
                    for (int ch = 0; ch < 4; ++ch) {
                        uint4 v = make_uint4(0u, 0u, 0u, 0u), w = make_uint4(0u, 0u, 0u, 0u);
                        if (8 * ch < lrs && live) {
                            v = ld_shared_v4(buf + STG_FQ + t * SLOT + 16 * ch);
                            w = ld_shared_v4(buf + STG_FK + t * SLOT + 16 * ch);
                        }
                        if (8 * ch < lrs) st_shared_v4(base + Ly.fq + sw_chunk(t, ch), v.x, v.y, v.z, v.w);
                        uint32_t *dst = ch < 2 ? fk0 + 4 * ch : fk1 + 4 * (ch - 2);
                        dst[0] = w.x;
                        dst[1] = w.y;
                        dst[2] = w.z;
                        dst[3] = w.w;
                    }
                    stn<8>(tlane + T_FK, fk0);
                    stn<8>(tlane + T_FK + 8, fk1);
                } else
#pragma unroll
                for (int g = 0; g < LRMAX / 16; ++g) {  // 16 features (8 TMEM columns) at a time
                    uint32_t fk[8];  // phi(K) row t as bf16 pairs
#pragma unroll
                    for (int hc = 0; hc < 2; ++hc) {
                        const int ch = 2 * g + hc;
                        uint4 v = make_uint4(0u, 0u, 0u, 0u), w = make_uint4(0u, 0u, 0u, 0u);
                        if (8 * ch < lrs && live) {
                            v = ld_shared_v4(buf + STG_FQ + t * SLOT + 16 * ch);
                            w = ld_shared_v4(buf + STG_FK + t * SLOT + 16 * ch);
                        }
                        if (8 * ch < lrs) st_shared_v4(base + Ly.fq + sw_chunk(t, ch), v.x, v.y, v.z, v.w);
                        fk[4 * hc] = w.x;
                        fk[4 * hc + 1] = w.y;
                        fk[4 * hc + 2] = w.z;
                        fk[4 * hc + 3] = w.w;
                    }
                    stn<8>(tlane + T_FK + 8 * g, fk);
                }
                const float cv = live ? reinterpret_cast<const float *>(sm + Ly.stage + par * STG + STG_C)[t] : 0.f;
                if (k + 1 < nchunk) stage_rows(k + 1);
                const float mcv = -cv;
                const bf16 mhi = __float2bfloat16_rn(mcv);
                const bf16 mlo = __float2bfloat16_rn(mcv - __bfloat162float(mhi));
                unsigned char *mt = sm + Ly.ncm + (t >> 6) * 2048;
                *reinterpret_cast<bf16 *>(mt + sw_elem(0, t & 63)) = mhi;
                *reinterpret_cast<bf16 *>(mt + sw_elem(1, t & 63)) = mlo;
                cvec[t] = cv;
                wait_st();
            } else {
                // this thread's K row: 1 / |k| as stored, z = W k from the projection, u = tanh(z / |k|)
                inv = live ? reinterpret_cast<const float *>(sm + Ly.stage + par * STG + STG_KI)[t] : 0.f;
                if (k + 1 < nchunk) stage_rows(k + 1);
                if (!wait_phase(bar(B_PROJ), par, abort)) break;
                fence_after();
                float z[LPZ];
                {
                    float a[LPZ];
                    ld_cols<LPZ>(tlane + T_ZK, a);
#pragma unroll
                    for (int j = 0; j < LPZ; ++j) z[j] = a[j];
                    if constexpr (MERGE_PROJ) {  // + the lo hyperplanes' part
                        ld_cols<LPZ>(tlane + T_ZK + LPP, a);
#pragma unroll
                        for (int j = 0; j < LPZ; ++j) z[j] += a[j];
                    }
                }
#pragma unroll
                for (int j = 0; j < LPZ; ++j) {
                    if (j < LP) zk_s[j * C + t] = z[j];
                    if constexpr (LT > 0) uk[j] = j < LP ? tc::tanh_abs(z[j] * inv) : 0.f;
                }
            }
            if (!group_sync(bar(B_CS1), par, abort)) break;  // c_t visible to every compute warp
            warp_signal(bar(B_FEAT));
            // masks over this half's 64 query columns t': P2 = (F_K F'_Q^T)[j][t'] and
            // M2 = (V dO^T)[j][t'] - c_t' for t' >= j (j = this thread's row), written in place
            if (!wait_phase(bar(B_A), par, abort)) break;
            fence_after();
            {
                const int j0 = 64 * h;
#pragma unroll
                for (int pass = 0; pass < 2; ++pass) {
                    const int tb = j0 + 32 * pass;
                    uint32_t sa[32], sd[32];
                    const bool need = tb + 31 >= 32 * q4;  // warp-uniform: some lane keeps a column
                    if (need) {
                        ld32_nw(tlane + T_SC + tb, sa);
                        ld32_nw(tlane + T_DV + tb, sd);
                    }
                    wait_ld();
                    reg_fence(sa);
                    reg_fence(sd);
#pragma unroll
                    for (int b = 0; b < 2; ++b) {
                        uint32_t pw[8], mw[8];
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            const int e = 16 * b + 2 * j, q0 = tb + e;
                            const bool k0 = need && q0 >= t, k1 = need && q0 + 1 >= t;
                            pw[j] = bfp::pack_bf16(k0 ? uf(sa[e]) : 0.f, k1 ? uf(sa[e + 1]) : 0.f);
                            mw[j] = bfp::pack_bf16(k0 ? uf(sd[e]) - cvec[q0] : 0.f, k1 ? uf(sd[e + 1]) - cvec[q0 + 1] : 0.f);
                        }
                        // bf16 pairs of this half's 64 columns go to its own first 32 columns
                        stn<8>(tlane + T_SC + j0 + 16 * pass + 8 * b, pw);
                        stn<8>(tlane + T_DV + j0 + 16 * pass + 8 * b, mw);
                    }
                }
            }
            wait_st();
            warp_signal(bar(B_MASK));
            if (h == 0) {
                // the gradient sketch with this chunk added -> the next chunk's bf16 operand and G_B
                // (its update was issued right after group A and ran during the masks)
                if (!wait_phase(bar(B_G), par, abort)) break;
                fence_after();
                convert_g(par ^ 1);
                warp_signal(bar(B_GOP));
            }
            if (!wait_phase(bar(B_B), par, abort)) break;
            fence_after();
            float zdz = 0.f;  // x . dxhat of the K row
            if (h == 1) {
                // park the K row in TMEM (the score columns are free once group B is done) so that
                // the K tile can take the next chunk
#pragma unroll
                for (int j = 0; j < D / 8; j += 2) {
                    const uint4 w0 = ld_shared_v4(base + Ly.k + (j >> 3) * BLK + sw_chunk(t, j & 7));
                    const uint4 w1 = ld_shared_v4(base + Ly.k + ((j + 1) >> 3) * BLK + sw_chunk(t, (j + 1) & 7));
                    const uint32_t r[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
                    stn<8>(tlane + T_SC + 4 * j, r);
                }
                // key-side Jacobian: dphi_K + G_B -> dz (bf16 pairs in TMEM)
                float dph[LRMAX == 32 ? 32 : 1];
                if constexpr (LRMAX == 32) {  // dphi_K's hi part (with M2 F'_Q^T) + its lo part + G_B
                    float a[32];
                    ld32(tlane + T_DP, a);
#pragma unroll
                    for (int j = 0; j < 32; ++j) dph[j] = a[j] + gb[LRMAX * par + j];
                    ld32(tlane + T_DP + 32, a);
#pragma unroll
                    for (int j = 0; j < 32; ++j) dph[j] += a[j];
                }
                float dz[LPP];
#pragma unroll
                for (int j = 0; j < LPP; ++j) dz[j] = 0.f;
#pragma unroll
                for (int l = 0; l < LMAX; ++l) {
                    if (l < L && l * R < LRMAX) {
                        float u[P], ph[R], dp[R];
#pragma unroll
                        for (int p = 0; p < P; ++p)
                            u[p] = LT > 0 ? uk[(l * P + p) % (LT > 0 ? LPZ : 1)] : tc::tanh_abs(zk_s[(l * P + p) * C + t] * inv);
                        tc::bucket_probs<P>(u, beta, ph);
                        if constexpr (LRMAX == 32) {
#pragma unroll
                            for (int r = 0; r < R; ++r) dp[r] = l * R + r < LRMAX ? dph[(l * R + r) % 32] : 0.f;
                        } else {  // this table's R columns only (wider sketches keep one table in registers)
                            ld_cols<R>(tlane + T_DP + l * R, dp);
#pragma unroll
                            for (int r = 0; r < R; ++r) dp[r] += gb[LRMAX * par + l * R + r];
                        }
                        float tmp[P];
                        table_backward<P, DB>(u, ph, dp, beta, tmp, &db);
#pragma unroll
                        for (int p = 0; p < P; ++p) dz[l * P + p] = tmp[p];
                    }
                }
                uint32_t r[8];
#pragma unroll
                for (int b = 0; b < 2; ++b) {
#pragma unroll
                    for (int j = 0; j < 8; ++j) r[j] = bfp::pack_bf16(dz[16 * b + 2 * j], dz[16 * b + 2 * j + 1]);
                    stn<8>(tlane + T_DZ + 8 * b, r);
                }
                // dxhat = W^T dz (dz rounded to bf16 as the product sees it), so x . dxhat = z . dz
#pragma unroll
                for (int j = 0; j < LMAX * P; ++j)
                    if (j < LP) zdz = fmaf(__bfloat162float(__float2bfloat16_rn(dz[j])), zk_s[j * C + t], zdz);
                wait_st();
                warp_signal(bar(B_JAC));
                if (Dm.dzk != nullptr && live) {  // d(loss)/d(W): this K row's dz / |k| (zeros past L P)
                    float4 *o = reinterpret_cast<float4 *>(Dm.dzk + (bh * Dm.N + n0 + t) * Dm.dzld);
#pragma unroll
                    for (int q = 0; q < LPP / 4; ++q)
                        if (4 * q < Dm.dzld)
                            o[q] = make_float4(dz[4 * q] * inv, dz[4 * q + 1] * inv, dz[4 * q + 2] * inv, dz[4 * q + 3] * inv);
                }
            } else {
                // dV row t = F_K G_A + P2 dO, straight to global memory
                bf16 *dst = dV + off + (n0 + t) * D;
#pragma unroll
                for (int pass = 0; pass < D / 32; ++pass) {
                    uint32_t v[32];
                    ld32_nw(tlane + T_DVV + 32 * pass, v);
                    wait_ld();
                    reg_fence(v);
                    uint32_t o[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j) o[j] = bfp::pack_bf16(uf(v[2 * j]), uf(v[2 * j + 1]));
                    if (live) store_row32(dst + 32 * pass, o, wide);
                }
                fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(B_DVR));  // dV columns (shared with z) read
            }
            if (h == 1) {
                // dK row t = inv (dxhat - x inv^2 (x . dxhat)), x parked in TMEM; straight to global memory
                if (!wait_phase(bar(B_C), par, abort)) break;
                fence_after();
                const float kk = inv * inv * zdz;
                bf16 *dst = dK + off + (n0 + t) * D;
#pragma unroll
                for (int pass = 0; pass < D / 32; ++pass) {
                    uint32_t v[32], xr[16];
                    ld32_nw(tlane + T_DV + 32 * pass, v);
                    ld16_nw(tlane + T_SC + 16 * pass, xr);
                    wait_ld();
                    reg_fence(v);
                    reg_fence(xr);
                    uint32_t o[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        o[j] = bfp::pack_bf16(inv * (uf(v[2 * j]) - bf_lo(xr[j]) * kk), inv * (uf(v[2 * j + 1]) - bf_hi(xr[j]) * kk));
                    if (live) store_row32(dst + 32 * pass, o, wide);
                }
            }
            fence_before();
            if (!group_sync(bar(B_CS2), par, abort)) break;  // gb / TMEM reads done before the next chunk
        }
    }
    cp_async_wait_all();  // no copy into the staging buffers outlives the CTA (after an abort)
    if constexpr (DB) {  // this CTA's d(loss)/d(beta) partial, summed in a fixed order
        const float sdb = block_sum_fixed(db, cvec);
        if (tid == 0) dbpart[bh * gridDim.x + blockIdx.x] = sdb;
    }
    fence_before();
    __syncthreads();
    if (warp == 0) {
        fence_after();
        tmem_dealloc(tmem, T_COLS);
    }
}

}  // namespace c5b

// ------------------------------------------------------------------ query side (forward order)
//
// With S_t the inclusive prefix sketch [A | B], B_t its mass row and g_t = A_t dO_t:
//   den_t = phi(Q_t) . B_t,   c_t = phi(Q_t) . g_t / den_t,   dphi_Q(t) = (g_t - B_t c_t) / den_t
// In chunks of C = 128 tokens walked forward, with S_prev the sketch of every earlier token:
//   g   = dO A_prev^T + mask_{j <= t}(dO V^T) F_K
//   B_t = B_prev + (tril 1) F_K
// then the query-side feature Jacobian gives dQ; the pass also writes {1 / den_t, c_t} per token
// and the segment's gradient-sketch sum G = sum_t F'_Q(t)^T [dO_t | -c_t] for the key side, and
// carries S (A^T += V^T F_K, B += F_K^T 1) in TMEM.
// The keys' features F_K come from the rows the forward's segment-sum pass stored (L R bf16 per
// token), not from K.
// Roles: warp 8 issues TMA and MMA; warps 0-3 own the Q rows (x kept in TMEM, den, c, the
// Jacobian, dQ); warps 4-7 copy the F_K rows into their tile and convert S to its bf16 operand
// copy.

namespace c5q {

using namespace race::nc5;

constexpr int NTHW = NTH + 32;

// TMEM columns (512 allocated) for sketch widths L R <= LRM (32, or 64 when d = 64); with LRM = 64
// the lower-triangular ones operand moves to shared memory.
template <int D, int LRM>
struct QCols {
    static constexpr bool TRIL_TMEM = LRM == 32;
    static constexpr uint32_t ZQ = 0;                        // projections of the Q tile, 32 columns
    // g: L R <= 32 takes dO S^T with the hi and lo halves of S as one N = 64 product, so g's
    // columns 0..31 hold the hi part (plus M1 F_K) and 32..63 the lo part; L R <= 64, L R columns
    static constexpr uint32_t G = LRM == 32 ? 32 : 160;
    static constexpr uint32_t DV = LRM == 32 ? 96 : 32;      // dO V^T, then M1 as bf16 pairs (in place), then dxhat
    static constexpr uint32_t BT = DV + 128 > G + 64 ? DV + 128 : G + 64;  // (tril 1) F_K
    static constexpr uint32_t TRIL = BT + LRM;               // lower-triangular ones as bf16 pairs (A operand), 64 columns
    static constexpr uint32_t DZ = TRIL_TMEM ? TRIL + 64 : TRIL;  // dz as bf16 pairs (A operand), 16 columns
    static constexpr uint32_t ST = DZ + 16;                  // A^T (lanes = d)
    static constexpr uint32_t MS = ST + LRM;                 // B (lanes = sketch row), column 0
    static constexpr uint32_t GT = MS + 16;                  // G^T (lanes = d)
    static constexpr uint32_t GB = GT + LRM;                 // G_B (lanes = sketch row), columns 0 + 1 (c split hi / lo)
    static constexpr uint32_t X = GB + 16;                   // the Q row as stored (bf16 pairs), D / 2 columns
    static_assert(X + D / 2 <= 512, "query-side TMEM budget");
};
constexpr uint32_t T_COLS = 512;

enum : uint32_t { B_QK, B_V, B_DO, B_PROJ, B_A, B_B, B_C, B_FEAT, B_MASK, B_JAC, B_SOP, B_CS, B_G, B_COUNT };

constexpr uint32_t STG_FK = C * 128;  // one staging buffer of F_K rows (128-byte slots)

struct QLayout {
    uint32_t q, stage, v, dO, fk, fq, shi, slo, whi, wlo, ncm, ones, tril, bprev, invq, red, bar, slot, bytes, kbb;
    __host__ __device__ QLayout(int D, int LRM)
    {
        kbb = (uint32_t)(D / 64) * BLK;
        q = 0;
        stage = q + kbb;  // two F_K staging buffers
        v = stage + 2 * STG_FK;
        dO = v + kbb;
        fk = dO + kbb;   // F_K [j][lr]
        fq = fk + BLK;   // F'_Q [t][lr]
        shi = fq + BLK;  // S operand [d rows][lr] (MN-major B of dO A^T)
        slo = shi + BLK;  // (L R <= 32: S lo sits in shi's columns 32..63 and this block is unused)
        whi = slo + BLK;  // W in pair layout (hi and lo blocks interleaved); wlo = its first lo block
        wlo = whi + WBLK;
        ncm = whi + 2 * (uint32_t)(D / 64) * WBLK;
        ones = ncm + 4096;
        tril = ones + 4096;   // LRM = 64: lower-triangular ones, K-major [t][j] in two 64-column blocks
        bprev = tril + (LRM == 64 ? 2 * BLK : 0);  // B_prev fp32 [2 parities][LRM]
        invq = bprev + 8 * LRM;   // 1 / |Q row| fp32 [C]
        red = invq + 4 * C;   // inv^2 (x . dxhat) of the Q rows, fp32 [C]
        bar = red + 4 * C;
        slot = bar + 128;
        bytes = slot + 16;
    }
};

// DB: also the CTA's query-side d(loss)/d(beta) partial to dbpart[bh][blockIdx.x].  LRM: the
// widest L R the instance supports (32, or 64 when d = 64).
template <int D, int P, int LT, int LRM, bool DB>
__global__ void __launch_bounds__(NTHW, 1)
    k_causal_bwdq5(const __grid_constant__ CUtensorMap tmQ, const bf16 *__restrict__ fk_in,
                   const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO, Dims Dm,
                   const float *__restrict__ W, const float *__restrict__ S0, int64_t seg_len, int nseg,
                   bf16 *__restrict__ dQ, float2 *__restrict__ aux, bf16 *__restrict__ fq_out,
                   float *__restrict__ Gseg, unsigned *__restrict__ err, float *__restrict__ dbpart)
{
    constexpr int KB = D / 64;
    constexpr int R = 1 << P;
    constexpr int LMAX = LPP / P;
    constexpr int LRMAX = LRM;
    using Cols = QCols<D, LRM>;
    // the Q projection as one N = 64 product: the lo part lands in g's columns, free until group A
    constexpr bool MERGE_PROJ = LRM == 32;
    static_assert(!MERGE_PROJ || QCols<D, LRM>::G == QCols<D, LRM>::ZQ + LPP, "lo projection in g's columns");
    constexpr uint32_t T_ZQ = Cols::ZQ, T_DV = Cols::DV, T_G = Cols::G, T_BT = Cols::BT, T_TRIL = Cols::TRIL;
    constexpr uint32_t T_DZ = Cols::DZ, T_ST = Cols::ST, T_MS = Cols::MS, T_GT = Cols::GT, T_GB = Cols::GB;
    constexpr uint32_t T_X = Cols::X;
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023) & ~1023u;
    unsigned char *sm = smem_raw + (base - raw);
    const QLayout Ly(D, LRM);
    auto bar = [&](uint32_t i) { return base + Ly.bar + 8 * i; };
    volatile int *abort = reinterpret_cast<volatile int *>(sm + Ly.slot + 8);
    float *bprev = reinterpret_cast<float *>(sm + Ly.bprev);
    float *invq_s = reinterpret_cast<float *>(sm + Ly.invq);
    float *red = reinterpret_cast<float *>(sm + Ly.red);
    const bool wide = (reinterpret_cast<uintptr_t>(dQ) & 31) == 0;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, q4 = warp & 3, h = (warp >> 2) & 1;
    const bool compute = warp < 8;
    const int t = 32 * q4 + lane;
    const int s = blockIdx.x;
    const int64_t bh = blockIdx.y;
    const int64_t n_begin = (int64_t)s * seg_len;
    const int64_t n_end = min(Dm.N, n_begin + seg_len);
    const int nchunk = n_end > n_begin ? (int)((n_end - n_begin + C - 1) / C) : 0;
    // LT > 0: the table count is a compile-time constant, so the per-table loops unroll without
    // run-time guards and the tables' independent chains interleave
    const int L = LT > 0 ? LT : Dm.L;
    const int LR = LT > 0 ? LT * (1 << P) : Dm.LR;
    const int LP = L * P;
    const float beta = Dm.beta;
    const int64_t off = bh * Dm.N * D;

    // ---- set-up
    if (warp == 0) tmem_alloc(base + Ly.slot, T_COLS);
    if (compute) {
        zero_region(sm + Ly.fk, 4 * BLK);  // F_K, F'_Q, S hi, S lo
        init_mass_tile(sm + Ly.ncm, false);
        init_mass_tile(sm + Ly.ones, true);
        load_w_pair<D>(head_w(W, Dm, bh), Dm.LP, sm + Ly.whi);
    }
    if (tid == NTH) {
        for (uint32_t i = 0; i < B_COUNT; ++i) {
            uint32_t cnt = 1;
            if (i == B_FEAT || i == B_MASK) cnt = 8;
            if (i == B_JAC || i == B_SOP) cnt = 4;
            if (i == B_CS) cnt = NTH;
            mbar_init(bar(i), cnt);
        }
        *abort = 0;
        tc::fence_mbar_init();
        prefetch_tmap(&tmQ);
        prefetch_tmap(&tmV);
        prefetch_tmap(&tmdO);
    }
    tc::fence_proxy_async();
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(sm + Ly.slot);
    const uint32_t tlane = tmem + ((uint32_t)(32 * q4) << 16);

    // sketch at the segment start, zero gradient sketch, and the lower-triangular ones operand
    if (compute) {
        const uint32_t zr[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        if (h == 0) {
            const float *Sb = S0 + ((int64_t)bh * nseg + s) * LR * (D + 1);
            for (int c0 = 0; c0 < LRMAX; c0 += 8) {
                uint32_t r[8];
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    r[j] = __float_as_uint((t < D && c0 + j < LR) ? Sb[(c0 + j) * (D + 1) + t] : 0.f);
                stn<8>(tlane + T_ST + c0, r);
                stn<8>(tlane + T_GT + c0, zr);
            }
            const uint32_t m[2] = {__float_as_uint(t < LR ? Sb[t * (D + 1) + D] : 0.f), 0u};
            stn<2>(tlane + T_MS, m);
            stn<8>(tlane + T_GB, zr);
        }
        // tril[t][j] = 1 for j <= t: half h writes the columns of keys 64 h .. 64 h + 63
        if constexpr (Cols::TRIL_TMEM) {
            for (int c0 = 32 * h; c0 < 32 * h + 32; c0 += 8) {
                uint32_t r[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int k0 = 2 * (c0 + j);
                    r[j] = (k0 <= t ? 0x3F80u : 0u) | (k0 + 1 <= t ? 0x3F800000u : 0u);
                }
                stn<8>(tlane + T_TRIL + c0, r);
            }
        } else {
            for (int ch = 0; ch < 8; ++ch) {
                uint32_t r[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int k0 = 64 * h + 8 * ch + 2 * j;
                    r[j] = (k0 <= t ? 0x3F80u : 0u) | (k0 + 1 <= t ? 0x3F800000u : 0u);
                }
                st_shared_v4(base + Ly.tril + h * BLK + sw_chunk(t, ch), r[0], r[1], r[2], r[3]);
            }
        }
        wait_st();
    }
    fence_before();
    __syncthreads();
    fence_after();

    // S (TMEM) -> bf16 hi / lo operand rows d (32 sketch columns at a time) and fp32 B_prev;
    // warps 4-7
    auto convert_s = [&](int par_out) {
        if constexpr (LRMAX == 32) {
            uint32_t ar[32], mv = 0;
            if (t < D) ld32_nw(tlane + T_ST, ar);
            if (q4 == 0) ld1_nw(tlane + T_MS, mv);
            wait_ld();
            reg_fence(ar);
            reg_fence1(mv);
            if (t < D) {
                float a[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) a[j] = uf(ar[j]);
                uint32_t hw[16], lw[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const float x0 = 2 * j < LR ? a[2 * j] : 0.f, x1 = 2 * j + 1 < LR ? a[2 * j + 1] : 0.f;
                    const bf16 h0 = __float2bfloat16_rn(x0), h1 = __float2bfloat16_rn(x1);
                    hw[j] = bfp::pack_bf16(__bfloat162float(h0), __bfloat162float(h1));
                    lw[j] = bfp::pack_bf16(x0 - __bfloat162float(h0), x1 - __bfloat162float(h1));
                }
#pragma unroll
                for (int c = 0; c < 4; ++c) {  // hi in columns 0..31, lo in 32..63 of one block
                    st_shared_v4(base + Ly.shi + sw_chunk(t, c), hw[4 * c], hw[4 * c + 1], hw[4 * c + 2], hw[4 * c + 3]);
                    st_shared_v4(base + Ly.shi + sw_chunk(t, 4 + c), lw[4 * c], lw[4 * c + 1], lw[4 * c + 2], lw[4 * c + 3]);
                }
            }
            if (q4 == 0) bprev[32 * par_out + lane] = lane < LR ? uf(mv) : 0.f;
        } else {
#pragma unroll
            for (int half = 0; half < LRMAX / 32; ++half) {
                uint32_t ar[32];
                if (t < D) ld32_nw(tlane + T_ST + 32 * half, ar);
                wait_ld();
                reg_fence(ar);
                if (t < D) {
                    uint32_t hw[16], lw[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int c0 = 32 * half + 2 * j;
                        const float x0 = c0 < LR ? uf(ar[2 * j]) : 0.f, x1 = c0 + 1 < LR ? uf(ar[2 * j + 1]) : 0.f;
                        const bf16 h0 = __float2bfloat16_rn(x0), h1 = __float2bfloat16_rn(x1);
                        hw[j] = bfp::pack_bf16(__bfloat162float(h0), __bfloat162float(h1));
                        lw[j] = bfp::pack_bf16(x0 - __bfloat162float(h0), x1 - __bfloat162float(h1));
                    }
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const int ch = 4 * half + c;
                        st_shared_v4(base + Ly.shi + sw_chunk(t, ch), hw[4 * c], hw[4 * c + 1], hw[4 * c + 2], hw[4 * c + 3]);
                        st_shared_v4(base + Ly.slo + sw_chunk(t, ch), lw[4 * c], lw[4 * c + 1], lw[4 * c + 2], lw[4 * c + 3]);
                    }
                }
            }
            if (32 * q4 < LRMAX) {  // lane = sketch row
                uint32_t mv = 0;
                ld1_nw(tlane + T_MS, mv);
                wait_ld();
                reg_fence1(mv);
                bprev[LRMAX * par_out + t] = t < LR ? uf(mv) : 0.f;
            }
        }
    };

    float db = 0.f;  // this thread's d(loss)/d(beta) share (DB only)
    if (!compute) {
        // ---------------------------------------------------------------- control warp
        if (lane == 0) {
            auto load_tiles = [&](int c, uint32_t which) {  // which: 1 = Q  2 = V  4 = dO
                const int y = (int)(n_begin + (int64_t)c * C);
                if (which & 1) {
                    mbar_arrive_expect_tx(bar(B_QK), KB * BLK);
#pragma unroll
                    for (int kb = 0; kb < KB; ++kb) tma_load(base + Ly.q + kb * BLK, &tmQ, 64 * kb, y, (int)bh, bar(B_QK));
                }
                if (which & 2) {
                    mbar_arrive_expect_tx(bar(B_V), KB * BLK);
#pragma unroll
                    for (int kb = 0; kb < KB; ++kb) tma_load(base + Ly.v + kb * BLK, &tmV, 64 * kb, y, (int)bh, bar(B_V));
                }
                if (which & 4) {
                    mbar_arrive_expect_tx(bar(B_DO), KB * BLK);
#pragma unroll
                    for (int kb = 0; kb < KB; ++kb)
                        tma_load(base + Ly.dO + kb * BLK, &tmdO, 64 * kb, y, (int)bh, bar(B_DO));
                }
            };
            int issued[3] = {0, 0, 0}, done[3] = {0, 0, 0};
            if (nchunk > 0) {
                load_tiles(0, 7);
                issued[0] = issued[1] = issued[2] = 1;
            }
            constexpr uint32_t id_dv = idesc_bf16(128, 128, 0, 0);
            constexpr uint32_t id_g1 = idesc_bf16(128, LRMAX, 0, 1);
            constexpr uint32_t id_g64 = idesc_bf16(128, 64, 0, 1);
            constexpr uint32_t id_bt = idesc_bf16(128, LRMAX, 0, 1);
            constexpr uint32_t id_x = idesc_bf16(128, D, 0, 1);
            constexpr uint32_t id_gt = idesc_bf16(128, LRMAX, 1, 1);
            constexpr uint32_t id_m16 = idesc_bf16(128, 16, 1, 0);
            // MN-major A operands with M = 128 read a second 64-column block at start + BLK; beyond
            // d (d = 64) or beyond the sketch rows it feeds accumulator lanes nobody reads
            const uint64_t d_v_k = desc_k(base + Ly.v), d_do_k = desc_k(base + Ly.dO);
            const uint64_t d_v_mt = desc_mn(base + Ly.v, BLK), d_do_mt = desc_mn(base + Ly.dO, BLK);
            const uint64_t d_fk_mn = desc_mn(base + Ly.fk, BLK), d_fq_mn = desc_mn(base + Ly.fq, BLK);
            const uint64_t d_shi = desc_mn(base + Ly.shi, BLK), d_slo = desc_mn(base + Ly.slo, BLK);
            const uint64_t d_ncm = desc_k(base + Ly.ncm), d_ones = desc_k(base + Ly.ones);
            const uint64_t d_whi = desc_mn(base + Ly.whi, 2 * WBLK), d_wlo = desc_mn(base + Ly.wlo, 2 * WBLK);
            bool ok = true;
            for (int c = 0; c < nchunk && ok; ++c) {
                const uint32_t par = c & 1;
                if (!(ok = wait_phase(bar(B_QK), par, abort))) break;
                ++done[0];
                fence_after();
                issue_projection_pair<D, MERGE_PROJ>(tmem + T_ZQ, base + Ly.q, base + Ly.whi);
                commit(bar(B_PROJ));
                if (!(ok = wait_phase(bar(B_FEAT), par, abort))) break;
                if (!(ok = wait_phase(bar(B_SOP), par, abort))) break;
                if (!(ok = wait_phase(bar(B_V), par, abort))) break;
                ++done[1];
                if (!(ok = wait_phase(bar(B_DO), par, abort))) break;
                ++done[2];
                fence_after();
                // group A: dO V^T, g = dO A_prev^T, (tril 1) F_K
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint64_t ko = (uint64_t)((ks >> 2) * BLK + (ks & 3) * 32) >> 4;
                    umma(tmem + T_DV, d_do_k + ko, d_v_k + ko, id_dv, ks > 0);
                    if constexpr (LRMAX == 32) {  // S hi and lo as one N = 64 operand
                        umma(tmem + T_G, d_do_k + ko, d_shi + (uint64_t)(ks * 128), id_g64, ks > 0);
                    } else {
                        umma(tmem + T_G, d_do_k + ko, d_shi + (uint64_t)(ks * 128), id_g1, ks > 0);
                        umma(tmem + T_G, d_do_k + ko, d_slo + (uint64_t)(ks * 128), id_g1, true);
                    }
                }
#pragma unroll
                for (int ks = 0; ks < C / 16; ++ks) {
                    if constexpr (Cols::TRIL_TMEM) {
                        umma_ts(tmem + T_BT, tmem + T_TRIL + 8 * ks, d_fk_mn + (uint64_t)(ks * 128), id_bt, ks > 0);
                    } else {
                        const uint64_t ko = (uint64_t)((ks >> 2) * BLK + (ks & 3) * 32) >> 4;
                        umma(tmem + T_BT, desc_k(base + Ly.tril) + ko, d_fk_mn + (uint64_t)(ks * 128), id_bt, ks > 0);
                    }
                }
                commit(bar(B_A));
                if (c + 1 < nchunk) {  // projections and norms have read the Q / K tiles; issued after
                    load_tiles(c + 1, 1);  // group A, which waits on this warp
                    ++issued[0];
                }
                // sketch update A^T += V^T F_K and B += F_K^T 1 while the mask is applied (this chunk's
                // products read the sketch from its shared copy; group B's commit covers these)
#pragma unroll
                for (int ks = 0; ks < C / 16; ++ks) {
                    const uint64_t ko = (uint64_t)(ks * 2048) >> 4, kk = (uint64_t)((ks >> 2) * 2048 + (ks & 3) * 32) >> 4;
                    umma(tmem + T_ST, d_v_mt + ko, d_fk_mn + ko, id_gt, true);
                    umma(tmem + T_MS, d_fk_mn + ko, d_ones + kk, id_m16, true);
                }
                // group B: g += M1 F_K
                if (!(ok = wait_phase(bar(B_MASK), par, abort))) break;
                fence_after();
#pragma unroll
                for (int ks = 0; ks < C / 16; ++ks) {
                    const uint32_t ac = (ks < 4 ? 8 * ks : 64 + 8 * (ks - 4));
                    umma_ts(tmem + T_G, tmem + T_DV + ac, d_fk_mn + (uint64_t)(ks * 128), id_bt, true);
                }
                commit(bar(B_B));
                if (c + 1 < nchunk) {  // V is last read by group B
                    if (!(ok = wait_phase(bar(B_B), par, abort))) break;
                    load_tiles(c + 1, 2);
                    ++issued[1];
                }
                // group C: dxhat (the dQ epilogue starts on it), then the gradient sketch update
                // G += F'_Q^T [dO | -c], which runs during the epilogue under its own commit
                if (!(ok = wait_phase(bar(B_JAC), par, abort))) break;
                fence_after();
                for (int ks = 0; ks < LPP / 16; ++ks) {
                    umma_ts(tmem + T_DV, tmem + T_DZ + 8 * ks, d_whi + (uint64_t)(ks * 128), id_x, ks > 0);
                    umma_ts(tmem + T_DV, tmem + T_DZ + 8 * ks, d_wlo + (uint64_t)(ks * 128), id_x, true);
                }
                commit(bar(B_C));
#pragma unroll
                for (int ks = 0; ks < C / 16; ++ks) {
                    const uint64_t ko = (uint64_t)(ks * 2048) >> 4, kk = (uint64_t)((ks >> 2) * 2048 + (ks & 3) * 32) >> 4;
                    umma(tmem + T_GT, d_do_mt + ko, d_fq_mn + ko, id_gt, true);
                    umma(tmem + T_GB, d_fq_mn + ko, d_ncm + kk, id_m16, true);
                }
                commit(bar(B_G));
                if (c + 1 < nchunk) {  // dO is last read by the gradient sketch update
                    if (!(ok = wait_phase(bar(B_G), par, abort))) break;
                    load_tiles(c + 1, 4);
                    ++issued[2];
                }
            }
            if (!ok) {
                atomicOr(err, kErrTimeout);
                *abort = 1;
                const uint32_t bars[3] = {bar(B_QK), bar(B_V), bar(B_DO)};
#pragma unroll
                for (int b = 0; b < 3; ++b)
                    if (issued[b] > done[b]) mbar_wait(bars[b], done[b] & 1);
            }
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------------------- compute warps
        if (h == 1) {
            convert_s(0);
            warp_signal(bar(B_SOP));
        }
        // F_K rows of chunk c -> staging buffer c & 1, by the thread that owns the row (warps 4-7)
        const int lrs = feature_row_stride(LR);
        const bf16 *fk_bh = fk_in + bh * Dm.N * lrs;
        auto stage_rows = [&](int c) {
            const int64_t row = n_begin + (int64_t)c * C + t;
            if (row < n_end) {
                const uint32_t buf = base + Ly.stage + (uint32_t)(c & 1) * STG_FK;
#pragma unroll
                for (int ch = 0; ch < LRMAX / 8; ++ch)
                    if (8 * ch < lrs) cp_async16(buf + t * 128 + 16 * ch, fk_bh + row * lrs + 8 * ch);
            }
            cp_async_commit();
        };
        if (h == 1 && nchunk > 0) stage_rows(0);
        bool ok = group_sync(bar(B_CS), 0, abort);  // B_prev visible to the Q warps
        for (int c = 0; c < nchunk && ok; ++c) {
            const uint32_t par = c & 1;
            const int64_t n0 = n_begin + (int64_t)c * C;
            const int cnt = (int)min((int64_t)C, n_end - n0);
            const bool live = t < cnt;
            float uq[LPP];  // Q rows keep u for the Jacobian
            if (h == 0) {
                if (!(ok = wait_phase(bar(B_QK), par, abort))) break;
                float inv;
                {
                    float ss = 0.f;
#pragma unroll
                    for (int j = 0; j < D / 8; j += 2) {
                        const uint4 w0 = ld_shared_v4(base + Ly.q + (j >> 3) * BLK + sw_chunk(t, j & 7));
                        const uint4 w1 = ld_shared_v4(base + Ly.q + ((j + 1) >> 3) * BLK + sw_chunk(t, (j + 1) & 7));
                        ss += sumsq8(w0) + sumsq8(w1);
                        // keep the Q row in TMEM for the dQ epilogue
                        const uint32_t r[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
                        stn<8>(tlane + T_X + 4 * j, r);
                    }
                    inv = ss > 0.f ? rsqrtf(ss) : 0.f;
                    invq_s[t] = inv;
                }
                if (!(ok = wait_phase(bar(B_PROJ), par, abort))) break;
                fence_after();
                float z[LPP];
                {
                    float a[32];
                    ld32(tlane + T_ZQ, a);
#pragma unroll
                    for (int j = 0; j < LPP; ++j) z[j] = a[j];
                    if constexpr (MERGE_PROJ) {  // + the lo hyperplanes' part (in g's columns until group A),
                        ld32(tlane + T_ZQ + LPP, a);  // and the sum back for the Jacobian's z . dz
#pragma unroll
                        for (int j = 0; j < LPP; ++j) z[j] += a[j];
#pragma unroll
                        for (int b = 0; b < LPP / 8; ++b) {
                            uint32_t r[8];
#pragma unroll
                            for (int j = 0; j < 8; ++j) r[j] = __float_as_uint(z[8 * b + j]);
                            stn<8>(tlane + T_ZQ + 8 * b, r);
                        }
                    }
                }
#pragma unroll
                for (int j = 0; j < LPP; ++j) uq[j] = j < LP ? tc::tanh_abs(z[j] * inv) : 0.f;
            } else {
                // the F_K row t (zero past the end) -> shared F_K tile; then the next chunk's rows
                cp_async_wait_all();
                const uint32_t buf = base + Ly.stage + par * STG_FK;
#pragma unroll
                for (int ch = 0; ch < LRMAX / 8; ++ch) {
                    if (8 * ch < lrs) {
                        const uint4 v = live ? ld_shared_v4(buf + t * 128 + 16 * ch) : make_uint4(0u, 0u, 0u, 0u);
                        st_shared_v4(base + Ly.fk + sw_chunk(t, ch), v.x, v.y, v.z, v.w);
                    }
                }
                if (c + 1 < nchunk) stage_rows(c + 1);
            }
            wait_st();
            warp_signal(bar(B_FEAT));
            // M1 = mask_{j <= t}(dO V^T) on this half's 64 key columns, bf16 in place
            if (!(ok = wait_phase(bar(B_A), par, abort))) break;
            fence_after();
            {
                const int j0 = 64 * h;
#pragma unroll
                for (int pass = 0; pass < 2; ++pass) {
                    const int jb = j0 + 32 * pass;
                    const bool need = jb <= 32 * q4 + 31;  // warp-uniform: some lane keeps a column
                    uint32_t a[32];
                    if (need) ld32_nw(tlane + T_DV + jb, a);
                    wait_ld();
                    reg_fence(a);
#pragma unroll
                    for (int b = 0; b < 2; ++b) {
                        uint32_t w[8];
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            const int e = 16 * b + 2 * j;
                            w[j] = bfp::pack_bf16(need && jb + e <= t ? uf(a[e]) : 0.f,
                                                  need && jb + e + 1 <= t ? uf(a[e + 1]) : 0.f);
                        }
                        stn<8>(tlane + T_DV + j0 + 16 * pass + 8 * b, w);
                    }
                }
            }
            wait_st();
            warp_signal(bar(B_MASK));
            if (!(ok = wait_phase(bar(B_B), par, abort))) break;
            fence_after();
            if (h == 0) {
                // den, c, dphi_Q and the feature Jacobian; F'_Q, -c and {1/den, c}, table by table
                auto write_fq = [&](int l, const float (&ph)[R], float rd) {  // F'_Q = phi / den, one table
                    if constexpr (R >= 8) {
#pragma unroll
                        for (int j = 0; j < R / 8; ++j) {
                            const int ch = l * (R / 8) + j;
                            st_shared_v4(base + Ly.fq + sw_chunk(t, ch), bfp::pack_bf16(ph[8 * j] * rd, ph[8 * j + 1] * rd),
                                         bfp::pack_bf16(ph[8 * j + 2] * rd, ph[8 * j + 3] * rd),
                                         bfp::pack_bf16(ph[8 * j + 4] * rd, ph[8 * j + 5] * rd),
                                         bfp::pack_bf16(ph[8 * j + 6] * rd, ph[8 * j + 7] * rd));
                        }
                    } else {
#pragma unroll
                        for (int r = 0; r < R; r += 2) {
                            const uint32_t w = bfp::pack_bf16(ph[r] * rd, ph[r + 1] * rd);
                            asm volatile("st.shared.b32 [%0], %1;\n" ::"r"(base + Ly.fq + sw_elem(t, l * R + r)), "r"(w)
                                         : "memory");
                        }
                    }
                };
                float dz[LPP];
#pragma unroll
                for (int j = 0; j < LPP; ++j) dz[j] = 0.f;
                float rd = 0.f, cc = 0.f;
                if constexpr (LRMAX == 32) {
                    uint32_t gr[32], br[32];
                    {
                        uint32_t gl[32];  // g = its hi part (with M1 F_K) + its lo part
                        ld32_nw(tlane + T_G, gr);
                        ld32_nw(tlane + T_G + 32, gl);
                        ld32_nw(tlane + T_BT, br);
                        wait_ld();
                        reg_fence(gr);
                        reg_fence(gl);
                        reg_fence(br);
#pragma unroll
                        for (int j = 0; j < 32; ++j) gr[j] = __float_as_uint(uf(gr[j]) + uf(gl[j]));
                    }
                    float den = 0.f, pg = 0.f;
                    float phq[LT > 0 ? LRMAX : 1];  // with L compiled in: the row's bucket probabilities
#pragma unroll
                    for (int l = 0; l < LMAX; ++l) {
                        if (l < L && l * R < LRMAX) {
                            float u[P], ph[R];
#pragma unroll
                            for (int p = 0; p < P; ++p) u[p] = uq[l * P + p];
                            tc::bucket_probs<P>(u, beta, ph);
#pragma unroll
                            for (int r = 0; r < R; ++r) {
                                const int lr = l * R + r < 32 ? l * R + r : 31;
                                if constexpr (LT > 0) phq[lr] = ph[r];
                                den = fmaf(ph[r], bprev[32 * par + lr] + uf(br[lr]), den);
                                pg = fmaf(ph[r], uf(gr[lr]), pg);
                            }
                        }
                    }
                    rd = live ? __frcp_rn(den) : 0.f;
                    cc = pg * rd;
                    if (live) aux[bh * Dm.N + n0 + t] = make_float2(rd, cc);
#pragma unroll
                    for (int l = 0; l < LMAX; ++l) {
                        if (l < L && l * R < LRMAX) {
                            float u[P], ph[R], g[R];
#pragma unroll
                            for (int p = 0; p < P; ++p) u[p] = uq[l * P + p];
                            if constexpr (LT > 0) {
#pragma unroll
                                for (int r = 0; r < R; ++r) ph[r] = phq[l * R + r < 32 ? l * R + r : 31];
                            } else {
                                tc::bucket_probs<P>(u, beta, ph);
                            }
#pragma unroll
                            for (int r = 0; r < R; ++r) {
                                const int lr = l * R + r < 32 ? l * R + r : 31;
                                g[r] = (uf(gr[lr]) - (bprev[32 * par + lr] + uf(br[lr])) * cc) * rd;
                            }
                            float tmp[P];
                            table_backward<P, DB>(u, ph, g, beta, tmp, &db);
#pragma unroll
                            for (int p = 0; p < P; ++p) dz[l * P + p] = tmp[p];
                            write_fq(l, ph, rd);
                        }
                    }
                } else {
                    // wider sketches: one table's g and B_t columns at a time, in two passes (den and
                    // c need every table before any table's gradient)
                    float den = 0.f, pg = 0.f;
#pragma unroll
                    for (int l = 0; l < LMAX; ++l) {
                        if (l < L && l * R < LRMAX) {
                            float u[P], ph[R], gg[R], bb[R];
#pragma unroll
                            for (int p = 0; p < P; ++p) u[p] = uq[l * P + p];
                            tc::bucket_probs<P>(u, beta, ph);
                            ld_cols<R>(tlane + T_G + l * R, gg);
                            ld_cols<R>(tlane + T_BT + l * R, bb);
#pragma unroll
                            for (int r = 0; r < R; ++r) {
                                den = fmaf(ph[r], bprev[LRMAX * par + l * R + r] + bb[r], den);
                                pg = fmaf(ph[r], gg[r], pg);
                            }
                        }
                    }
                    rd = live ? __frcp_rn(den) : 0.f;
                    cc = pg * rd;
                    if (live) aux[bh * Dm.N + n0 + t] = make_float2(rd, cc);
#pragma unroll
                    for (int l = 0; l < LMAX; ++l) {
                        if (l < L && l * R < LRMAX) {
                            float u[P], ph[R], gg[R], bb[R], g[R];
#pragma unroll
                            for (int p = 0; p < P; ++p) u[p] = uq[l * P + p];
                            tc::bucket_probs<P>(u, beta, ph);
                            ld_cols<R>(tlane + T_G + l * R, gg);
                            ld_cols<R>(tlane + T_BT + l * R, bb);
#pragma unroll
                            for (int r = 0; r < R; ++r) g[r] = (gg[r] - (bprev[LRMAX * par + l * R + r] + bb[r]) * cc) * rd;
                            float tmp[P];
                            table_backward<P, DB>(u, ph, g, beta, tmp, &db);
#pragma unroll
                            for (int p = 0; p < P; ++p) dz[l * P + p] = tmp[p];
                            write_fq(l, ph, rd);
                        }
                    }
                }
                if (live) {  // the row of F'_Q the key-side pass reads instead of recomputing it
                    const int lrs = feature_row_stride(LR);
                    bf16 *dst = fq_out + (bh * Dm.N + n0 + t) * lrs;
#pragma unroll
                    for (int ch = 0; ch < LRMAX / 8; ++ch)
                        if (8 * ch < lrs) st_global_v4(dst + 8 * ch, ld_shared_v4(base + Ly.fq + sw_chunk(t, ch)));
                }
                uint32_t r[8];
#pragma unroll
                for (int b = 0; b < 2; ++b) {
#pragma unroll
                    for (int j = 0; j < 8; ++j) r[j] = bfp::pack_bf16(dz[16 * b + 2 * j], dz[16 * b + 2 * j + 1]);
                    stn<8>(tlane + T_DZ + 8 * b, r);
                }
                {
                    // dxhat = W^T dz (dz rounded to bf16 as the product sees it), so x . dxhat = z . dz
                    // with z = W x, still in TMEM
                    float zq[32], zdz = 0.f;
                    ld32(tlane + T_ZQ, zq);
#pragma unroll
                    for (int j = 0; j < LPP; ++j)
                        if (j < LP) zdz = fmaf(__bfloat162float(__float2bfloat16_rn(dz[j])), zq[j], zdz);
                    red[t] = invq_s[t] * invq_s[t] * zdz;
                }
                const float mcv = -cc;
                const bf16 mhi = __float2bfloat16_rn(mcv);
                const bf16 mlo = __float2bfloat16_rn(mcv - __bfloat162float(mhi));
                unsigned char *mt = sm + Ly.ncm + (t >> 6) * 2048;
                *reinterpret_cast<bf16 *>(mt + sw_elem(0, t & 63)) = mhi;
                *reinterpret_cast<bf16 *>(mt + sw_elem(1, t & 63)) = mlo;
                wait_st();
                warp_signal(bar(B_JAC));
                if (Dm.dzq != nullptr && live) {  // d(loss)/d(W): this Q row's dz / |q| (zeros past L P)
                    float4 *o = reinterpret_cast<float4 *>(Dm.dzq + (bh * Dm.N + n0 + t) * Dm.dzld);
                    const float iq = invq_s[t];
#pragma unroll
                    for (int q = 0; q < LPP / 4; ++q)
                        if (4 * q < Dm.dzld)
                            o[q] = make_float4(dz[4 * q] * iq, dz[4 * q + 1] * iq, dz[4 * q + 2] * iq, dz[4 * q + 3] * iq);
                }
            } else {
                // the sketch after this chunk -> bf16 operand and B_prev of the next chunk
                convert_s(par ^ 1);
                warp_signal(bar(B_SOP));
            }
            if (!(ok = wait_phase(bar(B_C), par, abort))) break;
            fence_after();
            {
                // dQ row t = inv (dxhat - x inv^2 (x . dxhat)); half h takes columns h D/2 .. (h+1) D/2.
                // inv^2 (x . dxhat) comes from the Q row's thread, published before its JAC arrival
                if (h == 1 && !(ok = wait_phase(bar(B_JAC), par, abort))) break;
                const float iq = invq_s[t];
                const float kk = red[t];
                bf16 *dst = dQ + off + (n0 + t) * D + h * (D / 2);
#pragma unroll
                for (int pass = 0; pass < D / 64; ++pass) {
                    uint32_t v[32], xr[16];
                    ld32_nw(tlane + T_DV + h * (D / 2) + 32 * pass, v);
                    ld16_nw(tlane + T_X + h * (D / 4) + 16 * pass, xr);
                    wait_ld();
                    reg_fence(v);
                    reg_fence(xr);
                    uint32_t o[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        o[j] = bfp::pack_bf16(iq * (uf(v[2 * j]) - bf_lo(xr[j]) * kk), iq * (uf(v[2 * j + 1]) - bf_hi(xr[j]) * kk));
                    if (live) store_row32(dst + 32 * pass, o, wide);
                }
            }
            fence_before();
            if (!(ok = group_sync(bar(B_CS), (c + 1) & 1, abort))) break;  // B_prev, TMEM reads: next chunk
        }
        // the segment's gradient-sketch sum: G^T (lanes d) and G_B (lanes = sketch row, hi + lo)
        if (ok && nchunk > 0) ok = wait_phase(bar(B_G), (nchunk - 1) & 1, abort);
        if (ok) {
            fence_after();
            float *out = Gseg + ((int64_t)bh * nseg + s) * LR * (D + 1);
            if (h == 0 && t < D) {
#pragma unroll
                for (int half = 0; half < LRMAX / 32; ++half) {
                    float a[32];
                    ld32(tlane + T_GT + 32 * half, a);
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (32 * half + j < LR) out[(int64_t)(32 * half + j) * (D + 1) + t] = a[j];
                }
            }
            if (h == 1) {
                float m[2];
                ldn<2>(tlane + T_GB, m);
                if (t < LR) out[(int64_t)t * (D + 1) + D] = m[0] + m[1];
            }
        }
    }
    cp_async_wait_all();  // no copy into the staging buffers outlives the CTA (after an abort)
    if constexpr (DB) {  // this CTA's d(loss)/d(beta) partial, summed in a fixed order
        const float sdb = block_sum_fixed(db, red);
        if (tid == 0) dbpart[bh * gridDim.x + blockIdx.x] = sdb;
    }
    fence_before();
    __syncthreads();
    if (warp == 0) {
        fence_after();
        tmem_dealloc(tmem, T_COLS);
    }
}

}  // namespace c5q

// ------------------------------------------------------------------ host side

cudaError_t make_token_map(CUtensorMap *map, const void *base, const Dims &D);

size_t c5_feature_rows_bytes(const Dims &D)
{
    return (size_t)D.BH * D.N * nc5::feature_row_stride(D.LR) * sizeof(bf16_t);
}

bool c5_bwd_supported(const Dims &D)
{
    // L R <= 32 at d = 64 or 128; L R <= 64 at d = 64 (the TMEM budget of the key side: 512 columns)
    const bool width = D.LR <= 32 || (D.d == 64 && D.LR <= 64);
    return (D.d == 64 || D.d == 128) && D.P >= 1 && D.P <= (D.d == 64 ? 6 : 5) && D.LP <= nc5::LPP && width &&
           D.N <= 0x7FFFFFFF;
}

namespace {

template <int D, int P, int LT, int LRM>
cudaError_t bwdkv5_launch(const Dims &Dm, const bf16_t *fq, const bf16_t *fk, const float *kinv, const CUtensorMap &mk,
                          const CUtensorMap &mv, const CUtensorMap &mdo, const float *W, const float2 *aux,
                          const float *G0, int64_t seg_len, int nseg, bf16_t *dK, bf16_t *dV, unsigned *err,
                          float *dbpart, cudaStream_t st)
{
    const c5b::BwdLayout Ly(D, LRM);
    const size_t smem = Ly.bytes + 1024;
    auto kern = dbpart ? c5b::k_causal_bwdkv5<D, P, LT, LRM, true> : c5b::k_causal_bwdkv5<D, P, LT, LRM, false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return launch_kernel("tc5_causal_bwd_kv", kern, dim3((unsigned)nseg, (unsigned)Dm.BH), dim3(c5b::NTHW), smem,
                         st, fq, fk, kinv, mk, mv, mdo, Dm, W, aux, G0, seg_len, nseg, dK, dV, err, dbpart);
}

// (d, P, L) = (128, 3, 3) runs with L compiled in; every other shape with L at run time.  L R > 32
// (d = 64 only) takes the LRM = 64 instances (with L compiled in they spill three times as much).
template <int D, int P>
cudaError_t bwdkv5_inst(const Dims &Dm, const bf16_t *fq, const bf16_t *fk, const float *kinv, const CUtensorMap &mk,
                        const CUtensorMap &mv, const CUtensorMap &mdo, const float *W, const float2 *aux,
                        const float *G0, int64_t seg_len, int nseg, bf16_t *dK, bf16_t *dV, unsigned *err,
                        float *dbpart, cudaStream_t st)
{
#define RACE_KV_ARGS Dm, fq, fk, kinv, mk, mv, mdo, W, aux, G0, seg_len, nseg, dK, dV, err, dbpart, st
    if constexpr (D == 64 && P >= 2) {
        if (Dm.LR > 32) return bwdkv5_launch<D, P, 0, 64>(RACE_KV_ARGS);
    }
    if constexpr (D == 128 && P == 3)
        if (Dm.L == 3) return bwdkv5_launch<D, P, 3, 32>(RACE_KV_ARGS);
    if constexpr (P <= 5) return bwdkv5_launch<D, P, 0, 32>(RACE_KV_ARGS);
    return cudaErrorInvalidValue;
#undef RACE_KV_ARGS
}

template <int D, int P, int LT, int LRM>
cudaError_t bwdq5_launch(const Dims &Dm, const CUtensorMap &mq, const bf16_t *fk, const CUtensorMap &mv,
                         const CUtensorMap &mdo, const float *W, const float *S0, int64_t seg_len, int nseg,
                         bf16_t *dQ, float2 *aux, bf16_t *fq, float *Gseg, unsigned *err, float *dbpart,
                         cudaStream_t st)
{
    const c5q::QLayout Ly(D, LRM);
    const size_t smem = Ly.bytes + 1024;
    auto kern = dbpart ? c5q::k_causal_bwdq5<D, P, LT, LRM, true> : c5q::k_causal_bwdq5<D, P, LT, LRM, false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return launch_kernel("tc5_causal_bwd_q", kern, dim3((unsigned)nseg, (unsigned)Dm.BH), dim3(c5q::NTHW), smem, st,
                         mq, fk, mv, mdo, Dm, W, S0, seg_len, nseg, dQ, aux, fq, Gseg, err, dbpart);
}

// (d, P, L) = (128, 3, 3) runs with L compiled in; every other shape with L at run time.  L R > 32
// (d = 64 only) takes the LRM = 64 instances (with L compiled in they spill three times as much).
template <int D, int P>
cudaError_t bwdq5_inst(const Dims &Dm, const CUtensorMap &mq, const bf16_t *fk, const CUtensorMap &mv,
                       const CUtensorMap &mdo, const float *W, const float *S0, int64_t seg_len, int nseg,
                       bf16_t *dQ, float2 *aux, bf16_t *fq, float *Gseg, unsigned *err, float *dbpart,
                       cudaStream_t st)
{
#define RACE_Q_ARGS Dm, mq, fk, mv, mdo, W, S0, seg_len, nseg, dQ, aux, fq, Gseg, err, dbpart, st
    if constexpr (D == 64 && P >= 2) {
        if (Dm.LR > 32) return bwdq5_launch<D, P, 0, 64>(RACE_Q_ARGS);
    }
    if constexpr (D == 128 && P == 3)
        if (Dm.L == 3) return bwdq5_launch<D, P, 3, 32>(RACE_Q_ARGS);
    if constexpr (P <= 5) return bwdq5_launch<D, P, 0, 32>(RACE_Q_ARGS);
    return cudaErrorInvalidValue;
#undef RACE_Q_ARGS
}

}  // namespace

#define RACE_C5B_SHAPES(X) \
    X(64, 1) X(64, 2) X(64, 3) X(64, 4) X(64, 5) X(64, 6) X(128, 1) X(128, 2) X(128, 3) X(128, 4) X(128, 5)

cudaError_t launch_c5_bwd_q(const Dims &Dm, const bf16_t *Q, const bf16_t *fk, const bf16_t *V, const bf16_t *dO,
                            const float *W, const float *S0, int64_t seg_len, int nseg, bf16_t *dQ, float2 *aux,
                            bf16_t *fq, float *Gseg, unsigned *err, float *dbpart, cudaStream_t st)
{
    CUtensorMap mq, mv, mdo;
    cudaError_t e = make_token_map(&mq, Q, Dm);
    if (e == cudaSuccess) e = make_token_map(&mv, V, Dm);
    if (e == cudaSuccess) e = make_token_map(&mdo, dO, Dm);
    if (e != cudaSuccess) return e;
#define RACE_C5Q_CASE(DD, PP) \
    case DD * 16 + PP: return bwdq5_inst<DD, PP>(Dm, mq, fk, mv, mdo, W, S0, seg_len, nseg, dQ, aux, fq, Gseg, err, dbpart, st);
    switch (Dm.d * 16 + Dm.P) {
        RACE_C5B_SHAPES(RACE_C5Q_CASE)
        default: return cudaErrorInvalidValue;
    }
#undef RACE_C5Q_CASE
}

cudaError_t launch_c5_bwd_kv(const Dims &Dm, const bf16_t *fq, const bf16_t *fk, const float *kinv, const bf16_t *K,
                             const bf16_t *V, const bf16_t *dO, const float2 *aux, const float *W, const float *G0,
                             int64_t seg_len, int nseg, bf16_t *dK, bf16_t *dV, unsigned *err, float *dbpart,
                             cudaStream_t st)
{
    CUtensorMap mk, mv, mdo;
    cudaError_t e = make_token_map(&mk, K, Dm);
    if (e == cudaSuccess) e = make_token_map(&mv, V, Dm);
    if (e == cudaSuccess) e = make_token_map(&mdo, dO, Dm);
    if (e != cudaSuccess) return e;
#define RACE_C5KV_CASE(DD, PP) \
    case DD * 16 + PP: return bwdkv5_inst<DD, PP>(Dm, fq, fk, kinv, mk, mv, mdo, W, aux, G0, seg_len, nseg, dK, dV, err, dbpart, st);
    switch (Dm.d * 16 + Dm.P) {
        RACE_C5B_SHAPES(RACE_C5KV_CASE)
        default: return cudaErrorInvalidValue;
    }
#undef RACE_C5KV_CASE
}
#undef RACE_C5B_SHAPES

}  // namespace race
