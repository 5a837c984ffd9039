// race_c5_fwd.cu -- tcgen05 (TMEM accumulator) causal RACE attention forward, bf16 tensors.
//
// Algorithm 2 of the paper ("RACE Attention" slides, frame "Causality is a prefix update of the
// same statistics"; reading notes section 2.6) evaluated in chunks of C = 128 tokens.  With F the
// concatenated bucket features (L R columns) of a chunk and S = [A | B] the sketch of every
// earlier token (A: L R x d content, B: L R mass):
//
//   [num | den] = mask_{j <= t}(F_Q F_K^T) [V | 1]  +  F_Q [A | B]      O = num / den
//   A += F_K^T V,   B += F_K^T 1
//
// One CTA walks one segment of a (batch, head) sequence; the sketch at the segment start comes
// from the segment sums (the non-causal sketch kernel restricted to each segment) and an
// exclusive scan over segments.  The segment-sum pass also stores every key's bucket features
// F_K (L R bf16 per token), which this kernel reads instead of K.  Per chunk, on the tensor
// cores (M = 128, fp32 in TMEM):
//   z = Q (W_hi + W_lo)^T;
//   scores F_Q F_K^T with F_Q in TMEM (A operand) and F_K in a swizzled shared tile;
//   P = the causally masked scores, written back to TMEM as bf16 (A operand);
//   [num | den] = P V and P 1 plus F_Q [A | B], with [A | B] in shared memory as bf16 hi + lo
//   (about 16 mantissa bits);
//   A^T += V^T F_K (M = d, N = L R) and B += F_K^T 1 (M = L R), both accumulating in TMEM over
//   the whole segment.
// On CUDA cores: Q row norms and bucket features (tanh, products of sigmoids), the copy of the F_K
// rows into their tile, the causal mask, the num / den epilogue, and the conversion of the TMEM
// sketch to its bf16 operand copy.  The Q tile is single-buffered (refilled once the projection
// has read it); V tiles are double-buffered and each also stages its chunk's output for the TMA
// store; the F_K rows come in a chunk ahead (cp.async by the row's thread) into two staging
// buffers.
#include "race_launch.h"
#include "race_nc5_common.cuh"

namespace race {
namespace c5 {

using namespace race::nc5;

// TMEM columns (512 allocated).
constexpr uint32_t T_O = 0;      // [num | den]: d + 16 columns
constexpr uint32_t T_ST = 144;   // A^T (lanes = d), L R (<= 64) columns
constexpr uint32_t T_MS = 208;   // B (lanes = sketch row), 16 columns (column 0 used)
constexpr uint32_t T_ZQ = 224;   // projections of the Q tile
constexpr uint32_t T_FQ = 288;   // F_Q as bf16 pairs (A operand), L R / 2 columns
constexpr uint32_t T_SC = 320;   // scores, 128 columns
constexpr uint32_t T_P = 448;    // masked scores as bf16 pairs (A operand), 64 columns
constexpr uint32_t T_COLS = 512;

constexpr uint32_t STG_FK = C * 128;  // one staging buffer of F_K rows (128-byte slots: L R <= 64)

struct FwdLayout {
    uint32_t q, stage, v, fk, shi, slo, whi, wlo, ones, zero, bar, slot, bytes, kbb, sblk;
    __host__ __device__ FwdLayout(int D)
    {
        kbb = (uint32_t)(D / 64) * BLK;  // bytes of one token tile
        sblk = (uint32_t)(D + 16) * 128;
        q = 0;
        stage = q + kbb;   // two F_K staging buffers
        v = stage + 2 * STG_FK;  // two stages
        fk = v + 2 * kbb;  // two 64-column blocks (the second stays zero)
        shi = fk + 2 * BLK;
        slo = shi + sblk;
        whi = slo + sblk;
        wlo = whi + (uint32_t)(D / 64) * WBLK;
        ones = wlo + (uint32_t)(D / 64) * WBLK;
        zero = ones + 4096;  // a zero 64-column block (d = 64: the upper half of V^T)
        bar = zero + (D == 64 ? BLK : 0);
        slot = bar + 128;
        bytes = slot + 16;
    }
};

__device__ __forceinline__ void st_shared_b16(uint32_t addr, bf16 v)
{
    asm volatile("st.shared.b16 [%0], %1;\n" ::"r"(addr), "h"(*reinterpret_cast<unsigned short *>(&v)) : "memory");
}

__device__ __forceinline__ float bf16_rest(float x) { return x - __bfloat162float(__float2bfloat16_rn(x)); }

// Writes this thread's lane of the fp32 TMEM sketch (row d of A^T, row lr of B) into the bf16
// read-out operand: K-major rows n = output column (rows 0 .. d-1 content, row d mass), the 64
// columns = sketch rows.  h = 0 writes the hi copy, h = 1 the lo copy (x - bf16(x)).
template <int D>
__device__ __forceinline__ void sketch_to_operand(uint32_t tlane, int q4, int lane, int h, int LR, int lrp,
                                                  uint32_t shi, uint32_t slo)
{
    const int row = 32 * q4 + lane;
    const uint32_t dst = h ? slo : shi;
    const bool content = 32 * q4 < D, mass = 32 * q4 < lrp;  // warp-uniform
    // one pass per 32 sketch columns so that only 32 values are in flight per wait
    for (int half = 0; half < (lrp > 32 ? 2 : 1); ++half) {
        uint32_t a[32], m0 = 0;
        if (content) ld32_nw(tlane + T_ST + 32 * half, a);
        if (mass && half == 0) ld1_nw(tlane + T_MS, m0);
        wait_ld();
        reg_fence(a);
        reg_fence1(m0);
        if (content) {  // lane = d
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int cg = 4 * half + c;  // 8-column chunk of the operand row
                if (8 * cg < lrp) {
                    uint32_t w[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int k0 = 8 * c + 2 * j;
                        float x0 = 32 * half + k0 < LR ? uf(a[k0]) : 0.f;
                        float x1 = 32 * half + k0 + 1 < LR ? uf(a[k0 + 1]) : 0.f;
                        if (h) {
                            x0 = bf16_rest(x0);
                            x1 = bf16_rest(x1);
                        }
                        w[j] = bfp::pack_bf16(x0, x1);
                    }
                    st_shared_v4(dst + sw_chunk(row, cg), w[0], w[1], w[2], w[3]);
                }
            }
        }
        if (mass && half == 0) {  // lane = sketch row
            float x = row < LR ? uf(m0) : 0.f;
            if (h) x = bf16_rest(x);
            st_shared_b16(dst + sw_elem(D, row), __float2bfloat16_rn(x));
        }
    }
}

constexpr int NTHW = NTH + 32;  // 8 compute warps + 1 control warp (TMA and MMA issue)

// Barrier slots (8 bytes each) after FwdLayout::bar.
enum : uint32_t { B_QK, B_PROJ, B_SC, B_MMA, B_FEAT, B_MASK, B_SOP, B_V0, B_V1, B_COUNT };

template <int D, int P, int LT>
__global__ void __launch_bounds__(NTHW, 1)
    k_causal_fwd5(const __grid_constant__ CUtensorMap tmQ, const bf16 *__restrict__ fk_in,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO, Dims Dm,
                  const float *__restrict__ W, const float *__restrict__ S0, int64_t seg_len, int nseg,
                  unsigned *__restrict__ err)
{
    constexpr int KB = D / 64;
    constexpr int R = 1 << P;
    constexpr int LMAX = LPP / P;
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023) & ~1023u;
    unsigned char *sm = smem_raw + (base - raw);
    const FwdLayout Ly(D);
    auto bar = [&](uint32_t i) { return base + Ly.bar + 8 * i; };
    volatile int *abort = reinterpret_cast<volatile int *>(sm + Ly.slot + 8);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, q4 = warp & 3, h = (warp >> 2) & 1;
    const bool compute = warp < 8;
    const int t = 32 * q4 + lane;  // token row (TMEM lane) of a compute thread
    const int s = blockIdx.x;
    const int64_t bh = blockIdx.y;
    const int64_t n_begin = (int64_t)s * seg_len;
    const int64_t n_end = min(Dm.N, n_begin + seg_len);
    const int nchunk = n_end > n_begin ? (int)((n_end - n_begin + C - 1) / C) : 0;
    // LT > 0: the table count is a compile-time constant (per-table loops unroll without guards)
    const int L = LT > 0 ? LT : Dm.L;
    const int LR = LT > 0 ? LT * (1 << P) : Dm.LR, lrp = (LR + 15) & ~15;
    const float beta = Dm.beta;
    // L R <= 32: the features of consecutive chunks use alternate buffers (F_Q: 16 TMEM columns
    // each, F_K: one 16 KB tile each), so chunk c featurises while chunk c - 1's products run
    const bool pipe = lrp <= 32;

    // ---- set-up
    if (warp == 0) tmem_alloc(base + Ly.slot, T_COLS);
    if (compute) {
        zero_region(sm + Ly.fk, 2 * BLK);
        zero_region(sm + Ly.shi, 2 * Ly.sblk);
        init_mass_tile(sm + Ly.ones, true);
        if (D == 64) zero_region(sm + Ly.zero, BLK);
        load_w_tiles<D>(head_w(W, Dm, bh), Dm.LP, sm + Ly.whi, sm + Ly.wlo);
    }
    if (tid == NTH) {
        for (uint32_t i = 0; i < B_COUNT; ++i) mbar_init(bar(i), (i == B_FEAT || i == B_MASK || i == B_SOP) ? 8 : 1);
        *abort = 0;
        tc::fence_mbar_init();
        prefetch_tmap(&tmQ);
        prefetch_tmap(&tmV);
        prefetch_tmap(&tmO);
    }
    tc::fence_proxy_async();
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(sm + Ly.slot);
    const uint32_t tlane = tmem + ((uint32_t)(32 * q4) << 16);

    // sketch at the segment start -> TMEM accumulators (A^T lanes = d, B lanes = sketch row); the
    // F_Q operand columns past L R stay zero
    if (compute) {
        const float *Sb = S0 + ((int64_t)bh * nseg + s) * LR * (D + 1);
        if (h == 0) {
            if (t < D) {
                for (int c0 = 0; c0 < lrp; c0 += 8) {
                    uint32_t r[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j) r[j] = __float_as_uint(c0 + j < LR ? Sb[(c0 + j) * (D + 1) + t] : 0.f);
                    stn<8>(tlane + T_ST + c0, r);
                }
            }
            const uint32_t m[1] = {__float_as_uint(t < LR ? Sb[t * (D + 1) + D] : 0.f)};
            stn<1>(tlane + T_MS, m);
        } else {
            const uint32_t zr[8] = {0, 0, 0, 0, 0, 0, 0, 0};
            for (int c0 = 0; c0 < 32; c0 += 8) stn<8>(tlane + T_FQ + c0, zr);
        }
        wait_st();
    }
    fence_before();
    __syncthreads();
    fence_after();

    if (!compute) {
        // ---------------------------------------------------------------- control warp
        if (lane == 0) {
            auto load_qk = [&](int c) {  // the Q tile (the keys arrive as feature rows)
                const int y = (int)(n_begin + (int64_t)c * C);
                mbar_arrive_expect_tx(bar(B_QK), KB * BLK);
#pragma unroll
                for (int kb = 0; kb < KB; ++kb) tma_load(base + Ly.q + kb * BLK, &tmQ, 64 * kb, y, (int)bh, bar(B_QK));
            };
            auto load_v = [&](int c) {
                const int y = (int)(n_begin + (int64_t)c * C);
                const uint32_t b = bar(B_V0 + (c & 1));
                mbar_arrive_expect_tx(b, KB * BLK);
#pragma unroll
                for (int kb = 0; kb < KB; ++kb)
                    tma_load(base + Ly.v + (c & 1) * Ly.kbb + kb * BLK, &tmV, 64 * kb, y, (int)bh, b);
            };
            auto store_out = [&](int c) {
                const uint32_t stage = base + Ly.v + (c & 1) * Ly.kbb;
                const int y = (int)(n_begin + (int64_t)c * C);
#pragma unroll
                for (int kb = 0; kb < KB; ++kb) tma_store(&tmO, 64 * kb, y, (int)bh, stage + kb * BLK);
                bulk_commit();
            };
            // loads issued and completions waited for, per barrier (to drain after an abort)
            int qk_issued = 0, qk_done = 0;
            Counts<2> v_issued, v_done;
            if (nchunk > 0) {
                // withhold (a test of the failure path): the first Q / K tiles are never requested,
                // so every wait on them runs out and the CTA takes the abort path below
                if (!Dm.withhold) {
                    load_qk(0);
                    ++qk_issued;
                }
                load_v(0);
                v_issued.inc(0);
                if (nchunk > 1) {
                    load_v(1);
                    v_issued.inc(1);
                }
            }
            constexpr uint32_t id_s = idesc_bf16(128, 128, 0, 0);
            constexpr uint32_t id_pv = idesc_bf16(128, D, 0, 1);
            constexpr uint32_t id_p1 = idesc_bf16(128, 16, 0, 0);
            constexpr uint32_t id_ro = idesc_bf16(128, D + 16, 0, 0);
            constexpr uint32_t id_ms = idesc_bf16(128, 16, 1, 0);
            const uint32_t id_up = idesc_bf16(128, lrp, 1, 1);
            const uint64_t d_ones = desc_k(base + Ly.ones);
            const uint64_t d_shi = desc_k(base + Ly.shi), d_slo = desc_k(base + Ly.slo);
            auto project = [&](int c) {
                fence_after();
                issue_projection<D>(tmem + T_ZQ, base + Ly.q, base + Ly.whi, base + Ly.wlo);
                commit(bar(B_PROJ));
            };
            bool ok = true, projected = false;  // projected: this chunk's projection went out early
            for (int c = 0; c < nchunk && ok; ++c) {
                const uint32_t vst = base + Ly.v + (c & 1) * Ly.kbb;
                const uint32_t fq = T_FQ + (pipe ? 16u * (c & 1) : 0u);
                const uint32_t fk = base + Ly.fk + (pipe ? (uint32_t)(c & 1) * BLK : 0u);
                const uint64_t d_fk_k = desc_k(fk);
                const uint64_t d_fk_mn = desc_mn(fk, BLK);       // B operand: one 64-column block
                const uint64_t d_fk_mt = desc_mn(fk, base + Ly.shi - fk);  // A, M = 128: rows 64+ unread
                if (!projected) {
                    if (!(ok = wait_phase(bar(B_QK), c & 1, abort))) break;
                    ++qk_done;
                    project(c);
                }
                projected = false;
                // scores once the features are in; then the Q / K tiles (read by the projection and
                // the norms) take the next chunk
                if (!(ok = wait_phase(bar(B_FEAT), c & 1, abort))) break;
                fence_after();
                for (int ks = 0; ks < lrp / 16; ++ks)
                    umma_ts(tmem + T_SC, tmem + fq + 8 * ks, d_fk_k + (uint64_t)(ks * 2), id_s, ks > 0);
                commit(bar(B_SC));
                if (c + 1 < nchunk) {
                    load_qk(c + 1);
                    ++qk_issued;
                }
                // the previous chunk's output is staged and this chunk's sketch operand is written
                if (!(ok = wait_phase(bar(B_SOP), c & 1, abort))) break;
                if (c >= 1) store_out(c - 1);
                if (!(ok = wait_phase(bar(B_V0 + (c & 1)), (c >> 1) & 1, abort))) break;
                v_done.inc(c & 1);
                fence_after();
                const uint64_t d_v = desc_mn(vst, BLK);
                const uint64_t d_vt = desc_mn(vst, D == 128 ? BLK : (Ly.zero - (Ly.v + (c & 1) * Ly.kbb)));
                // the sketch update needs only V and F_K, and the operand copy has read the sketch:
                // it runs while the mask is applied (the products' commit below covers it)
#pragma unroll
                for (int ks = 0; ks < C / 16; ++ks) {
                    const uint64_t ko = (uint64_t)(ks * 2048) >> 4, kk = (uint64_t)((ks >> 2) * 2048 + (ks & 3) * 32) >> 4;
                    umma(tmem + T_ST, d_vt + ko, d_fk_mn + ko, id_up, true);
                    umma(tmem + T_MS, d_fk_mt + ko, d_ones + kk, id_ms, true);
                }
                if (!(ok = wait_phase(bar(B_MASK), c & 1, abort))) break;
                // the next chunk's projection ahead of this chunk's products when its tiles are in,
                // so its features are computed while these run
                if (pipe && c + 1 < nchunk && mbar_test(bar(B_QK), (c + 1) & 1)) {
                    ++qk_done;
                    project(c + 1);
                    projected = true;
                }
                fence_after();
#pragma unroll
                for (int ks = 0; ks < C / 16; ++ks) {
                    const uint64_t ko = (uint64_t)(ks * 2048) >> 4, kk = (uint64_t)((ks >> 2) * 2048 + (ks & 3) * 32) >> 4;
                    umma_ts(tmem + T_O, tmem + T_P + 8 * ks, d_v + ko, id_pv, ks > 0);
                    umma_ts(tmem + T_O + D, tmem + T_P + 8 * ks, d_ones + kk, id_p1, ks > 0);
                }
                for (int ks = 0; ks < lrp / 16; ++ks) {
                    umma_ts(tmem + T_O, tmem + fq + 8 * ks, d_shi + (uint64_t)(ks * 2), id_ro, true);
                    umma_ts(tmem + T_O, tmem + fq + 8 * ks, d_slo + (uint64_t)(ks * 2), id_ro, true);
                }
                commit(bar(B_MMA));
                // V stage (c + 1) & 1 held chunk c - 1, whose output store must have read it
                if (c >= 1 && c + 1 < nchunk) {
                    bulk_wait_read0();
                    load_v(c + 1);
                    v_issued.inc((c + 1) & 1);
                }
            }
            if (ok && nchunk > 0) {
                ok = wait_phase(bar(B_SOP), nchunk & 1, abort);
                if (ok) store_out(nchunk - 1);
            }
            if (!ok) {
                atomicOr(err, kErrTimeout);
                *abort = 1;
                // let copies still in flight land before the CTA's shared memory goes away
                if (qk_issued > qk_done) mbar_wait(bar(B_QK), qk_done & 1);
#pragma unroll
                for (int b = 0; b < 2; ++b)
                    if (v_issued.v[b] > v_done.v[b]) mbar_wait(bar(B_V0 + b), v_done.v[b] & 1);
            }
            bulk_wait0();
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------------------- compute warps
        sketch_to_operand<D>(tlane, q4, lane, h, LR, lrp, base + Ly.shi, base + Ly.slo);
        warp_signal(bar(B_SOP));

        // output epilogue of chunk c: O = num / den (this half's columns), staged in V stage c & 1
        auto epilogue = [&](int c) {
            const uint32_t stage = base + Ly.v + (c & 1) * Ly.kbb;
            // this half's D / 2 columns in 32-column passes; den rides on the first
            float rd = 0.f;
#pragma unroll
            for (int pass = 0; pass < D / 64; ++pass) {
                uint32_t v[32], dn = 0;
                ld32_nw(tlane + T_O + h * (D / 2) + 32 * pass, v);
                if (pass == 0) ld1_nw(tlane + T_O + D, dn);
                wait_ld();
                reg_fence(v);
                reg_fence1(dn);
                if (pass == 0) {
                    rd = __frcp_rn(uf(dn));
                    if (h == 0 && t < (int)min((int64_t)C, n_end - n_begin - (int64_t)c * C)) flag_den(uf(dn), err);
                }
#pragma unroll
                for (int j = 0; j < 4; ++j) {  // 8-column chunks of this pass
                    const int ch = h * (D / 16) + 4 * pass + j;
                    float x[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) x[e] = uf(v[8 * j + e]) * rd;
                    st_shared_v4(stage + (ch >> 3) * BLK + sw_chunk(t, ch & 7), bfp::pack_bf16(x[0], x[1]),
                                 bfp::pack_bf16(x[2], x[3]), bfp::pack_bf16(x[4], x[5]), bfp::pack_bf16(x[6], x[7]));
                }
            }
        };

        // output of the previous chunk, and the sketch operand for this chunk's read-out
        auto previous = [&](int c) {
            if (!wait_phase(bar(B_MMA), (c - 1) & 1, abort)) return false;
            fence_after();
            epilogue(c - 1);
            sketch_to_operand<D>(tlane, q4, lane, h, LR, lrp, base + Ly.shi, base + Ly.slo);
            warp_signal(bar(B_SOP));
            return true;
        };

        // F_K rows of chunk c -> staging buffer c & 1, by the thread that owns the row (warps 4-7)
        const int lrs = feature_row_stride(LR);
        const bf16 *fk_bh = fk_in + bh * Dm.N * lrs;
        auto stage_rows = [&](int c) {
            const int64_t row = n_begin + (int64_t)c * C + t;
            if (row < n_end) {
                const uint32_t buf = base + Ly.stage + (uint32_t)(c & 1) * STG_FK;
#pragma unroll
                for (int ch = 0; ch < 8; ++ch)
                    if (8 * ch < lrs) cp_async16(buf + t * 128 + 16 * ch, fk_bh + row * lrs + 8 * ch);
            }
            cp_async_commit();
        };
        if (h == 1 && nchunk > 0) stage_rows(0);

        for (int c = 0; c < nchunk; ++c) {
            const int64_t n0 = n_begin + (int64_t)c * C;
            const int cnt = (int)min((int64_t)C, n_end - n0);
            const uint32_t fq = T_FQ + (pipe ? 16u * (c & 1) : 0u);
            const uint32_t fk = base + Ly.fk + (pipe ? (uint32_t)(c & 1) * BLK : 0u);
            // row norm of this thread's Q row (warps 0-3)
            float inv = 0.f;
            if (h == 0) {
                if (!wait_phase(bar(B_QK), c & 1, abort)) break;
                const float ss = half_sumsq<D>(base + Ly.q, t, 0) + half_sumsq<D>(base + Ly.q, t, 1);
                inv = ss > 0.f ? rsqrtf(ss) : 0.f;
            }
            if (!pipe && c >= 1 && !previous(c)) break;
            if (h == 0) {
                // features of the Q row t -> TMEM
                if (!wait_phase(bar(B_PROJ), c & 1, abort)) break;
                fence_after();
                float z[LPP];
                {
                    float a[32];
                    ld32(tlane + T_ZQ, a);
#pragma unroll
                    for (int k = 0; k < LPP; ++k) z[k] = a[k];
                }
#pragma unroll
                for (int l = 0; l < LMAX; ++l) {
                    if (l < L) {
                        float u[P], ph[R];
#pragma unroll
                        for (int p = 0; p < P; ++p) u[p] = tc::tanh_abs(z[l * P + p] * inv);
                        tc::bucket_probs<P>(u, beta, ph);
                        if constexpr (R >= 16) {
#pragma unroll
                            for (int b = 0; b < R / 16; ++b) {
                                uint32_t r[8];
#pragma unroll
                                for (int j = 0; j < 8; ++j) r[j] = bfp::pack_bf16(ph[16 * b + 2 * j], ph[16 * b + 2 * j + 1]);
                                stn<8>(tlane + fq + (l * R) / 2 + 8 * b, r);
                            }
                        } else {
                            uint32_t r[R / 2];
#pragma unroll
                            for (int j = 0; j < R / 2; ++j) r[j] = bfp::pack_bf16(ph[2 * j], ph[2 * j + 1]);
                            stn<R / 2>(tlane + fq + (l * R) / 2, r);
                        }
                    }
                }
            } else {
                // the F_K row t (zero past the end) -> shared F_K tile; then the next chunk's rows
                cp_async_wait_all();
                const bool live = t < cnt;
                const uint32_t buf = base + Ly.stage + (uint32_t)(c & 1) * STG_FK;
#pragma unroll
                for (int ch = 0; ch < 8; ++ch) {
                    if (8 * ch < lrs) {
                        const uint4 v = live ? ld_shared_v4(buf + t * 128 + 16 * ch) : make_uint4(0u, 0u, 0u, 0u);
                        st_shared_v4(fk + sw_chunk(t, ch), v.x, v.y, v.z, v.w);
                    }
                }
                if (c + 1 < nchunk) stage_rows(c + 1);
            }
            wait_st();
            warp_signal(bar(B_FEAT));
            if (pipe && c >= 1 && !previous(c)) break;
            // causal mask j <= t on this half's 64 key columns -> bf16 P in TMEM
            if (!wait_phase(bar(B_SC), c & 1, abort)) break;
            fence_after();
            {
                const int j0 = 64 * h;
                const bool need0 = j0 <= 32 * q4 + 31, need1 = j0 + 32 <= 32 * q4 + 31;  // warp-uniform
                uint32_t a0[32], a1[32];
                if (need0) ld32_nw(tlane + T_SC + j0, a0);
                if (need1) ld32_nw(tlane + T_SC + j0 + 32, a1);
                wait_ld();
                reg_fence(a0);
                reg_fence(a1);
#pragma unroll
                for (int b = 0; b < 2; ++b) {
                    const int jb = j0 + 32 * b;
                    uint32_t r0[8], r1[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const int jj = jb + 2 * j;
                        const uint32_t x0 = b ? a1[2 * j] : a0[2 * j], x1 = b ? a1[2 * j + 1] : a0[2 * j + 1];
                        const uint32_t x2 = b ? a1[16 + 2 * j] : a0[16 + 2 * j], x3 = b ? a1[17 + 2 * j] : a0[17 + 2 * j];
                        r0[j] = bfp::pack_bf16(jj <= t ? uf(x0) : 0.f, jj + 1 <= t ? uf(x1) : 0.f);
                        r1[j] = bfp::pack_bf16(jj + 16 <= t ? uf(x2) : 0.f, jj + 17 <= t ? uf(x3) : 0.f);
                    }
                    stn<8>(tlane + T_P + jb / 2, r0);
                    stn<8>(tlane + T_P + jb / 2 + 8, r1);
                }
            }
            wait_st();
            warp_signal(bar(B_MASK));
        }
        if (nchunk > 0 && wait_phase(bar(B_MMA), (nchunk - 1) & 1, abort)) {
            fence_after();
            epilogue(nchunk - 1);
            warp_signal(bar(B_SOP));
        }
        cp_async_wait_all();  // no copy into the staging buffers outlives the CTA (after an abort)
    }
    fence_before();
    __syncthreads();
    if (warp == 0) {
        fence_after();
        tmem_dealloc(tmem, T_COLS);
    }
}

}  // namespace c5

// ------------------------------------------------------------------ host side

cudaError_t make_token_map(CUtensorMap *map, const void *base, const Dims &D);

bool c5_supported(const Dims &D)
{
    return (D.d == 64 || D.d == 128) && D.P >= 1 && D.P <= 6 && D.LP <= nc5::LPP && D.LR <= 64 &&
           D.N <= 0x7FFFFFFF;
}

namespace {

template <int D, int P, int LT>
cudaError_t causal_fwd5_launch(const Dims &Dm, const CUtensorMap &mq, const bf16_t *fk, const CUtensorMap &mv,
                               const CUtensorMap &mo, const float *W, const float *S0, int64_t seg_len, int nseg,
                               unsigned *err, cudaStream_t st)
{
    const c5::FwdLayout Ly(D);
    const size_t smem = Ly.bytes + 1024;
    auto kern = c5::k_causal_fwd5<D, P, LT>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return launch_kernel("tc5_causal_fwd", kern, dim3((unsigned)nseg, (unsigned)Dm.BH), dim3(c5::NTHW), smem, st, mq,
                         fk, mv, mo, Dm, W, S0, seg_len, nseg, err);
}

// (d, P, L) = (128, 3, 3) runs with L compiled in; every other shape with L at run time.
template <int D, int P>
cudaError_t causal_fwd5_inst(const Dims &Dm, const CUtensorMap &mq, const bf16_t *fk, const CUtensorMap &mv,
                             const CUtensorMap &mo, const float *W, const float *S0, int64_t seg_len, int nseg,
                             unsigned *err, cudaStream_t st)
{
    if constexpr (D == 128 && P == 3)
        if (Dm.L == 3) return causal_fwd5_launch<D, P, 3>(Dm, mq, fk, mv, mo, W, S0, seg_len, nseg, err, st);
    return causal_fwd5_launch<D, P, 0>(Dm, mq, fk, mv, mo, W, S0, seg_len, nseg, err, st);
}

}  // namespace

cudaError_t launch_c5_fwd(const Dims &Dm, const bf16_t *Q, const bf16_t *fk, const bf16_t *V, const float *W,
                          const float *S0, int64_t seg_len, int nseg, bf16_t *O, unsigned *err, cudaStream_t st)
{
    CUtensorMap mq, mv, mo;
    cudaError_t e = make_token_map(&mq, Q, Dm);
    if (e == cudaSuccess) e = make_token_map(&mv, V, Dm);
    if (e == cudaSuccess) e = make_token_map(&mo, O, Dm);
    if (e != cudaSuccess) return e;
    switch (Dm.d * 16 + Dm.P) {
        case 64 * 16 + 1: return causal_fwd5_inst<64, 1>(Dm, mq, fk, mv, mo, W, S0, seg_len, nseg, err, st);
        case 64 * 16 + 2: return causal_fwd5_inst<64, 2>(Dm, mq, fk, mv, mo, W, S0, seg_len, nseg, err, st);
        case 64 * 16 + 3: return causal_fwd5_inst<64, 3>(Dm, mq, fk, mv, mo, W, S0, seg_len, nseg, err, st);
        case 64 * 16 + 4: return causal_fwd5_inst<64, 4>(Dm, mq, fk, mv, mo, W, S0, seg_len, nseg, err, st);
        case 64 * 16 + 5: return causal_fwd5_inst<64, 5>(Dm, mq, fk, mv, mo, W, S0, seg_len, nseg, err, st);
        case 64 * 16 + 6: return causal_fwd5_inst<64, 6>(Dm, mq, fk, mv, mo, W, S0, seg_len, nseg, err, st);
        case 128 * 16 + 1: return causal_fwd5_inst<128, 1>(Dm, mq, fk, mv, mo, W, S0, seg_len, nseg, err, st);
        case 128 * 16 + 2: return causal_fwd5_inst<128, 2>(Dm, mq, fk, mv, mo, W, S0, seg_len, nseg, err, st);
        case 128 * 16 + 3: return causal_fwd5_inst<128, 3>(Dm, mq, fk, mv, mo, W, S0, seg_len, nseg, err, st);
        case 128 * 16 + 4: return causal_fwd5_inst<128, 4>(Dm, mq, fk, mv, mo, W, S0, seg_len, nseg, err, st);
        case 128 * 16 + 5: return causal_fwd5_inst<128, 5>(Dm, mq, fk, mv, mo, W, S0, seg_len, nseg, err, st);
        case 128 * 16 + 6: return causal_fwd5_inst<128, 6>(Dm, mq, fk, mv, mo, W, S0, seg_len, nseg, err, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace race
