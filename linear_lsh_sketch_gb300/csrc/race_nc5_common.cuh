// race_nc5_common.cuh -- pieces shared by the tcgen05 (TMEM accumulator) RACE kernels: tile
// geometry, the hyperplane operand tiles, row norms, the bucket-feature writer and bounded
// mbarrier waits.
//
// Token tiles are C = 128 rows of a [N, d] slice, loaded by TMA as d / 64 SW128 column blocks
// (race_tc5.cuh).  Eight warps share a tile: warp w reads TMEM lanes 32 (w % 4) .. + 31, so
// thread (w, lane) owns token row t = 32 (w % 4) + lane, and the two warps of a lane quadrant
// (half h = w / 4) split that row's work.
#pragma once

#include "race_common.cuh"
#include "race_tc5.cuh"

namespace race {
namespace nc5 {

using bf16 = __nv_bfloat16;
using namespace race::tc5;

constexpr int C = 128;           // tokens per tile
constexpr int NTH = 256;         // threads per CTA
constexpr uint32_t BLK = C * 128;  // bytes of one SW128 column block of a token tile
constexpr int LPP = 32;          // projection columns (L * P <= 32): z occupies 32 TMEM columns
constexpr uint32_t WBLK = LPP * 128;  // bytes of one SW128 column block of a hyperplane tile

// Hyperplanes as bf16 hi and lo SW128 tiles [D / 64][LPP rows][64]: row p = W row p (p < L P),
// zero rows after; hi + lo == W to about 2^-16 relative.
template <int D>
__device__ __forceinline__ void load_w_tiles(const float *__restrict__ W, int LP, unsigned char *whi,
                                             unsigned char *wlo)
{
    for (int i = threadIdx.x; i < LPP * (D / 8); i += NTH) {
        const int row = i / (D / 8), c = i - row * (D / 8);  // 8-element chunk c of row `row`
        uint32_t h[4], l[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            float w0 = 0.f, w1 = 0.f;
            if (row < LP) {
                w0 = W[row * D + 8 * c + 2 * j];
                w1 = W[row * D + 8 * c + 2 * j + 1];
            }
            const bf16 h0 = __float2bfloat16_rn(w0), h1 = __float2bfloat16_rn(w1);
            h[j] = bfp::pack_bf16(__bfloat162float(h0), __bfloat162float(h1));
            l[j] = bfp::pack_bf16(w0 - __bfloat162float(h0), w1 - __bfloat162float(h1));
        }
        const uint32_t off = (c >> 3) * WBLK + sw_chunk(row, c & 7);
        st_shared_v4(smem_addr(whi) + off, h[0], h[1], h[2], h[3]);
        st_shared_v4(smem_addr(wlo) + off, l[0], l[1], l[2], l[3]);
    }
}

__device__ __forceinline__ void zero_region(unsigned char *p, uint32_t nbytes)
{
    for (uint32_t i = threadIdx.x * 16; i < nbytes; i += NTH * 16) st_shared_v4(smem_addr(p) + i, 0, 0, 0, 0);
}

// The 4 KB mass operand (K-major, N = 16 rows, K = 128 tokens as two 64-token SW128 blocks of
// 2 KB): row 0 all ones when `ones`, every other element zero.  Row 0 of a swizzle atom is not
// permuted, so it is the first 128 bytes of each block.  Each address has one writer.
__device__ __forceinline__ void init_mass_tile(unsigned char *p, bool ones)
{
    const uint32_t one2 = ones ? 0x3F803F80u : 0u;
    for (uint32_t i = threadIdx.x * 16; i < 4096; i += NTH * 16) {
        const uint32_t v = (i & 2047) < 128 ? one2 : 0u;
        st_shared_v4(smem_addr(p) + i, v, v, v, v);
    }
}

// Half h's share of sum_k x[t][k]^2 for row t of a token tile at `tile` (D / 64 column blocks).
template <int D>
__device__ __forceinline__ float half_sumsq(uint32_t tile, int t, int h)
{
    uint4 w[D / 16];  // all loads first, then four independent accumulation chains
#pragma unroll
    for (int j = 0; j < D / 16; ++j) {
        const int c = h * (D / 16) + j;
        w[j] = ld_shared_v4(tile + (c >> 3) * BLK + sw_chunk(t, c & 7));
    }
    float s[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int j = 0; j < D / 16; ++j) {
        const uint32_t q[4] = {w[j].x, w[j].y, w[j].z, w[j].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float lo = __uint_as_float(q[i] << 16), hi = __uint_as_float(q[i] & 0xFFFF0000u);
            s[i] = fmaf(lo, lo, fmaf(hi, hi, s[i]));
        }
    }
    return (s[0] + s[1]) + (s[2] + s[3]);
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(bar) : "memory");
}

// Bounded wait for the phase with parity `parity` that also gives up as soon as another thread
// of the CTA has raised `*abort`.  A wait that runs out (tc::kWaitLimitNs or 2^22 polls) raises
// `*abort` itself.  Returns true when the phase completed.
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, volatile int *abort)
{
    if (tc::mbar_try(bar, parity)) return true;
    const uint64_t t0 = tc::globaltimer_ns();
    for (int i = 1; i < (1 << 22); ++i) {
        if (tc::mbar_try(bar, parity)) return true;
        if ((i & 15) == 0) {
            if (*abort) return false;
            if (tc::globaltimer_ns() - t0 > tc::kWaitLimitNs) break;
        }
    }
    *abort = 1;
    return false;
}

// wait_phase for a converged warp: every lane polls and all lanes return the same result, so the
// warp stays converged for the elect.sync issue that follows.
__device__ __forceinline__ bool wait_phase_w(uint32_t bar, uint32_t parity, volatile int *abort)
{
    if (__all_sync(0xffffffffu, tc::mbar_try(bar, parity))) return true;
    const uint64_t t0 = tc::globaltimer_ns();
    for (int i = 1; i < (1 << 22); ++i) {
        if (__all_sync(0xffffffffu, tc::mbar_try(bar, parity))) return true;
        if ((i & 15) == 0) {
            if (__any_sync(0xffffffffu, *abort != 0)) return false;
            if (__any_sync(0xffffffffu, tc::globaltimer_ns() - t0 > tc::kWaitLimitNs)) break;
        }
    }
    *abort = 1;
    return false;
}

// Per-barrier counts of copies issued or waited for (to drain the copies in flight after an
// abort), kept in registers: a run-time index into a plain array would put it in local memory,
// whose lines the small L1 left beside a large shared-memory carve-out does not keep.
template <int N>
struct Counts {
    int v[N];
    __device__ __forceinline__ Counts()
    {
#pragma unroll
        for (int j = 0; j < N; ++j) v[j] = 0;
    }
    __device__ __forceinline__ void inc(int b)
    {
#pragma unroll
        for (int j = 0; j < N; ++j) v[j] += j == b ? 1 : 0;
    }
};

// Non-blocking check of the phase with parity `parity`.
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Hands the warp's finished work to the issuing thread: every lane orders its shared-memory
// writes before later async-proxy reads and its TMEM stores before the hand-off; lane 0 then
// arrives once on `bar` (whose count is the number of handing-off warps).
__device__ __forceinline__ void warp_signal(uint32_t bar)
{
    tc::fence_proxy_async();
    fence_before();
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
}

// Barrier among the threads that share `bar` (its count): arrive, then a bounded wait for the
// phase with parity `parity`.  Unlike bar.sync it cannot strand a thread when another has left
// its loop after an abort.
__device__ __forceinline__ bool group_sync(uint32_t bar, uint32_t parity, volatile int *abort)
{
    mbar_arrive(bar);
    return wait_phase(bar, parity, abort);
}

// Bounded wait by every thread, then a CTA-wide vote: true if any thread's wait ran out.
__device__ __forceinline__ bool wait_all(uint32_t bar, uint32_t parity)
{
    const bool ok = mbar_wait(bar, parity);
    return __syncthreads_or(!ok) != 0;
}

// 16 bytes from global memory that no kernel writes while this one runs (no L1 allocation).
__device__ __forceinline__ uint4 ld_global_nc_v4(const void *p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.b32 {%0, %1, %2, %3}, [%4];\n"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// Asynchronous global -> shared copies that complete per thread (cp.async): 16 bytes (L2 only),
// 8 or 4 bytes; commit closes this thread's group, wait_all waits for all of its groups.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async8(uint32_t dst, const void *src)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;\n" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async4(uint32_t dst, const void *src)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;\n" ::: "memory"); }

// 16 bytes to global memory without allocating in L1.
__device__ __forceinline__ void st_global_v4(void *p, uint4 v)
{
    asm volatile("st.global.L1::no_allocate.v4.b32 [%0], {%1, %2, %3, %4};\n" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
}

// Stored bucket-feature rows (phi(K) of the keys, F'_Q of the causal backward) hold L R bf16 values
// padded with zeros to a multiple of 8, so that every row is a whole number of 16-byte chunks.
__host__ __device__ constexpr int feature_row_stride(int LR) { return (LR + 7) & ~7; }

// The P projections of table l (run time, warp-uniform) from the register array z, by selects:
// indexing z with a run-time l would move it to local memory.
template <int P>
__device__ __forceinline__ void table_z(const float (&z)[LPP], int l, float (&zl)[P])
{
    constexpr int LMAX = LPP / P;
#pragma unroll
    for (int p = 0; p < P; ++p) zl[p] = z[p];
#pragma unroll
    for (int j = 1; j < LMAX; ++j) {
        if (l == j) {
#pragma unroll
            for (int p = 0; p < P; ++p) zl[p] = z[j * P + p];
        }
    }
}

// Writes one token row of bucket features into an SW128 feature tile ([lr / 64][C][64] bf16,
// lr = l R + r), for the tables half h owns: tables l with l % 2 == h when R >= 8, else 16-byte
// chunks (8 / R tables each) with chunk % 2 == h.  z holds the row's projections W x (LPP
// columns), inv = 1 / |x|; phi^(l)_r = prod_t sigmoid(2 beta u_t v_{r,t}) with
// u = tanh(z inv) (the softmax over hypercube corners in product form), times `scale`.
// Tables >= L inside a written chunk are zero.  grow (may be null): the token's stored feature
// row in global memory (feature_row_stride(L R) bf16), which receives the same 16-byte chunks.
// ROLL: one copy of the per-table code, looped over the tables at run time (with 32 or more
// buckets per table the unrolled copies overflow the instruction cache).
template <int P, bool ROLL = (1 << P) >= 32>
__device__ __forceinline__ void write_features(const float (&z)[LPP], float inv, float beta, int L, int h,
                                               float scale, int t, uint32_t ftile, bf16 *grow = nullptr)
{
    constexpr int R = 1 << P;
    constexpr int LMAX = LPP / P;
    if constexpr (R >= 8) {
        auto table = [&](int l) {
            float u[P], ph[R], zl[P];
            table_z<P>(z, l, zl);
#pragma unroll
            for (int p = 0; p < P; ++p) u[p] = tc::tanh_abs(zl[p] * inv);
            tc::bucket_probs<P>(u, beta, ph);
#pragma unroll
            for (int j = 0; j < R / 8; ++j) {
                const int c = l * (R / 8) + j;
                const uint4 v = make_uint4(bfp::pack_bf16(ph[8 * j] * scale, ph[8 * j + 1] * scale),
                                           bfp::pack_bf16(ph[8 * j + 2] * scale, ph[8 * j + 3] * scale),
                                           bfp::pack_bf16(ph[8 * j + 4] * scale, ph[8 * j + 5] * scale),
                                           bfp::pack_bf16(ph[8 * j + 6] * scale, ph[8 * j + 7] * scale));
                st_shared_v4(ftile + (c >> 3) * BLK + sw_chunk(t, c & 7), v.x, v.y, v.z, v.w);
                if (grow) st_global_v4(grow + 8 * c, v);
            }
        };
        if constexpr (ROLL) {
#pragma unroll 1
            for (int l = h; l < L; l += 2) table(l);
        } else {
#pragma unroll
            for (int l = 0; l < LMAX; ++l)
                if (l < L && (l & 1) == h) table(l);
        }
    } else {
        constexpr int TPC = 8 / R;
        constexpr int NCH = (LMAX + TPC - 1) / TPC;
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
            if (c * TPC < L && (c & 1) == h) {
                float v[8];
#pragma unroll
                for (int k = 0; k < TPC; ++k) {
                    const int l = c * TPC + k;
                    float ph[R];
                    if (l < L && l < LMAX) {
                        float u[P];
#pragma unroll
                        for (int p = 0; p < P; ++p) u[p] = tc::tanh_abs(z[(l < LMAX ? l : 0) * P + p] * inv);
                        tc::bucket_probs<P>(u, beta, ph);
                    } else {
#pragma unroll
                        for (int r = 0; r < R; ++r) ph[r] = 0.f;
                    }
#pragma unroll
                    for (int r = 0; r < R; ++r) v[k * R + r] = ph[r] * scale;
                }
                const uint4 w = make_uint4(bfp::pack_bf16(v[0], v[1]), bfp::pack_bf16(v[2], v[3]),
                                           bfp::pack_bf16(v[4], v[5]), bfp::pack_bf16(v[6], v[7]));
                st_shared_v4(ftile + (c >> 3) * BLK + sw_chunk(t, c & 7), w.x, w.y, w.z, w.w);
                if (grow) st_global_v4(grow + 8 * c, w);
            }
        }
    }
}

// Chain rule from dphi (one table, R values, phi recomputed from u) to the table's P
// projection gradients dz_p = beta * sum_r phi_r (dphi_r - phi . dphi) v_{r,p} * (1 - u_p^2).
// DB: also adds the table's d(loss)/d(beta) share to *db.  The logits are beta (u . v_r), so
// that share is sum_r ds_r (u . v_r) = sum_p u_p du_p with du_p = sum_r ds_r v_{r,p}, the sum
// formed here before the scaling by beta.
template <int P, bool DB = false>
__device__ __forceinline__ void table_backward(const float (&u)[P], const float (&ph)[1 << P],
                                               const float (&dph)[1 << P], float beta, float *dz,
                                               float *db = nullptr)
{
    constexpr int R = 1 << P;
    float s = 0.f;
#pragma unroll
    for (int r = 0; r < R; ++r) s = fmaf(ph[r], dph[r], s);
    float du[P];
    if constexpr (P >= 4) {
        // du_p = (sum over corners with bit p set) - (sum over the others), folding the hypercube
        // one bit at a time from the highest: 3 (R - 1) additions instead of R P
        float ds[R];
#pragma unroll
        for (int r = 0; r < R; ++r) ds[r] = ph[r] * (dph[r] - s);
#pragma unroll
        for (int p = P - 1; p >= 0; --p) {
            const int half = 1 << p;
            float hi = 0.f, lo = 0.f;
#pragma unroll
            for (int r = 0; r < (R >> 1); ++r) {
                if (r < half) {
                    hi += ds[r + half];
                    lo += ds[r];
                    ds[r] += ds[r + half];
                }
            }
            du[p] = hi - lo;
        }
    } else {
#pragma unroll
        for (int p = 0; p < P; ++p) du[p] = 0.f;
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const float ds = ph[r] * (dph[r] - s);
#pragma unroll
            for (int p = 0; p < P; ++p) du[p] += ((r >> p) & 1) ? ds : -ds;
        }
    }
    if constexpr (DB) {
        float a = *db;
#pragma unroll
        for (int p = 0; p < P; ++p) a = fmaf(u[p], du[p], a);
        *db = a;
    }
#pragma unroll
    for (int p = 0; p < P; ++p) dz[p] = beta * du[p] * (1.f - u[p] * u[p]);
}

// R consecutive fp32 TMEM columns of this thread's lane.
template <int R>
__device__ __forceinline__ void ld_cols(uint32_t taddr, float (&v)[R])
{
    if constexpr (R <= 16) {
        ldn<R>(taddr, v);
    } else {
#pragma unroll
        for (int k = 0; k < R / 32; ++k) {
            float a[32];
            ld32(taddr + 32 * k, a);
#pragma unroll
            for (int j = 0; j < 32; ++j) v[32 * k + j] = a[j];
        }
    }
}

// Instruction descriptors.
__host__ __device__ constexpr uint32_t idesc_proj() { return idesc_bf16(128, LPP, 0, 0); }

// 32 bf16 (64 bytes, packed pairs in o) of one output row to global memory: two 32-byte stores
// when `wide` (the tensor's base is 32-byte aligned, so every row segment is), else four 16-byte
// stores.  Full 32-byte sectors halve the store instructions of a row-per-thread epilogue.  The
// stores do not allocate in L1: with most of L1 given to shared memory, output lines would evict
// the few lines that hold register spills.
__device__ __forceinline__ void store_row32(bf16 *dst, const uint32_t (&o)[16], bool wide)
{
    if (wide) {
        asm volatile("st.global.L1::no_allocate.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};\n" ::"l"(dst), "r"(o[0]),
                     "r"(o[1]), "r"(o[2]), "r"(o[3]), "r"(o[4]), "r"(o[5]), "r"(o[6]), "r"(o[7])
                     : "memory");
        asm volatile("st.global.L1::no_allocate.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};\n" ::"l"(dst + 16),
                     "r"(o[8]), "r"(o[9]), "r"(o[10]), "r"(o[11]), "r"(o[12]), "r"(o[13]), "r"(o[14]), "r"(o[15])
                     : "memory");
    } else {
#pragma unroll
        for (int q = 0; q < 4; ++q)
            asm volatile("st.global.L1::no_allocate.v4.b32 [%0], {%1, %2, %3, %4};\n" ::"l"(dst + 8 * q), "r"(o[4 * q]),
                         "r"(o[4 * q + 1]), "r"(o[4 * q + 2]), "r"(o[4 * q + 3])
                         : "memory");
    }
}

// Issues z = X (W_hi + W_lo)^T for a token tile (D / 16 K steps per hyperplane copy).
template <int D>
__device__ __forceinline__ void issue_projection(uint32_t tz, uint32_t xtile, uint32_t whi, uint32_t wlo)
{
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
        const uint32_t ko = (ks >> 2) * BLK + (ks & 3) * 32, kw = (ks >> 2) * WBLK + (ks & 3) * 32;
        umma(tz, desc_k(xtile + ko), desc_k(whi + kw), idesc_proj(), ks > 0);
    }
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
        const uint32_t ko = (ks >> 2) * BLK + (ks & 3) * 32, kw = (ks >> 2) * WBLK + (ks & 3) * 32;
        umma(tz, desc_k(xtile + ko), desc_k(wlo + kw), idesc_proj(), true);
    }
}

// Hyperplane tiles in pair layout: per 64-column block kb, the hi rows then the lo rows,
// [D / 64][hi 32 rows | lo 32 rows][64] (2 WBLK bytes per block), so that one K-major operand of
// N = 64 rows holds both halves.
template <int D>
__device__ __forceinline__ void load_w_pair(const float *__restrict__ W, int LP, unsigned char *wp)
{
    for (int i = threadIdx.x; i < LPP * (D / 8); i += NTH) {
        const int row = i / (D / 8), c = i - row * (D / 8);
        uint32_t h[4], l[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            float w0 = 0.f, w1 = 0.f;
            if (row < LP) {
                w0 = W[row * D + 8 * c + 2 * j];
                w1 = W[row * D + 8 * c + 2 * j + 1];
            }
            const bf16 h0 = __float2bfloat16_rn(w0), h1 = __float2bfloat16_rn(w1);
            h[j] = bfp::pack_bf16(__bfloat162float(h0), __bfloat162float(h1));
            l[j] = bfp::pack_bf16(w0 - __bfloat162float(h0), w1 - __bfloat162float(h1));
        }
        const uint32_t off = (c >> 3) * 2 * WBLK + sw_chunk(row, c & 7);
        st_shared_v4(smem_addr(wp) + off, h[0], h[1], h[2], h[3]);
        st_shared_v4(smem_addr(wp) + off + WBLK, l[0], l[1], l[2], l[3]);
    }
}

// z = X (W_hi + W_lo)^T from pair-layout tiles.  MERGED: one N = 64 product per K step that
// leaves X W_hi^T in columns tz .. tz + 31 and X W_lo^T in tz + 32 .. tz + 63 (the reader adds
// them); otherwise both into tz .. tz + 31.
template <int D, bool MERGED>
__device__ __forceinline__ void issue_projection_pair(uint32_t tz, uint32_t xtile, uint32_t wp)
{
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
        const uint32_t ko = (ks >> 2) * BLK + (ks & 3) * 32, kw = (ks >> 2) * 2 * WBLK + (ks & 3) * 32;
        if constexpr (MERGED) {
            umma(tz, desc_k(xtile + ko), desc_k(wp + kw), idesc_bf16(128, 2 * LPP, 0, 0), ks > 0);
        } else {
            umma(tz, desc_k(xtile + ko), desc_k(wp + kw), idesc_proj(), ks > 0);
            umma(tz, desc_k(xtile + ko), desc_k(wp + kw + WBLK), idesc_proj(), true);
        }
    }
}

// The same, issued by a converged warp (one elected lane).
template <int D>
__device__ __forceinline__ void issue_projection_w(uint32_t tz, uint32_t xtile, uint32_t whi, uint32_t wlo)
{
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
        const uint32_t ko = (ks >> 2) * BLK + (ks & 3) * 32, kw = (ks >> 2) * WBLK + (ks & 3) * 32;
        umma_w(tz, desc_k(xtile + ko), desc_k(whi + kw), idesc_proj(), ks > 0);
    }
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
        const uint32_t ko = (ks >> 2) * BLK + (ks & 3) * 32, kw = (ks >> 2) * WBLK + (ks & 3) * 32;
        umma_w(tz, desc_k(xtile + ko), desc_k(wlo + kw), idesc_proj(), true);
    }
}

}  // namespace nc5
}  // namespace race
