// race_common.cuh -- types shared by the RACE attention kernels and their host launchers.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace race {

using bf16_t = __nv_bfloat16;

constexpr int kMaxP = 8;     // hyperplanes per table
constexpr int kMaxL = 16;    // tables
constexpr int kMaxLR = 256;  // L * 2^P, the width of the concatenated bucket-feature vector
constexpr int kMaxD = 128;   // head dimension

// Problem dimensions as the kernels see them.  dv = d + 1: a sketch row holds the d content
// columns (A = Phi_K^T V) followed by the mass column (B = Phi_K^T 1).
struct Dims {
    int64_t BH;  // B * H independent (batch, head) problems
    int64_t N;   // tokens per problem
    int d, L, P, R, LR, LP, dv;
    float beta;
    int64_t H;       // heads (problem bh is head bh % H)
    int w_per_head;  // 0: one W [L, P, d] for every head; 1: W is [H, L, P, d]
    int sms;         // streaming multiprocessors of the device the work is planned for
    int withhold;    // failure-path test hook: the causal tcgen05 forward skips its first tile load
    // d(loss)/d(W) (null unless asked for): every backward kernel writes each Q row's (dzq) and K
    // row's (dzk) projection gradient dz / |x| as L P floats, [BH][N][dzld] (dzld = L P rounded up
    // to a multiple of 4, so that rows start on 16 bytes); a reduction then forms
    // dW = sum over rows of (dz / |x|) x^T
    float *dzq, *dzk;
    int dzld;
};

// Bits of the device status word (the first word of a workspace): a bounded wait ran out, or a
// read-out met a denominator that is zero, negative or not finite (its output row is 0/0).
constexpr unsigned kErrTimeout = 1u;
constexpr unsigned kErrNumeric = 2u;

// Records a degenerate denominator of one output row in the status word (err may be null).
__device__ __forceinline__ void flag_den(float den, unsigned *err)
{
    if (err != nullptr && !(den > 0.f && den <= 3.402823466e38f)) atomicOr(err, kErrNumeric);
}

// The hyperplanes problem bh hashes with: the shared W, or its head's slice of a per-head W.
__host__ __device__ inline const float *head_w(const float *W, const Dims &D, int64_t bh)
{
    return D.w_per_head ? W + (bh % D.H) * (int64_t)D.LP * D.d : W;
}

__device__ __forceinline__ float ld_f(const float *p, int64_t i) { return p[i]; }
__device__ __forceinline__ float ld_f(const __nv_bfloat16 *p, int64_t i) { return __bfloat162float(p[i]); }
__device__ __forceinline__ void st_f(float *p, int64_t i, float v) { p[i] = v; }
__device__ __forceinline__ void st_f(__nv_bfloat16 *p, int64_t i, float v) { p[i] = __float2bfloat16_rn(v); }

// Sum of one float per thread over the CTA in a fixed order (butterflies within each warp, then
// the warps in index order), so that a reduction gives the same bits on every run.  Every
// thread of the block calls it; `scratch` holds one float per warp and may be in use until the
// call.  The total is returned in thread 0.
__device__ __forceinline__ float block_sum_fixed(float v, float *scratch)
{
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
    const int warp = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
    __syncthreads();
    if ((threadIdx.x & 31) == 0) scratch[warp] = v;
    __syncthreads();
    float s = 0.f;
    if (threadIdx.x == 0)
        for (int w = 0; w < nw; ++w) s += scratch[w];
    return s;
}

// Bump allocator for dynamic shared memory layouts, usable on host (to size the launch) and
// device (to find the regions); every region starts on a 16-byte boundary.
struct SmemLayout {
    int used = 0;  // in floats
    __host__ __device__ int take(int nfloats) {
        int at = used;
        used += (nfloats + 3) & ~3;
        return at;
    }
    __host__ __device__ size_t bytes() const { return (size_t)used * sizeof(float); }
};

}  // namespace race
