// race_tc_common.cuh -- pieces shared by the tcgen05 kernels: mbarriers with bounded waits, the
// global timer, and the nonlinearities of the bucket features (tanh, sigmoid pairs, the product
// form of the corner softmax).
#pragma once

#include "race_common.cuh"
#include "race_bf16.cuh"

namespace race {
namespace tc {

using bf16 = __nv_bfloat16;

// ------------------------------------------------------------------ mbarriers

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

}  // namespace tc
}  // namespace race
