// race_bf16.cuh -- packing of float pairs into bf16x2 words (round to nearest even), the form in
// which the kernels write tensor-core operands to shared memory and TMEM.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

namespace race {
namespace bfp {

// Two floats as one bf16x2 word: lo in the low half, hi in the high half.
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi)
{
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

}  // namespace bfp
}  // namespace race
