// Elementwise pieces of the fused epilogue shared by the GEMM kernel and the
// K == 0 path: activations and the bf16 output conversion.
#pragma once

#include <cuda_bf16.h>

#include <cstdint>

namespace tg {

// Two fp32 bit patterns -> two bf16 (round to nearest even), low half first.
__device__ __forceinline__ uint32_t pack_bf16x2(uint32_t lo, uint32_t hi)
{
    const __nv_bfloat162 h = __floats2bfloat162_rn(__uint_as_float(lo), __uint_as_float(hi));
    return *reinterpret_cast<const uint32_t *>(&h);
}

// Activations of the fused epilogue (codes as in tg_activation).
__device__ __forceinline__ float activation(float x, int32_t act)
{
    switch (act) {
        case 1:  // relu
            return fmaxf(x, 0.0f);
        case 2: {  // gelu, tanh form
            const float u = 0.7978845608028654f * (x + 0.044715f * x * x * x);
            return 0.5f * x * (1.0f + tanhf(u));
        }
        case 3:  // silu
            return x / (1.0f + expf(-x));
        default:
            return x;
    }
}

}  // namespace tg
