// Shared device helpers of the GDN prefill library (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "../../include/gdn.h"

namespace gdn {

// Kernels whose waits are bounded keep an error word in their own translation
// unit (`static __device__ int`, no relocatable device code): when a wait runs
// out they record a code there and return early; gdn_sync_status() reads and
// clears every such word through the unit's host accessor.
enum : int { ERR_NONE = 0, ERR_WAIT_TIMEOUT = 1 };

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
    return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

__device__ __forceinline__ uint16_t float_to_bf16_bits(float f) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

__device__ __forceinline__ uint16_t code_to_f16_bits(int q) {
    return __half_as_ushort(__int2half_rn(q));
}

// int8 quantisation code of w for the row scale s (s = amax/127):
// clamp(rne(w / s), -127, 127) with an IEEE-correct fp32 divide; s == 0 -> 0.
__device__ __forceinline__ int quant_code(float w, float s) {
    if (s == 0.0f) return 0;
    int q = __float2int_rn(__fdiv_rn(w, s));
    return max(-127, min(127, q));
}

__device__ __forceinline__ float silu_f(float u) { return u / (1.0f + expf(-u)); }

// fp32 -> tf32 (10 explicit mantissa bits), round to nearest, ties away; as fp32 bits.
__device__ __forceinline__ uint32_t tf32_bits(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}
__device__ __forceinline__ float round_tf32(float x) { return __uint_as_float(tf32_bits(x)); }

// Block-wide max of a non-negative value; all threads get the result.
// `red` must hold 32 floats of shared memory.
__device__ __forceinline__ float block_max(float v, float* red) {
    v = warp_max(v);
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    __syncthreads();
    if (l == 0) red[w] = v;
    __syncthreads();
    const int nw = (blockDim.x + 31) >> 5;
    float r = (l < nw) ? red[l] : 0.0f;
    return warp_max(r);
}

}  // namespace gdn
