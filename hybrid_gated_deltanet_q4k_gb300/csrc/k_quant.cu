// Step 1b: per-token int8 quantisation of the bf16 activations.
//
// The int8 projections of the pages (sparkinfer PR #464, Summary) take int8
// rows with one fp32 scale each; the activation side is quantised the same
// way as the weights: scale = amax/127, code = clamp(rne(x/scale), -127, 127),
// IEEE fp32.  One CTA per row; the row (<= 16384 values) stays in registers
// between the amax reduction and the quantisation, so the kernel reads each
// input byte once and writes each code once, with 16-byte accesses.
#include "common.cuh"

namespace gdn {

constexpr int QR_THREADS = 256;
constexpr int QR_MAX_VEC = 16384 / 8 / QR_THREADS;  // 16-byte vectors per thread

__global__ void __launch_bounds__(QR_THREADS)
quant_rows_bf16_kernel(const uint16_t* __restrict__ x, int cols, uint16_t* __restrict__ codes,
                       float* __restrict__ scale) {
    __shared__ float red[32];
    const int64_t row = blockIdx.x;
    const int nvec = cols >> 3;
    const uint4* src = reinterpret_cast<const uint4*>(x + row * cols);
    uint4 v[QR_MAX_VEC];
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < QR_MAX_VEC; ++i) {
        const int j = threadIdx.x + i * QR_THREADS;
        if (j < nvec) {
            v[i] = __ldg(src + j);
            const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                amax = fmaxf(amax, fabsf(__uint_as_float(w[e] << 16)));
                amax = fmaxf(amax, fabsf(__uint_as_float(w[e] & 0xffff0000u)));
            }
        }
    }
    amax = block_max(amax, red);
    const float s = __fdiv_rn(amax, 127.0f);
    if (threadIdx.x == 0) scale[row] = s;
    uint4* dst = reinterpret_cast<uint4*>(codes + row * cols);
#pragma unroll
    for (int i = 0; i < QR_MAX_VEC; ++i) {
        const int j = threadIdx.x + i * QR_THREADS;
        if (j < nvec) {
            const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
            uint32_t o[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int q0 = quant_code(__uint_as_float(w[e] << 16), s);
                const int q1 = quant_code(__uint_as_float(w[e] & 0xffff0000u), s);
                o[e] = static_cast<uint32_t>(code_to_f16_bits(q0)) | (static_cast<uint32_t>(code_to_f16_bits(q1)) << 16);
            }
            dst[j] = make_uint4(o[0], o[1], o[2], o[3]);
        }
    }
}

cudaError_t launch_quant_rows(const uint16_t* x, int64_t rows, int64_t cols, uint16_t* codes, float* scale,
                              cudaStream_t st) {
    quant_rows_bf16_kernel<<<static_cast<unsigned>(rows), QR_THREADS, 0, st>>>(x, static_cast<int>(cols), codes, scale);
    return cudaGetLastError();
}

}  // namespace gdn
