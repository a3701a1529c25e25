// Step 1b: per-token int8 quantisation of the bf16 activations.
//
// The int8 projections of the pages (sparkinfer PR #464, Summary) take int8
// rows with one fp32 scale each; the activation side is quantised the same
// way as the weights: scale = amax/127, code = clamp(rne(x/scale), -127, 127),
// IEEE fp32 (the fast quantiser of common.cuh returns exactly those codes).
// One CTA per row with up to QR_VEC 16-byte vectors per thread, all loads
// issued before the first use; the row stays in registers between the amax
// reduction and the quantisation, so the kernel reads each input byte once and
// writes each code once.  Rows of up to 4096 values take 64-thread CTAs (two
// warps per row, up to 32 rows resident per SM), longer rows 256 threads.
#include "common.cuh"
#include "qk_decode.cuh"

namespace gdn {

static __device__ int g_quant_error;   // index checks of the debug build

constexpr int QR_VEC = 8;   // 16-byte vectors per thread

template <int THREADS>
__global__ void __launch_bounds__(THREADS)
quant_rows_bf16_kernel(const uint16_t* __restrict__ x, int64_t rows, int cols, uint16_t* __restrict__ codes,
                       float* __restrict__ scale) {
    pdl_trigger();
    __shared__ float red[32];
    const int64_t row = blockIdx.x;
    const int nvec = cols >> 3;
    const uint4* src = reinterpret_cast<const uint4*>(x + row * cols);
    uint4 v[QR_VEC];
#pragma unroll
    for (int i = 0; i < QR_VEC; ++i) {
        const int j = threadIdx.x + i * THREADS;
        if (j < nvec) v[i] = __ldg(src + j);
    }
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < QR_VEC; ++i) {
        if (static_cast<int>(threadIdx.x) + i * THREADS < nvec) {
            const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                amax = fmaxf(amax, fabsf(__uint_as_float(w[e] << 16)));
                amax = fmaxf(amax, fabsf(__uint_as_float(w[e] & 0xffff0000u)));
            }
        }
    }
    amax = block_max(amax, red);
    const QScale qsc = make_qscale(amax);
    const bool row_ok = GDN_IN_RANGE(g_quant_error, row < rows);
    if (threadIdx.x == 0 && row_ok) scale[row] = qsc.s;
    uint4* dst = reinterpret_cast<uint4*>(codes + row * cols);
#pragma unroll
    for (int i = 0; i < QR_VEC; ++i) {
        const int j = threadIdx.x + i * THREADS;
        if (j < nvec && row_ok) {
            const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
            float xv[8], c[8];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                xv[2 * e] = __uint_as_float(w[e] << 16);
                xv[2 * e + 1] = __uint_as_float(w[e] & 0xffff0000u);
            }
            quantise8(xv, qsc, c);
            dst[j] = make_uint4(codes_to_f16x2(c[0], c[1]), codes_to_f16x2(c[2], c[3]), codes_to_f16x2(c[4], c[5]),
                                codes_to_f16x2(c[6], c[7]));
        }
    }
}

cudaError_t launch_quant_rows(const uint16_t* x, int64_t rows, int64_t cols, uint16_t* codes, float* scale,
                              cudaStream_t st) {
    static_assert(16384 / 8 <= QR_VEC * 256, "the widest row must fit a 256-thread CTA");
    if (cols <= QR_VEC * 64 * 8)
        quant_rows_bf16_kernel<64><<<static_cast<unsigned>(rows), 64, 0, st>>>(x, rows, static_cast<int>(cols), codes, scale);
    else
        quant_rows_bf16_kernel<256><<<static_cast<unsigned>(rows), 256, 0, st>>>(x, rows, static_cast<int>(cols), codes, scale);
    return cudaGetLastError();
}

int read_and_clear_quant_error() {
    int v = 0, z = 0;
    cudaMemcpyFromSymbol(&v, g_quant_error, sizeof(int));
    if (v) cudaMemcpyToSymbol(g_quant_error, &z, sizeof(int));
    return v;
}

}  // namespace gdn
