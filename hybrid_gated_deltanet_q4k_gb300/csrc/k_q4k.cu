// Step 1a: Q4_K superblocks -> int8 rows with one fp32 scale per row.
//
// sparkinfer PR #464 ("fused Q4K/Q6K->int8 dequant + token-parallel GDN conv
// ..."), Summary, "Fused Q4_K/Q6_K -> int8-row dequant": one block per weight
// row decodes the superblocks in registers and writes int8 + a per-row scale
// directly, with no bf16 scratch; the quantisation starts from the exact fp32
// decode (same page, Correctness paragraph).
//
// Layout of one 144-byte superblock (GGUF Q4_K): fp16 d, fp16 dmin, 12 bytes of
// 6-bit scales/mins, 128 bytes of 4-bit codes; sub-block j of 32 weights
// decodes as d*sc_j*q - dmin*m_j.  Weight 64p+l (l<32) is the low nibble of
// code byte 32p+l, weight 64p+32+l its high nibble.
//
// Thread mapping: a thread owns 16 weights of one superblock -- 8 code bytes
// at 32p + 8i (i = 0..3), i.e. 8 weights of sub-block 2p (low nibbles) and 8 of
// sub-block 2p+1 (high nibbles).  Superblocks are 16-byte aligned (144 = 9*16),
// so the header is one 16-byte load and the 8 code bytes one 8-byte load.
// The row's weights stay in registers between the amax reduction and the
// quantisation: HBM traffic is the 144 B/256 weights read plus the codes
// written, nothing else.
#include "common.cuh"

namespace gdn {

constexpr int DEQ_THREADS = 256;
constexpr int DEQ_MAX_COLS = 16384;                              // 64 superblocks
constexpr int DEQ_MAX_GROUPS = DEQ_MAX_COLS / 16 / DEQ_THREADS;  // 16-weight groups per thread

// Byte i (0..11) of the 12 scale bytes, held in three little-endian words.
__device__ __forceinline__ int scale_byte(uint32_t y, uint32_t z, uint32_t w, int i) {
    const uint32_t word = i < 4 ? y : (i < 8 ? z : w);
    return static_cast<int>((word >> (8 * (i & 3))) & 0xffu);
}

// 6-bit scale and min of sub-block j.
__device__ __forceinline__ void q4k_scale_min(uint32_t y, uint32_t z, uint32_t w, int j, int& sc, int& m) {
    if (j < 4) {
        sc = scale_byte(y, z, w, j) & 63;
        m = scale_byte(y, z, w, j + 4) & 63;
    } else {
        const int hi = scale_byte(y, z, w, j + 4);
        sc = (hi & 15) | ((scale_byte(y, z, w, j - 4) >> 6) << 4);
        m = (hi >> 4) | ((scale_byte(y, z, w, j) >> 6) << 4);
    }
}

template <typename OutT>
__device__ __forceinline__ void store8(OutT* dst, const int* q);

template <>
__device__ __forceinline__ void store8<int8_t>(int8_t* dst, const int* q) {
    uint32_t lo = 0, hi = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        lo |= (static_cast<uint32_t>(q[i]) & 0xffu) << (8 * i);
        hi |= (static_cast<uint32_t>(q[i + 4]) & 0xffu) << (8 * i);
    }
    *reinterpret_cast<uint2*>(dst) = make_uint2(lo, hi);
}

template <>
__device__ __forceinline__ void store8<uint16_t>(uint16_t* dst, const int* q) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
        w[i] = static_cast<uint32_t>(code_to_f16_bits(q[2 * i])) |
               (static_cast<uint32_t>(code_to_f16_bits(q[2 * i + 1])) << 16);
    *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
}

template <typename OutT>
__global__ void __launch_bounds__(DEQ_THREADS)
q4k_deq_rows_kernel(const uint8_t* __restrict__ blocks, int cols, OutT* __restrict__ codes,
                    float* __restrict__ row_scale) {
    __shared__ float red[32];
    const int64_t row = blockIdx.x;
    const int nsb = cols >> 8;
    const int ngroups = nsb * 16;
    const uint8_t* rb = blocks + row * static_cast<int64_t>(nsb) * 144;

    float v[DEQ_MAX_GROUPS][16];
    float amax = 0.0f;
#pragma unroll
    for (int it = 0; it < DEQ_MAX_GROUPS; ++it) {
        const int g = threadIdx.x + it * DEQ_THREADS;
        if (g < ngroups) {
            const int sb = g >> 4, i16 = g & 15, p = i16 >> 2, l0 = (i16 & 3) * 8;
            const uint8_t* blk = rb + sb * 144;
            const uint4 hdr = __ldg(reinterpret_cast<const uint4*>(blk));
            const uint2 qs = __ldg(reinterpret_cast<const uint2*>(blk + 16 + 32 * p + l0));
            const float d = __half2float(__ushort_as_half(static_cast<uint16_t>(hdr.x & 0xffffu)));
            const float dmin = __half2float(__ushort_as_half(static_cast<uint16_t>(hdr.x >> 16)));
            int sc0, m0, sc1, m1;
            q4k_scale_min(hdr.y, hdr.z, hdr.w, 2 * p, sc0, m0);
            q4k_scale_min(hdr.y, hdr.z, hdr.w, 2 * p + 1, sc1, m1);
            // d*sc and dmin*m are exact in fp32 (11-bit x 6-bit significands);
            // one fused multiply-add gives the single rounding of d*sc*q - dmin*m.
            const float ds0 = __fmul_rn(d, static_cast<float>(sc0)), dm0 = __fmul_rn(dmin, static_cast<float>(m0));
            const float ds1 = __fmul_rn(d, static_cast<float>(sc1)), dm1 = __fmul_rn(dmin, static_cast<float>(m1));
            const uint32_t qw[2] = {qs.x, qs.y};
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const uint32_t byte = (qw[j >> 2] >> (8 * (j & 3))) & 0xffu;
                v[it][j] = __fmaf_rn(ds0, static_cast<float>(byte & 15u), -dm0);
                v[it][8 + j] = __fmaf_rn(ds1, static_cast<float>(byte >> 4), -dm1);
                amax = fmaxf(amax, fmaxf(fabsf(v[it][j]), fabsf(v[it][8 + j])));
            }
        }
    }
    amax = block_max(amax, red);
    const float s = __fdiv_rn(amax, 127.0f);
    if (threadIdx.x == 0) row_scale[row] = s;
    OutT* out = codes + row * static_cast<int64_t>(cols);
#pragma unroll
    for (int it = 0; it < DEQ_MAX_GROUPS; ++it) {
        const int g = threadIdx.x + it * DEQ_THREADS;
        if (g < ngroups) {
            const int sb = g >> 4, i16 = g & 15, p = i16 >> 2, l0 = (i16 & 3) * 8;
            int q[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) q[j] = quant_code(v[it][j], s);
            const int base = sb * 256 + 64 * p + l0;
            store8<OutT>(out + base, q);
            store8<OutT>(out + base + 32, q + 8);
        }
    }
}

cudaError_t launch_q4k_deq_i8(const void* blocks, int64_t rows, int64_t cols, int8_t* q, float* s,
                              cudaStream_t st) {
    q4k_deq_rows_kernel<int8_t><<<static_cast<unsigned>(rows), DEQ_THREADS, 0, st>>>(
        static_cast<const uint8_t*>(blocks), static_cast<int>(cols), q, s);
    return cudaGetLastError();
}

cudaError_t launch_q4k_deq_codes(const void* blocks, int64_t rows, int64_t cols, uint16_t* q, float* s,
                                 cudaStream_t st) {
    q4k_deq_rows_kernel<uint16_t><<<static_cast<unsigned>(rows), DEQ_THREADS, 0, st>>>(
        static_cast<const uint8_t*>(blocks), static_cast<int>(cols), q, s);
    return cudaGetLastError();
}

}  // namespace gdn
