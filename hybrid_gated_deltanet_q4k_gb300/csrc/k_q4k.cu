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
#include "qk_decode.cuh"

namespace gdn {

constexpr int DEQ_THREADS = 256;
constexpr int DEQ_MAX_COLS = 16384;                              // 64 superblocks
constexpr int DEQ_MAX_GROUPS = DEQ_MAX_COLS / 16 / DEQ_THREADS;  // 16-weight groups per thread


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

// Warp-per-row variant for rows of at most DEQ_WARP_MAX_SB superblocks (4096
// weights): in iteration i the warp decodes superblock i, lane l the 8 weights
// 8l .. 8l+7 (sub-block l/4, the low or high nibbles of 8 code bytes).
// Pass 1 finds the row amax without decoding every weight: d*sc*q - dmin*m,
// rounded once, is monotonic in q, so the largest magnitude of a lane's 8
// weights is at its smallest or largest 4-bit code (byte-wise SIMD min/max).
// The amax is a warp reduction (no block barrier).  Pass 2 reloads the lane's
// 16-byte header and 8 code bytes (L1 hits) and writes its 8 codes as one
// 16-byte vector: consecutive lanes write consecutive 16 bytes.  Nothing is
// held across the passes, so the kernel runs at full occupancy.  One launch
// covers two matrices (the rows of the second follow those of the first), so
// a layer's two weight matrices share one grid and one tail.
constexpr int DEQ_WARP_MAX_SB = 16;
constexpr int DEQ_WARP_THREADS = 256;

struct DeqJob {
    const uint8_t* blocks;
    int64_t rows;
    int cols;
    uint16_t* codes;
    float* scale;
};

__global__ void __launch_bounds__(DEQ_WARP_THREADS, 4)
q4k_deq_rows_warp_kernel(DeqJob j0, DeqJob j1) {
    const int lane = threadIdx.x & 31;
    int64_t row = static_cast<int64_t>(blockIdx.x) * (DEQ_WARP_THREADS / 32) + (threadIdx.x >> 5);
    const bool second = row >= j0.rows;
    const DeqJob j = second ? j1 : j0;
    if (second) row -= j0.rows;
    if (row >= j.rows) return;
    const int nsb = j.cols >> 8;
    const uint8_t* rb = j.blocks + row * static_cast<int64_t>(nsb) * 144;
    const int sub = lane >> 2, p = sub >> 1, l0 = (lane & 3) * 8;
    const int shift = (sub & 1) * 4;    // high nibbles for odd sub-blocks
    const uint8_t* my_hdr = rb;
    const uint8_t* my_qs = rb + 16 + 32 * p + l0;

    float amax = 0.0f;
#pragma unroll 8
    for (int i = 0; i < nsb; ++i) {
        const uint4 hdr = __ldg(reinterpret_cast<const uint4*>(my_hdr + i * 144));
        const uint2 qs = __ldg(reinterpret_cast<const uint2*>(my_qs + i * 144));
        float ds, dm;
        q4k_sub_affine(hdr, sub, ds, dm);
        const uint32_t n0 = (qs.x >> shift) & 0x0f0f0f0fu, n1 = (qs.y >> shift) & 0x0f0f0f0fu;
        uint32_t mn = __vminu4(n0, n1), mx = __vmaxu4(n0, n1);
        mn = __vminu4(mn, mn >> 16);
        mx = __vmaxu4(mx, mx >> 16);
        mn = __vminu4(mn, mn >> 8) & 0xffu;
        mx = __vmaxu4(mx, mx >> 8) & 0xffu;
        const float w0 = __fmaf_rn(ds, static_cast<float>(mn), -dm);
        const float w1 = __fmaf_rn(ds, static_cast<float>(mx), -dm);
        amax = fmaxf(amax, fmaxf(fabsf(w0), fabsf(w1)));
    }
    amax = warp_max(amax);
    const QScale qsc = make_qscale(amax);
    if (lane == 0) j.scale[row] = qsc.s;
    uint16_t* out = j.codes + row * static_cast<int64_t>(j.cols) + lane * 8;
#pragma unroll 4
    for (int i = 0; i < nsb; ++i) {
        const uint4 hdr = __ldg(reinterpret_cast<const uint4*>(my_hdr + i * 144));
        const uint2 qs = __ldg(reinterpret_cast<const uint2*>(my_qs + i * 144));
        float ds, dm;
        q4k_sub_affine(hdr, sub, ds, dm);
        float w[8], c[8];
        bool redo = !qsc.fast;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const uint32_t q = ((e < 4 ? qs.x : qs.y) >> (8 * (e & 3) + shift)) & 15u;
            w[e] = __fmaf_rn(ds, static_cast<float>(q), -dm);
            c[e] = qcode_fast(w[e], qsc, redo);
        }
        if (redo) {
#pragma unroll
            for (int e = 0; e < 8; ++e) c[e] = qcode_exact(w[e], qsc.s);
        }
        *reinterpret_cast<uint4*>(out + i * 256) = make_uint4(codes_to_f16x2(c[0], c[1]), codes_to_f16x2(c[2], c[3]),
                                                              codes_to_f16x2(c[4], c[5]), codes_to_f16x2(c[6], c[7]));
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
    if (cols <= DEQ_WARP_MAX_SB * 256) {
        const DeqJob j0{static_cast<const uint8_t*>(blocks), rows, static_cast<int>(cols), q, s};
        const DeqJob j1{nullptr, 0, 256, nullptr, nullptr};
        const int64_t wpb = DEQ_WARP_THREADS / 32;
        q4k_deq_rows_warp_kernel<<<static_cast<unsigned>((rows + wpb - 1) / wpb), DEQ_WARP_THREADS, 0, st>>>(j0, j1);
        return cudaGetLastError();
    }
    q4k_deq_rows_kernel<uint16_t><<<static_cast<unsigned>(rows), DEQ_THREADS, 0, st>>>(
        static_cast<const uint8_t*>(blocks), static_cast<int>(cols), q, s);
    return cudaGetLastError();
}

// Both weight matrices of a layer in one launch (each falls back to its own
// CTA-per-row launch when its rows are longer than the warp variant takes).
cudaError_t launch_q4k_deq_codes2(const void* b0, int64_t rows0, int64_t cols0, uint16_t* q0, float* s0,
                                  const void* b1, int64_t rows1, int64_t cols1, uint16_t* q1, float* s1,
                                  cudaStream_t st) {
    if (cols0 > DEQ_WARP_MAX_SB * 256 || cols1 > DEQ_WARP_MAX_SB * 256) {
        cudaError_t e = launch_q4k_deq_codes(b0, rows0, cols0, q0, s0, st);
        if (e != cudaSuccess) return e;
        return launch_q4k_deq_codes(b1, rows1, cols1, q1, s1, st);
    }
    const DeqJob j0{static_cast<const uint8_t*>(b0), rows0, static_cast<int>(cols0), q0, s0};
    const DeqJob j1{static_cast<const uint8_t*>(b1), rows1, static_cast<int>(cols1), q1, s1};
    const int64_t wpb = DEQ_WARP_THREADS / 32;
    q4k_deq_rows_warp_kernel<<<static_cast<unsigned>((rows0 + rows1 + wpb - 1) / wpb), DEQ_WARP_THREADS, 0, st>>>(j0, j1);
    return cudaGetLastError();
}

}  // namespace gdn
