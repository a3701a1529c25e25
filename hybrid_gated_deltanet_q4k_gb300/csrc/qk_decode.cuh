// Decoding of GGUF Q4_K and Q6_K superblocks, shared by the kernels that
// read them (step 1a to int8 codes, and the fused decode-and-dot of the
// decode step), so that every path yields the same codes bit for bit.
//
// Q4_K (144 B): fp16 d | fp16 dmin | 12 bytes of 6-bit scales/mins | 128 bytes
// of 4-bit codes; sub-block j (32 weights) decodes as d*sc_j*q - dmin*m_j.
// Lane l of a warp takes the 8 weights 8l .. 8l+7 of a superblock: sub-block
// l/4, the low (even sub-block) or high (odd) nibbles of code bytes
// 32(l/8) + 8(l%4) .. +7.
//
// Q6_K (210 B): ql[128] | qh[64] | int8 scales[16] | fp16 d; weight v decodes
// as d*scales[v/16]*(c - 32) with c's low 4 bits in nibble g/2 of
// ql[64h + 32(g%2) + l] and its high 2 bits in bits 2g, 2g+1 of qh[32h + l]
// (h = v/128, g = (v%128)/32, l = v%32).  Lane L takes the 8 weights 8L .. 8L+7:
// they share h, g and one scale.
#pragma once

#include "common.cuh"

namespace gdn {

// 6-bit scale and min of Q4_K sub-block j from the 12 scale bytes, held in
// three little-endian words y, z, w: sub-blocks 0..3 take the low six bits of
// bytes j and j + 4; 4..7 take the nibbles of byte j + 4 and the top two bits
// of bytes j - 4 and j.  Byte permutes pick byte j % 4 of each word, with no
// branch on j.
__device__ __forceinline__ void q4k_scale_min(uint32_t y, uint32_t z, uint32_t w, int j, int& sc, int& m) {
    const int k = j & 3;
    const uint32_t yk = __byte_perm(y, 0u, 0x4440 + k), zk = __byte_perm(z, 0u, 0x4440 + k);
    const uint32_t wk = __byte_perm(w, 0u, 0x4440 + k);
    const bool lo = j < 4;
    sc = static_cast<int>(lo ? (yk & 63u) : ((wk & 15u) | ((yk >> 2) & 0x30u)));
    m = static_cast<int>(lo ? (zk & 63u) : ((wk >> 4) | ((zk >> 2) & 0x30u)));
}

// d*sc and dmin*m of Q4_K sub-block `sub` of a superblock header; both products
// are exact in fp32 (11-bit x 6-bit significands).
__device__ __forceinline__ void q4k_sub_affine(const uint4& hdr, int sub, float& ds, float& dm) {
    const float d = __half2float(__ushort_as_half(static_cast<uint16_t>(hdr.x & 0xffffu)));
    const float dmin = __half2float(__ushort_as_half(static_cast<uint16_t>(hdr.x >> 16)));
    int sc, m;
    q4k_scale_min(hdr.y, hdr.z, hdr.w, sub, sc, m);
    ds = __fmul_rn(d, small_uint_to_float(static_cast<uint32_t>(sc)));
    dm = __fmul_rn(dmin, small_uint_to_float(static_cast<uint32_t>(m)));
}

// Loads of the decoders: read-only global loads (G = true) or plain loads (G =
// false, e.g. from shared memory).
template <bool G, typename T>
__device__ __forceinline__ T ldq(const T* p) {
    if constexpr (G) return __ldg(p);
    else return *p;
}

// Q4_K: the lane's 8 weights of the superblock at blk (16-byte aligned), exact
// single roundings of d*sc*q - dmin*m; amax: just their largest magnitude (at
// the smallest or largest code: the decode is monotonic in q).
template <bool G>
struct Q4KLaneT {
    static constexpr int BYTES = 144;
    __device__ __forceinline__ static float amax(const uint8_t* blk, int lane) {
        const int sub = lane >> 2, p = sub >> 1, l0 = (lane & 3) * 8, shift = (sub & 1) * 4;
        const uint4 hdr = ldq<G>(reinterpret_cast<const uint4*>(blk));
        const uint2 qs = ldq<G>(reinterpret_cast<const uint2*>(blk + 16 + 32 * p + l0));
        float ds, dm;
        q4k_sub_affine(hdr, sub, ds, dm);
        const uint32_t n0 = (qs.x >> shift) & 0x0f0f0f0fu, n1 = (qs.y >> shift) & 0x0f0f0f0fu;
        uint32_t mn = __vminu4(n0, n1), mx = __vmaxu4(n0, n1);
        mn = __vminu4(mn, mn >> 16);
        mx = __vmaxu4(mx, mx >> 16);
        mn = __vminu4(mn, mn >> 8) & 0xffu;
        mx = __vmaxu4(mx, mx >> 8) & 0xffu;
        const float w0 = __fmaf_rn(ds, small_uint_to_float(mn), -dm);
        const float w1 = __fmaf_rn(ds, small_uint_to_float(mx), -dm);
        return fmaxf(fabsf(w0), fabsf(w1));
    }
    __device__ __forceinline__ static void decode(const uint8_t* blk, int lane, float (&w)[8]) {
        const int sub = lane >> 2, p = sub >> 1, l0 = (lane & 3) * 8, shift = (sub & 1) * 4;
        const uint4 hdr = ldq<G>(reinterpret_cast<const uint4*>(blk));
        const uint2 qs = ldq<G>(reinterpret_cast<const uint2*>(blk + 16 + 32 * p + l0));
        float ds, dm;
        q4k_sub_affine(hdr, sub, ds, dm);
        // the lane's 8 nibbles, one per byte, then each byte as 2^23 + q (byte
        // permutes); q = (2^23 + q) - 2^23 and the fma on the packed f32x2
        // instructions, two weights at a time (each half rounds as the scalar
        // instruction would)
        const uint32_t n0 = (qs.x >> shift) & 0x0f0f0f0fu, n1 = (qs.y >> shift) & 0x0f0f0f0fu;
        const F2 two23 = f2(8388608.0f, 8388608.0f), ds2 = f2(ds, ds), ndm2 = f2(-dm, -dm);
#pragma unroll
        for (int e = 0; e < 8; e += 2) {
            const uint32_t b0 = __byte_perm(e < 4 ? n0 : n1, 0x4B000000u, 0x7440 + (e & 3));
            const uint32_t b1 = __byte_perm(e < 4 ? n0 : n1, 0x4B000000u, 0x7440 + ((e + 1) & 3));
            const F2 q = f2_sub(f2(__uint_as_float(b0), __uint_as_float(b1)), two23);
            f2_split(f2_fma(ds2, q, ndm2), w[e], w[e + 1]);
        }
    }
};
using Q4KLane = Q4KLaneT<true>;

// Q6_K: the lane's 8 six-bit codes c (0..63, weight = d*scale*(c - 32)) and its
// d * scale (exact); the superblock is only 2-byte aligned (210 = 2 * 105),
// so it is read in 16-bit words.
template <bool G>
__device__ __forceinline__ void q6k_lane(const uint8_t* blk, int lane, uint32_t (&c)[8], float& ds) {
    const int v0 = 8 * lane, h = v0 >> 7, g = (v0 & 127) >> 5, l0 = v0 & 31;
    const uint16_t* ql = reinterpret_cast<const uint16_t*>(blk + 64 * h + 32 * (g & 1) + l0);
    const uint16_t* qh = reinterpret_cast<const uint16_t*>(blk + 128 + 32 * h + l0);
    const int nsh = 4 * (g >> 1), hsh = 2 * g;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint32_t lw = ldq<G>(ql + k), hw = ldq<G>(qh + k);
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const uint32_t lo = (lw >> (8 * e + nsh)) & 15u;
            const uint32_t hi = (hw >> (8 * e + hsh)) & 3u;
            c[2 * k + e] = lo | (hi << 4);
        }
    }
    const int8_t sc = static_cast<int8_t>(ldq<G>(blk + 192 + (v0 >> 4)));
    const float d = __half2float(__ushort_as_half(ldq<G>(reinterpret_cast<const uint16_t*>(blk + 208))));
    ds = __fmul_rn(d, static_cast<float>(sc));
}

template <bool G>
struct Q6KLaneT {
    static constexpr int BYTES = 210;
    __device__ __forceinline__ static float amax(const uint8_t* blk, int lane) {
        uint32_t c[8];
        float ds;
        q6k_lane<G>(blk, lane, c, ds);
        int m = 0;
#pragma unroll
        for (int e = 0; e < 8; ++e) m = max(m, abs(static_cast<int>(c[e]) - 32));
        return fabsf(__fmul_rn(ds, small_uint_to_float(static_cast<uint32_t>(m))));   // the largest |w| of the 8, exact
    }
    __device__ __forceinline__ static void decode(const uint8_t* blk, int lane, float (&w)[8]) {
        uint32_t c[8];
        float ds;
        q6k_lane<G>(blk, lane, c, ds);
        // c - 32 exactly: (2^23 + c) - (2^23 + 32); the product with d*scale is
        // exact (packed f32x2 instructions, two weights at a time)
        const F2 off = f2(8388640.0f, 8388640.0f), ds2 = f2(ds, ds);
#pragma unroll
        for (int e = 0; e < 8; e += 2) {
            const F2 cm = f2_sub(f2(__uint_as_float(0x4B000000u | c[e]), __uint_as_float(0x4B000000u | c[e + 1])), off);
            f2_split(f2_mul(ds2, cm), w[e], w[e + 1]);
        }
    }
};
using Q6KLane = Q6KLaneT<true>;

// The int8 codes of 8 decoded weights for the row's scale, as magic floats:
// the fast quantiser, with the exact fallback where it may round differently
// (results equal qcode_exact for every weight).
// The fast path is qcode_fast on the packed f32x2 instructions, two weights
// at a time: the same roundings, so the same codes and the same fallbacks.
__device__ __forceinline__ void quantise8(const float (&w)[8], const QScale& qsc, float (&c)[8]) {
    bool redo = !qsc.fast;
    const F2 rs = f2(qsc.rs, qsc.rs), mg = f2(QCODE_MAGIC, QCODE_MAGIC);
#pragma unroll
    for (int e = 0; e < 8; e += 2) {
        const F2 y = f2_mul(f2(w[e], w[e + 1]), rs);
        const F2 t = f2_add(y, mg);
        float d0, d1;
        f2_split(f2_sub(y, f2_sub(t, mg)), d0, d1);
        redo |= !(fabsf(d0) <= 0.499f) || !(fabsf(d1) <= 0.499f);
        f2_split(t, c[e], c[e + 1]);
    }
    if (redo) {
#pragma unroll
        for (int e = 0; e < 8; ++e) c[e] = qcode_exact(w[e], qsc.s);
    }
}

// 8 magic-float codes stored as fp16 patterns (16 bytes) or int8 (8 bytes).
template <typename OutT>
__device__ __forceinline__ void store_codes8(OutT* dst, const float (&c)[8]);

template <>
__device__ __forceinline__ void store_codes8<uint16_t>(uint16_t* dst, const float (&c)[8]) {
    *reinterpret_cast<uint4*>(dst) = make_uint4(codes_to_f16x2(c[0], c[1]), codes_to_f16x2(c[2], c[3]),
                                                codes_to_f16x2(c[4], c[5]), codes_to_f16x2(c[6], c[7]));
}

template <>
__device__ __forceinline__ void store_codes8<int8_t>(int8_t* dst, const float (&c)[8]) {
    *reinterpret_cast<uint2*>(dst) = make_uint2(codes_to_i8x4(c[0], c[1], c[2], c[3]), codes_to_i8x4(c[4], c[5], c[6], c[7]));
}

}  // namespace gdn
