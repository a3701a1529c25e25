// q4k_pack, q6k_pack: fp32 weights -> GGUF Q4_K / Q6_K superblocks (host,
// plain encoders).
//
// Q4_K (plain min-max):
// The pages only ever decode Q4_K (sparkinfer PR #464, "Fused Q4_K/Q6_K ->
// int8-row dequant"); the weights here are synthetic, so they are encoded with
// the simplest encoder the format admits.  Per 32-weight sub-block j the range
// [min(0, min w), max w] is split into 15 steps: step_j = (max - min)/15,
// min_j = -min(0, min w).  The superblock's d and dmin are the largest step_j
// and min_j divided by 63, rounded to fp16 (a zero of either sign stored as
// +0).  sc_j = clamp(rne(step_j / d), 0, 63), m_j = clamp(rne(min_j / dmin), 0,
// 63), and each code q = clamp(rne((w + dmin*m_j) / (d*sc_j)), 0, 15); a zero
// divisor gives 0.  All arithmetic is IEEE fp32 with nearest-even rounding and
// no contraction (built with -ffp-contract=off), so the bytes do not depend on
// the host CPU.
//
// Block layout (144 bytes): fp16 d | fp16 dmin | 12 bytes of 6-bit fields |
// 128 bytes of 4-bit codes.  6-bit fields: bytes 0-3 hold sc_0..3 in bits 0-5
// and the top two bits of sc_4..7 in bits 6-7; bytes 4-7 likewise for m_0..3
// and m_4..7; bytes 8-11 hold the low nibbles of sc_4..7 (bits 0-3) and of
// m_4..7 (bits 4-7).  Code byte 32p + l holds weight 64p + l in its low nibble
// and weight 64p + 32 + l in its high nibble.
//
// Q6_K (plain absmax; the pages name Q6_K beside Q4_K in the same summary):
// per 16-weight sub-block j, step_j = max|w| / 31; d = max_j step_j / 127
// rounded to fp16 (+0 for a zero); scale_j = clamp(rne(step_j / d), 0, 127);
// q = clamp(rne(w / (d * scale_j)), -32, 31), a zero divisor giving 0.
// Block layout (210 bytes): ql[128] | qh[64] | int8 scales[16] | fp16 d.  The
// 6-bit code c = q + 32 of weight v (half h = v / 128, group g = (v % 128) /
// 32, lane l = v % 32) keeps its low 4 bits in nibble g / 2 of ql[64h +
// 32(g % 2) + l] and its high 2 bits in bits 2g, 2g+1 of qh[32h + l].
#include <cmath>
#include <cstdint>
#include <cstring>

#include "../../include/gdn.h"

namespace {

uint16_t f32_to_f16_rne(float f) {
    uint32_t x;
    std::memcpy(&x, &f, 4);
    const uint32_t sign = (x >> 16) & 0x8000u;
    const uint32_t ax = x & 0x7fffffffu;
    if (ax >= 0x7f800000u) return static_cast<uint16_t>(sign | 0x7c00u | (ax > 0x7f800000u ? 0x200u : 0u));
    if (ax >= 0x477ff000u) return static_cast<uint16_t>(sign | 0x7c00u);  // >= 65520 rounds to infinity
    if (ax < 0x38800000u) {                                                  // below 2^-14: subnormal or zero
        if (ax <= 0x33000000u) return static_cast<uint16_t>(sign);           // <= 2^-25 rounds to zero
        const uint32_t mant = (ax & 0x7fffffu) | 0x800000u;
        const int e = static_cast<int>(ax >> 23) - 127;                      // -25 .. -15
        const int sh = -(e + 1);                                             // 14 .. 24
        uint32_t h = mant >> sh;
        const uint32_t rem = mant & ((1u << sh) - 1u), half = 1u << (sh - 1);
        if (rem > half || (rem == half && (h & 1u))) ++h;
        return static_cast<uint16_t>(sign | h);
    }
    const uint32_t mant = ax & 0x7fffffu;
    uint32_t h = ((static_cast<uint32_t>(static_cast<int>(ax >> 23) - 127 + 15)) << 10) | (mant >> 13);
    const uint32_t rem = mant & 0x1fffu;
    if (rem > 0x1000u || (rem == 0x1000u && (h & 1u))) ++h;
    return static_cast<uint16_t>(sign | h);
}

float f16_to_f32(uint16_t h) {
    const uint32_t sign = static_cast<uint32_t>(h & 0x8000u) << 16;
    const uint32_t e = (h >> 10) & 31u, m = h & 0x3ffu;
    float v;
    if (e == 0)
        v = std::ldexp(static_cast<float>(m), -24);
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = std::ldexp(static_cast<float>(m | 0x400u), static_cast<int>(e) - 25);
    uint32_t bits;
    std::memcpy(&bits, &v, 4);
    bits |= sign;
    std::memcpy(&v, &bits, 4);
    return v;
}

inline int clamp_rne(float v, int lo, int hi) {
    const float r = std::nearbyint(v);
    if (!(r >= static_cast<float>(lo))) return lo;
    if (r > static_cast<float>(hi)) return hi;
    return static_cast<int>(r);
}

void pack_superblock(const float* x, uint8_t* out) {
    float step[8], mins[8];
    for (int j = 0; j < 8; ++j) {
        float mn = x[32 * j], mx = x[32 * j];
        for (int i = 1; i < 32; ++i) {
            const float v = x[32 * j + i];
            if (v < mn) mn = v;
            if (v > mx) mx = v;
        }
        if (!(mn < 0.0f)) mn = 0.0f;
        step[j] = (mx - mn) / 15.0f;
        mins[j] = -mn;
    }
    float max_step = step[0], max_min = mins[0];
    for (int j = 1; j < 8; ++j) {
        if (step[j] > max_step) max_step = step[j];
        if (mins[j] > max_min) max_min = mins[j];
    }
    uint16_t d16 = f32_to_f16_rne(max_step / 63.0f);
    uint16_t dm16 = f32_to_f16_rne(max_min / 63.0f);
    if ((d16 & 0x7fffu) == 0) d16 = 0;
    if ((dm16 & 0x7fffu) == 0) dm16 = 0;
    const float d = f16_to_f32(d16), dm = f16_to_f32(dm16);
    int sc[8], m[8];
    for (int j = 0; j < 8; ++j) {
        sc[j] = d > 0.0f ? clamp_rne(step[j] / d, 0, 63) : 0;
        m[j] = dm > 0.0f ? clamp_rne(mins[j] / dm, 0, 63) : 0;
    }
    std::memcpy(out, &d16, 2);
    std::memcpy(out + 2, &dm16, 2);
    uint8_t* s = out + 4;
    for (int j = 0; j < 4; ++j) {
        s[j] = static_cast<uint8_t>((sc[j] & 63) | ((sc[j + 4] >> 4) << 6));
        s[j + 4] = static_cast<uint8_t>((m[j] & 63) | ((m[j + 4] >> 4) << 6));
        s[j + 8] = static_cast<uint8_t>((sc[j + 4] & 15) | ((m[j + 4] & 15) << 4));
    }
    uint8_t q[256];
    for (int j = 0; j < 8; ++j) {
        const float ds = d * static_cast<float>(sc[j]);
        const float dms = dm * static_cast<float>(m[j]);
        for (int i = 0; i < 32; ++i) {
            const float num = x[32 * j + i] + dms;
            q[32 * j + i] = static_cast<uint8_t>(ds > 0.0f ? clamp_rne(num / ds, 0, 15) : 0);
        }
    }
    uint8_t* qs = out + 16;
    for (int p = 0; p < 4; ++p)
        for (int l = 0; l < 32; ++l)
            qs[32 * p + l] = static_cast<uint8_t>(q[64 * p + l] | (q[64 * p + 32 + l] << 4));
}

void pack_q6k_superblock(const float* x, uint8_t* out) {
    float step[16];
    for (int j = 0; j < 16; ++j) {
        float amax = 0.0f;
        for (int i = 0; i < 16; ++i) {
            const float a = std::fabs(x[16 * j + i]);
            if (a > amax) amax = a;
        }
        step[j] = amax / 31.0f;
    }
    float max_step = step[0];
    for (int j = 1; j < 16; ++j)
        if (step[j] > max_step) max_step = step[j];
    uint16_t d16 = f32_to_f16_rne(max_step / 127.0f);
    if ((d16 & 0x7fffu) == 0) d16 = 0;
    const float d = f16_to_f32(d16);
    int sc[16];
    for (int j = 0; j < 16; ++j) sc[j] = d > 0.0f ? clamp_rne(step[j] / d, 0, 127) : 0;
    uint8_t* ql = out;
    uint8_t* qh = out + 128;
    std::memset(out, 0, 192);
    for (int v = 0; v < 256; ++v) {
        const float ds = d * static_cast<float>(sc[v / 16]);
        const int q = ds > 0.0f ? clamp_rne(x[v] / ds, -32, 31) : 0;
        const int c = q + 32, h = v / 128, g = (v % 128) / 32, l = v % 32;
        ql[64 * h + 32 * (g % 2) + l] |= static_cast<uint8_t>((c & 15) << (4 * (g / 2)));
        qh[32 * h + l] |= static_cast<uint8_t>((c >> 4) << (2 * g));
    }
    for (int j = 0; j < 16; ++j) out[192 + j] = static_cast<uint8_t>(static_cast<int8_t>(sc[j]));
    std::memcpy(out + 208, &d16, 2);
}

}  // namespace

extern "C" int q6k_pack(const float* w, int64_t rows, int64_t cols, void* blocks) {
    if (w == nullptr || blocks == nullptr || rows < 0 || cols <= 0 || cols % 256 != 0) return GDN_EINVAL;
    const int64_t nsb = cols / 256;
    uint8_t* out = static_cast<uint8_t*>(blocks);
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t b = 0; b < nsb; ++b) pack_q6k_superblock(w + r * cols + b * 256, out + (r * nsb + b) * 210);
    return GDN_OK;
}

extern "C" int q4k_pack(const float* w, int64_t rows, int64_t cols, void* blocks) {
    if (w == nullptr || blocks == nullptr || rows < 0 || cols <= 0 || cols % 256 != 0) return GDN_EINVAL;
    const int64_t nsb = cols / 256;
    uint8_t* out = static_cast<uint8_t*>(blocks);
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t b = 0; b < nsb; ++b) pack_superblock(w + r * cols + b * 256, out + (r * nsb + b) * 144);
    return GDN_OK;
}
