// Shared device helpers of the GDN prefill library (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "../../include/gdn.h"

#include <mutex>

namespace gdn {

// Host: kernel attributes (dynamic shared memory, carveout) and device
// queries belong to one device, so a launcher's one-time setup runs once per
// device, on the first call made with that device current.  run(f) calls
// f(device) at most once per device ordinal below MAX_DEVICES and returns the
// current device, or -1 (nothing run) for an ordinal past the table.
constexpr int MAX_DEVICES = 256;
struct PerDeviceOnce {
    std::once_flag flag[MAX_DEVICES];
    template <class F>
    int run(F&& f) {
        int d = -1;
        if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= MAX_DEVICES) return -1;
        std::call_once(flag[d], f, d);
        return d;
    }
};

// Kernels whose waits are bounded keep an error word in their own translation
// unit (`static __device__ int`, no relocatable device code): when a wait runs
// out they record a code there and return early; gdn_sync_status() reads and
// clears every such word through the unit's host accessor.
enum : int { ERR_NONE = 0, ERR_WAIT_TIMEOUT = 1, ERR_RANGE = 2, ERR_INDEX = 3 };

// Index checks of the debug build (compiled with GDN_DEBUG): a global store
// whose index lies outside the extent its kernel was given records ERR_INDEX
// in the unit's error word and is skipped (gdn_sync_status then reports
// GDN_EINDEX), where a sanitizer would have reported an out-of-bounds access.
// Release builds compile the checks away: GDN_IN_RANGE is `true`.
#ifdef GDN_DEBUG
__device__ __forceinline__ bool gdn_debug_in_range(int& word, bool ok) {
    if (!ok) atomicCAS(&word, 0, static_cast<int>(ERR_INDEX));
    return ok;
}
#define GDN_IN_RANGE(word, cond) ::gdn::gdn_debug_in_range((word), (cond))
#else
#define GDN_IN_RANGE(word, cond) true
#endif

// The sequences of one call, passed to kernels as a __grid_constant__
// parameter (2 KB, no device memory): sequence s holds tokens [tok[s],
// tok[s+1]) of the call's token rows and the work units [unit[s], unit[s+1])
// of the kernel that reads it (chunks of the delta rule, token runs of the
// conv), numbered across all sequences in order.  One sequence of n tokens is
// {1, {0, n}, {0, units(n)}}.
struct SeqTable {
    int n;
    int tok[GDN_MAX_SEQS + 1];
    int unit[GDN_MAX_SEQS + 1];
};

// Recurrent-state snapshots taken during a prefill: after every `every_chunks`
// chunks (counted from the start of the prompt, of which this call's first
// chunk is number chunk_base), the state S goes to
// state[(chunks done) / every_chunks - 1], each [Hv][dv][dk] fp32.
struct DeltaCkpt {
    float* state;
    int every_chunks;
    int chunk_base;
};

// Test of the bounded waits (gdn_test_delta_wait_timeout): the delta rule's
// prep runs alone and issues no copy of its [Q; K] tile, so its wait for that
// copy runs out after wait_ns; the kernel records the timeout, frees its TMEM
// and returns.
struct DeltaFault {
    uint64_t wait_ns;
};

// The sequence holding work unit u: the last s with unit[s] <= u (an empty
// sequence owns no unit, so it is passed over).
__device__ __forceinline__ int seq_of_unit(const SeqTable& t, int u) {
    int lo = 0, hi = t.n - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (t.unit[mid] <= u) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// Host: the table of the sequences cu[0..n_seqs] (token offsets) with units
// of `per` tokens.
inline SeqTable make_seq_table(const int64_t* cu, int n_seqs, int per) {
    SeqTable t{};
    t.n = n_seqs;
    for (int s = 0; s <= n_seqs; ++s) {
        t.tok[s] = static_cast<int>(cu[s]);
        t.unit[s] = s == 0 ? 0 : t.unit[s - 1] + static_cast<int>((cu[s] - cu[s - 1] + per - 1) / per);
    }
    return t;
}
inline SeqTable one_seq_table(int64_t n, int per) {
    const int64_t cu[2] = {0, n};
    return make_seq_table(cu, 1, per);
}

// Let the next kernel in the stream, when it is launched as a programmatic
// dependent, start now (its CTAs wait with griddepcontrol.wait before they
// read anything this kernel writes); no effect otherwise.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

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

// Codes are carried between the quantiser and the stores as "magic" floats
// t = q + QCODE_MAGIC (q the integer code).  QCODE_MAGIC = 1.5 * 2^23 + 0x6480
// puts t in [2^23, 2^24), where consecutive fp32 values are the integers, so
// the one addition that forms t rounds to the nearest integer with ties to
// even (QCODE_MAGIC is even), exactly as rint; and since fp32 bit patterns
// grow by one per integer there, the low 16 bits of t are 0x6480 + q, the fp16
// pattern of 1152 + q, and its low byte is (0x80 + q) mod 256.  The stores
// take the code from those bits with byte permutes and one packed fp16
// subtraction, so no instruction converts between integer and float.
constexpr float QCODE_MAGIC = 12608640.0f;

// The code of w by the IEEE divide, clamp(rne(w / s), -127, 127) (s == 0 or a
// NaN quotient: 0), as a magic float.
__device__ __forceinline__ float qcode_exact(float w, float s) {
    if (s == 0.0f) return QCODE_MAGIC;
    const float r = rintf(__fdiv_rn(w, s));
    if (r != r) return QCODE_MAGIC;
    return __fadd_rn(fminf(fmaxf(r, -127.0f), 127.0f), QCODE_MAGIC);
}

// The integer value of a magic-float code.
__device__ __forceinline__ float qcode_value(float t) { return __fsub_rn(t, QCODE_MAGIC); }

// Row scale s = amax/127 with its reciprocal for the fast quantiser.
struct QScale {
    float s, rs;
    bool fast;   // s and 1/s are normal numbers far from overflow
};
__device__ __forceinline__ QScale make_qscale(float amax) {
    QScale q;
    q.s = __fdiv_rn(amax, 127.0f);
    q.rs = __frcp_rn(q.s);
    q.fast = q.s >= 1e-30f && q.s <= 1e30f;
    return q;
}

// Fast quantiser: y = w * fl(1/s) is within 2^-22 (relative) of w/s, and |w/s|
// <= 127.5 in a row whose amax gave s, so y and fl(w/s) lie within 3e-5 of each
// other; rounding to nearest can tell them apart only when they straddle a
// half-integer.  When y is within 1e-3 of one (or is not a number), `redo` is
// set and the caller recomputes with qcode_exact, so the result always equals
// qcode_exact(w, s).  No clamp is needed: |w| <= amax and s = fl(amax/127)
// give |y| <= 127 (1 + 2^-22) < 127.5, so |rint(y)| <= 127.  Returns the
// magic float of rint(y); every step is an explicitly rounded fp32 operation
// (no contraction), and none is a conversion.
__device__ __forceinline__ float qcode_fast(float w, const QScale& q, bool& redo) {
    const float y = __fmul_rn(w, q.rs);
    const float t = __fadd_rn(y, QCODE_MAGIC);
    redo |= !(fabsf(__fsub_rn(y, qcode_value(t))) <= 0.499f);
    return t;
}

// Two floats as a pair of fp16 values (rounded to nearest), low half first.
__device__ __forceinline__ uint32_t f16x2_bits(float lo, float hi) {
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
}

// Two magic-float codes as a pair of fp16 values, low half first: the fp16
// patterns of 1152 + q (the low halves of the magic floats) minus 1152, exact.
__device__ __forceinline__ uint32_t codes_to_f16x2(float t0, float t1) {
    const uint32_t b = __byte_perm(__float_as_uint(t0), __float_as_uint(t1), 0x5410);
    const __half2 h = __hsub2(*reinterpret_cast<const __half2*>(&b), __half2half2(__ushort_as_half(0x6480)));
    return *reinterpret_cast<const uint32_t*>(&h);
}

// Four magic-float codes as four int8 bytes, the first in the lowest byte:
// the low bytes (0x80 + q) mod 256 of the magic floats, with the top bit flipped.
__device__ __forceinline__ uint32_t codes_to_i8x4(float t0, float t1, float t2, float t3) {
    const uint32_t lo = __byte_perm(__float_as_uint(t0), __float_as_uint(t1), 0x0040);
    const uint32_t hi = __byte_perm(__float_as_uint(t2), __float_as_uint(t3), 0x0040);
    return __byte_perm(lo, hi, 0x5410) ^ 0x80808080u;
}

// An integer 0 <= v < 2^23 as a float, exactly, without a conversion
// instruction: 2^23 + v has the pattern 0x4B000000 | v.
__device__ __forceinline__ float small_uint_to_float(uint32_t v) {
    return __fsub_rn(__uint_as_float(0x4B000000u | v), 8388608.0f);
}

// max(a, b), a NaN if either is one
__device__ __forceinline__ float fmaxf_nan(float a, float b) {
    float r;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    return r;
}

// The hardware base-2 exponential and reciprocal (MUFU; a few ulp), with
// subnormal inputs and results flushed to zero, which skips the scaling the
// subnormal-preserving forms add around the operation.
__device__ __forceinline__ float ex2_ftz(float x) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}
__device__ __forceinline__ float rcp_ftz(float x) {
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

// SiLU(u) = u / (1 + e^-u) = u * 1/(1 + 2^(-u log2 e)) with the hardware
// exponential and reciprocal (a few ulp; its consumers round to fp16 or to
// int8 codes).  u << 0 gives 2^(-u log2 e) = inf, a reciprocal of 0 and the
// product -0; e^-u below fp32's normal range (u > 87) flushes to 0, where
// 1 + e^-u is 1 either way.
__device__ __forceinline__ float silu_f(float u) {
    return u * rcp_ftz(1.0f + ex2_ftz(u * -1.4426950408889634f));
}

// The causal depthwise conv of one channel at token t (taps w.x .. w.w on
// x_{t-3} .. x_t) followed by SiLU.  Every kernel that evaluates the conv calls
// this one function, so their results agree bit for bit.
__device__ __forceinline__ float conv4_silu(const float4 w, float xm3, float xm2, float xm1, float x) {
    float u = w.x * xm3;
    u = fmaf(w.y, xm2, u);
    u = fmaf(w.z, xm1, u);
    u = fmaf(w.w, x, u);
    return silu_f(u);
}

// Two fp32 values in one 64-bit register pair, for the packed fp32
// instructions (mul / add / sub / fma .rn.f32x2: each half rounds as the scalar
// instruction does, so a packed evaluation gives the scalar one's bits).
struct F2 {
    unsigned long long v;
};
__device__ __forceinline__ F2 f2(float lo, float hi) {
    F2 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r.v) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f2_split(F2 a, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(a.v));
}
__device__ __forceinline__ F2 f2_mul(F2 a, F2 b) {
    F2 r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r.v) : "l"(a.v), "l"(b.v));
    return r;
}
__device__ __forceinline__ F2 f2_add(F2 a, F2 b) {
    F2 r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r.v) : "l"(a.v), "l"(b.v));
    return r;
}
__device__ __forceinline__ F2 f2_sub(F2 a, F2 b) {
    F2 r;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r.v) : "l"(a.v), "l"(b.v));
    return r;
}
__device__ __forceinline__ F2 f2_fma(F2 a, F2 b, F2 c) {
    F2 r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r.v) : "l"(a.v), "l"(b.v), "l"(c.v));
    return r;
}

// Gates of one value head from the projection's beta and alpha columns:
// log a = -exp(A_log) * softplus(alpha + dt_bias), b = sigmoid(beta).
__device__ __forceinline__ void gate_values(float beta, float alpha, float A_log, float dt_bias, float& log_a,
                                            float& b) {
    const float u = alpha + dt_bias;
    const float sp = fmaxf(u, 0.0f) + log1pf(expf(-fabsf(u)));
    log_a = -expf(A_log) * sp;
    b = 1.0f / (1.0f + expf(-beta));
}

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
