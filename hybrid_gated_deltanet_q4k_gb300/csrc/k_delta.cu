// Step 3: the gated delta rule, chunked (WY/UT form) with the state carried
// across chunks, on tensor cores.
//
// Per value head h (key head hk = h / (Hv/Hk)) the rule of Gated DeltaNet is
//     S_t = a_t S_{t-1} (I - b_t k_t k_t^T) + b_t v_t k_t^T,   o_t = S_t q_t,
// S a dv x dk matrix.  The pages name the chunked tensor-core form ("Verbs Are
// Fast" epic #3598, parked ticket "chunk-resident delta-rule scan vs the
// WY-chunked (tensor-core) form"; sparkinfer PR #511 "chunk-parallel GDN
// scan") and, as prior art, llama.cpp's token loop with the state in
// registers ("CRUX parity spike" #4220, technique table row 1).
//
// Within a chunk of C tokens entering with state S, gamma_i = sum_{j<=i} log a_j:
//     L_ij = b_i e^{gamma_i-gamma_j} k_i.k_j (j < i),   T = (I + L)^{-1}
//     R = diag(b) V - diag(b e^gamma) K S^T             (C x dv)
//     Delta = T R                                        (= U - W S^T of the WY form)
//     O = diag(e^gamma) Q S^T + A Delta,   A_ij = e^{gamma_i-gamma_j} q_i.k_j (j <= i)
//     S <- e^{gamma_C} S + Delta^T diag(e^{gamma_C - gamma}) K
// All exponents are <= 0.  Tokens past N are padded with log a = 0, b = 0,
// which leaves S unchanged.
//
// Two kernels, both on the fifth-generation tensor cores (tcgen05.mma
// kind::f16 with fp16 operands, fp32 accumulators in TMEM, operands staged by
// TMA):
//   delta_prep   one CTA per (chunk, key head), all chunks in parallel: the
//                Gram products Q K^T and K K^T once (the value heads of a key
//                head share them), K^T for the state pass, then per value
//                head gamma, the masked A, T = (I + L)^{-1} by recursive
//                doubling on the block-triangular structure, and A T.  Writes
//                [A T; T] and K^T (fp16, in the state pass's shared-memory
//                operand image) and a gate table (gamma, e^gamma, b,
//                e^{gamma_C - gamma}).
//   delta_state  one CTA per (head, 32 rows of S): the chunks in order.  Rows
//                of S evolve independently (row i only reads v[i]), so the
//                rows split across CTAs with no communication.  The fp32 state
//                stays in registers; its fp16 image is the B operand of the
//                next chunk's products.  A producer warp copies every operand
//                of chunk c+1 into shared memory (TMA boxes of 64 tokens x 64
//                halfs with the 128-byte swizzle for Q, K, V; bulk copies of
//                the prep images) as soon as chunk c has released its buffer.
// Products take fp16 operands rounded to nearest (the conv writes q, k, v in
// fp16; T, A T, S, R, Delta are rounded where they are produced) and
// accumulate in fp32; everything else is fp32.  fp16 keeps the 11 significant
// bits tf32 keeps, so o and S stay within ~5e-4 (relative L2) of the exact
// recurrence on the test workloads.  Its range ends at 65504: q and k are unit
// or smaller and A is bounded by |q||k|, but T, A T, S, R and Delta are
// checked where they are rounded, as is the output o (written in fp16), and a
// value out of range sets ERR_RANGE in this unit's error word (the result is
// then not to be used).
#include "common.cuh"
#include "tma.cuh"
#include "tcgen05.cuh"
#include "streams.h"

#include <algorithm>
#include <mutex>

namespace gdn {

static __device__ int g_delta_error;

constexpr int DC = GDN_CHUNK;  // 64
constexpr int DELTA_THREADS = 256;            // prep; compute warps of the state pass
constexpr int STATE_THREADS = DELTA_THREADS + 64;  // + TMA producer warp + MMA warp
constexpr int NV = 32;         // rows of S per state CTA
constexpr float F16_MAX = 65504.0f;

struct DeltaArgs {
    const uint16_t* qkv;  // [n][c_conv] fp16: q | k | v
    const float* log_a;   // [n][hv]
    const float* b;       // [n][hv]
    int n, hv, ratio, c_qk, c_conv, c_v;
    int chunk0, nchunks;  // the chunks [chunk0, chunk0 + nchunks) of this launch (indices are absolute)
    int nch_total;        // chunks of all sequences: the extent of the scratch tables
    uint16_t* TA;  // [nchunks][hv][2*DC][DC] [A T; T], fp16, in the swizzled operand image
    float* G;      // [nchunks][hv][DC][4]    gamma, e^gamma, b, e^{gamma_C - gamma}
    uint16_t* KT;  // [nchunks][hk][D][DC]    K^T, fp16, in the swizzled operand image
    const float* state_in;  // [hv][D][D] or null
    float* state_out;
    uint16_t* o;   // [n][c_v] fp16
    DeltaCkpt ckpt;  // state snapshots (ckpt.state null: none); one sequence only
    uint64_t prep_wait_ns;  // limit of the prep's wait for its [Q; K] copy
    int prep_no_copy;       // test only: the prep issues no copy, so that wait runs out
};

// Eight floats as eight fp16 (16 bytes, first value in the lowest half).
__device__ __forceinline__ uint4 f16x8(const float (&v)[8]) {
    return make_uint4(f16x2_bits(v[0], v[1]), f16x2_bits(v[2], v[3]), f16x2_bits(v[4], v[5]), f16x2_bits(v[6], v[7]));
}

// true when x is not a finite value fp16 can hold
__device__ __forceinline__ bool f16_out_of_range(float x) { return !(fabsf(x) <= F16_MAX); }


// ------------------------------------------------------------------ prep

constexpr int PREP_MAX_RATIO = 8;  // value heads per key head handled by one CTA
constexpr int PL = DC + 4;         // row pitch (floats) of L, T and the block temporaries

__host__ __device__ constexpr int align1k(int x) { return (x + 1023) & ~1023; }

template <int D>
struct PrepSmem {
    static constexpr int SLAB = DC * 128;          // 64 rows x 64 halfs, 128-byte swizzle
    static constexpr int NSLAB = D / 64;
    static constexpr int QK0 = 0;                  // [Q; K] [2*DC][D]: NSLAB slabs of Q rows then K rows (TMA)
    static constexpr int L0 = QK0 + NSLAB * 2 * SLAB;    // L  [DC][PL]
    static constexpr int T0 = L0 + DC * PL * 4;          // T  [DC][PL]
    static constexpr int W0 = T0 + DC * PL * 4;          // block temporaries [DC/2][PL]
    static constexpr int GL0 = W0 + DC / 2 * PL * 4;     // gamma [PREP_MAX_RATIO][DC]
    static constexpr int BB0 = GL0 + PREP_MAX_RATIO * DC * 4;  // b [PREP_MAX_RATIO][DC]
    static constexpr int EN0 = BB0 + PREP_MAX_RATIO * DC * 4;  // e^{-gamma} [PREP_MAX_RATIO][DC]
    // 8 KB pieces 0-5 of operand and output images once the Gram product is
    // done: the [Q; K] region, extended by a region of its own.
    static constexpr int NPIECE = 6;
    static constexpr int EX0 = align1k(EN0 + PREP_MAX_RATIO * DC * 4);
    static constexpr int B0 = EX0 + (NPIECE - 2 * NSLAB) * SLAB;   // mbarriers: TMA, MMA
    static constexpr int MISC0 = B0 + 16;                          // TMEM base address
    static constexpr int BYTES = MISC0 + 16;
    static __device__ __forceinline__ int piece(int p) { return p < 2 * NSLAB ? QK0 + p * SLAB : EX0 + (p - 2 * NSLAB) * SLAB; }
    static constexpr int AI = 0;    // A operand [DC][DC] (piece 0; piece 1 unused)
    // [A T; T] output staging [2*DC][DC], two buffers (pieces 2-3 and 4-5, one
    // 16 KB slab each) used by alternate value heads; the second buffer first
    // stages K^T (key rows 64p .. 64p+63 in piece 4 + p).
    static __device__ __forceinline__ int out(int j) { return piece(2 + 2 * (j & 1)); }
    static __device__ __forceinline__ int kt_stage(int p) { return piece(4 + p); }
};

// C = s * A B for blocks of the fp32 matrices in shared memory (row pitch PL):
// A is R x KK at a, B is KK x Cc at b, C at c; one 2 x 2 output tile per
// thread, threads 0 .. (R/2)(Cc/2) - 1 of the range given by t take part.
template <int R, int KK, int Cc>
__device__ __forceinline__ void block_mm(const float* a, const float* b, float* c, float s, int t) {
    constexpr int TC = Cc / 2;
    if (t < 0 || t >= (R / 2) * TC) return;
    const int r0 = 2 * (t / TC), c0 = 2 * (t % TC);
    float c00 = 0.f, c01 = 0.f, c10 = 0.f, c11 = 0.f;
#pragma unroll 8
    for (int k = 0; k < KK; ++k) {
        const float a0 = a[r0 * PL + k], a1 = a[(r0 + 1) * PL + k];
        const float2 bv = *reinterpret_cast<const float2*>(b + k * PL + c0);
        c00 = fmaf(a0, bv.x, c00);
        c01 = fmaf(a0, bv.y, c01);
        c10 = fmaf(a1, bv.x, c10);
        c11 = fmaf(a1, bv.y, c11);
    }
    *reinterpret_cast<float2*>(c + r0 * PL + c0) = make_float2(s * c00, s * c01);
    *reinterpret_cast<float2*>(c + (r0 + 1) * PL + c0) = make_float2(s * c10, s * c11);
}

// The same with one 2 x 4 output tile per thread (threads 0 .. (R/2)(Cc/4) - 1):
// per k a warp reads four rows of A and 128 contiguous bytes of B, half the
// shared-memory wavefronts of the 2 x 2 tiling for the same products.
// TRI 1: B is lower triangular (B[k][j] = 0 for k < j) and a warp's tiles
// share their columns, so its k loop starts at its first column; TRI 2: A is
// lower triangular (A[i][k] = 0 for k > i), so a warp's k loop ends past its
// last row.  The products skipped are exact zeros added to a sum that is
// still +0 (TRI 1) or to the finished sum (TRI 2): the results do not change.
template <int R, int KK, int Cc, int TRI = 0>
__device__ __forceinline__ void block_mm24(const float* a, const float* b, float* c, float s, int t) {
    constexpr int TC = Cc / 4, TR = R / 2;
    if (t < 0 || t >= TR * TC) return;
    const int r0 = TRI == 1 ? 2 * (t % TR) : 2 * (t / TC), c0 = TRI == 1 ? 4 * (t / TR) : 4 * (t % TC);
    const int tw0 = t & ~31, tw1 = min(t | 31, TR * TC - 1);   // the warp's first and last active thread
    const int k0 = TRI == 1 ? 4 * (tw0 / TR) : 0;
    const int k1 = TRI == 2 ? min(KK, 2 * (tw1 / TC) + 2) : KK;
    // the four sums of a row in two packed pairs (fma.rn.f32x2: each half
    // rounds as fmaf does, so the products and sums are those of the scalar form)
    F2 x[2][2] = {{f2(0.f, 0.f), f2(0.f, 0.f)}, {f2(0.f, 0.f), f2(0.f, 0.f)}};
#pragma unroll 8
    for (int k = k0; k < k1; ++k) {
        const float a0 = a[r0 * PL + k], a1 = a[(r0 + 1) * PL + k];
        const float4 bv = *reinterpret_cast<const float4*>(b + k * PL + c0);
        const F2 b01 = f2(bv.x, bv.y), b23 = f2(bv.z, bv.w), a00 = f2(a0, a0), a11 = f2(a1, a1);
        x[0][0] = f2_fma(a00, b01, x[0][0]);
        x[0][1] = f2_fma(a00, b23, x[0][1]);
        x[1][0] = f2_fma(a11, b01, x[1][0]);
        x[1][1] = f2_fma(a11, b23, x[1][1]);
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        float v0, v1, v2, v3;
        f2_split(x[i][0], v0, v1);
        f2_split(x[i][1], v2, v3);
        *reinterpret_cast<float4*>(c + (r0 + i) * PL + c0) = make_float4(s * v0, s * v1, s * v2, s * v3);
    }
}

// One CTA per (chunk, key head), 256 threads:
//   - TMA loads the chunk's Q and K rows of the key head as one stacked
//     [Q; K] operand; one tcgen05 product [Q; K] K^T (M = 128, N = 64) leaves
//     q_i.k_j in TMEM lanes 0-63 and k_i.k_j in lanes 64-127 (all value heads
//     of the key head share them).  Warp w then holds row 32(w%4) + lane,
//     columns 32(w/4) .. +31, in registers.
//   - K^T, in the state pass's operand image, by 8 x 8 transposes of the K
//     rows (ldmatrix.trans, stmatrix).
//   - For each value head (gates differ): the gate prefix sums gamma; the
//     masked A (rows of lanes 0-63) as an fp16 operand image; L (rows of
//     lanes 64-127) into shared memory; T = (I + L)^-1 by recursive doubling
//     on the block triangular structure:
//         16 x 16 diagonal blocks by substitution (one column per lane),
//         inv [[A, 0], [C, B]] = [[A^-1, 0], [-B^-1 C A^-1, B^-1]]
//     for 32 x 32 and then 64 x 64, every block product in fp32 on the CUDA
//     cores; A T on the tensor cores; [A T; T] (fp16) and the gate table to
//     global memory.  Alternate heads stage their output in alternate
//     buffers, so a head never waits for the previous head's store.
// 88 registers a thread: a prep CTA then fits on an SM beside a state CTA,
// so the prep of the next token segment runs in the shadow of the state
// pass.  Registers are allocated per SM sub-partition (16K each, warps spread
// over the four): three state warps (112 registers a thread once rounded)
// leave 5632 registers, two prep warps of 88.
template <int D>
__global__ void __maxnreg__(88) delta_prep_kernel(const __grid_constant__ CUtensorMap qkv_map, DeltaArgs a,
                                                   const __grid_constant__ SeqTable sq) {
    using L = PrepSmem<D>;
    extern __shared__ __align__(1024) unsigned char smb[];
    unsigned char* base = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smb) + 1023) & ~uintptr_t(1023));
    float* Ls = reinterpret_cast<float*>(base + L::L0);
    float* Ts = reinterpret_cast<float*>(base + L::T0);
    float* Ws = reinterpret_cast<float*>(base + L::W0);
    uint64_t* bars = reinterpret_cast<uint64_t*>(base + L::B0);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(base + L::MISC0);

    // chunk chunk0 + blockIdx.x of sequence blockIdx.z (none past its end)
    const int sq_i = blockIdx.z, local = a.chunk0 + blockIdx.x;
    if (local >= sq.unit[sq_i + 1] - sq.unit[sq_i]) return;
    const int chunk = sq.unit[sq_i] + local, hk = blockIdx.y;
    if (!GDN_IN_RANGE(g_delta_error, chunk < a.nch_total && (hk + 1) * a.ratio <= a.hv)) return;
    const int t0 = sq.tok[sq_i] + local * DC, t_end = sq.tok[sq_i + 1];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int r = a.ratio;

    if (tid == 0) {
        mbar_init_cta(bars + 0, 1);
        mbar_init_cta(bars + 1, 1);
        mbar_init_fence();
        if (!a.prep_no_copy) {
            mbar_expect_tx(bars + 0, 2 * L::NSLAB * L::SLAB);
            for (int sl = 0; sl < L::NSLAB; ++sl) {
                unsigned char* dst = base + L::QK0 + sl * 2 * L::SLAB;
                tma_load_2d_tile(dst, &qkv_map, bars + 0, hk * D + 64 * sl, t0);
                tma_load_2d_tile(dst + L::SLAB, &qkv_map, bars + 0, a.c_qk + hk * D + 64 * sl, t0);
            }
        }
    }
    if (warp == 0) t5::alloc(tslot, 128);
    // T's blocks (rows 0-15, cols 16-31) and (rows 32-47, cols 48-63) stay zero: the
    // 32 x 32 diagonal blocks of T are read whole by the last doubling step
    for (int idx = tid; idx < 2 * 16 * 16; idx += DELTA_THREADS) {
        const int o = 32 * (idx >> 8), rr = (idx >> 4) & 15, cc = idx & 15;
        Ts[(o + rr) * PL + o + 16 + cc] = 0.f;
    }
    // gates of the value heads h = hk*r + j: log a -> inclusive prefix sum gamma
    // and e^{-gamma} (one warp per head)
    for (int j = warp; j < r; j += DELTA_THREADS / 32) {
        const int h = hk * r + j;
        float* gl = reinterpret_cast<float*>(base + L::GL0) + j * DC;
        float* bb = reinterpret_cast<float*>(base + L::BB0) + j * DC;
        float* en = reinterpret_cast<float*>(base + L::EN0) + j * DC;
        float x0 = 0.f, x1 = 0.f;
        const int ta = t0 + 2 * lane, tb = ta + 1;
        if (ta < t_end) x0 = a.log_a[static_cast<int64_t>(ta) * a.hv + h];
        if (tb < t_end) x1 = a.log_a[static_cast<int64_t>(tb) * a.hv + h];
        bb[2 * lane] = ta < t_end ? a.b[static_cast<int64_t>(ta) * a.hv + h] : 0.f;
        bb[2 * lane + 1] = tb < t_end ? a.b[static_cast<int64_t>(tb) * a.hv + h] : 0.f;
        float s = x0 + x1;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float y = __shfl_up_sync(0xffffffffu, s, o);
            if (lane >= o) s += y;
        }
        gl[2 * lane] = s - x1;
        gl[2 * lane + 1] = s;
        en[2 * lane] = __expf(x1 - s);
        en[2 * lane + 1] = __expf(-s);
    }
    t5::fence_before();
    __syncthreads();
    t5::fence_after();
    const uint32_t tmem = *tslot;

    bool ok = true;
    if (tid == 0) {
        ok = mbar_wait_bounded(bars + 0, 0, &g_delta_error, ERR_WAIT_TIMEOUT, a.prep_wait_ns);
        if (ok) {
            t5::fence_after();
            const uint32_t sb = smem_addr(base);
            const uint64_t dA = t5::desc_sw128(sb + L::QK0), dB = t5::desc_sw128(sb + L::QK0 + L::SLAB);
            constexpr uint32_t ID = t5::idesc_f16(128, DC);
#pragma unroll
            for (int k = 0; k < D / 16; ++k) {
                const uint64_t off = static_cast<uint64_t>((k >> 2) * (2 * L::SLAB >> 4) + 2 * (k & 3));
                t5::mma_f16(tmem, dA + off, dB + off, ID, k > 0 ? 1u : 0u);
            }
            t5::commit(bars + 1);
        }
    }
    ok = __syncthreads_and(ok);
    if (!ok) {
        // the copy never landed: nothing was issued; give the copy (bounded) time to land
        if (tid == 0) mbar_wait_bounded(bars + 0, 0, nullptr, 0, 20000000ull);
        t5::fence_before();
        __syncthreads();
        if (warp == 0) t5::dealloc(tmem, 128);
        return;
    }

    // ---- K^T image for the state pass: warp task = tokens 8tb .. 8tb+7 x key
    // rows 32dq .. 32dq+31, four 8 x 8 blocks transposed; written to its staging
    // while the Gram product runs, then by bulk copies.  Every thread observes
    // the copy's completion itself (it has completed: this returns at once).
    mbar_wait_bounded(bars + 0, 0, &g_delta_error, ERR_WAIT_TIMEOUT);
    for (int task = warp; task < (DC / 8) * (D / 32); task += DELTA_THREADS / 32) {
        const int tb = task % (DC / 8), dq = task / (DC / 8);
        const int d = 32 * dq + 8 * (lane >> 3), rr = lane & 7;   // block of this lane's address, row rr of it
        uint32_t f[4];
        ldsm_x4_trans(smem_addr(base + L::QK0 + (d >> 6) * 2 * L::SLAB + L::SLAB + sw128_f16(8 * tb + rr, d & 63)), f);
        const int dr = d + rr;
        stsm_x4(smem_addr(base + L::kt_stage(dr >> 6) + sw128_f16(dr & 63, 8 * tb)), f);
    }

    // ---- the Gram rows of this thread
    const int q = warp & 3, half = warp >> 2;
    const bool qrow = q < 2;                 // lanes 0-63: q_i.k_j; lanes 64-127: k_i.k_j
    const int row = 32 * (q & 1) + lane;     // token i of this row
    const int c0 = 32 * half;                // first column (token j)
    const bool upper = (q & 1) == 0 && half == 1;   // rows 0-31 x columns 32-63: every j > i, masked
    float g[32];
    if (!mbar_wait_bounded(bars + 1, 0, &g_delta_error, ERR_WAIT_TIMEOUT)) ok = false;
    ok = __all_sync(0xffffffffu, ok);
    if (ok) {
        t5::fence_after();
        t5::ld32(tmem + (static_cast<uint32_t>(32 * q) << 16) + c0, g);
    }
    fence_proxy_async_smem();               // the K^T staging goes to the bulk copies
    ok = __syncthreads_and(ok);
    if (!ok) {
        if (tid == 0) mbar_wait_bounded(bars + 1, 0, nullptr, 0, 200000000ull);
        t5::fence_before();
        __syncthreads();
        if (warp == 0) t5::dealloc(tmem, 128);
        return;
    }
    if (tid == 0) {
        uint16_t* kt = a.KT + (static_cast<int64_t>(chunk) * gridDim.y + hk) * D * DC;
        for (int p = 0; p < L::NSLAB; ++p) bulk_store_1d(kt + p * (64 * DC), base + L::kt_stage(p), L::SLAB);
        bulk_commit();
    }

    bool bad = false;   // a T or A T value outside the fp16 range
    for (int j = 0; j < r; ++j) {
        const int h = hk * r + j;
        const int64_t cb = static_cast<int64_t>(chunk) * a.hv + h;
        const float* gl = reinterpret_cast<const float*>(base + L::GL0) + j * DC;
        const float* bb = reinterpret_cast<const float*>(base + L::BB0) + j * DC;
        const float* en = reinterpret_cast<const float*>(base + L::EN0) + j * DC;
        const float gi = gl[row];
        // this head's output buffer was last read by the store two heads back
        // (or, for head 1, by the K^T store): let that read finish first
        if (tid == 0 && j >= 1) bulk_wait_read_but_last();
        // The decay e^{gamma_i - gamma_j} of an entry (j <= i, so at most 1): as
        // e^{gamma_i} e^{-gamma_j} when the chunk's whole decay gamma_C >= -64, so
        // that every factor is a normal fp32 value, else by its own exponential.
        auto entries = [&](auto decay) {
            if (qrow) {
                // A_ij = e^{gamma_i - gamma_j} q_i.k_j (j <= i), |A_ij| <= |q_i||k_j| <= 1:
                // half of one 128-byte row of the swizzled image (zeros above the diagonal block)
                unsigned char* arow = base + L::piece(L::AI) + row * 128;
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    uint4 w = make_uint4(0u, 0u, 0u, 0u);
                    if (!upper) {
                        float v[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const int c = c0 + 8 * m + e;
                            v[e] = c <= row ? decay(c) * g[8 * m + e] : 0.f;
                        }
                        w = f16x8(v);
                    }
                    *reinterpret_cast<uint4*>(arow + ((((c0 >> 3) + m) ^ (row & 7)) << 4)) = w;
                }
            } else {
                // L_ij = b_i e^{gamma_i - gamma_j} k_i.k_j (j < i)
                const float bi = bb[row];
#pragma unroll
                for (int m = 0; m < 8; ++m) {
                    float v[4] = {0.f, 0.f, 0.f, 0.f};
                    if (!upper) {
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int c = c0 + 4 * m + e;
                            v[e] = c < row ? bi * decay(c) * g[4 * m + e] : 0.f;
                        }
                    }
                    *reinterpret_cast<float4*>(Ls + row * PL + c0 + 4 * m) = make_float4(v[0], v[1], v[2], v[3]);
                }
            }
        };
        if (gl[DC - 1] >= -64.f) {
            const float egi = __expf(gi);
            entries([&](int c) { return egi * en[c]; });
        } else {
            entries([&](int c) { return __expf(gi - gl[c]); });
        }
        __syncthreads();
        // 16 x 16 diagonal blocks of T: warp 0 blocks 0, 1; warp 1 blocks 2, 3; lane = column.
        // Right-looking: once t_k is final it is folded into the sums of the rows below,
        // so each step waits on one product, not on a sum over k.
        if (warp < 2) {
            const int blk = 2 * warp + (lane >> 4), cc = lane & 15, o = 16 * blk;
            float t[16], sum[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) sum[i] = 0.f;
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                t[k] = k < cc ? 0.f : (k == cc ? 1.f : -sum[k]);
#pragma unroll
                for (int i = k + 1; i < 16; ++i) sum[i] = fmaf(Ls[(o + i) * PL + o + k], t[k], sum[i]);
            }
#pragma unroll
            for (int rr = 0; rr < 16; ++rr) Ts[(o + rr) * PL + o + cc] = t[rr];
        }
        __syncthreads();
        // 32 x 32 blocks: T21 = -T22 (L21 T11), T43 = -T44 (L43 T33)
        {
            const int p = tid >> 6, o = 32 * p;   // threads 0-63: rows 16-31; 64-127: rows 48-63
            block_mm<16, 16, 16>(Ls + (o + 16) * PL + o, Ts + o * PL + o, Ws + 16 * p * PL, 1.f, p < 2 ? (tid & 63) : -1);
            __syncthreads();
            block_mm<16, 16, 16>(Ts + (o + 16) * PL + o + 16, Ws + 16 * p * PL, Ts + (o + 16) * PL + o, -1.f,
                                 p < 2 ? (tid & 63) : -1);
            __syncthreads();
        }
        // 64 x 64: T[32:64, 0:32] = -T[32:64, 32:64] (L[32:64, 0:32] T[0:32, 0:32])
        block_mm24<32, 32, 32, 1>(Ls + 32 * PL, Ts, Ws, 1.f, tid);
        __syncthreads();
        block_mm24<32, 32, 32, 2>(Ts + 32 * PL + 32, Ws, Ts + 32 * PL, -1.f, tid);
        __syncthreads();
        // The T rows of the output (rows 64-127 of [A T; T]), fp16, which are also
        // the B operand of A T (MN-major: row k holds T_k0 .. T_k63); thread -> row
        // tid%64, columns 16(tid/64) ..
        {
            const int rr = tid & 63, cq = 16 * (tid >> 6);
            unsigned char* orow = base + L::out(j) + (DC + rr) * 128;
            float mx = 0.f;
#pragma unroll
            for (int m = 0; m < 2; ++m) {
                const int c = cq + 8 * m;
                const float4 r0 = *reinterpret_cast<const float4*>(Ts + rr * PL + c);
                const float4 r1 = *reinterpret_cast<const float4*>(Ts + rr * PL + c + 4);
                const float rv[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
                float v[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    v[e] = c + e <= rr ? rv[e] : 0.f;
                    mx = fmaxf_nan(mx, fabsf(v[e]));
                }
                *reinterpret_cast<uint4*>(orow + ((((c >> 3) ^ (rr & 7)) & 7) << 4)) = f16x8(v);
            }
            bad |= !(mx <= F16_MAX);
        }
        if (tid < DC) {
            const float gv = gl[tid];
            *reinterpret_cast<float4*>(a.G + (cb * DC + tid) * 4) = make_float4(gv, expf(gv), bb[tid], expf(gl[DC - 1] - gv));
        }
        fence_proxy_async_smem();
        t5::fence_before();
        __syncthreads();
        // A T on the tensor cores (M = 64, N = 64, K = 64) into TMEM columns 64-127;
        // B = the T rows, MN-major (bit 16 of the instruction descriptor).  With N =
        // 64 fp16, one 128-byte swizzle atom wide, its descriptor is the K-major one
        // (8-row groups 1024 bytes apart); a K step of 16 rows is 2048 bytes further.
        bool mok = true;
        if (tid == 0) {
            t5::fence_after();
            const uint32_t sb = smem_addr(base);
            const uint64_t dA = t5::desc_sw128(sb + L::piece(L::AI)), dB = t5::desc_sw128(sb + L::out(j) + DC * 128);
            constexpr uint32_t ID = t5::idesc_f16(64, DC) | (1u << 16);
#pragma unroll
            for (int k = 0; k < DC / 16; ++k)
                t5::mma_f16(tmem + 64, dA + 2 * k, dB + static_cast<uint64_t>(k * (2048 >> 4)), ID, k > 0 ? 1u : 0u);
            t5::commit(bars + 1);
        }
        if (!mbar_wait_bounded(bars + 1, (j + 1) & 1, &g_delta_error, ERR_WAIT_TIMEOUT)) mok = false;
        mok = __all_sync(0xffffffffu, mok);
        if (mok) {
            // rows 0-63 of the output: A T, row i in lane 32(i/16) + i%16 (M = 64)
            t5::fence_after();
            float at[32];
            t5::ld32(tmem + (static_cast<uint32_t>(32 * q) << 16) + 64 + c0, at);
            if (lane < 16) {
                const int ri = 16 * q + lane;
                unsigned char* orow = base + L::out(j) + ri * 128;
                float mx = 0.f;
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    float v[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        v[e] = at[8 * m + e];
                        mx = fmaxf_nan(mx, fabsf(v[e]));
                    }
                    *reinterpret_cast<uint4*>(orow + ((((c0 >> 3) + m) ^ (ri & 7)) << 4)) = f16x8(v);
                }
                bad |= !(mx <= F16_MAX);
            }
        }
        fence_proxy_async_smem();
        t5::fence_before();
        mok = __syncthreads_and(mok);   // also: A and L are free for the next head
        if (tid == 0 && mok) {
            bulk_store_1d(a.TA + cb * 2 * DC * DC, base + L::out(j), 2 * L::SLAB);
            bulk_commit();
        }
        if (!mok) break;
    }
    if (bad) atomicCAS(&g_delta_error, 0, ERR_RANGE);
    if (tid == 0) bulk_wait_all();
    t5::fence_before();
    __syncthreads();
    if (warp == 0) t5::dealloc(tmem, 128);
}

// ------------------------------------------------------------------ state pass

// Shared-memory layout of the state pass (byte offsets; every operand base is
// 1024-byte aligned, as the 128-byte swizzle requires).  Operands are slabs of
// rows of 64 fp16 (128 bytes) with the 128-byte swizzle, K-major for the
// tensor cores: the image a 2-D TMA box with SWIZZLE_128B writes, and the one
// delta_prep writes for [A T; T] and K^T.
template <int D>
struct StateSmem {
    static constexpr int SLAB = DC * 128;          // 64 rows x 64 halfs
    static constexpr int NSLAB = D / 64;
    static constexpr int QK_SLAB = 2 * SLAB;       // Q rows 0-63, K rows 64-127
    static constexpr int SOP = NV * 128;           // 32 rows x 64 halfs
    static constexpr int KT_BYTES = D * 128;       // one K^T [D][DC]
    static constexpr int QK0 = 0;                  // [Q; K] [2*DC][D]  (TMA)
    static constexpr int KT0 = QK0 + NSLAB * QK_SLAB;   // K^T [2][D][DC] (bulk copies)
    static constexpr int TA0 = KT0 + 2 * KT_BYTES; // [A T; T] [2*DC][DC] (bulk copy of the prep image)
    static constexpr int V0 = TA0 + QK_SLAB;       // V [DC][64]        (TMA; this CTA's NV columns at i0 % 64)
    // the three B operands the compute warps write are stored MN-major (row =
    // K index, NV = 32 fp16 of 64 bytes each, 64-byte swizzle), so a thread
    // holding 16 consecutive v of one K index writes two 16-byte chunks
    static constexpr int S0 = V0 + SLAB;           // S [D][NV]         fp16 operand of X, Y
    static constexpr int R0 = S0 + NSLAB * SOP;    // R [DC][NV]
    static constexpr int E0 = R0 + SOP;            // Delta~ [DC][NV]
    static constexpr int G0 = E0 + SOP;            // gate table [2][DC] x (gamma, e^gamma, b, e^{gamma_C-gamma})
    static constexpr int B0 = G0 + 2 * DC * 16;    // mbarriers
    static constexpr int NBAR = 14;
    static constexpr int MISC0 = B0 + NBAR * 8;    // TMEM base address, abort flag
    static constexpr int BYTES = MISC0 + 16;
    static_assert(BYTES + 1024 <= 227 * 1024, "state pass shared memory");
};

// TMEM columns (fp32 accumulators of NV = 32 columns).  [Q; K] S^T is
// double-buffered: the output reads Y of chunk c while X, Y of chunk c+1 run.
// Its eight K steps alternate between two accumulators (the second TM_XY2
// columns further on), summed when read: two chains of four dependent
// products complete sooner than one of eight.  256 columns, so a prep CTA
// (128) still fits beside a state CTA.
constexpr uint32_t TM_XY = 0, TM_DZ = 64, TM_U = 96, TM_XY2 = 128;
constexpr uint32_t TM_COLS = 256;

enum StateBar : int {
    F_QK, F_KT0, F_KT1, F_V, F_TA,       // copies landed (tx bytes)
    E_QK, E_KT0, E_KT1, E_V, E_TA,       // buffer free again
    M_XY, M_DZ, M_U,                     // MMA groups complete (tcgen05.commit)
    M_FIN,                               // every MMA of the CTA complete (shutdown)
};

// Bounded wait on an mbarrier phase that also gives up when another role of
// the CTA has aborted.
__device__ __forceinline__ bool state_wait(uint64_t* bar, uint32_t parity, volatile int* abort) {
    if (mbar_test(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (mbar_test(bar, parity)) return true;
        if (*abort) return false;
        if (globaltimer_ns() - t0 > 2000000000ull) {
            atomicCAS(&g_delta_error, 0, ERR_WAIT_TIMEOUT);
            *abort = 1;
            return false;
        }
    }
}

// Named barriers between the compute warps (which write operands) and the
// MMA warp (which then issues the products).  Both sides wait (bar.sync), so
// no thread can reach a barrier a second time before it has completed.
enum StateNamedBar : int { NB_S = 1, NB_R = 2, NB_D = 3 };
__device__ __forceinline__ void nb_sync(int id) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "n"(DELTA_THREADS + 32) : "memory");
}

__device__ __forceinline__ void mbar_arrive_cta(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// Issue the k steps [0, NK) of one MMA chain with a K-major A operand (a K
// step is 16 fp16 = 32 bytes, four per 128-byte swizzle row, then the next
// slab) and an MN-major B operand (desc_sw64_mn): a K step of 16 rows of
// 64 bytes is 1024 bytes further on.
template <int NK, int A_SLAB>
__device__ __forceinline__ void mma_chain_bmn(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc) {
#pragma unroll
    for (int k = 0; k < NK; ++k)
        t5::mma_f16(d_tmem, adesc + static_cast<uint64_t>((k >> 2) * (A_SLAB >> 4) + 2 * (k & 3)),
                    bdesc + static_cast<uint64_t>(k * (1024 >> 4)), idesc, k > 0 ? 1u : 0u);
}

// The same with the even K steps into d_tmem and the odd ones into d_tmem +
// TM_XY2 (each accumulator's first step overwrites it).
template <int NK, int A_SLAB>
__device__ __forceinline__ void mma_chain_bmn_split(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc) {
#pragma unroll
    for (int k = 0; k < NK; ++k)
        t5::mma_f16(d_tmem + ((k & 1) ? TM_XY2 : 0u), adesc + static_cast<uint64_t>((k >> 2) * (A_SLAB >> 4) + 2 * (k & 3)),
                    bdesc + static_cast<uint64_t>(k * (1024 >> 4)), idesc, k > 1 ? 1u : 0u);
}

// One CTA per (value head, NV rows of S); 320 threads:
//   warps 0-7  compute.  Warp w reads TMEM lanes 32*(w%4) .. +31 and columns
//              16*(w/4) .. +15 of each 32-column accumulator.
//   warp 8     producer: TMA boxes of Q, K, V; bulk copies of K^T, [A T; T],
//              gates.
//   warp 9     TMEM owner and MMA issuer: meets the compute warps at a named
//              barrier once they have written an operand, then issues (one
//              thread).
// Per chunk, with S the NV x D slice of the state (fp16 operands, fp32 sums):
//   MMA  [Y; X] = [Q; K] S^T          (M = 128: Y in lanes 0-63, X in 64-127;
//        even and odd K steps in two accumulators, added when read)
//   warps 2,3,6,7 (lanes 64-127)  R = diag(b)(V - diag(e^gamma) X) -> R^T
//   MMA  [Z; Delta] = [A T; T] R      (M = 128: Z = A Delta in lanes 0-63,
//        Delta in lanes 64-127; delta_prep folds A T, so A Delta costs no
//        extra product)
//   warps 2,3,6,7  Delta~^T = (diag(e^{gamma_C-gamma}) Delta)^T
//   MMA  U = K^T Delta~               (M = D: row d in lane d, or 32*(d/16)+d%16)
//   warps  S <- e^{gamma_C} S + U in fp32 registers, its fp16 image -> S
//   MMA  next chunk's [Q; K] S^T
//   warps 0,1,4,5 (lanes 0-63)  O = diag(e^gamma) Y + Z, while it runs.
// The state's chain per chunk is four dependent steps (X, R, Delta, U); the
// output stays off it.  Every thread meets every named barrier of
// every chunk, also after a wait ran out (it then skips the work, and the MMA
// warp issues nothing once its own check has seen the abort), so no barrier is
// ever left waiting.
// At most 112 registers a thread: three of this CTA's warps share a
// sub-partition's 16K registers, and 112 leaves room for two warps of a prep
// CTA (88 registers) beside them, so the next segment's prep runs in the
// shadow of this pass; without the cap the compiler may take more.
template <int D>
__global__ void __maxnreg__(112)
delta_state_kernel(const __grid_constant__ CUtensorMap qkv_map, DeltaArgs a, const __grid_constant__ SeqTable sq) {
    using L = StateSmem<D>;
    extern __shared__ __align__(1024) unsigned char smb[];
    unsigned char* base = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smb) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(base + L::B0);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(base + L::MISC0);
    volatile int* abort = reinterpret_cast<volatile int*>(base + L::MISC0 + 4);

    const int h = blockIdx.x, i0 = blockIdx.y * NV, hk = h / a.ratio;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (!GDN_IN_RANGE(g_delta_error, h < a.hv && i0 + NV <= D)) return;
    const uint32_t sbase = smem_addr(base);
    // chunks chunk0 .. chunk0 + nchunks - 1 of sequence blockIdx.z, those it has
    const int sq_i = blockIdx.z;
    const int nch = min(a.nchunks, sq.unit[sq_i + 1] - sq.unit[sq_i] - a.chunk0);
    if (nch <= 0) return;
    const int cg0 = sq.unit[sq_i] + a.chunk0;            // global index of the first (scratch tables)
    const int tc0 = sq.tok[sq_i] + a.chunk0 * DC;        // its first token
    const int t_end = sq.tok[sq_i + 1];
    const int64_t sq_off = static_cast<int64_t>(sq_i) * a.hv * D * D;
    // the sequence's state before the first chunk: the caller's (or zero) at
    // its start, else what the previous token segment left in state_out
    const float* st_in = a.chunk0 == 0 ? (a.state_in ? a.state_in + sq_off : nullptr) : a.state_out + sq_off;
    float* st_out = a.state_out + sq_off;

    if (tid == 0) {
        for (int i = F_QK; i <= F_TA; ++i) mbar_init_cta(bars + i, 1);
        for (int i = E_QK; i <= E_TA; ++i) mbar_init_cta(bars + i, 1);
        mbar_init_cta(bars + E_V, DELTA_THREADS / 32);
        for (int i = M_XY; i <= M_FIN; ++i) mbar_init_cta(bars + i, 1);
        mbar_init_fence();
        *abort = 0;
    }
    if (warp == 9) t5::alloc(tslot, TM_COLS);
    t5::fence_before();
    __syncthreads();
    t5::fence_after();
    const uint32_t tmem = *tslot;

    if (warp == 8) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            auto cb = [&](int c) { return static_cast<int64_t>(c) * a.hv + h; };
            for (int j = 0; j < nch; ++j) {
                const int c = cg0 + j, tc = tc0 + j * DC;
                if (!GDN_IN_RANGE(g_delta_error, c < a.nch_total)) {
                    *abort = 1;
                    break;
                }
                const uint32_t pp = (j - 1) & 1;   // phase of the previous chunk's release
                if (j >= 1 && !state_wait(bars + E_QK, pp, abort)) break;
                mbar_expect_tx(bars + F_QK, 2 * L::NSLAB * L::SLAB);
                for (int sl = 0; sl < L::NSLAB; ++sl) {
                    unsigned char* dst = base + L::QK0 + sl * L::QK_SLAB;
                    tma_load_2d_tile(dst, &qkv_map, bars + F_QK, hk * D + 64 * sl, tc);
                    tma_load_2d_tile(dst + L::SLAB, &qkv_map, bars + F_QK, a.c_qk + hk * D + 64 * sl, tc);
                }
                const int kb = j & 1;
                if (j >= 2 && !state_wait(bars + E_KT0 + kb, ((j - 2) >> 1) & 1, abort)) break;
                mbar_expect_tx(bars + F_KT0 + kb, L::KT_BYTES);
                bulk_load_1d(base + L::KT0 + kb * L::KT_BYTES,
                             a.KT + (static_cast<int64_t>(c) * (a.hv / a.ratio) + hk) * D * DC, L::KT_BYTES,
                             bars + F_KT0 + kb);
                if (j >= 1 && !state_wait(bars + E_V, pp, abort)) break;
                mbar_expect_tx(bars + F_V, L::SLAB + DC * 16);
                tma_load_2d_tile(base + L::V0, &qkv_map, bars + F_V, 2 * a.c_qk + h * D + (i0 & ~63), tc);
                bulk_load_1d(base + L::G0 + (j & 1) * DC * 16, a.G + cb(c) * DC * 4, DC * 16, bars + F_V);
                if (j >= 1 && !state_wait(bars + E_TA, pp, abort)) break;
                mbar_expect_tx(bars + F_TA, L::QK_SLAB);
                bulk_load_1d(base + L::TA0, a.TA + cb(c) * 2 * DC * DC, L::QK_SLAB, bars + F_TA);
            }
        }
    } else if (warp == 9) {
        // ------------------------------------------------------------ MMA issuer
        // B operands MN-major (bit 16 of the instruction descriptor)
        constexpr uint32_t ID128 = t5::idesc_f16(128, NV) | (1u << 16);
        constexpr uint32_t IDU = t5::idesc_f16(D, NV) | (1u << 16);
        const uint64_t dQK = t5::desc_sw128(sbase + L::QK0), dS = t5::desc_sw64_mn(sbase + L::S0);
        const uint64_t dTA = t5::desc_sw128(sbase + L::TA0), dR = t5::desc_sw64_mn(sbase + L::R0);
        const uint64_t dE = t5::desc_sw64_mn(sbase + L::E0);
        const uint64_t dKT = t5::desc_sw128(sbase + L::KT0);
        const bool leader = lane == 0;
        // Leader only: the copy a product reads has landed and nothing has failed.
        // It is checked before the named barrier, while the compute warps still
        // write their operand, so that after the barrier only the tcgen05 fence
        // stands between it and the issue.  (A wait that ran out sets the abort
        // flag; products issued after another role aborted read stale operands,
        // which is harmless: nothing reads their results.)
        auto ready = [&](int bar, uint32_t parity) {
            bool ok = false;
            if (leader) ok = !*abort && state_wait(bars + bar, parity, abort);
            __syncwarp();
            return ok;
        };
        for (int j = 0; j < nch; ++j) {
            const uint32_t ph = j & 1;
            bool go = ready(F_QK, ph);
            nb_sync(NB_S);                      // S of chunk j written
            if (go) {
                t5::fence_after();
                mma_chain_bmn_split<D / 16, L::QK_SLAB>(tmem + TM_XY + 32 * ph, dQK, dS, ID128);
                t5::commit(bars + M_XY);
                t5::commit(bars + E_QK);
            }
            go = ready(F_TA, ph);
            nb_sync(NB_R);                      // R^T written
            if (go) {
                t5::fence_after();
                mma_chain_bmn<DC / 16, L::QK_SLAB>(tmem + TM_DZ, dTA, dR, ID128);
                t5::commit(bars + M_DZ);
                t5::commit(bars + E_TA);
            }
            go = ready(F_KT0 + ph, (j >> 1) & 1);
            nb_sync(NB_D);                      // Delta~^T written
            if (go) {
                t5::fence_after();
                mma_chain_bmn<DC / 16, L::KT_BYTES>(tmem + TM_U, dKT + ph * (L::KT_BYTES >> 4), dE, IDU);
                t5::commit(bars + M_U);
                t5::commit(bars + E_KT0 + ph);
            }
        }
        __syncwarp();
        if (leader) {
            // every MMA issued above has completed before TMEM is released
            t5::commit(bars + M_FIN);
            mbar_wait_bounded(bars + M_FIN, 0, nullptr, 0, 200000000ull);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ compute
        const int q = warp & 3, hc = warp >> 2;
        const int v0 = 16 * hc;
        const bool xw = q >= 2;                 // lanes 64-127: X rows; lanes 0-63: Y rows
        const int tok = 32 * (q & 1) + lane;    // token of this lane in the M = 128 products
        const bool act = lane < 16;             // lanes holding rows of an M = 64 product
        const uint32_t tl = tmem + (static_cast<uint32_t>(32 * q) << 16) + v0;   // this warp's lanes, columns v0..
        // key-dimension row d of U owned by this thread (all lanes for D = 128, lanes 0-15 for D = 64)
        const bool own_d = D == 128 ? true : act;
        const int d = D == 128 ? 32 * q + lane : 16 * q + lane;
        const int vc = (i0 & 63) + v0;          // first V column of this warp in the 64-column V box
        bool bad = false;                       // an S, R, Delta~ or o value outside the fp16 range

        float S[16];
#pragma unroll
        for (int v = 0; v < 16; ++v)
            S[v] = (own_d && st_in) ? st_in[(static_cast<int64_t>(h) * D + i0 + v0 + v) * D + d] : 0.f;
        // values v0 .. v0+15 of row k of an MN-major [K][NV] operand at off: two
        // 16-byte chunks of the 64-byte row, placed by the 64-byte swizzle
        auto write_row = [&](int off, int k, const float (&x)[16]) {
            float m = 0.0f;
#pragma unroll
            for (int v = 0; v < 16; ++v) m = fmaxf_nan(m, fabsf(x[v]));
            bad |= !(m <= F16_MAX);              // an infinity, a NaN or a value past the fp16 range
            float lo[8], hi[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                lo[e] = x[e];
                hi[e] = x[8 + e];
            }
            unsigned char* row = base + off + k * 64;
            const int c0 = v0 >> 3, sw = (k >> 1) & 3;
            *reinterpret_cast<uint4*>(row + ((c0 ^ sw) << 4)) = f16x8(lo);
            *reinterpret_cast<uint4*>(row + (((c0 + 1) ^ sw) << 4)) = f16x8(hi);
        };
        auto write_s = [&]() {
            if (own_d) write_row(L::S0, d, S);
        };
        // the row of token t of an [DC][NV] operand (R, Delta~)
        auto write_col = [&](int off, int t, const float (&x)[16]) { write_row(off, t, x); };
        // the operands this thread wrote go to the tensor cores
        auto handover = [&](int id) {
            fence_proxy_async_smem();
            t5::fence_before();
            nb_sync(id);
        };
        // an MMA group has completed (warp-uniform; false once anything failed)
        auto mma_done = [&](int bar, uint32_t parity) {
            bool ok = state_wait(bars + bar, parity, abort);
            ok = __all_sync(0xffffffffu, ok);
            if (ok) t5::fence_after();
            return ok;
        };

        write_s();
        handover(NB_S);
        for (int j = 0; j < nch; ++j) {
            const int tc = tc0 + j * DC;
            const uint32_t ph = j & 1;
            const float4* G = reinterpret_cast<const float4*>(base + L::G0 + ph * DC * 16);
            float4 gt = make_float4(0.f, 0.f, 0.f, 0.f);
            float dec = 0.f;
            if (!*abort && state_wait(bars + F_V, ph, abort)) {
                gt = G[tok];            // gates of this lane's token: gamma, e^gamma, b, e^{gamma_C - gamma}
                dec = G[DC - 1].y;      // e^{gamma_C}
            }

            // ---- R = diag(b) (V - diag(e^gamma) X), stored as R^T (X rows: lanes 64-127);
            // this lane's V columns are read before the product's wait
            uint4 vraw[2];
            if (xw) {
#pragma unroll
                for (int m = 0; m < 2; ++m) vraw[m] = *reinterpret_cast<const uint4*>(base + L::V0 + sw128_f16(tok, vc + 8 * m));
            }
            if (xw && mma_done(M_XY, ph)) {
                float x[16], x2[16];
                t5::ld16x2(tl + TM_XY + 32 * ph, x, tl + TM_XY2 + TM_XY + 32 * ph, x2);
#pragma unroll
                for (int v = 0; v < 16; ++v) x[v] += x2[v];
#pragma unroll
                for (int m = 0; m < 2; ++m) {
                    const uint32_t w4[4] = {vraw[m].x, vraw[m].y, vraw[m].z, vraw[m].w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 vv = __half22float2(*reinterpret_cast<const __half2*>(&w4[e]));
                        const int i = 8 * m + 2 * e;
                        x[i] = gt.z * (vv.x - gt.y * x[i]);
                        x[i + 1] = gt.z * (vv.y - gt.y * x[i + 1]);
                    }
                }
                write_col(L::R0, tok, x);
            }
            // V and this chunk's gate reads are done (every lane's values are in
            // registers): one arrival per compute warp
            __syncwarp();
            if (lane == 0) mbar_arrive_cta(bars + E_V);
            handover(NB_R);

            // ---- [Z; Delta] = [A T; T] R -> Delta~^T (Delta rows: lanes 64-127)
            if (xw && mma_done(M_DZ, ph)) {
                float dl[16];
                t5::ld16(tl + TM_DZ, dl);
#pragma unroll
                for (int v = 0; v < 16; ++v) dl[v] *= gt.w;
                write_col(L::E0, tok, dl);
            }
            handover(NB_D);

            // ---- S <- e^{gamma_C} S + U
            if (mma_done(M_U, ph)) {
                float u[16];
                t5::ld16(tl + TM_U, u);
#pragma unroll
                for (int v = 0; v < 16; ++v) S[v] = fmaf(dec, S[v], u[v]);
                write_s();
                // a snapshot of the state after a whole chunk that ends on a multiple of the interval
                const int done = a.ckpt.chunk_base + a.chunk0 + j + 1;
                if (a.ckpt.state && own_d && tc + DC <= t_end && done % a.ckpt.every_chunks == 0) {
                    float* cp = a.ckpt.state + static_cast<int64_t>(done / a.ckpt.every_chunks - 1) * a.hv * D * D;
#pragma unroll
                    for (int v = 0; v < 16; ++v) cp[(static_cast<int64_t>(h) * D + i0 + v0 + v) * D + d] = S[v];
                }
            }
            if (j + 1 < nch) handover(NB_S);

            // ---- O = diag(e^gamma) Y + Z (Y rows: lanes 0-63), while the next X, Y run;
            // written in fp16 (|o_i| <= max|S| |q|_1 <= 65504 for |q| <= d^-1/2; checked)
            if (!xw && mma_done(M_DZ, ph)) {
                float y[16], z[16];
                t5::ld16x2(tl + TM_XY + 32 * ph, y, tl + TM_DZ, z);
                {
                    float y2[16];
                    t5::ld16(tl + TM_XY2 + TM_XY + 32 * ph, y2);
#pragma unroll
                    for (int v = 0; v < 16; ++v) y[v] += y2[v];
                }
                const int t = tc + tok;
                if (t < t_end && GDN_IN_RANGE(g_delta_error, t < a.n && h * D + i0 + v0 + 16 <= a.c_v)) {
                    float ov[2][8];
#pragma unroll
                    for (int v = 0; v < 16; ++v) {
                        ov[v >> 3][v & 7] = fmaf(gt.y, y[v], z[v]);
                        bad |= f16_out_of_range(ov[v >> 3][v & 7]);
                    }
                    uint4* dst = reinterpret_cast<uint4*>(a.o + static_cast<int64_t>(t) * a.c_v + h * D + i0 + v0);
                    dst[0] = f16x8(ov[0]);
                    dst[1] = f16x8(ov[1]);
                }
            }
        }
        if (!*abort && own_d) {
#pragma unroll
            for (int v = 0; v < 16; ++v) st_out[(static_cast<int64_t>(h) * D + i0 + v0 + v) * D + d] = S[v];
        }
        if (bad) atomicCAS(&g_delta_error, 0, ERR_RANGE);
    }

    if (*abort && tid == 0) {
        // A wait ran out.  Copies already issued land in their own time; let them
        // finish (bounded) before the CTA's shared memory is released.
        for (int i = F_QK; i <= F_TA; ++i)
            for (uint32_t par = 0; par < 2; ++par) mbar_wait_bounded(bars + i, par, nullptr, 0, 20000000ull);
    }
    t5::fence_before();
    __syncthreads();
    if (warp == 9) {
        t5::fence_after();
        t5::dealloc(tmem, TM_COLS);
    }
}

// Scratch per chunk: [A T; T] (fp16) and the gate table per value head, K^T
// (fp16) per key head; every piece is a multiple of 1 KB.
size_t delta_scratch_bytes(int hv, int hk, int d, int64_t n) {
    const int64_t nch = (n + DC - 1) / DC;
    const int64_t per = static_cast<int64_t>(hv) * (2 * DC * DC * 2 + DC * 16) + static_cast<int64_t>(hk) * d * DC * 2;
    return static_cast<size_t>(nch * per);
}

static PFN_cuTensorMapEncodeTiled_v12000 delta_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        cudaDriverEntryPointQueryResult q;
        void* p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// fp16 qkv [n][c_conv]: boxes of DC tokens x 64 halfs, 128-byte swizzle, zero fill.
static bool make_qkv_map(CUtensorMap* map, const uint16_t* qkv, int64_t n, int c_conv) {
    auto enc = delta_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(c_conv), static_cast<cuuint64_t>(n)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(c_conv) * 2};
    cuuint32_t box[2] = {64, static_cast<cuuint32_t>(DC)};
    cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<uint16_t*>(qkv), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int read_and_clear_delta_error() {
    int v = 0, z = 0;
    cudaMemcpyFromSymbol(&v, g_delta_error, sizeof(int));
    if (v) cudaMemcpyToSymbol(g_delta_error, &z, sizeof(int));
    return v;
}

// Token segments of DELTA_SEG_CHUNKS chunks of every sequence (twice that
// in calls of at least 512 chunks, below).  With more
// than one, the prep of segment i+1 runs on the library's low-priority stream
// while the state pass of segment i runs on its high-priority one (the state
// is carried between segments in state_out, fp32, so the results are those of
// one launch).  Both are forked from the caller's stream and joined back to
// it.  Each launch covers all sequences (grid z); a CTA past the end of its
// sequence returns at once.
constexpr int DELTA_SEG_CHUNKS = 64;
template <int D>
static void launch_prep(const CUtensorMap& map, const DeltaArgs& a, const SeqTable& sq, cudaStream_t st) {
    delta_prep_kernel<D><<<dim3(a.nchunks, a.hv / a.ratio, sq.n), DELTA_THREADS, PrepSmem<D>::BYTES + 1024, st>>>(map, a, sq);
}
template <int D>
static void launch_state(const CUtensorMap& map, const DeltaArgs& a, const SeqTable& sq, cudaStream_t st) {
    delta_state_kernel<D><<<dim3(a.hv, D / NV, sq.n), STATE_THREADS, StateSmem<D>::BYTES + 1024, st>>>(map, a, sq);
}

// after_state (may be null): work on each segment's output tokens, enqueued on
// the low-priority stream once that segment's state pass is done (after all
// the preps, so it never delays one), so that it too runs beside the later
// state segments; without segments it runs on st after the state pass.  With
// several sequences a segment's tokens are not contiguous, and the hook runs
// once over all tokens after the last state segment.
// prep_only: the prep alone, one launch (the wait-expiry test).
template <int D>
static cudaError_t launch_delta_d(DeltaArgs& a, const SeqTable& sq, cudaStream_t st, bool overlap,
                                  const TokenRangeHook* after_state, bool prep_only) {
    static PerDeviceOnce attr_once;
    const int dev = attr_once.run([](int) {
        cudaFuncSetAttribute(delta_prep_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, PrepSmem<D>::BYTES + 1024);
        cudaFuncSetAttribute(delta_state_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, StateSmem<D>::BYTES + 1024);
        // the whole unified L1 as shared memory, so that a state CTA and a prep CTA fit on one SM
        cudaFuncSetAttribute(delta_prep_kernel<D>, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
        cudaFuncSetAttribute(delta_state_kernel<D>, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
    });
    if (dev < 0) return cudaErrorInvalidDevice;
    CUtensorMap map;
    if (!make_qkv_map(&map, a.qkv, a.n, a.c_conv)) return cudaErrorInvalidValue;
    int nch = 0;  // chunks of the longest sequence
    for (int i = 0; i < sq.n; ++i) nch = std::max(nch, sq.unit[i + 1] - sq.unit[i]);
    a.chunk0 = 0;
    a.nchunks = nch;
    if (nch == 0) return cudaSuccess;
    if (prep_only) {
        launch_prep<D>(map, a, sq, st);
        return cudaGetLastError();
    }
    if (!overlap || nch <= DELTA_SEG_CHUNKS) {
        launch_prep<D>(map, a, sq, st);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        launch_state<D>(map, a, sq, st);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        return after_state ? (*after_state)(0, a.n, st) : cudaSuccess;
    }
    const bool per_segment_hook = after_state && sq.n == 1;
    std::lock_guard<std::mutex> lock(lib_streams_mutex());
    LibStreams* ls = nullptr;
    cudaError_t e = lib_streams(&ls);
    if (e != cudaSuccess) return e;
    cudaStream_t prep_st = ls->lo, state_st = ls->hi;
    if ((e = cudaEventRecord(ls->ev_a, st)) != cudaSuccess) return e;
    if ((e = cudaStreamWaitEvent(prep_st, ls->ev_a, 0)) != cudaSuccess) return e;
    if ((e = cudaStreamWaitEvent(state_st, ls->ev_a, 0)) != cudaSuccess) return e;
    // Every segment boundary costs a state-pass launch, its start and its
    // drain, against the prep of the first segment, which nothing hides: calls
    // of at least 512 chunks take segments of twice the length (at 32768
    // tokens four of 128 chunks beat eight of 64 and two of 256).
    const int seg = nch >= 512 ? 2 * DELTA_SEG_CHUNKS : DELTA_SEG_CHUNKS;
    cudaError_t first = cudaSuccess;
    int nseg = 0;
    for (int c0 = 0; c0 < nch && first == cudaSuccess; c0 += seg) {
        DeltaArgs s = a;
        s.chunk0 = c0;
        s.nchunks = nch - c0 < seg ? nch - c0 : seg;
        // the second prep waits for the first to complete, so that the first
        // state segment (high priority) and it become ready together and the
        // state pass takes its SMs before the prep's CTAs fill them
        if (c0 == seg && (first = cudaStreamWaitEvent(prep_st, ls->ev_a, 0)) != cudaSuccess) break;
        launch_prep<D>(map, s, sq, prep_st);
        if ((first = cudaGetLastError()) != cudaSuccess) break;
        if ((first = cudaEventRecord(ls->ev_b, prep_st)) != cudaSuccess) break;
        if ((first = cudaStreamWaitEvent(state_st, ls->ev_b, 0)) != cudaSuccess) break;
        if (c0 == 0 && (first = cudaEventRecord(ls->ev_a, state_st)) != cudaSuccess) break;   // passed once prep 0 is done
        launch_state<D>(map, s, sq, state_st);
        if ((first = cudaGetLastError()) != cudaSuccess) break;
        if (per_segment_hook && nseg < LIB_EVENT_POOL) first = cudaEventRecord(ls->pool[nseg], state_st);
        ++nseg;
    }
    if (per_segment_hook && first == cudaSuccess) {
        // segments past the event pool wait for the last state segment
        if (nseg > LIB_EVENT_POOL) first = cudaEventRecord(ls->ev_a, state_st);
        for (int i = 0; i < nseg && first == cudaSuccess; ++i) {
            first = cudaStreamWaitEvent(prep_st, i < LIB_EVENT_POOL ? ls->pool[i] : ls->ev_a, 0);
            if (first != cudaSuccess) break;
            const int64_t tb = static_cast<int64_t>(i) * seg * DC;
            const int64_t te = std::min<int64_t>(a.n, tb + static_cast<int64_t>(seg) * DC);
            first = (*after_state)(tb, te, prep_st);
        }
    }
    // join both library streams back to the caller's stream, also after a failure
    e = cudaEventRecord(ls->ev_b, prep_st);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(state_st, ls->ev_b, 0);
    if (e == cudaSuccess) e = cudaEventRecord(ls->ev_a, state_st);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(st, ls->ev_a, 0);
    if (first == cudaSuccess && e == cudaSuccess && after_state && !per_segment_hook) first = (*after_state)(0, a.n, st);
    return first != cudaSuccess ? first : e;
}

cudaError_t launch_delta(const gdn_layer& L, const uint16_t* qkv, const float* log_a, const float* b, int64_t n,
                         const float* state_in, float* state_out, uint16_t* o, void* scratch, cudaStream_t st,
                         bool overlap, const TokenRangeHook* after_state, const int64_t* cu_seqlens, int n_seqs,
                         const DeltaCkpt* ckpt, const DeltaFault* fault) {
    DeltaArgs a;
    const int d = L.dk;
    // the call's sequences (host token offsets; null: one sequence of n tokens),
    // each chunked from its first token; the states are [n_seqs][hv][D][D]
    const SeqTable sq = cu_seqlens ? make_seq_table(cu_seqlens, n_seqs, DC) : one_seq_table(n, DC);
    a.qkv = qkv;
    a.log_a = log_a;
    a.b = b;
    a.n = static_cast<int>(n);
    a.hv = L.n_v_heads;
    a.ratio = L.n_v_heads / L.n_qk_heads;
    a.c_qk = L.n_qk_heads * d;
    a.c_v = L.n_v_heads * d;
    a.c_conv = 2 * a.c_qk + a.c_v;
    a.chunk0 = 0;
    a.nchunks = 0;
    const int64_t nch = sq.unit[sq.n];   // chunks of all sequences: the scratch tables' extent
    a.nch_total = static_cast<int>(nch);
    unsigned char* base = static_cast<unsigned char*>(scratch);
    a.TA = reinterpret_cast<uint16_t*>(base);
    a.G = reinterpret_cast<float*>(base + nch * a.hv * 2 * DC * DC * 2);
    a.KT = reinterpret_cast<uint16_t*>(base + nch * a.hv * (2 * DC * DC * 2 + DC * 16));
    a.state_in = state_in;
    a.state_out = state_out;
    a.o = o;
    a.ckpt = ckpt && !cu_seqlens ? *ckpt : DeltaCkpt{nullptr, 1, 0};
    a.prep_wait_ns = fault ? fault->wait_ns : 2000000000ull;
    a.prep_no_copy = fault ? 1 : 0;
    const bool prep_only = fault != nullptr;
    return d == 128 ? launch_delta_d<128>(a, sq, st, overlap, after_state, prep_only)
                    : launch_delta_d<64>(a, sq, st, overlap, after_state, prep_only);
}

}  // namespace gdn
