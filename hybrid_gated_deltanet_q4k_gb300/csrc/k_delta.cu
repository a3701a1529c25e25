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
// Two kernels:
//   delta_prep   one CTA per (chunk, key head), all chunks in parallel: K K^T
//                and Q K^T once on tensor cores, then per value head gamma,
//                the masked A, and T by
//                blocked inversion of the unit lower-triangular I + L (16x16
//                diagonal blocks by substitution, off-diagonal blocks by
//                block products).  Writes T and A (tf32-rounded) and a gate
//                table (gamma, e^gamma, b, e^{gamma_C - gamma}) per token:
//                33 KB per (chunk, head).
//   delta_state  one CTA per (head, 32 rows of S): the chunks in order.  Rows
//                of S evolve independently (row i only reads v[i]), so the
//                rows split across CTAs with no communication.  The fp32 state
//                stays in registers as the accumulator fragments of the
//                update product.  Every operand of chunk c+1 is copied into
//                shared memory by TMA (issued by a producer warp, completion
//                on mbarriers) while chunk c computes: each copy is issued
//                right after the operand's last use in chunk c (K and Q, used
//                in the first phase, are double-buffered).  K, Q, V arrive as 2-D
//                boxes of 64 tokens x 32 floats with the 128-byte swizzle; T
//                and A are written by delta_prep in that same swizzled image,
//                so a 1-D bulk copy lands them ready.
// Products use mma.sync m16n8k8 with tf32 operands rounded to nearest (the
// conv writes q, k, v already rounded; T, A, S, R, Delta are rounded where
// they are produced) and fp32 accumulation; everything else is fp32.
// Rounding every operand to tf32 keeps o and S within ~5e-4 (relative L2) of
// the exact recurrence on the test workloads.
#include "common.cuh"
#include "tma.cuh"
#include "tcgen05.cuh"

#include <mutex>

namespace gdn {

static __device__ int g_delta_error;

constexpr int DC = GDN_CHUNK;  // 64
constexpr int DELTA_THREADS = 256;            // prep; compute warps of the state pass
constexpr int STATE_THREADS = DELTA_THREADS + 64;  // + TMA producer warp + MMA warp
constexpr int NV = 32;         // rows of S per state CTA

struct DeltaArgs {
    const float* qkv;     // [n][c_conv] fp32: q | k | v
    const float* log_a;   // [n][hv]
    const float* b;       // [n][hv]
    int n, hv, ratio, c_qk, c_conv, c_v;
    int nchunks;
    float* T;      // [nchunks][hv][DC][DC]   tf32-rounded
    float* A;      // [nchunks][hv][DC][DC]   tf32-rounded
    float* G;      // [nchunks][hv][DC][4]    gamma, e^gamma, b, e^{gamma_C - gamma}
    float* KT;     // [nchunks][hk][D][DC]    K^T, in the swizzled operand image
    const float* state_in;  // [hv][D][D] or null
    float* state_out;
    float* o;      // [n][c_v]
};

__device__ __forceinline__ uint32_t to_tf32(float x) { return tf32_bits(x); }
__device__ __forceinline__ float tf32f(float x) { return round_tf32(x); }

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, bool valid) {
    const uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(s), "l"(gmem), "r"(valid ? 16 : 0) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// D += A(16x8, row) * B(8x8, col); fragments as in the PTX m16n8k8 .tf32 layout:
// a0 (g, t) a1 (g+8, t) a2 (g, t+4) a3 (g+8, t+4); b0 (k=t, n=g) b1 (k=t+4, n=g);
// c0 (g, 2t) c1 (g, 2t+1) c2 (g+8, 2t) c3 (g+8, 2t+1), g = lane/4, t = lane%4.
__device__ __forceinline__ void mma_tf32(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t lds_u32(const float* p) { return __float_as_uint(*p); }

// ldmatrix on fp32 data: an 8x4 block of fp32 is an 8x8 block of b16 pairs, and
// the b16 fragment of thread l (row l/4, elements 2(l%4), 2(l%4)+1) is exactly
// fp32 element (l/4, l%4) -- the tf32 m16n8k8 fragment position.  Lane l passes
// the address of row l%8 of matrix l/8.
__device__ __forceinline__ void ldsm_x4(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3, const float* p) {
    const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(p));
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(a));
}
// A fragment (16x8 tile at row0, col0 of a row-major [m][k] array with pitch P).
template <int P>
__device__ __forceinline__ const float* a_frag_addr(const float* base, int row0, int col0, int lane) {
    const int mat = lane >> 3, r = lane & 7;
    return base + (row0 + r + 8 * (mat & 1)) * P + col0 + 4 * (mat >> 1);
}
// Two B fragments (n-tiles n0 and n0+8, k-block col0) of an [n][k] array with pitch P.
template <int P>
__device__ __forceinline__ const float* b2_frag_addr(const float* base, int n0, int col0, int lane) {
    const int mat = lane >> 3, r = lane & 7;
    return base + (n0 + r + 8 * (mat >> 1)) * P + col0 + 4 * (mat & 1);
}

// Float index of element (r, c) of a [DC][DC] matrix stored as the shared-memory
// image the state pass reads: two slabs of DC rows x 32 floats (c / 32), each
// with 128-byte rows and the 128-byte swizzle.
__device__ __forceinline__ int swz64(int r, int c) {
    return (c >> 5) * (DC * 32) + static_cast<int>(sw128_f32(r, c & 31) >> 2);
}

// ------------------------------------------------------------------ prep

constexpr int PREP_MAX_RATIO = 8;  // value heads per key head handled by one CTA

template <int D>
struct PrepSmem {
    static constexpr int P = D + 4;    // K, Q row pitch (floats)
    static constexpr int PL = DC + 4;  // KK, QK, L, T row pitch (floats)
    static constexpr int K0 = 0;                      // Ks[DC][P]   (later: Ls, Ts)
    static constexpr int Q0 = K0 + DC * P;            // Qs[DC][P]
    static constexpr int L0 = K0;                     // Ls[DC][PL]  aliases Ks after the products
    static constexpr int T0 = L0 + DC * PL;           // Ts[DC][PL]
    static constexpr int KK0 = Q0 + DC * P;           // KK[DC][PL]  k_i . k_j (lower triangle)
    static constexpr int QK0 = KK0 + DC * PL;         // QK[DC][PL]  q_i . k_j (lower triangle)
    static constexpr int Z0 = QK0 + DC * PL;          // Zs[3][256]
    static constexpr int GL0 = Z0 + 3 * 256;          // gamma[PREP_MAX_RATIO][DC]
    static constexpr int BB0 = GL0 + PREP_MAX_RATIO * DC;  // b[PREP_MAX_RATIO][DC]
    static constexpr int FLOATS = BB0 + PREP_MAX_RATIO * DC;
    static_assert(2 * DC * PL <= 2 * DC * P, "L and T must fit in the K and Q region");
};

// One CTA per (chunk, key head): K K^T and Q K^T once (the value heads of a key
// head share them), then for each of its value heads the gated L, T = (I+L)^-1,
// the masked A and the gate table.
template <int D>
__global__ void __launch_bounds__(DELTA_THREADS, 2) delta_prep_kernel(DeltaArgs a) {
    using L = PrepSmem<D>;
    constexpr int P = L::P, PL = L::PL;
    extern __shared__ __align__(16) float sm[];
    float* Ks = sm + L::K0;
    float* Qs = sm + L::Q0;
    float* Ls = sm + L::L0;
    float* Ts = sm + L::T0;
    float* KK = sm + L::KK0;
    float* QK = sm + L::QK0;
    float* Zs = sm + L::Z0;

    const int chunk = blockIdx.x, hk = blockIdx.y;
    const int t0 = chunk * DC;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, tg = lane & 3;
    const int r = a.ratio;

    // K and Q rows (tf32 values from the conv) by asynchronous copies; rows past n are zero.
    for (int idx = tid; idx < 2 * DC * (D / 4); idx += DELTA_THREADS) {
        const int which = idx / (DC * (D / 4)), rem = idx % (DC * (D / 4));
        const int row = rem / (D / 4), c4 = rem % (D / 4), t = t0 + row;
        const bool ok = t < a.n;
        const int col = (which == 0 ? a.c_qk : 0) + hk * D + 4 * c4;
        const float* src = ok ? a.qkv + static_cast<int64_t>(t) * a.c_conv + col : a.qkv;
        cp_async16((which == 0 ? Ks : Qs) + row * P + 4 * c4, src, ok);
    }
    cp_async_commit();
    // gates of the value heads h = hk*r + j: log a -> inclusive prefix sum (one warp per head)
    for (int j = warp; j < r; j += DELTA_THREADS / 32) {
        const int h = hk * r + j;
        float* gl = sm + L::GL0 + j * DC;
        float* bb = sm + L::BB0 + j * DC;
        float x0 = 0.f, x1 = 0.f;
        const int ta = t0 + 2 * lane, tb = ta + 1;
        if (ta < a.n) x0 = a.log_a[static_cast<int64_t>(ta) * a.hv + h];
        if (tb < a.n) x1 = a.log_a[static_cast<int64_t>(tb) * a.hv + h];
        bb[2 * lane] = ta < a.n ? a.b[static_cast<int64_t>(ta) * a.hv + h] : 0.f;
        bb[2 * lane + 1] = tb < a.n ? a.b[static_cast<int64_t>(tb) * a.hv + h] : 0.f;
        float s = x0 + x1;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float y = __shfl_up_sync(0xffffffffu, s, o);
            if (lane >= o) s += y;
        }
        gl[2 * lane] = s - x1;
        gl[2 * lane + 1] = s;
    }
    cp_async_wait<0>();
    __syncthreads();

    // K K^T and Q K^T on the lower-triangular 16x8 tiles: warp -> m-tile warp/2,
    // n-tiles 4*(warp%2) .. +3 (skipping tiles wholly above the diagonal).
    {
        const int mt = warp >> 1, nt0 = 4 * (warp & 1);
        float ck[4][4] = {}, cq[4][4] = {};
        const float* ka = a_frag_addr<P>(Ks, 16 * mt, 0, lane);
        const float* qa = a_frag_addr<P>(Qs, 16 * mt, 0, lane);
        const float* kb0 = b2_frag_addr<P>(Ks, 8 * nt0, 0, lane);
        const float* kb1 = b2_frag_addr<P>(Ks, 8 * nt0 + 16, 0, lane);
        const bool live01 = 8 * nt0 <= 16 * mt + 15, live23 = 8 * (nt0 + 2) <= 16 * mt + 15;
#pragma unroll 4
        for (int ks = 0; ks < D / 8; ++ks) {
            const int c = 8 * ks;
            uint32_t k0, k1, k2, k3, q0, q1, q2, q3, b0, b1, b2, b3;
            ldsm_x4(k0, k1, k2, k3, ka + c);
            ldsm_x4(q0, q1, q2, q3, qa + c);
            if (live01) {
                ldsm_x4(b0, b1, b2, b3, kb0 + c);
                mma_tf32(ck[0], k0, k1, k2, k3, b0, b1);
                mma_tf32(cq[0], q0, q1, q2, q3, b0, b1);
                mma_tf32(ck[1], k0, k1, k2, k3, b2, b3);
                mma_tf32(cq[1], q0, q1, q2, q3, b2, b3);
            }
            if (live23) {
                ldsm_x4(b0, b1, b2, b3, kb1 + c);
                mma_tf32(ck[2], k0, k1, k2, k3, b0, b1);
                mma_tf32(cq[2], q0, q1, q2, q3, b0, b1);
                mma_tf32(ck[3], k0, k1, k2, k3, b2, b3);
                mma_tf32(cq[3], q0, q1, q2, q3, b2, b3);
            }
        }
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int i = 16 * mt + g + (e >> 1) * 8, jj = 8 * (nt0 + j) + 2 * tg + (e & 1);
                KK[i * PL + jj] = ck[j][e];
                QK[i * PL + jj] = cq[j][e];
            }
    }
    // K^T of this (chunk, key head) for the state pass's update product, in its
    // shared-memory operand image: two slabs (tokens 0-31, 32-63) of D rows of
    // 32 floats with the 128-byte swizzle.  Lanes take consecutive d, so the
    // column reads of Ks are conflict-free.
    {
        float* kt = a.KT + (static_cast<int64_t>(chunk) * gridDim.y + hk) * D * DC;
        for (int idx = tid; idx < D * (DC / 4); idx += DELTA_THREADS) {
            const int d = idx % D, t = 4 * (idx / D);
            const float4 v = make_float4(Ks[t * P + d], Ks[(t + 1) * P + d], Ks[(t + 2) * P + d], Ks[(t + 3) * P + d]);
            *reinterpret_cast<float4*>(kt + (t >> 5) * (D * 32) + (sw128_f32(d, t & 31) >> 2)) = v;
        }
    }
    __syncthreads();   // K and Q are no longer needed: L and T reuse their space

    for (int j = 0; j < r; ++j) {
        const int h = hk * r + j;
        const int64_t cb = static_cast<int64_t>(chunk) * a.hv + h;
        const float* gl = sm + L::GL0 + j * DC;
        const float* bb = sm + L::BB0 + j * DC;
        float* aout = a.A + cb * DC * DC;
        for (int idx = tid; idx < DC * DC; idx += DELTA_THREADS) {
            const int i = idx / DC, jj = idx % DC;
            const float dec = jj <= i ? expf(gl[i] - gl[jj]) : 0.f;
            Ls[i * PL + jj] = jj < i ? bb[i] * dec * KK[i * PL + jj] : 0.f;
            Ts[i * PL + jj] = 0.f;
            aout[swz64(i, jj)] = tf32f(dec * QK[i * PL + jj]);
        }
        __syncthreads();
        // T = (I + L)^{-1}: diagonal 16x16 blocks by substitution, one column per thread.
        if (tid < 64) {
            const int blk = tid >> 4, c = tid & 15, o = 16 * blk;
            float col[16];
#pragma unroll
            for (int rr = 0; rr < 16; ++rr) {
                float v;
                if (rr < c) {
                    v = 0.f;
                } else if (rr == c) {
                    v = 1.f;
                } else {
                    float s = 0.f;
#pragma unroll
                    for (int k = 0; k < rr; ++k)
                        if (k >= c) s = fmaf(Ls[(o + rr) * PL + o + k], col[k], s);
                    v = -s;
                }
                col[rr] = v;
            }
#pragma unroll
            for (int rr = 0; rr < 16; ++rr) Ts[(o + rr) * PL + o + c] = col[rr];
        }
        __syncthreads();
        // Off-diagonal blocks, block row by block row:
        //   T_IJ = -T_II * sum_{K=J}^{I-1} L_IK T_KJ   (J < I)
        for (int I = 1; I < 4; ++I) {
            for (int e = tid; e < I * 256; e += DELTA_THREADS) {
                const int J = e >> 8, rr = (e >> 4) & 15, c = e & 15;
                float z = 0.f;
                for (int K = J; K < I; ++K)
#pragma unroll
                    for (int m = 0; m < 16; ++m)
                        z = fmaf(Ls[(16 * I + rr) * PL + 16 * K + m], Ts[(16 * K + m) * PL + 16 * J + c], z);
                Zs[J * 256 + rr * 16 + c] = z;
            }
            __syncthreads();
            for (int e = tid; e < I * 256; e += DELTA_THREADS) {
                const int J = e >> 8, rr = (e >> 4) & 15, c = e & 15;
                float s = 0.f;
#pragma unroll
                for (int m = 0; m < 16; ++m) s = fmaf(Ts[(16 * I + rr) * PL + 16 * I + m], Zs[J * 256 + m * 16 + c], s);
                Ts[(16 * I + rr) * PL + 16 * J + c] = -s;
            }
            __syncthreads();
        }
        float* tout = a.T + cb * DC * DC;
        for (int idx = tid; idx < DC * DC; idx += DELTA_THREADS) {
            const int rr = idx / DC, c = idx % DC;
            tout[swz64(rr, c)] = tf32f(Ts[rr * PL + c]);
        }
        if (tid < DC) {
            const float gv = gl[tid];
            *reinterpret_cast<float4*>(a.G + (cb * DC + tid) * 4) = make_float4(gv, expf(gv), bb[tid], expf(gl[DC - 1] - gv));
        }
        __syncthreads();   // before the next head overwrites L and T
    }
}

// ------------------------------------------------------------------ state pass

// Shared-memory layout of the state pass (byte offsets; every operand base is
// 1024-byte aligned, as the 128-byte swizzle requires).  Operands are slabs of
// rows of 32 fp32 (128 bytes) with the 128-byte swizzle, K-major for the
// tensor cores: the image a 2-D TMA box with SWIZZLE_128B writes, and the one
// delta_prep writes for T, A and K^T.
template <int D>
struct StateSmem {
    static constexpr int SLAB = DC * 128;          // 64 rows x 32 floats
    static constexpr int NSLAB = D / 32;
    static constexpr int QK_SLAB = 2 * SLAB;       // Q rows 0-63, K rows 64-127
    static constexpr int SOP = NV * 128;           // 32 rows x 32 floats
    static constexpr int KT_SLAB = D * 128;        // D rows x 32 floats
    static constexpr int KT_BYTES = 2 * KT_SLAB;   // one K^T [D][DC]
    static constexpr int QK0 = 0;                  // [Q; K] [2*DC][D]  (TMA)
    static constexpr int KT0 = QK0 + NSLAB * QK_SLAB;   // K^T [2][D][DC] (bulk copies)
    static constexpr int T0 = KT0 + 2 * KT_BYTES;  // T [DC][DC]        (bulk copy)
    static constexpr int A0 = T0 + 2 * SLAB;       // [A; 0] [2*DC][DC] (bulk copies into the upper rows)
    static constexpr int V0 = A0 + 2 * QK_SLAB;    // V [DC][NV]        (TMA)
    static constexpr int S0 = V0 + SLAB;           // S [NV][D]         tf32 operand of X, Y
    static constexpr int R0 = S0 + NSLAB * SOP;    // R^T, then Delta^T [NV][DC]
    static constexpr int E0 = R0 + 2 * SOP;        // Delta~^T [NV][DC]
    static constexpr int G0 = E0 + 2 * SOP;        // gate table [2][DC] x (gamma, e^gamma, b, e^{gamma_C-gamma})
    static constexpr int B0 = G0 + 2 * DC * 16;    // mbarriers
    static constexpr int NBAR = 17;
    static constexpr int MISC0 = B0 + NBAR * 8;    // TMEM base address, abort flag
    static constexpr int BYTES = MISC0 + 16;
    static_assert(BYTES + 1024 <= 227 * 1024, "state pass shared memory");
};

// TMEM columns (fp32 accumulators of NV = 32 columns).  [Q; K] S^T is
// double-buffered: the output reads Y of chunk c while X, Y of chunk c+1 run.
constexpr uint32_t TM_XY = 0, TM_D = 64, TM_U = 96, TM_Z = 128;
constexpr uint32_t TM_COLS = 256;

enum StateBar : int {
    F_QK, F_KT0, F_KT1, F_V, F_T, F_A,   // copies landed (tx bytes)
    E_QK, E_KT0, E_KT1, E_V, E_T, E_A,   // buffer free again
    M_XY, M_D, M_U, M_Z,                 // MMA groups complete (tcgen05.commit)
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

// Issue the k steps [0, NK) of one MMA chain; a K step is 8 fp32 = 32 bytes,
// four per 128-byte swizzle row, then the next slab.
template <int NK, int A_SLAB, int B_SLAB>
__device__ __forceinline__ void mma_chain(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc) {
#pragma unroll
    for (int k = 0; k < NK; ++k)
        t5::mma_tf32(d_tmem, adesc + static_cast<uint64_t>((k >> 2) * (A_SLAB >> 4) + 2 * (k & 3)),
                     bdesc + static_cast<uint64_t>((k >> 2) * (B_SLAB >> 4) + 2 * (k & 3)), idesc, k > 0 ? 1u : 0u);
}

// One CTA per (value head, NV rows of S); 320 threads:
//   warps 0-7  compute.  Warp w reads TMEM lanes 32*(w%4) .. +31 and columns
//              16*(w/4) .. +15 of each 32-column accumulator.
//   warp 8     producer: TMA boxes of Q, K, V; bulk copies of K^T, T, A, gates.
//   warp 9     TMEM owner and MMA issuer: meets the compute warps at a named
//              barrier once they have written an operand, then issues (one
//              thread).
// Per chunk, with S the NV x D slice of the state (tf32 operands, fp32 sums):
//   MMA  [Y; X] = [Q; K] S^T          (M = 128: Y in lanes 0-63, X in 64-127)
//   warps 2,3,6,7 (lanes 64-127)  R = diag(b)(V - diag(e^gamma) X) -> R^T
//   MMA  Delta = T R                  (M = 64: row j in lane 32*(j/16) + j%16)
//   lanes 0-15  Delta^T and Delta~^T = (diag(e^{gamma_C-gamma}) Delta)^T
//   MMA  U = K^T Delta~               (M = D: row d in lane d, or 32*(d/16)+d%16)
//   MMA  [Z; 0] = [A; 0] Delta        (M = 128: Z in lanes 0-63, next to Y)
//   warps  S <- e^{gamma_C} S + U in fp32 registers, its tf32 image -> S
//   MMA  next chunk's [Q; K] S^T
//   warps 0,1,4,5 (lanes 0-63)  O = diag(e^gamma) Y + Z, while it runs.
// The state's chain per chunk is four dependent steps (X, R, Delta, U); the
// output products stay off it.  Every thread meets every named barrier of
// every chunk, also after a wait ran out (it then skips the work, and the MMA
// warp issues nothing more), so no barrier is ever left waiting.
template <int D>
__global__ void __launch_bounds__(STATE_THREADS, 1)
delta_state_kernel(const __grid_constant__ CUtensorMap qkv_map, DeltaArgs a) {
    using L = StateSmem<D>;
    extern __shared__ __align__(1024) unsigned char smb[];
    unsigned char* base = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smb) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(base + L::B0);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(base + L::MISC0);
    volatile int* abort = reinterpret_cast<volatile int*>(base + L::MISC0 + 4);

    const int h = blockIdx.x, i0 = blockIdx.y * NV, hk = h / a.ratio;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t sbase = smem_addr(base);

    if (tid == 0) {
        for (int i = F_QK; i <= F_A; ++i) mbar_init_cta(bars + i, 1);
        for (int i = E_QK; i <= E_A; ++i) mbar_init_cta(bars + i, 1);
        mbar_init_cta(bars + E_V, DELTA_THREADS);
        for (int i = M_XY; i <= M_FIN; ++i) mbar_init_cta(bars + i, 1);
        mbar_init_fence();
        *abort = 0;
    }
    // the zero rows 64-127 of the [A; 0] operand
    for (int idx = tid; idx < 2 * L::SLAB / 16; idx += STATE_THREADS) {
        const int sl = idx / (L::SLAB / 16), off = idx % (L::SLAB / 16);
        *reinterpret_cast<uint4*>(base + L::A0 + sl * L::QK_SLAB + L::SLAB + 16 * off) = make_uint4(0u, 0u, 0u, 0u);
    }
    fence_proxy_async_smem();
    if (warp == 9) t5::alloc(tslot, TM_COLS);
    t5::fence_before();
    __syncthreads();
    t5::fence_after();
    const uint32_t tmem = *tslot;

    if (warp == 8) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            auto cb = [&](int c) { return static_cast<int64_t>(c) * a.hv + h; };
            for (int c = 0; c < a.nchunks; ++c) {
                const uint32_t pp = (c - 1) & 1;   // phase of the previous chunk's release
                if (c >= 1 && !state_wait(bars + E_QK, pp, abort)) break;
                mbar_expect_tx(bars + F_QK, 2 * L::NSLAB * L::SLAB);
                for (int sl = 0; sl < L::NSLAB; ++sl) {
                    unsigned char* dst = base + L::QK0 + sl * L::QK_SLAB;
                    tma_load_2d_tile(dst, &qkv_map, bars + F_QK, hk * D + 32 * sl, c * DC);
                    tma_load_2d_tile(dst + L::SLAB, &qkv_map, bars + F_QK, a.c_qk + hk * D + 32 * sl, c * DC);
                }
                const int kb = c & 1;
                if (c >= 2 && !state_wait(bars + E_KT0 + kb, ((c - 2) >> 1) & 1, abort)) break;
                mbar_expect_tx(bars + F_KT0 + kb, L::KT_BYTES);
                bulk_load_1d(base + L::KT0 + kb * L::KT_BYTES,
                             a.KT + (static_cast<int64_t>(c) * (a.hv / a.ratio) + hk) * D * DC, L::KT_BYTES,
                             bars + F_KT0 + kb);
                if (c >= 1 && !state_wait(bars + E_V, pp, abort)) break;
                mbar_expect_tx(bars + F_V, L::SLAB + DC * 16);
                tma_load_2d_tile(base + L::V0, &qkv_map, bars + F_V, 2 * a.c_qk + h * D + i0, c * DC);
                bulk_load_1d(base + L::G0 + (c & 1) * DC * 16, a.G + cb(c) * DC * 4, DC * 16, bars + F_V);
                if (c >= 1 && !state_wait(bars + E_T, pp, abort)) break;
                mbar_expect_tx(bars + F_T, 2 * L::SLAB);
                bulk_load_1d(base + L::T0, a.T + cb(c) * DC * DC, 2 * L::SLAB, bars + F_T);
                if (c >= 1 && !state_wait(bars + E_A, pp, abort)) break;
                mbar_expect_tx(bars + F_A, 2 * L::SLAB);
                for (int sl = 0; sl < 2; ++sl)
                    bulk_load_1d(base + L::A0 + sl * L::QK_SLAB, a.A + cb(c) * DC * DC + sl * (DC * 32), L::SLAB,
                                 bars + F_A);
            }
        }
    } else if (warp == 9) {
        // ------------------------------------------------------------ MMA issuer
        constexpr uint32_t ID64 = t5::idesc_tf32(64, NV);
        constexpr uint32_t ID128 = t5::idesc_tf32(128, NV);
        constexpr uint32_t IDU = t5::idesc_tf32(D, NV);
        const uint64_t dQK = t5::desc_sw128(sbase + L::QK0), dS = t5::desc_sw128(sbase + L::S0);
        const uint64_t dT = t5::desc_sw128(sbase + L::T0), dR = t5::desc_sw128(sbase + L::R0);
        const uint64_t dA = t5::desc_sw128(sbase + L::A0), dE = t5::desc_sw128(sbase + L::E0);
        const uint64_t dKT = t5::desc_sw128(sbase + L::KT0);
        const bool leader = lane == 0;
        // leader only: the copy has landed and nothing has failed
        auto ready = [&](int bar, uint32_t parity) {
            if (*abort || !state_wait(bars + bar, parity, abort)) return false;
            t5::fence_after();
            return true;
        };
        for (int c = 0; c < a.nchunks; ++c) {
            const uint32_t ph = c & 1;
            nb_sync(NB_S);                      // S of chunk c written
            if (leader && ready(F_QK, ph)) {
                mma_chain<D / 8, L::QK_SLAB, L::SOP>(tmem + TM_XY + 32 * ph, dQK, dS, ID128);
                t5::commit(bars + M_XY);
                t5::commit(bars + E_QK);
            }
            __syncwarp();
            nb_sync(NB_R);                      // R^T written
            if (leader && ready(F_T, ph)) {
                mma_chain<DC / 8, L::SLAB, L::SOP>(tmem + TM_D, dT, dR, ID64);
                t5::commit(bars + M_D);
                t5::commit(bars + E_T);
            }
            __syncwarp();
            nb_sync(NB_D);                      // Delta^T, Delta~^T written
            if (leader && ready(F_KT0 + ph, (c >> 1) & 1)) {
                mma_chain<DC / 8, L::KT_SLAB, L::SOP>(tmem + TM_U, dKT + ph * (L::KT_BYTES >> 4), dE, IDU);
                t5::commit(bars + M_U);
                t5::commit(bars + E_KT0 + ph);
                if (ready(F_A, ph)) {
                    mma_chain<DC / 8, L::QK_SLAB, L::SOP>(tmem + TM_Z, dA, dR, ID128);
                    t5::commit(bars + M_Z);
                    t5::commit(bars + E_A);
                }
            }
            __syncwarp();
        }
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
        const bool act = lane < 16;             // owns token j = 16q + lane of the M = 64 product
        const int j = 16 * q + lane;
        const uint32_t tl = tmem + (static_cast<uint32_t>(32 * q) << 16) + v0;   // this warp's lanes, columns v0..
        // key-dimension row d of U owned by this thread (all lanes for D = 128, lanes 0-15 for D = 64)
        const bool own_d = D == 128 ? true : act;
        const int d = D == 128 ? 32 * q + lane : 16 * q + lane;

        float S[16];
#pragma unroll
        for (int v = 0; v < 16; ++v)
            S[v] = (own_d && a.state_in) ? a.state_in[(static_cast<int64_t>(h) * D + i0 + v0 + v) * D + d] : 0.f;
        auto write_s = [&]() {
            if (own_d) {
                unsigned char* sp = base + L::S0 + (d >> 5) * L::SOP;
#pragma unroll
                for (int v = 0; v < 16; ++v)
                    *reinterpret_cast<float*>(sp + sw128_f32(v0 + v, d & 31)) = tf32f(S[v]);
            }
        };
        // column t of an [NV][DC] operand (R^T, Delta^T, Delta~^T), rows v0 .. v0+15
        auto write_col = [&](int off, int t, const float (&x)[16]) {
            unsigned char* cp = base + off + (t >> 5) * L::SOP;
#pragma unroll
            for (int v = 0; v < 16; ++v) *reinterpret_cast<float*>(cp + sw128_f32(v0 + v, t & 31)) = x[v];
        };
        // the operands this thread wrote go to the tensor cores
        auto handover = [&](int id) {
            fence_proxy_async_smem();
            t5::fence_before();
            nb_sync(id);
        };
        // an MMA group has completed (warp-uniform; false once anything failed)
        auto mma_done = [&](int bar, uint32_t parity) {
            bool ok = !*abort && state_wait(bars + bar, parity, abort);
            ok = __all_sync(0xffffffffu, ok);
            if (ok) t5::fence_after();
            return ok;
        };

        write_s();
        handover(NB_S);
        for (int c = 0; c < a.nchunks; ++c) {
            const uint32_t ph = c & 1;
            const float4* G = reinterpret_cast<const float4*>(base + L::G0 + ph * DC * 16);
            float4 gt = make_float4(0.f, 0.f, 0.f, 0.f);
            float sc = 0.f, dec = 0.f;
            if (!*abort && state_wait(bars + F_V, ph, abort)) {
                gt = G[tok];            // gates of this lane's token (M = 128 products)
                sc = G[j].w;            // e^{gamma_C - gamma_j}
                dec = G[DC - 1].y;      // e^{gamma_C}
            }

            // ---- R = diag(b) (V - diag(e^gamma) X), stored as R^T (X rows: lanes 64-127)
            if (xw && mma_done(M_XY, ph)) {
                float x[16];
                t5::ld16(tl + TM_XY + 32 * ph, x);
                const unsigned char* vp = base + L::V0;
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const float4 vv = *reinterpret_cast<const float4*>(vp + sw128_f32(tok, v0 + 4 * m));
                    x[4 * m + 0] = tf32f(gt.z * (vv.x - gt.y * x[4 * m + 0]));
                    x[4 * m + 1] = tf32f(gt.z * (vv.y - gt.y * x[4 * m + 1]));
                    x[4 * m + 2] = tf32f(gt.z * (vv.z - gt.y * x[4 * m + 2]));
                    x[4 * m + 3] = tf32f(gt.z * (vv.w - gt.y * x[4 * m + 3]));
                }
                write_col(L::R0, tok, x);
            }
            mbar_arrive_cta(bars + E_V);         // V and this chunk's gate reads are done
            handover(NB_R);

            // ---- Delta = T R -> Delta^T (over R^T) and Delta~^T
            if (mma_done(M_D, ph)) {
                float dl[16];
                t5::ld16(tl + TM_D, dl);
                if (act) {
                    float de[16];
#pragma unroll
                    for (int v = 0; v < 16; ++v) {
                        de[v] = tf32f(dl[v] * sc);
                        dl[v] = tf32f(dl[v]);
                    }
                    write_col(L::R0, j, dl);
                    write_col(L::E0, j, de);
                }
            }
            handover(NB_D);

            // ---- S <- e^{gamma_C} S + U
            if (mma_done(M_U, ph)) {
                float u[16];
                t5::ld16(tl + TM_U, u);
#pragma unroll
                for (int v = 0; v < 16; ++v) S[v] = fmaf(dec, S[v], u[v]);
                write_s();
            }
            if (c + 1 < a.nchunks) handover(NB_S);

            // ---- O = diag(e^gamma) Y + Z (Y rows: lanes 0-63), while the next X, Y run
            if (!xw && mma_done(M_Z, ph)) {
                float y[16], z[16];
                t5::ld16x2(tl + TM_XY + 32 * ph, y, tl + TM_Z, z);
                const int t = c * DC + tok;
                if (t < a.n) {
                    float4* dst = reinterpret_cast<float4*>(a.o + static_cast<int64_t>(t) * a.c_v + h * D + i0 + v0);
#pragma unroll
                    for (int m = 0; m < 4; ++m)
                        dst[m] = make_float4(fmaf(gt.y, y[4 * m], z[4 * m]), fmaf(gt.y, y[4 * m + 1], z[4 * m + 1]),
                                             fmaf(gt.y, y[4 * m + 2], z[4 * m + 2]),
                                             fmaf(gt.y, y[4 * m + 3], z[4 * m + 3]));
                }
            }
        }
        if (!*abort && own_d) {
#pragma unroll
            for (int v = 0; v < 16; ++v) a.state_out[(static_cast<int64_t>(h) * D + i0 + v0 + v) * D + d] = S[v];
        }
    }

    if (*abort && tid == 0) {
        // A wait ran out.  Copies already issued land in their own time; let them
        // finish (bounded) before the CTA's shared memory is released.
        for (int i = F_QK; i <= F_A; ++i)
            for (uint32_t par = 0; par < 2; ++par) mbar_wait_bounded(bars + i, par, nullptr, 0, 20000000ull);
    }
    t5::fence_before();
    __syncthreads();
    if (warp == 9) {
        t5::fence_after();
        t5::dealloc(tmem, TM_COLS);
    }
}

size_t delta_scratch_bytes(int hv, int hk, int d, int64_t n) {
    const int64_t nch = (n + DC - 1) / DC;
    const int64_t per = static_cast<int64_t>(hv) * DC * (2 * DC + 4) + static_cast<int64_t>(hk) * d * DC;
    return static_cast<size_t>(nch * per) * sizeof(float);
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

// fp32 qkv [n][c_conv]: boxes of DC tokens x 32 floats, 128-byte swizzle, zero fill.
static bool make_qkv_map(CUtensorMap* map, const float* qkv, int64_t n, int c_conv) {
    auto enc = delta_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(c_conv), static_cast<cuuint64_t>(n)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(c_conv) * 4};
    cuuint32_t box[2] = {32, static_cast<cuuint32_t>(DC)};
    cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(qkv), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int read_and_clear_delta_error() {
    int v = 0, z = 0;
    cudaMemcpyFromSymbol(&v, g_delta_error, sizeof(int));
    if (v) cudaMemcpyToSymbol(g_delta_error, &z, sizeof(int));
    return v;
}

template <int D>
static cudaError_t launch_delta_d(DeltaArgs& a, cudaStream_t st) {
    const size_t prep_smem = PrepSmem<D>::FLOATS * sizeof(float);
    const size_t state_smem = StateSmem<D>::BYTES + 1024;
    static bool attr = false;
    if (!attr) {
        cudaFuncSetAttribute(delta_prep_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(prep_smem));
        cudaFuncSetAttribute(delta_state_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(state_smem));
        attr = true;
    }
    delta_prep_kernel<D><<<dim3(a.nchunks, a.hv / a.ratio), DELTA_THREADS, prep_smem, st>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    CUtensorMap map;
    if (!make_qkv_map(&map, a.qkv, a.n, a.c_conv)) return cudaErrorInvalidValue;
    delta_state_kernel<D><<<dim3(a.hv, D / NV), STATE_THREADS, state_smem, st>>>(map, a);
    return cudaGetLastError();
}

cudaError_t launch_delta(const gdn_layer& L, const float* qkv, const float* log_a, const float* b, int64_t n,
                         const float* state_in, float* state_out, float* o, void* scratch, cudaStream_t st) {
    DeltaArgs a;
    const int d = L.dk;
    a.qkv = qkv;
    a.log_a = log_a;
    a.b = b;
    a.n = static_cast<int>(n);
    a.hv = L.n_v_heads;
    a.ratio = L.n_v_heads / L.n_qk_heads;
    a.c_qk = L.n_qk_heads * d;
    a.c_v = L.n_v_heads * d;
    a.c_conv = 2 * a.c_qk + a.c_v;
    a.nchunks = static_cast<int>((n + DC - 1) / DC);
    const int64_t nch = a.nchunks;
    float* base = static_cast<float*>(scratch);
    a.T = base;
    a.A = a.T + nch * a.hv * DC * DC;
    a.G = a.A + nch * a.hv * DC * DC;
    a.KT = a.G + nch * a.hv * DC * 4;
    a.state_in = state_in;
    a.state_out = state_out;
    a.o = o;
    return d == 128 ? launch_delta_d<128>(a, st) : launch_delta_d<64>(a, st);
}

}  // namespace gdn
