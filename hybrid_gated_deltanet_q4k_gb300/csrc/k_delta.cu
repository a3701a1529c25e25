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

#include <mutex>

namespace gdn {

static __device__ int g_delta_error;

constexpr int DC = GDN_CHUNK;  // 64
constexpr int DELTA_THREADS = 256;            // prep; compute warps of the state pass
constexpr int STATE_THREADS = DELTA_THREADS + 32;  // + one TMA producer warp
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

template <int D>
struct StateSmem {
    // byte offsets; every TMA destination is 1024-byte aligned
    static constexpr int SLAB = DC * 128;          // 64 token rows x 32 floats
    static constexpr int NSLAB = D / 32;
    static constexpr int KQ_BYTES = NSLAB * SLAB;  // one K or Q tile
    static constexpr int P = D + 4;                // S row pitch (floats)
    static constexpr int PT = DC + 4;              // R^T, Delta^T row pitch (floats)
    static constexpr int K0 = 0;                               // Ks[2]
    static constexpr int Q0 = K0 + 2 * KQ_BYTES;               // Qs[2]
    static constexpr int T0 = Q0 + 2 * KQ_BYTES;               // Ts (2 slabs)
    static constexpr int A0 = T0 + 2 * SLAB;                   // As (2 slabs)
    static constexpr int V0 = A0 + 2 * SLAB;                   // Vs (1 slab: NV = 32 floats)
    static constexpr int G0 = V0 + SLAB;                       // Gs[2][DC][4]
    static constexpr int S0 = G0 + 2 * DC * 16;                // Ss[NV][P]
    static constexpr int R0 = S0 + NV * P * 4;                 // Rt[NV][PT]
    static constexpr int E0 = R0 + NV * PT * 4;                // Et[NV][PT]
    static constexpr int B0 = E0 + NV * PT * 4;                // mbarriers: full KQ[2], V, T, A; freed KQ[2], V, T, A
    static constexpr int BYTES = B0 + 128;
};

// One chunk step in three phases, each a set of independent MMA chains:
//   A: X = K S^T and Y = Q S^T together (k split in even/odd halves);
//      R = diag(b) (V - diag(e^gamma) X), stored transposed
//   B: Delta = T R, stored transposed (plain and scaled by e^{gamma_C - gamma})
//   C: O = diag(e^gamma) Y + A Delta, and S <- e^{gamma_C} S + Delta~^T K
// Warps 0-7 compute; warp 8 is the TMA producer.  For each operand buffer a
// "full" mbarrier (TMA bytes) and a "freed" mbarrier (the 256 compute threads
// arrive after their last read) pace the producer: K and Q of chunk c+1
// (double-buffered) once chunk c-1 is done, V and the gate table after phase A,
// T after phase B, A after phase C.  The compute warps synchronise among
// themselves with a named barrier, so the producer never holds them up.
// Fragments come from shared memory by ldmatrix, except K in the update,
// whose [token][d] layout is the transpose of what ldmatrix delivers.
__device__ __forceinline__ void compute_sync() { asm volatile("bar.sync 1, %0;" ::"n"(DELTA_THREADS) : "memory"); }

__device__ __forceinline__ void mbar_arrive_cta(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

template <int D>
__global__ void __launch_bounds__(STATE_THREADS, 1)
delta_state_kernel(const __grid_constant__ CUtensorMap qkv_map, DeltaArgs a) {
    using L = StateSmem<D>;
    constexpr int P = L::P, PT = L::PT;
    constexpr int NT_D = D / 8;     // n-tiles across d
    constexpr int DW = NT_D / 4;    // n-tiles of d per warp in the update (4 warps across d)
    extern __shared__ __align__(1024) unsigned char smb[];
    unsigned char* base = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smb) + 1023) & ~uintptr_t(1023));
    float* Ss = reinterpret_cast<float*>(base + L::S0);
    float* Rt = reinterpret_cast<float*>(base + L::R0);
    float* Et = reinterpret_cast<float*>(base + L::E0);
    uint64_t* bars = reinterpret_cast<uint64_t*>(base + L::B0);
    uint64_t* fKQ = bars;       // full [2]
    uint64_t* fV = bars + 2;
    uint64_t* fT = bars + 3;
    uint64_t* fA = bars + 4;
    uint64_t* eKQ = bars + 5;   // freed [2]
    uint64_t* eV = bars + 7;
    uint64_t* eT = bars + 8;
    uint64_t* eA = bars + 9;
    __shared__ int abort_flag;

    const int h = blockIdx.x, i0 = blockIdx.y * NV, hk = h / a.ratio;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, tg = lane & 3;

    if (tid == 0) {
        for (int i = 0; i < 5; ++i) mbar_init_cta(bars + i, 1);
        for (int i = 5; i < 10; ++i) mbar_init_cta(bars + i, DELTA_THREADS);
        mbar_init_fence();
        abort_flag = 0;
    }
    __syncthreads();

    if (warp == DELTA_THREADS / 32) {
        // ------------------------------------------------------------ producer
        if (lane != 0) return;
        auto chunk_base = [&](int c) { return static_cast<int64_t>(c) * a.hv + h; };
        bool ok = true;
        auto wait_freed = [&](uint64_t* bar, uint32_t parity) {
            if (ok && !mbar_wait_bounded(bar, parity, &g_delta_error, ERR_WAIT_TIMEOUT)) ok = false;
            return ok;
        };
        for (int c = 0; c < a.nchunks && ok; ++c) {
            // K, Q of chunk c into buffer c&1: freed when chunk c-2 finished
            if (c >= 2 && !wait_freed(eKQ + (c & 1), ((c - 2) >> 1) & 1)) break;
            {
                uint64_t* bar = fKQ + (c & 1);
                unsigned char* kd = base + L::K0 + (c & 1) * L::KQ_BYTES;
                unsigned char* qd = base + L::Q0 + (c & 1) * L::KQ_BYTES;
                mbar_expect_tx(bar, 2 * L::KQ_BYTES);
                for (int sl = 0; sl < L::NSLAB; ++sl) {
                    tma_load_2d_tile(kd + sl * L::SLAB, &qkv_map, bar, a.c_qk + hk * D + 32 * sl, c * DC);
                    tma_load_2d_tile(qd + sl * L::SLAB, &qkv_map, bar, hk * D + 32 * sl, c * DC);
                }
            }
            // V and the gate table of chunk c: V freed after phase A of chunk c-1,
            // gate buffer c&1 after chunk c-2 (covered by the K/Q wait above)
            if (c >= 1 && !wait_freed(eV, (c - 1) & 1)) break;
            mbar_expect_tx(fV, L::SLAB + DC * 16);
            tma_load_2d_tile(base + L::V0, &qkv_map, fV, 2 * a.c_qk + h * D + i0, c * DC);
            bulk_load_1d(base + L::G0 + (c & 1) * DC * 16, a.G + chunk_base(c) * DC * 4, DC * 16, fV);
            // T of chunk c: freed after phase B of chunk c-1
            if (c >= 1 && !wait_freed(eT, (c - 1) & 1)) break;
            mbar_expect_tx(fT, 2 * L::SLAB);
            bulk_load_1d(base + L::T0, a.T + chunk_base(c) * DC * DC, 2 * L::SLAB, fT);
            // A of chunk c: freed after phase C of chunk c-1
            if (c >= 1 && !wait_freed(eA, (c - 1) & 1)) break;
            mbar_expect_tx(fA, 2 * L::SLAB);
            bulk_load_1d(base + L::A0, a.A + chunk_base(c) * DC * DC, 2 * L::SLAB, fA);
        }
        if (!ok) abort_flag = 1;
        return;
    }

    // ---------------------------------------------------------------- compute
    auto wait = [&](uint64_t* bar, uint32_t parity) {
        if (!mbar_wait_bounded(bar, parity, &g_delta_error, ERR_WAIT_TIMEOUT)) abort_flag = 1;
    };
    // fp32 element (r, c) of a swizzled tile of 32-float slabs, as a float pointer
    auto tile = [&](int off, int r, int c) {
        return reinterpret_cast<const float*>(base + off + (c >> 5) * L::SLAB + sw128_f32(r, c & 31));
    };

    // State fragments: warp owns rows 16*(warp/4) .. +15 of the tile and d columns
    // 8*DW*(warp%4) .. +8*DW-1, as m16n8 accumulators.
    const int smt = warp >> 2, snt0 = DW * (warp & 3);
    float S[DW][4];
#pragma unroll
    for (int j = 0; j < DW; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int i = 16 * smt + g + (e >> 1) * 8, d = 8 * (snt0 + j) + 2 * tg + (e & 1);
            S[j][e] = a.state_in ? a.state_in[(static_cast<int64_t>(h) * D + i0 + i) * D + d] : 0.f;
        }
    // Output-tile ownership for the C x NV products: m-tile warp/2, n-tiles 2*(warp%2), +1.
    const int omt = warp >> 1, ont0 = 2 * (warp & 1);
    // ldmatrix row of this lane: matrix lane/8, row lane%8
    const int lm = lane >> 3, lr = lane & 7;

    for (int chunk = 0; chunk < a.nchunks; ++chunk) {
        const int t0 = chunk * DC;
        const int KO = L::K0 + (chunk & 1) * L::KQ_BYTES;
        const int QO = L::Q0 + (chunk & 1) * L::KQ_BYTES;
        const float* Gs = reinterpret_cast<const float*>(base + L::G0 + (chunk & 1) * DC * 16);
#pragma unroll
        for (int j = 0; j < DW; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int i = 16 * smt + g + (e >> 1) * 8, d = 8 * (snt0 + j) + 2 * tg + (e & 1);
                Ss[i * P + d] = tf32f(S[j][e]);
            }
        wait(fKQ + (chunk & 1), (chunk >> 1) & 1);
        wait(fV, chunk & 1);
        compute_sync();
        if (abort_flag) break;     // uniform: read after a barrier

        // ---- phase A: X = K S^T, Y = Q S^T; R = diag(b) (V - diag(e^gamma) X)
        float y[2][4];
        {
            float xa[2][2][4] = {}, ya[2][2][4] = {};
            const int arow = 16 * omt + lr + 8 * (lm & 1);
            const float* sb = b2_frag_addr<P>(Ss, 8 * ont0, 0, lane);
#pragma unroll 2
            for (int ks = 0; ks < D / 8; ks += 2) {
#pragma unroll
                for (int p = 0; p < 2; ++p) {
                    const int c = 8 * (ks + p) + 4 * (lm >> 1);
                    uint32_t k0, k1, k2, k3, q0, q1, q2, q3, b0, b1, b2, b3;
                    ldsm_x4(k0, k1, k2, k3, tile(KO, arow, c));
                    ldsm_x4(q0, q1, q2, q3, tile(QO, arow, c));
                    ldsm_x4(b0, b1, b2, b3, sb + 8 * (ks + p));
                    mma_tf32(xa[0][p], k0, k1, k2, k3, b0, b1);
                    mma_tf32(ya[0][p], q0, q1, q2, q3, b0, b1);
                    mma_tf32(xa[1][p], k0, k1, k2, k3, b2, b3);
                    mma_tf32(ya[1][p], q0, q1, q2, q3, b2, b3);
                }
            }
            const float e_lo = Gs[4 * (16 * omt + g) + 1], e_hi = Gs[4 * (16 * omt + g + 8) + 1];
#pragma unroll
            for (int j = 0; j < 2; ++j)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int t = 16 * omt + g + (e >> 1) * 8, i = 8 * (ont0 + j) + 2 * tg + (e & 1);
                    const float ex = (e >> 1) ? e_hi : e_lo;
                    const float x = xa[j][0][e] + xa[j][1][e];
                    y[j][e] = ex * (ya[j][0][e] + ya[j][1][e]);
                    Rt[i * PT + t] = tf32f(Gs[4 * t + 2] * (*tile(L::V0, t, i) - ex * x));
                }
        }
        mbar_arrive_cta(eV);       // V of this chunk is consumed
        wait(fT, chunk & 1);
        compute_sync();
        if (abort_flag) break;

        // ---- phase B: Delta = T R (T unit lower triangular)
        {
            float dl[2][4] = {};
            const int arow = 16 * omt + lr + 8 * (lm & 1);
            const float* rb = b2_frag_addr<PT>(Rt, 8 * ont0, 0, lane);
            for (int ks = 0; ks < 2 * omt + 2; ++ks) {
                uint32_t a0, a1, a2, a3, b0, b1, b2, b3;
                ldsm_x4(a0, a1, a2, a3, tile(L::T0, arow, 8 * ks + 4 * (lm >> 1)));
                ldsm_x4(b0, b1, b2, b3, rb + 8 * ks);
                mma_tf32(dl[0], a0, a1, a2, a3, b0, b1);
                mma_tf32(dl[1], a0, a1, a2, a3, b2, b3);
            }
            mbar_arrive_cta(eT);   // T of this chunk is consumed
            compute_sync();        // every warp has read R
#pragma unroll
            for (int j = 0; j < 2; ++j)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int t = 16 * omt + g + (e >> 1) * 8, i = 8 * (ont0 + j) + 2 * tg + (e & 1);
                    Rt[i * PT + t] = tf32f(dl[j][e]);
                    Et[i * PT + t] = tf32f(dl[j][e] * Gs[4 * t + 3]);
                }
        }
        wait(fA, chunk & 1);
        compute_sync();
        if (abort_flag) break;

        // ---- phase C: O = Y + A Delta;  S <- e^{gamma_C} S + Delta~^T K
        {
            const int arow = 16 * omt + lr + 8 * (lm & 1);
            const float* db = b2_frag_addr<PT>(Rt, 8 * ont0, 0, lane);
            for (int ks = 0; ks < 2 * omt + 2; ++ks) {
                uint32_t a0, a1, a2, a3, b0, b1, b2, b3;
                ldsm_x4(a0, a1, a2, a3, tile(L::A0, arow, 8 * ks + 4 * (lm >> 1)));
                ldsm_x4(b0, b1, b2, b3, db + 8 * ks);
                mma_tf32(y[0], a0, a1, a2, a3, b0, b1);
                mma_tf32(y[1], a0, a1, a2, a3, b2, b3);
            }
            mbar_arrive_cta(eA);   // A of this chunk is consumed
            const float dec = Gs[4 * (DC - 1) + 1];
#pragma unroll
            for (int j = 0; j < DW; ++j)
#pragma unroll
                for (int e = 0; e < 4; ++e) S[j][e] *= dec;
            const float* ea = a_frag_addr<PT>(Et, 16 * smt, 0, lane);
            // B fragment (k = token tg / tg+4, n = d) of K(c): byte offsets within the swizzled
            // tile for ks = 0; token 8ks+r sits 1024*ks bytes further (same swizzle key r).
            const unsigned char* kbase = base + KO;
            uint32_t koff[DW][2];
#pragma unroll
            for (int j = 0; j < DW; ++j) {
                const int d = 8 * (snt0 + j) + g;
                koff[j][0] = (d >> 5) * L::SLAB + sw128_f32(tg, d & 31);
                koff[j][1] = (d >> 5) * L::SLAB + sw128_f32(tg + 4, d & 31);
            }
#pragma unroll 2
            for (int ks = 0; ks < DC / 8; ++ks) {
                uint32_t a0, a1, a2, a3;
                ldsm_x4(a0, a1, a2, a3, ea + 8 * ks);
                const unsigned char* kb = kbase + 1024 * ks;
#pragma unroll
                for (int j = 0; j < DW; ++j)
                    mma_tf32(S[j], a0, a1, a2, a3, *reinterpret_cast<const uint32_t*>(kb + koff[j][0]),
                             *reinterpret_cast<const uint32_t*>(kb + koff[j][1]));
            }
            mbar_arrive_cta(eKQ + (chunk & 1));   // K, Q and the gate table of this chunk are consumed
#pragma unroll
            for (int j = 0; j < 2; ++j)
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int t = 16 * omt + g + 8 * hh, i = 8 * (ont0 + j) + 2 * tg;
                    if (t0 + t < a.n)
                        *reinterpret_cast<float2*>(a.o + static_cast<int64_t>(t0 + t) * a.c_v + h * D + i0 + i) =
                            make_float2(y[j][2 * hh], y[j][2 * hh + 1]);
                }
        }
        compute_sync();            // every warp has read Delta and S before they are rewritten
    }
    if (abort_flag) {
        // A wait ran out.  Copies the producer issued for this CTA land in their own
        // time; let them finish (bounded) before the CTA's shared memory is released.
        if (tid == 0)
            for (int i = 0; i < 5; ++i)
                for (uint32_t par = 0; par < 2; ++par) mbar_wait_bounded(bars + i, par, nullptr, 0, 20000000ull);
        return;
    }
#pragma unroll
    for (int j = 0; j < DW; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int i = 16 * smt + g + (e >> 1) * 8, d = 8 * (snt0 + j) + 2 * tg + (e & 1);
            a.state_out[(static_cast<int64_t>(h) * D + i0 + i) * D + d] = S[j][e];
        }
}

size_t delta_scratch_bytes(int hv, int d, int64_t n) {
    (void)d;
    const int64_t nch = (n + DC - 1) / DC;
    const int64_t per = static_cast<int64_t>(hv) * DC * (2 * DC + 4);
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
    a.state_in = state_in;
    a.state_out = state_out;
    a.o = o;
    return d == 128 ? launch_delta_d<128>(a, st) : launch_delta_d<64>(a, st);
}

}  // namespace gdn
