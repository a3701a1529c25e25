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
//   delta_prep   one CTA per (chunk, head), all chunks in parallel: gamma,
//                K K^T and Q K^T on tensor cores, the masked A, and T by
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
//                shared memory with cp.async while chunk c computes: each
//                copy is issued right after the operand's last use in chunk c
//                (K and Q, used in the first phase, are double-buffered).
// Products use mma.sync m16n8k8 with tf32 operands rounded to nearest (the
// conv writes q, k, v already rounded; T, A, S, R, Delta are rounded where
// they are produced) and fp32 accumulation; everything else is fp32.
// Rounding every operand to tf32 keeps o and S within ~5e-4 (relative L2) of
// the exact recurrence on the test workloads.
#include "common.cuh"

namespace gdn {

constexpr int DC = GDN_CHUNK;  // 64
constexpr int DELTA_THREADS = 256;
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

// Load rows [t0, t0+DC) of a head slice of the fp32 qkv buffer into smem
// (pitch P floats), rounded to tf32; rows past n are zero.
template <int D, int P>
__device__ __forceinline__ void load_rows_tf32(float* dst, const float* qkv, int64_t ld, int col0, int t0, int n) {
    constexpr int V4 = D / 4;
    for (int idx = threadIdx.x; idx < DC * V4; idx += DELTA_THREADS) {
        const int r = idx / V4, c4 = idx % V4, t = t0 + r;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (t < n) v = *reinterpret_cast<const float4*>(qkv + static_cast<int64_t>(t) * ld + col0 + 4 * c4);
        float* d = dst + r * P + 4 * c4;
        d[0] = tf32f(v.x); d[1] = tf32f(v.y); d[2] = tf32f(v.z); d[3] = tf32f(v.w);
    }
}

// ------------------------------------------------------------------ prep

template <int D>
__global__ void __launch_bounds__(DELTA_THREADS, 2) delta_prep_kernel(DeltaArgs a) {
    constexpr int P = D + 4;        // row pitch of K, Q (conflict-free A/B fragment loads)
    constexpr int PL = DC + 4;      // row pitch of L, T
    extern __shared__ float sm[];
    float* Ks = sm;                 // [DC][P]
    float* Qs = Ks + DC * P;        // [DC][P]
    float* Ls = Qs + DC * P;        // [DC][PL]
    float* Ts = Ls + DC * PL;       // [DC][PL]
    float* Zs = Ts + DC * PL;       // [3][16][16]
    float* gl = Zs + 3 * 256;       // [DC] log a, then gamma
    float* bb = gl + DC;            // [DC]

    const int chunk = blockIdx.x, h = blockIdx.y, hk = h / a.ratio;
    const int t0 = chunk * DC;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, tg = lane & 3;

    load_rows_tf32<D, P>(Ks, a.qkv, a.c_conv, a.c_qk + hk * D, t0, a.n);
    load_rows_tf32<D, P>(Qs, a.qkv, a.c_conv, hk * D, t0, a.n);
    if (tid < DC) {
        const int t = t0 + tid;
        gl[tid] = t < a.n ? a.log_a[static_cast<int64_t>(t) * a.hv + h] : 0.f;
        bb[tid] = t < a.n ? a.b[static_cast<int64_t>(t) * a.hv + h] : 0.f;
    }
    for (int i = tid; i < DC * PL; i += DELTA_THREADS) Ts[i] = 0.f;
    __syncthreads();
    if (tid < 32) {  // inclusive prefix sum of log a over the chunk (2 per lane)
        const float x0 = gl[2 * tid], x1 = gl[2 * tid + 1];
        float s = x0 + x1;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float y = __shfl_up_sync(0xffffffffu, s, o);
            if (tid >= o) s += y;
        }
        gl[2 * tid] = s - x1;
        gl[2 * tid + 1] = s;
    }
    __syncthreads();

    // K K^T and Q K^T on the lower-triangular 16x8 tiles: warp -> m-tile warp/2,
    // n-tiles 4*(warp%2) .. +3 (skipping tiles wholly above the diagonal).
    {
        const int mt = warp >> 1, nt0 = 4 * (warp & 1);
        float ck[4][4] = {}, cq[4][4] = {};
        const float* ka = Ks + (16 * mt + g) * P + tg;
        const float* qa = Qs + (16 * mt + g) * P + tg;
#pragma unroll 4
        for (int ks = 0; ks < D / 8; ++ks) {
            const int c = 8 * ks;
            const uint32_t k0 = lds_u32(ka + c), k1 = lds_u32(ka + 8 * P + c), k2 = lds_u32(ka + c + 4),
                           k3 = lds_u32(ka + 8 * P + c + 4);
            const uint32_t q0 = lds_u32(qa + c), q1 = lds_u32(qa + 8 * P + c), q2 = lds_u32(qa + c + 4),
                           q3 = lds_u32(qa + 8 * P + c + 4);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int nt = nt0 + j;
                if (8 * nt <= 16 * mt + 15) {
                    const float* kb = Ks + (8 * nt + g) * P + c + tg;
                    const uint32_t b0 = lds_u32(kb), b1 = lds_u32(kb + 4);
                    mma_tf32(ck[j], k0, k1, k2, k3, b0, b1);
                    mma_tf32(cq[j], q0, q1, q2, q3, b0, b1);
                }
            }
        }
        float* aout = a.A + (static_cast<int64_t>(chunk) * a.hv + h) * DC * DC;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int nt = nt0 + j;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int i = 16 * mt + g + (e >> 1) * 8, jj = 8 * nt + 2 * tg + (e & 1);
                const bool live = 8 * nt <= 16 * mt + 15;
                const float dec = (live && jj <= i) ? expf(gl[i] - gl[jj]) : 0.f;
                Ls[i * PL + jj] = (jj < i) ? bb[i] * dec * ck[j][e] : 0.f;
                aout[i * DC + jj] = tf32f(dec * cq[j][e]);
            }
        }
    }
    __syncthreads();

    // T = (I + L)^{-1}: diagonal 16x16 blocks by substitution, one column per thread.
    if (tid < 64) {
        const int blk = tid >> 4, c = tid & 15, o = 16 * blk;
        float col[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            float v;
            if (r < c) {
                v = 0.f;
            } else if (r == c) {
                v = 1.f;
            } else {
                float s = 0.f;
#pragma unroll
                for (int k = 0; k < r; ++k)
                    if (k >= c) s = fmaf(Ls[(o + r) * PL + o + k], col[k], s);
                v = -s;
            }
            col[r] = v;
        }
#pragma unroll
        for (int r = 0; r < 16; ++r) Ts[(o + r) * PL + o + c] = col[r];
    }
    __syncthreads();
    // Off-diagonal blocks, block row by block row:
    //   T_IJ = -T_II * sum_{K=J}^{I-1} L_IK T_KJ   (J < I)
    for (int I = 1; I < 4; ++I) {
        for (int e = tid; e < I * 256; e += DELTA_THREADS) {
            const int J = e >> 8, r = (e >> 4) & 15, c = e & 15;
            float z = 0.f;
            for (int K = J; K < I; ++K)
#pragma unroll
                for (int m = 0; m < 16; ++m)
                    z = fmaf(Ls[(16 * I + r) * PL + 16 * K + m], Ts[(16 * K + m) * PL + 16 * J + c], z);
            Zs[J * 256 + r * 16 + c] = z;
        }
        __syncthreads();
        for (int e = tid; e < I * 256; e += DELTA_THREADS) {
            const int J = e >> 8, r = (e >> 4) & 15, c = e & 15;
            float s = 0.f;
#pragma unroll
            for (int m = 0; m < 16; ++m) s = fmaf(Ts[(16 * I + r) * PL + 16 * I + m], Zs[J * 256 + m * 16 + c], s);
            Ts[(16 * I + r) * PL + 16 * J + c] = -s;
        }
        __syncthreads();
    }
    float* tout = a.T + (static_cast<int64_t>(chunk) * a.hv + h) * DC * DC;
    for (int idx = tid; idx < DC * DC; idx += DELTA_THREADS) tout[idx] = tf32f(Ts[(idx / DC) * PL + idx % DC]);
    if (tid < DC) {
        const float gv = gl[tid];
        *reinterpret_cast<float4*>(a.G + ((static_cast<int64_t>(chunk) * a.hv + h) * DC + tid) * 4) =
            make_float4(gv, expf(gv), bb[tid], expf(gl[DC - 1] - gv));
    }
}

// ------------------------------------------------------------------ state pass

template <int D>
struct StateSmem {
    static constexpr int P = D + 4;    // K, Q, S row pitch (conflict-free fragment loads)
    static constexpr int PT = DC + 4;  // T, A row pitch
    static constexpr int PR = NV + 8;  // V, R/Delta row pitch (conflict-free in both orientations)
    static constexpr int K0 = 0;                   // Ks[2][DC][P]
    static constexpr int Q0 = K0 + 2 * DC * P;     // Qs[2][DC][P]
    static constexpr int S0 = Q0 + 2 * DC * P;     // Ss[NV][P]
    static constexpr int T0 = S0 + NV * P;         // Ts[DC][PT]
    static constexpr int A0 = T0 + DC * PT;        // As[DC][PT]
    static constexpr int V0 = A0 + DC * PT;        // Vs[DC][PR]
    static constexpr int R0 = V0 + DC * PR;        // Rs[DC][PR]
    static constexpr int G0 = R0 + DC * PR;        // Gs[2][DC][4]
    static constexpr int FLOATS = G0 + 2 * DC * 4;
};

// One chunk step in three phases, each a set of independent MMA chains:
//   A: X = K S^T and Y = Q S^T together (k split in even/odd halves);
//      R = diag(b) (V - diag(e^gamma) X)
//   B: Delta = T R
//   C: O = diag(e^gamma) Y + A Delta, and S <- e^{gamma_C} S + Delta~^T K
// Operand copies for chunk c+1: K and Q (double-buffered) at the start of
// chunk c, V and the gate table after phase A, T after B, A after C.
template <int D>
__global__ void __launch_bounds__(DELTA_THREADS, 1) delta_state_kernel(DeltaArgs a) {
    using L = StateSmem<D>;
    constexpr int P = L::P, PT = L::PT, PR = L::PR;
    constexpr int NT_D = D / 8;     // n-tiles across d
    constexpr int DW = NT_D / 4;    // n-tiles of d per warp in the update (4 warps across d)
    extern __shared__ __align__(16) float sm[];
    float* Ss = sm + L::S0;
    float* Ts = sm + L::T0;
    float* As = sm + L::A0;
    float* Vs = sm + L::V0;
    float* Rs = sm + L::R0;

    const int h = blockIdx.x, i0 = blockIdx.y * NV, hk = h / a.ratio;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, tg = lane & 3;

    // ---- asynchronous copies of one chunk's operands (rows past n are zero-filled)
    auto rows = [&](float* dst, int pitch, int col0, int width, int c) {   // token rows of qkv
        const int t0 = c * DC, w4 = width / 4;
        for (int idx = tid; idx < DC * w4; idx += DELTA_THREADS) {
            const int r = idx / w4, c4 = idx % w4, t = t0 + r;
            const bool ok = t < a.n;
            const float* src = ok ? a.qkv + static_cast<int64_t>(t) * a.c_conv + col0 + 4 * c4 : a.qkv;
            cp_async16(dst + r * pitch + 4 * c4, src, ok);
        }
    };
    auto mat = [&](float* dst, const float* src) {                        // a [DC][DC] scratch matrix
        for (int idx = tid; idx < DC * DC / 4; idx += DELTA_THREADS) {
            const int r = idx / (DC / 4), c4 = idx % (DC / 4);
            cp_async16(dst + r * PT + 4 * c4, src + 4 * idx, true);
        }
    };
    auto chunk_base = [&](int c) { return static_cast<int64_t>(c) * a.hv + h; };
    auto issue_KQ = [&](int c) {
        if (c < a.nchunks) {
            rows(sm + L::K0 + (c & 1) * DC * P, P, a.c_qk + hk * D, D, c);
            rows(sm + L::Q0 + (c & 1) * DC * P, P, hk * D, D, c);
        }
        cp_async_commit();
    };
    auto issue_VG = [&](int c) {
        if (c < a.nchunks) {
            rows(Vs, PR, 2 * a.c_qk + h * D + i0, NV, c);
            if (tid < DC) cp_async16(sm + L::G0 + (c & 1) * DC * 4 + 4 * tid, a.G + (chunk_base(c) * DC + tid) * 4, true);
        }
        cp_async_commit();
    };
    auto issue_T = [&](int c) {
        if (c < a.nchunks) mat(Ts, a.T + chunk_base(c) * DC * DC);
        cp_async_commit();
    };
    auto issue_A = [&](int c) {
        if (c < a.nchunks) mat(As, a.A + chunk_base(c) * DC * DC);
        cp_async_commit();
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

    issue_KQ(0);
    issue_VG(0);
    issue_T(0);
    issue_A(0);
    for (int chunk = 0; chunk < a.nchunks; ++chunk) {
        const int t0 = chunk * DC;
        const float* Ks = sm + L::K0 + (chunk & 1) * DC * P;
        const float* Qs = sm + L::Q0 + (chunk & 1) * DC * P;
        const float* Gs = sm + L::G0 + (chunk & 1) * DC * 4;
#pragma unroll
        for (int j = 0; j < DW; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int i = 16 * smt + g + (e >> 1) * 8, d = 8 * (snt0 + j) + 2 * tg + (e & 1);
                Ss[i * P + d] = tf32f(S[j][e]);
            }
        issue_KQ(chunk + 1);
        cp_async_wait<3>();        // K(c), Q(c), V(c), G(c) have landed
        __syncthreads();

        // ---- phase A: X = K S^T, Y = Q S^T; R = diag(b) (V - diag(e^gamma) X)
        float y[2][4];
        {
            float xa[2][2][4] = {}, ya[2][2][4] = {};
            const float* ka = Ks + (16 * omt + g) * P + tg;
            const float* qa = Qs + (16 * omt + g) * P + tg;
#pragma unroll 2
            for (int ks = 0; ks < D / 8; ks += 2) {
#pragma unroll
                for (int p = 0; p < 2; ++p) {
                    const int c = 8 * (ks + p);
                    const uint32_t k0 = lds_u32(ka + c), k1 = lds_u32(ka + 8 * P + c), k2 = lds_u32(ka + c + 4),
                                   k3 = lds_u32(ka + 8 * P + c + 4);
                    const uint32_t q0 = lds_u32(qa + c), q1 = lds_u32(qa + 8 * P + c), q2 = lds_u32(qa + c + 4),
                                   q3 = lds_u32(qa + 8 * P + c + 4);
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        const float* sb = Ss + (8 * (ont0 + j) + g) * P + c + tg;
                        const uint32_t b0 = lds_u32(sb), b1 = lds_u32(sb + 4);
                        mma_tf32(xa[j][p], k0, k1, k2, k3, b0, b1);
                        mma_tf32(ya[j][p], q0, q1, q2, q3, b0, b1);
                    }
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
                    Rs[t * PR + i] = tf32f(Gs[4 * t + 2] * (Vs[t * PR + i] - ex * x));
                }
        }
        __syncthreads();
        issue_VG(chunk + 1);
        cp_async_wait<3>();        // T(c) has landed
        __syncthreads();

        // ---- phase B: Delta = T R (T unit lower triangular)
        {
            float dl[2][4] = {};
            const float* ta = Ts + (16 * omt + g) * PT + tg;
            for (int ks = 0; ks < 2 * omt + 2; ++ks) {
                const int c = 8 * ks;
                const uint32_t a0 = lds_u32(ta + c), a1 = lds_u32(ta + 8 * PT + c), a2 = lds_u32(ta + c + 4),
                               a3 = lds_u32(ta + 8 * PT + c + 4);
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const float* rb = Rs + (c + tg) * PR + 8 * (ont0 + j) + g;
                    mma_tf32(dl[j], a0, a1, a2, a3, lds_u32(rb), lds_u32(rb + 4 * PR));
                }
            }
            __syncthreads();       // every warp has read R
#pragma unroll
            for (int j = 0; j < 2; ++j)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int t = 16 * omt + g + (e >> 1) * 8, i = 8 * (ont0 + j) + 2 * tg + (e & 1);
                    Rs[t * PR + i] = tf32f(dl[j][e]);
                }
        }
        __syncthreads();
        issue_T(chunk + 1);
        cp_async_wait<3>();        // A(c) has landed
        __syncthreads();

        // ---- phase C: O = Y + A Delta;  S <- e^{gamma_C} S + Delta~^T K
        {
            const float* aa = As + (16 * omt + g) * PT + tg;
            for (int ks = 0; ks < 2 * omt + 2; ++ks) {
                const int c = 8 * ks;
                const uint32_t a0 = lds_u32(aa + c), a1 = lds_u32(aa + 8 * PT + c), a2 = lds_u32(aa + c + 4),
                               a3 = lds_u32(aa + 8 * PT + c + 4);
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const float* rb = Rs + (c + tg) * PR + 8 * (ont0 + j) + g;
                    mma_tf32(y[j], a0, a1, a2, a3, lds_u32(rb), lds_u32(rb + 4 * PR));
                }
            }
            const float dec = Gs[4 * (DC - 1) + 1];
#pragma unroll
            for (int j = 0; j < DW; ++j)
#pragma unroll
                for (int e = 0; e < 4; ++e) S[j][e] *= dec;
#pragma unroll 2
            for (int ks = 0; ks < DC / 8; ++ks) {
                const int t = 8 * ks + tg;
                const float* da = Rs + t * PR + 16 * smt + g;
                const float k0 = Gs[4 * t + 3], k1 = Gs[4 * (t + 4) + 3];
                const uint32_t a0 = to_tf32(da[0] * k0), a1 = to_tf32(da[8] * k0), a2 = to_tf32(da[4 * PR] * k1),
                               a3 = to_tf32(da[4 * PR + 8] * k1);
#pragma unroll
                for (int j = 0; j < DW; ++j) {
                    const float* kb = Ks + t * P + 8 * (snt0 + j) + g;
                    mma_tf32(S[j], a0, a1, a2, a3, lds_u32(kb), lds_u32(kb + 4 * P));
                }
            }
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
        __syncthreads();           // every warp has read A, Delta, K(c), Q(c), S
        issue_A(chunk + 1);
    }
    cp_async_wait<0>();
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

template <int D>
static cudaError_t launch_delta_d(DeltaArgs& a, cudaStream_t st) {
    constexpr int P = D + 4;
    const size_t prep_smem = (2 * DC * P + 2 * DC * (DC + 4) + 3 * 256 + 2 * DC) * sizeof(float);
    const size_t state_smem = StateSmem<D>::FLOATS * sizeof(float);
    static bool attr = false;
    if (!attr) {
        cudaFuncSetAttribute(delta_prep_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(prep_smem));
        cudaFuncSetAttribute(delta_state_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(state_smem));
        attr = true;
    }
    delta_prep_kernel<D><<<dim3(a.nchunks, a.hv), DELTA_THREADS, prep_smem, st>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    delta_state_kernel<D><<<dim3(a.hv, D / NV), DELTA_THREADS, state_smem, st>>>(a);
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
