// Step 3: the gated delta rule, chunked (WY/UT form) with the state carried
// across chunks.
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
//     Lm_ij = b_i e^{gamma_i-gamma_j} k_i.k_j (j < i)
//     W = (I + Lm)^{-1} diag(b e^gamma) K,   U = (I + Lm)^{-1} diag(b) V
//     Delta = U - W S^T
//     O = diag(e^gamma) Q S^T + (M o Q K^T) Delta,   M_ij = e^{gamma_i-gamma_j} (j <= i)
//     S <- e^{gamma_C} S + Delta^T diag(e^{gamma_C - gamma}) K
// All exponents are <= 0.  Tokens past N are padded with log a = 0, b = 0,
// which leaves S unchanged.
//
// Two kernels:
//   delta_prep   one CTA per (chunk, head), all chunks in parallel: gamma,
//                K K^T and Q K^T, the masked A_qk = M o Q K^T, and W, U by
//                forward substitution of (I + Lm) X = rhs (each thread owns one
//                column of W or U, so the substitution needs no barriers).
//   delta_state  one CTA per (head, 16 rows of S): the chunks in order,
//                Delta, O and the state update; rows of S evolve
//                independently (row i only reads v[i]), so the rows split
//                across CTAs with no communication.
// fp32 throughout on the CUDA cores (no tensor cores in this form).
#include "common.cuh"

namespace gdn {

constexpr int DC = GDN_CHUNK;  // 64
constexpr int DELTA_THREADS = 256;
constexpr int STATE_NV = 16;   // rows of S per state-pass CTA

struct DeltaArgs {
    const float* qkv;     // [n][c_conv] fp32: q | k | v
    const float* log_a;   // [n][hv]
    const float* b;       // [n][hv]
    int n, hv, ratio, c_qk, c_conv, c_v;
    int nchunks;
    float* w;      // [nchunks][hv][DC][D]
    float* u;      // [nchunks][hv][DC][D]
    float* aqk;    // [nchunks][hv][DC][DC]
    float* gam;    // [nchunks][hv][DC]
    const float* state_in;  // [hv][D][D] or null
    float* state_out;
    float* o;      // [n][c_v]
};

template <int D>
__global__ void __launch_bounds__(DELTA_THREADS) delta_prep_kernel(DeltaArgs a) {
    constexpr int P = D + 1;
    extern __shared__ float sm[];
    float* Ks = sm;                 // [DC][P]
    float* Qs = Ks + DC * P;        // [DC][P]  (Q, later the W right-hand side / W)
    float* Vs = Qs + DC * P;        // [DC][P]  (V, later U)
    float* Lm = Vs + DC * P;        // [DC][DC + 1]
    float* gl = Lm + DC * (DC + 1); // [DC] log a, then gamma
    float* bb = gl + DC;            // [DC]

    const int chunk = blockIdx.x, h = blockIdx.y, hk = h / a.ratio;
    const int t0 = chunk * DC;
    const int tid = threadIdx.x;
    for (int idx = tid; idx < DC * D; idx += DELTA_THREADS) {
        const int i = idx / D, c = idx % D, t = t0 + i;
        float kq = 0.f, qq = 0.f, vv = 0.f;
        if (t < a.n) {
            const float* row = a.qkv + static_cast<int64_t>(t) * a.c_conv;
            qq = row[hk * D + c];
            kq = row[a.c_qk + hk * D + c];
            vv = row[2 * a.c_qk + h * D + c];
        }
        Ks[i * P + c] = kq;
        Qs[i * P + c] = qq;
        Vs[i * P + c] = vv;
    }
    if (tid < DC) {
        const int t = t0 + tid;
        gl[tid] = t < a.n ? a.log_a[static_cast<int64_t>(t) * a.hv + h] : 0.f;
        bb[tid] = t < a.n ? a.b[static_cast<int64_t>(t) * a.hv + h] : 0.f;
    }
    __syncthreads();
    if (tid < 32) {  // inclusive prefix sum of log a over the chunk (2 per lane)
        float x0 = gl[2 * tid], x1 = gl[2 * tid + 1];
        float s = x0 + x1;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float y = __shfl_up_sync(0xffffffffu, s, o);
            if (tid >= o) s += y;
        }
        const float excl = s - (x0 + x1);
        gl[2 * tid] = excl + x0;
        gl[2 * tid + 1] = s;
    }
    __syncthreads();

    // K K^T and Q K^T, 4x4 outputs per thread at rows ti+16r, cols tj+16c.
    const int ti = tid >> 4, tj = tid & 15;
    float* aqk = a.aqk + (static_cast<int64_t>(chunk) * a.hv + h) * DC * DC;
#pragma unroll 1
    for (int pass = 0; pass < 2; ++pass) {
        const float* A = pass == 0 ? Ks : Qs;
        float acc[4][4] = {};
#pragma unroll 4
        for (int c = 0; c < D; ++c) {
            float av[4], bv[4];
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                av[r] = A[(ti + 16 * r) * P + c];
                bv[r] = Ks[(tj + 16 * r) * P + c];
            }
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int q = 0; q < 4; ++q) acc[r][q] = fmaf(av[r], bv[q], acc[r][q]);
        }
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int i = ti + 16 * r, j = tj + 16 * q;
                const float dec = j <= i ? expf(gl[i] - gl[j]) : 0.f;
                if (pass == 0)
                    Lm[i * (DC + 1) + j] = j < i ? bb[i] * dec * acc[r][q] : 0.f;
                else
                    aqk[i * DC + j] = dec * acc[r][q];
            }
    }
    __syncthreads();
    // right-hand sides: W <- diag(b e^gamma) K (into Qs), U <- diag(b) V (in place)
    for (int idx = tid; idx < DC * D; idx += DELTA_THREADS) {
        const int i = idx / D, c = idx % D;
        Qs[i * P + c] = bb[i] * expf(gl[i]) * Ks[i * P + c];
        Vs[i * P + c] = bb[i] * Vs[i * P + c];
    }
    __syncthreads();
    // forward substitution (I + Lm) X = rhs, one column per thread
    if (tid < 2 * D) {
        float* X = tid < D ? Qs : Vs;
        const int c = tid < D ? tid : tid - D;
        for (int i = 1; i < DC; ++i) {
            float s = 0.f;
            for (int j = 0; j < i; ++j) s = fmaf(Lm[i * (DC + 1) + j], X[j * P + c], s);
            X[i * P + c] -= s;
        }
    }
    __syncthreads();
    float* wout = a.w + (static_cast<int64_t>(chunk) * a.hv + h) * DC * D;
    float* uout = a.u + (static_cast<int64_t>(chunk) * a.hv + h) * DC * D;
    for (int idx = tid; idx < DC * D; idx += DELTA_THREADS) {
        const int i = idx / D, c = idx % D;
        wout[idx] = Qs[i * P + c];
        uout[idx] = Vs[i * P + c];
    }
    if (tid < DC) a.gam[(static_cast<int64_t>(chunk) * a.hv + h) * DC + tid] = gl[tid];
}

template <int D>
__global__ void __launch_bounds__(DELTA_THREADS) delta_state_kernel(DeltaArgs a) {
    constexpr int NV = STATE_NV;
    constexpr int P = D + 1;
    extern __shared__ float sm[];
    float* S = sm;                  // [NV][P]
    float* Ws = S + NV * P;         // [DC][P]
    float* Qs = Ws + DC * P;        // [DC][P]
    float* Ks = Qs + DC * P;        // [DC][P]
    float* Aq = Ks + DC * P;        // [DC][DC + 1]
    float* Dl = Aq + DC * (DC + 1); // [DC][NV + 1]  U, then Delta
    float* gm = Dl + DC * (NV + 1); // [DC]
    float* kd = gm + DC;            // [DC] e^{gamma_C - gamma_t}

    const int h = blockIdx.x, i0 = blockIdx.y * NV, hk = h / a.ratio;
    const int tid = threadIdx.x;
    for (int idx = tid; idx < NV * D; idx += DELTA_THREADS) {
        const int i = idx / D, c = idx % D;
        S[i * P + c] = a.state_in ? a.state_in[(static_cast<int64_t>(h) * D + i0 + i) * D + c] : 0.f;
    }
    const int ci = tid & 15;          // column of S^T / row of S owned in the Delta and O phase
    const int trow = tid >> 4;        // tokens trow + 16k
    const int si = tid >> 4;          // row of S owned in the update phase
    const int sc = tid & 15;          // columns sc + 16m

    for (int chunk = 0; chunk < a.nchunks; ++chunk) {
        const int t0 = chunk * DC;
        const int64_t ch = static_cast<int64_t>(chunk) * a.hv + h;
        const float* wsrc = a.w + ch * DC * D;
        for (int idx = tid; idx < DC * D; idx += DELTA_THREADS) {
            const int i = idx / D, c = idx % D, t = t0 + i;
            Ws[i * P + c] = wsrc[idx];
            float qq = 0.f, kq = 0.f;
            if (t < a.n) {
                const float* row = a.qkv + static_cast<int64_t>(t) * a.c_conv;
                qq = row[hk * D + c];
                kq = row[a.c_qk + hk * D + c];
            }
            Qs[i * P + c] = qq;
            Ks[i * P + c] = kq;
        }
        const float* asrc = a.aqk + ch * DC * DC;
        for (int idx = tid; idx < DC * DC; idx += DELTA_THREADS) Aq[(idx / DC) * (DC + 1) + idx % DC] = asrc[idx];
        const float* usrc = a.u + ch * DC * D;
        for (int idx = tid; idx < DC * NV; idx += DELTA_THREADS) {
            const int t = idx / NV, i = idx % NV;
            Dl[t * (NV + 1) + i] = usrc[t * D + i0 + i];
        }
        if (tid < DC) gm[tid] = a.gam[ch * DC + tid];
        __syncthreads();
        if (tid < DC) kd[tid] = expf(gm[DC - 1] - gm[tid]);

        // Delta = U - W S^T and O_inter = diag(e^gamma) Q S^T for column ci, tokens trow+16k
        float dw[4] = {}, dq[4] = {};
#pragma unroll 4
        for (int c = 0; c < D; ++c) {
            const float s = S[ci * P + c];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                dw[k] = fmaf(Ws[(trow + 16 * k) * P + c], s, dw[k]);
                dq[k] = fmaf(Qs[(trow + 16 * k) * P + c], s, dq[k]);
            }
        }
        float oacc[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int t = trow + 16 * k;
            Dl[t * (NV + 1) + ci] -= dw[k];
            oacc[k] = expf(gm[t]) * dq[k];
        }
        __syncthreads();
        // O += (M o Q K^T) Delta  (A_qk already masked and decayed)
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int t = trow + 16 * k;
            float s = oacc[k];
            for (int j = 0; j <= t; ++j) s = fmaf(Aq[t * (DC + 1) + j], Dl[j * (NV + 1) + ci], s);
            if (t0 + t < a.n) a.o[static_cast<int64_t>(t0 + t) * a.c_v + h * D + i0 + ci] = s;
        }
        // S <- e^{gamma_C} S + Delta^T diag(e^{gamma_C - gamma}) K for row si, columns sc+16m
        const float decay = expf(gm[DC - 1]);
        float sn[D / 16];
#pragma unroll
        for (int m = 0; m < D / 16; ++m) sn[m] = decay * S[si * P + sc + 16 * m];
        for (int t = 0; t < DC; ++t) {
            const float coef = Dl[t * (NV + 1) + si] * kd[t];
#pragma unroll
            for (int m = 0; m < D / 16; ++m) sn[m] = fmaf(coef, Ks[t * P + sc + 16 * m], sn[m]);
        }
        __syncthreads();
#pragma unroll
        for (int m = 0; m < D / 16; ++m) S[si * P + sc + 16 * m] = sn[m];
        __syncthreads();
    }
    for (int idx = tid; idx < NV * D; idx += DELTA_THREADS) {
        const int i = idx / D, c = idx % D;
        a.state_out[(static_cast<int64_t>(h) * D + i0 + i) * D + c] = S[i * P + c];
    }
}

size_t delta_scratch_bytes(int hv, int d, int64_t n) {
    const int64_t nch = (n + DC - 1) / DC;
    const int64_t per = static_cast<int64_t>(hv) * DC * (2 * d + DC + 1);
    return static_cast<size_t>(nch * per) * sizeof(float);
}

template <int D>
static cudaError_t launch_delta_d(DeltaArgs& a, cudaStream_t st) {
    constexpr int P = D + 1;
    const size_t prep_smem = (3 * DC * P + DC * (DC + 1) + 2 * DC) * sizeof(float);
    const size_t state_smem = (STATE_NV * P + 3 * DC * P + DC * (DC + 1) + DC * (STATE_NV + 1) + 2 * DC) * sizeof(float);
    static bool attr = false;
    if (!attr) {
        cudaFuncSetAttribute(delta_prep_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(prep_smem));
        cudaFuncSetAttribute(delta_state_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(state_smem));
        attr = true;
    }
    delta_prep_kernel<D><<<dim3(a.nchunks, a.hv), DELTA_THREADS, prep_smem, st>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    delta_state_kernel<D><<<dim3(a.hv, D / STATE_NV), DELTA_THREADS, state_smem, st>>>(a);
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
    a.w = base;
    a.u = a.w + nch * a.hv * DC * d;
    a.aqk = a.u + nch * a.hv * DC * d;
    a.gam = a.aqk + nch * a.hv * DC * DC;
    a.state_in = state_in;
    a.state_out = state_out;
    a.o = o;
    return d == 128 ? launch_delta_d<128>(a, st) : launch_delta_d<64>(a, st);
}

}  // namespace gdn
