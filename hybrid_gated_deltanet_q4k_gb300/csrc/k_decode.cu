// The decode step of the layer: one new token for each of B sequences.
//
// Two kernels of its own, beside the prefill kernels it shares (activation
// quantisation, conv with one token per sequence, gated norm):
//
// gemv_codes_kernel -- the projections for a few tokens.  Decoding a whole
//   weight matrix to int8 codes in HBM (step 1a of the prefill) would move
//   3.5x the Q4_K bytes for one token; here each warp decodes one weight row
//   in registers (the same per-lane decode and quantiser as step 1a, so the
//   codes and the row scale are bit for bit the prefill's), and takes the
//   exact integer dot products with the tokens' int8 codes (dp4a, int32).
//   The epilogue ((float)acc * s_x) * s_w is the prefill GEMM's, so the
//   projections equal the prefill's bit for bit.  A decode GEMV is bound by
//   reading the quantised weights once ("Qwen3.5 speed: prefill and decode
//   parity with llama.cpp" #5305, child ticket #5221: decode GEMV bandwidth
//   against llama.cpp's quantised-activation GEMV, Q4_K and Q6_K).  Row pass 1 finds the amax (the row stays in L1), pass 2 decodes,
//   quantises and accumulates.  The tokens' codes sit in shared memory as
//   packed int8.
//
// decode_rule_kernel -- one token of the gated delta rule per sequence, in
//   fp32, the state read and written once:
//     S_i <- a S_i + b (v_i - a S_i.k) k^T,   o_i = S_i.q
//   for every row i of every value head (rows are independent).  One warp per
//   row: each lane holds D/32 consecutive entries; S_i.k, S_i.q and k.q are
//   warp sums of the old row, and o_i = a S_i.q + b (v_i - a S_i.k) (k.q)
//   needs no second pass.  The pages measure this step per decode call
//   (#5305, child ticket #5222: the GDN recurrence at 44.7 us per call against
//   llama.cpp's 2.5 us) and name llama.cpp's form as prior art (a token loop
//   with the state in registers, "CRUX parity spike" #4220, technique table
//   row 1).  o is written in fp16 (the gated norm's input
//   type); a value beyond its range sets ERR_RANGE.
#include "common.cuh"
#include "qk_decode.cuh"

namespace gdn {

static __device__ int g_decode_error;

constexpr int GEMV_THREADS = 256;
constexpr int GEMV_WARPS = GEMV_THREADS / 32;
constexpr int GEMV_TOKENS = GDN_DECODE_GEMV_TOKENS;   // tokens per launch (codes in shared memory)

struct GemvArgs {
    const uint8_t* blocks;   // [rows][cols/256] superblocks
    int rows, cols;
    const uint16_t* xc;      // [g][cols] int8 codes as fp16 patterns
    const float* sx;         // [g]
    int g;                   // tokens of this launch, 1 .. GEMV_TOKENS
    uint16_t* out_bf16;      // out[t][r] for r < n_bf16, at t * ld_bf16 + r
    int64_t ld_bf16;
    int n_bf16;
    float* out_f32;          // r >= n_bf16: at t * ld_f32 + r - n_bf16
    int64_t ld_f32;
};

__device__ __forceinline__ uint32_t pack_i8x4(float c0, float c1, float c2, float c3) {
    return (static_cast<uint32_t>(static_cast<int>(c0)) & 0xffu) | ((static_cast<uint32_t>(static_cast<int>(c1)) & 0xffu) << 8) |
           ((static_cast<uint32_t>(static_cast<int>(c2)) & 0xffu) << 16) | (static_cast<uint32_t>(static_cast<int>(c3)) << 24);
}

__device__ __forceinline__ int warp_sum_i(int v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

template <class Fmt>
__global__ void __launch_bounds__(GEMV_THREADS, 2) gemv_codes_kernel(GemvArgs a) {
    extern __shared__ __align__(16) uint32_t xs[];   // [g][cols / 4] packed int8
    const int kw = a.cols >> 2;
    for (int i = threadIdx.x; i < a.g * kw; i += GEMV_THREADS) {
        const int t = i / kw, k4 = i - t * kw;
        const uint2 h = __ldg(reinterpret_cast<const uint2*>(a.xc + static_cast<int64_t>(t) * a.cols + 4 * k4));
        const float2 f0 = __half22float2(*reinterpret_cast<const __half2*>(&h.x));
        const float2 f1 = __half22float2(*reinterpret_cast<const __half2*>(&h.y));
        xs[i] = pack_i8x4(f0.x, f0.y, f1.x, f1.y);
    }
    __syncthreads();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nsb = a.cols >> 8;
    for (int row = blockIdx.x * GEMV_WARPS + warp; row < a.rows; row += gridDim.x * GEMV_WARPS) {
        const uint8_t* rb = a.blocks + static_cast<int64_t>(row) * nsb * Fmt::BYTES;
        float amax = 0.0f;
#pragma unroll 4
        for (int i = 0; i < nsb; ++i) amax = fmaxf(amax, Fmt::amax(rb + i * Fmt::BYTES, lane));
        amax = warp_max(amax);
        const QScale qsc = make_qscale(amax);
        int acc[GEMV_TOKENS];
#pragma unroll
        for (int t = 0; t < GEMV_TOKENS; ++t) acc[t] = 0;
#pragma unroll 2
        for (int i = 0; i < nsb; ++i) {
            float w[8], c[8];
            Fmt::decode(rb + i * Fmt::BYTES, lane, w);
            quantise8(w, qsc, c);
            const int lo = static_cast<int>(pack_i8x4(c[0], c[1], c[2], c[3]));
            const int hi = static_cast<int>(pack_i8x4(c[4], c[5], c[6], c[7]));
            const uint32_t* xw = xs + 64 * i + 2 * lane;
#pragma unroll
            for (int t = 0; t < GEMV_TOKENS; ++t) {
                if (t < a.g) {
                    const uint2 xv = *reinterpret_cast<const uint2*>(xw + t * kw);
                    acc[t] = __dp4a(lo, static_cast<int>(xv.x), acc[t]);
                    acc[t] = __dp4a(hi, static_cast<int>(xv.y), acc[t]);
                }
            }
        }
        int mine = 0;
#pragma unroll
        for (int t = 0; t < GEMV_TOKENS; ++t) {
            if (t < a.g) {
                const int s = warp_sum_i(acc[t]);   // exact: |sum| <= 16384 * 127^2 < 2^31
                if (lane == t) mine = s;
            }
        }
        if (lane < a.g) {
            const float y = __fmul_rn(__fmul_rn(static_cast<float>(mine), a.sx[lane]), qsc.s);
            if (row < a.n_bf16)
                a.out_bf16[lane * a.ld_bf16 + row] = float_to_bf16_bits(y);
            else
                a.out_f32[lane * a.ld_f32 + (row - a.n_bf16)] = y;
        }
    }
}

// out = codes(x) . codes(W)^T rescaled, for n tokens in launches of at most
// GEMV_TOKENS; W in Q4_K (q6k false) or Q6_K.
cudaError_t launch_gemv_codes(const void* blocks, bool q6k, int64_t rows, int64_t cols, const uint16_t* xc,
                              const float* sx, int64_t n, uint16_t* out_bf16, int64_t ld_bf16, int64_t n_bf16,
                              float* out_f32, int64_t ld_f32, cudaStream_t st) {
    static int sms = 0;
    if (!sms) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        const int max_smem = GEMV_TOKENS * 16384;
        cudaFuncSetAttribute(gemv_codes_kernel<Q4KLane>, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
        cudaFuncSetAttribute(gemv_codes_kernel<Q6KLane>, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
    }
    const int64_t need_ctas = (rows + GEMV_WARPS - 1) / GEMV_WARPS;
    const unsigned grid = static_cast<unsigned>(need_ctas < 4LL * sms ? need_ctas : 4LL * sms);
    for (int64_t t0 = 0; t0 < n; t0 += GEMV_TOKENS) {
        GemvArgs a;
        a.blocks = static_cast<const uint8_t*>(blocks);
        a.rows = static_cast<int>(rows);
        a.cols = static_cast<int>(cols);
        a.xc = xc + t0 * cols;
        a.sx = sx + t0;
        a.g = static_cast<int>(n - t0 < GEMV_TOKENS ? n - t0 : GEMV_TOKENS);
        a.out_bf16 = out_bf16 ? out_bf16 + t0 * ld_bf16 : nullptr;
        a.ld_bf16 = ld_bf16;
        a.n_bf16 = static_cast<int>(n_bf16);
        a.out_f32 = out_f32 ? out_f32 + t0 * ld_f32 : nullptr;
        a.ld_f32 = ld_f32;
        const size_t smem = static_cast<size_t>(a.g) * cols;
        if (q6k)
            gemv_codes_kernel<Q6KLane><<<grid, GEMV_THREADS, smem, st>>>(a);
        else
            gemv_codes_kernel<Q4KLane><<<grid, GEMV_THREADS, smem, st>>>(a);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

// ------------------------------------------------------------ recurrence

struct DecodeArgs {
    const uint16_t* qkv;   // [B][c_conv] fp16: q | k | v
    const float* log_a;    // [B][hv]
    const float* b;        // [B][hv]
    float* state;          // [B][hv][D][D], in place
    uint16_t* o;           // [B][c_v] fp16
    int hv, ratio, c_qk, c_conv, c_v;
};

constexpr int DEC_WARPS = 8;

template <int D>
__global__ void __launch_bounds__(DEC_WARPS * 32) decode_rule_kernel(DecodeArgs a) {
    constexpr int E = D / 32;   // entries per lane
    const int lane = threadIdx.x & 31;
    const int gr = blockIdx.x * DEC_WARPS + (threadIdx.x >> 5);   // row of all heads: h * D + i
    const int sq = blockIdx.y;
    if (gr >= a.hv * D) return;
    const int h = gr / D, i = gr - h * D, hk = h / a.ratio;
    const uint16_t* tok = a.qkv + static_cast<int64_t>(sq) * a.c_conv;
    float q[E], k[E], s[E];
    {
        const uint16_t* qp = tok + hk * D + E * lane;
        const uint16_t* kp = tok + a.c_qk + hk * D + E * lane;
#pragma unroll
        for (int e = 0; e < E; e += 2) {
            const float2 qv = __half22float2(*reinterpret_cast<const __half2*>(qp + e));
            const float2 kv = __half22float2(*reinterpret_cast<const __half2*>(kp + e));
            q[e] = qv.x; q[e + 1] = qv.y;
            k[e] = kv.x; k[e + 1] = kv.y;
        }
    }
    float* sp = a.state + ((static_cast<int64_t>(sq) * a.hv + h) * D + i) * D + E * lane;
    if (E == 4) {
        const float4 v4 = *reinterpret_cast<const float4*>(sp);
        s[0] = v4.x; s[1 % E] = v4.y; s[2 % E] = v4.z; s[3 % E] = v4.w;
    } else {
        const float2 v2 = *reinterpret_cast<const float2*>(sp);
        s[0] = v2.x; s[1 % E] = v2.y;
    }
    float sk = 0.f, sq_ = 0.f, kq = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) {
        sk = fmaf(s[e], k[e], sk);
        sq_ = fmaf(s[e], q[e], sq_);
        kq = fmaf(k[e], q[e], kq);
    }
    sk = warp_sum(sk);
    sq_ = warp_sum(sq_);
    kq = warp_sum(kq);
    const int64_t gi = static_cast<int64_t>(sq) * a.hv + h;
    const float dec = expf(a.log_a[gi]), beta = a.b[gi];
    const float v = __half2float(__ushort_as_half(tok[2 * a.c_qk + h * D + i]));
    const float u = beta * (v - dec * sk);   // b (v_i - a S_i.k)
#pragma unroll
    for (int e = 0; e < E; ++e) s[e] = fmaf(u, k[e], dec * s[e]);
    if (E == 4)
        *reinterpret_cast<float4*>(sp) = make_float4(s[0], s[1 % E], s[2 % E], s[3 % E]);
    else
        *reinterpret_cast<float2*>(sp) = make_float2(s[0], s[1 % E]);
    if (lane == 0) {
        const float ov = fmaf(u, kq, dec * sq_);   // S_new . q
        if (!(fabsf(ov) <= 65504.0f)) atomicCAS(&g_decode_error, 0, ERR_RANGE);
        a.o[static_cast<int64_t>(sq) * a.c_v + h * D + i] = __half_as_ushort(__float2half_rn(ov));
    }
}

cudaError_t launch_decode_rule(const gdn_layer& L, const uint16_t* qkv, const float* log_a, const float* b,
                               int64_t n_seqs, float* state, uint16_t* o, cudaStream_t st) {
    DecodeArgs a;
    const int d = L.dk;
    a.qkv = qkv;
    a.log_a = log_a;
    a.b = b;
    a.state = state;
    a.o = o;
    a.hv = L.n_v_heads;
    a.ratio = L.n_v_heads / L.n_qk_heads;
    a.c_qk = L.n_qk_heads * d;
    a.c_v = L.n_v_heads * d;
    a.c_conv = 2 * a.c_qk + a.c_v;
    const dim3 grid(static_cast<unsigned>((a.hv * d + DEC_WARPS - 1) / DEC_WARPS), static_cast<unsigned>(n_seqs));
    if (d == 128)
        decode_rule_kernel<128><<<grid, DEC_WARPS * 32, 0, st>>>(a);
    else
        decode_rule_kernel<64><<<grid, DEC_WARPS * 32, 0, st>>>(a);
    return cudaGetLastError();
}

int read_and_clear_decode_error() {
    int v = 0, z = 0;
    cudaMemcpyFromSymbol(&v, g_decode_error, sizeof(int));
    if (v) cudaMemcpyToSymbol(g_decode_error, &z, sizeof(int));
    return v;
}

}  // namespace gdn
