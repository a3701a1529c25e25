// Step 2: token-parallel causal 4-tap depthwise conv + SiLU + per-head L2 norm,
// and the gates.
//
// sparkinfer PR #464 ("fused Q4K/Q6K->int8 dequant + token-parallel GDN conv
// ..."), Summary, "Token-parallel GDN conv": the causal 4-tap conv reads only
// the raw projected inputs, so every token is independent; the page runs one
// block per (token, head) with the taps, SiLU, L2 norm and conv-state layout
// of the sequential kernel it replaced.
//
// Here one warp owns one head (dk = dv = d channels, d/32 per lane) over a
// run of CONV_TOKENS consecutive tokens and keeps the last three raw inputs of
// its channels in registers, so each raw input is read from HBM once (plus a
// three-token halo per run).  The L2 norm of a q or k head is a warp
// reduction.  Inputs are the bf16 projection outputs; arithmetic is fp32 and
// the outputs are fp16 (rounded to nearest): the recurrence's tensor-core
// products take fp16 operands, so that kernel copies them into shared memory
// untouched.  fp16 keeps 11 significant bits, as tf32 does (bf16 keeps 8 and
// would move o by ~0.3%, which the int8 re-quantisation of the gated-norm
// output amplifies about threefold in y); its range ends at 65504, and a value
// beyond it is reported (ERR_RANGE in this unit's error word), never stored as
// infinity silently.
//
// Gates (when not drawn directly): log a = -exp(A_log) * softplus(alpha +
// dt_bias), b = sigmoid(beta), from the fp32 beta | alpha columns of the
// projection; computed by the extra blocks of the same launch.
#include "common.cuh"

namespace gdn {

static __device__ int g_conv_error;

constexpr int CONV_WARPS = 8;
constexpr int CONV_TOKENS = 16;

struct ConvArgs {
    const uint16_t* qkvz;
    int64_t ld_qkvz;
    int n;
    int c_qk;        // q channels (= k channels)
    int c_conv;
    int d;           // head dim (dk = dv)
    int n_heads;     // 2*Hk + Hv heads of d channels
    int n_qk_norm;   // heads 0 .. 2*Hk-1 are L2-normed
    int n_q;         // heads 0 .. Hk-1 are q (scaled)
    float eps;
    float q_scale;
    const float* conv_w;   // [c_conv][4]
    const float* tail;     // [n_seqs][c_conv][3]: per sequence, the raw inputs before its first token
    uint16_t* out;         // [n][c_conv] fp16
    // gates
    const float* ba;
    int64_t ld_ba;
    int hv;
    const float* A_log;
    const float* dt_bias;
    float* log_a;
    float* b;
    int conv_blocks_y;     // gridDim.y slices that run the conv; the rest run gates
};

// Tokens t0 .. t0+NT-1 (those below t1 are written) of one head, one warp,
// CPL channels per lane: xr holds the raw inputs of the tokens (packed bf16
// pairs), h0, h1, h2 the three raw inputs before t0.  The conv, SiLU, the L2
// norm of q and k heads (a warp reduction) and the fp16 store.
template <int CPL, int NT>
__device__ __forceinline__ void conv_head_tokens(const ConvArgs& a, int head, int t0, int t1,
                                                 const uint32_t (&xr)[NT][CPL / 2], float (&h0)[CPL], float (&h1)[CPL],
                                                 float (&h2)[CPL]) {
    const int lane = threadIdx.x & 31;
    const int c0 = head * a.d + lane * CPL;
    float4 w[CPL];
#pragma unroll
    for (int i = 0; i < CPL; ++i) w[i] = *reinterpret_cast<const float4*>(a.conv_w + static_cast<int64_t>(c0 + i) * 4);
    const bool norm = head < a.n_qk_norm;
    const float mul = head < a.n_q ? a.q_scale : 1.0f;
    // An L2-normed head has |y| <= |mul| whenever its sum of squares is finite,
    // so it is checked once per token (the sum, and mul once); every value of a
    // head that is not normed is checked.
    const bool mul_ok = fabsf(mul) <= 65504.0f;
    // Tokens in groups of G: the sums of squares of a group's tokens go through
    // the butterfly together, so their shuffles overlap (each token's sum is
    // formed in the same order as warp_sum's).
    constexpr int G = 4;
    static_assert(NT % G == 0, "token runs are whole groups");
#pragma unroll
    for (int k0 = 0; k0 < NT; k0 += G) {
        float y[G][CPL], ss[G];
#pragma unroll
        for (int g = 0; g < G; ++g) {
            ss[g] = 0.0f;
#pragma unroll
            for (int i = 0; i < CPL; ++i) {
                const uint32_t xw = xr[k0 + g][i >> 1];
                const float x = __uint_as_float((i & 1) ? (xw & 0xffff0000u) : (xw << 16));
                y[g][i] = conv4_silu(w[i], h0[i], h1[i], h2[i], x);
                ss[g] = fmaf(y[g][i], y[g][i], ss[g]);
                h0[i] = h1[i]; h1[i] = h2[i]; h2[i] = x;
            }
        }
        if (norm) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
                for (int g = 0; g < G; ++g) ss[g] += __shfl_xor_sync(0xffffffffu, ss[g], o);
            }
        }
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const int t = t0 + k0 + g;
            bool over;
            if (norm) {
                over = !(ss[g] <= 3.0e38f) || !mul_ok;
                const float r = rsqrtf(ss[g] + a.eps) * mul;
#pragma unroll
                for (int i = 0; i < CPL; ++i) y[g][i] *= r;
            } else {
                float m = 0.0f;
#pragma unroll
                for (int i = 0; i < CPL; ++i) m = fmaxf_nan(m, fabsf(y[g][i]));
                over = !(m <= 65504.0f);
            }
            if (t < t1 && GDN_IN_RANGE(g_conv_error, t < a.n && c0 + CPL <= a.c_conv)) {
                uint16_t* dst = a.out + static_cast<int64_t>(t) * a.c_conv + c0;
                if (over) atomicCAS(&g_conv_error, 0, ERR_RANGE);
                const uint32_t p0 = f16x2_bits(y[g][0], y[g][1 % CPL]);
                if (CPL == 4)
                    *reinterpret_cast<uint2*>(dst) = make_uint2(p0, f16x2_bits(y[g][2 % CPL], y[g][3 % CPL]));
                else
                    *reinterpret_cast<uint32_t*>(dst) = p0;
            }
        }
    }
}

// CPL raw inputs of a bf16 row at channel c0, as packed pairs.
template <int CPL>
__device__ __forceinline__ void load_raw(const uint16_t* src, uint32_t (&x)[CPL / 2]) {
    if (CPL == 4) {
        const uint2 u = __ldg(reinterpret_cast<const uint2*>(src));
        x[0] = u.x; x[1 % (CPL / 2)] = u.y;
    } else {
        x[0] = __ldg(reinterpret_cast<const uint32_t*>(src));
    }
}

// Tokens t0 .. t1-1 (at most CONV_TOKENS) of one head, of a sequence whose
// first token is ts and whose conv state is tail [c_conv][3].
template <int CPL>
__device__ __forceinline__ void conv_head_run(const ConvArgs& a, int head, int t0, int t1, int ts, const float* tail) {
    const int lane = threadIdx.x & 31;
    const int c0 = head * a.d + lane * CPL;
    float h0[CPL], h1[CPL], h2[CPL];  // x_{t-3}, x_{t-2}, x_{t-1}
    auto raw = [&](int t, int i) -> float {
        // raw input x_t of channel c0+i; a token before the sequence's first
        // reads its conv state (oldest first)
        if (t >= ts) return bf16_bits_to_float(a.qkvz[static_cast<int64_t>(t) * a.ld_qkvz + c0 + i]);
        if (!GDN_IN_RANGE(g_conv_error, t - ts >= -3 && c0 + i < a.c_conv)) return 0.0f;
        return tail[static_cast<int64_t>(c0 + i) * 3 + (3 + t - ts)];
    };
#pragma unroll
    for (int i = 0; i < CPL; ++i) {
        h0[i] = raw(t0 - 3, i);
        h1[i] = raw(t0 - 2, i);
        h2[i] = raw(t0 - 1, i);
    }
    // All CONV_TOKENS rows of the run are loaded (packed bf16 pairs) before the
    // first is used, so each warp keeps the whole run in flight.
    uint32_t xr[CONV_TOKENS][CPL / 2];
#pragma unroll
    for (int k = 0; k < CONV_TOKENS; ++k) {
        const int t = t0 + k;
        if (t < t1) {
            load_raw<CPL>(a.qkvz + static_cast<int64_t>(t) * a.ld_qkvz + c0, xr[k]);
        } else {
#pragma unroll
            for (int i = 0; i < CPL / 2; ++i) xr[k][i] = 0u;
        }
    }
    conv_head_tokens<CPL, CONV_TOKENS>(a, head, t0, t1, xr, h0, h1, h2);
}

// Block x: run blockIdx.x of the runs of CONV_TOKENS tokens that tile each
// sequence from its first token (sq: runs as units).
template <int CPL>
__global__ void __launch_bounds__(CONV_WARPS * 32, 3) conv_kernel(ConvArgs a, const __grid_constant__ SeqTable sq) {
    const int r = blockIdx.x, s = seq_of_unit(sq, r);
    const int ts = sq.tok[s];
    const int t0 = ts + (r - sq.unit[s]) * CONV_TOKENS;
    const int t1 = min(sq.tok[s + 1], t0 + CONV_TOKENS);
    if (static_cast<int>(blockIdx.y) < a.conv_blocks_y) {
        const int head = blockIdx.y * CONV_WARPS + (threadIdx.x >> 5);
        if (head < a.n_heads) conv_head_run<CPL>(a, head, t0, t1, ts, a.tail + static_cast<int64_t>(s) * a.c_conv * 3);
        return;
    }
    // gate block: tokens t0 .. t1-1, all value heads
    for (int i = threadIdx.x; i < (t1 - t0) * a.hv; i += blockDim.x) {
        const int t = t0 + i / a.hv, h = i % a.hv;
        const float beta = a.ba[static_cast<int64_t>(t) * a.ld_ba + h];
        const float alpha = a.ba[static_cast<int64_t>(t) * a.ld_ba + a.hv + h];
        if (GDN_IN_RANGE(g_conv_error, t < a.n))
            gate_values(beta, alpha, a.A_log[h], a.dt_bias[h], a.log_a[static_cast<int64_t>(t) * a.hv + h],
                        a.b[static_cast<int64_t>(t) * a.hv + h]);
    }
}

static ConvArgs conv_args(const gdn_layer& L, const uint16_t* qkvz, int64_t ld_qkvz, int64_t n, const float* tail,
                          const float* ba, int64_t ld_ba, uint16_t* out, float* log_a, float* b) {
    ConvArgs a;
    a.qkvz = qkvz;
    a.ld_qkvz = ld_qkvz;
    a.n = static_cast<int>(n);
    a.c_qk = L.n_qk_heads * L.dk;
    a.c_conv = 2 * a.c_qk + L.n_v_heads * L.dv;
    a.d = L.dk;
    a.n_heads = 2 * L.n_qk_heads + L.n_v_heads;
    a.n_qk_norm = 2 * L.n_qk_heads;
    a.n_q = L.n_qk_heads;
    a.eps = L.eps_l2;
    a.q_scale = L.q_scale;
    a.conv_w = L.conv_w;
    a.tail = tail;
    a.out = out;
    a.ba = ba;
    a.ld_ba = ld_ba;
    a.hv = L.n_v_heads;
    a.A_log = L.A_log;
    a.dt_bias = L.dt_bias;
    a.log_a = log_a;
    a.b = b;
    a.conv_blocks_y = (a.n_heads + CONV_WARPS - 1) / CONV_WARPS;
    return a;
}

// cu_seqlens: host token offsets [n_seqs + 1] of the call's sequences (null:
// one sequence of n tokens); tail then holds one conv state per sequence.
cudaError_t launch_conv(const gdn_layer& L, const uint16_t* qkvz, int64_t ld_qkvz, int64_t n, const float* tail,
                        const float* ba, int64_t ld_ba, uint16_t* out, float* log_a, float* b, cudaStream_t st,
                        const int64_t* cu_seqlens, int n_seqs) {
    const ConvArgs a = conv_args(L, qkvz, ld_qkvz, n, tail, ba, ld_ba, out, log_a, b);
    const bool gates = L.gate_log_a == nullptr;
    const SeqTable sq = cu_seqlens ? make_seq_table(cu_seqlens, n_seqs, CONV_TOKENS) : one_seq_table(n, CONV_TOKENS);
    if (sq.unit[sq.n] == 0) return cudaSuccess;
    dim3 grid(static_cast<unsigned>(sq.unit[sq.n]), static_cast<unsigned>(a.conv_blocks_y + (gates ? 1 : 0)));
    if (L.dk == 128)
        conv_kernel<4><<<grid, CONV_WARPS * 32, 0, st>>>(a, sq);
    else
        conv_kernel<2><<<grid, CONV_WARPS * 32, 0, st>>>(a, sq);
    return cudaGetLastError();
}

// conv_state of sequence blockIdx.y <- its last three raw inputs per channel
// (x_{N-3}, x_{N-2}, x_{N-1} of its N tokens), from the projection, or from the
// old state for N < 3 (an empty sequence keeps it).  One thread per channel
// reads its three old values before writing, so the update is in place.
__global__ void conv_state_kernel(const uint16_t* __restrict__ qkvz, int64_t ld, int c_conv, float* state,
                                  const __grid_constant__ SeqTable sq) {
    const int c = blockIdx.x * blockDim.x + threadIdx.x;
    if (c >= c_conv) return;
    const int s = blockIdx.y, ts = sq.tok[s], n = sq.tok[s + 1] - ts;
    if (!GDN_IN_RANGE(g_conv_error, s < sq.n)) return;
    float* st = state + static_cast<int64_t>(s) * c_conv * 3;
    float old[3] = {st[c * 3 + 0], st[c * 3 + 1], st[c * 3 + 2]};
    float nw[3];
#pragma unroll
    for (int j = 0; j < 3; ++j) {
        const int t = n - 3 + j;
        nw[j] = t >= 0 ? bf16_bits_to_float(qkvz[static_cast<int64_t>(ts + t) * ld + c]) : old[3 + t];
    }
#pragma unroll
    for (int j = 0; j < 3; ++j) st[c * 3 + j] = nw[j];
}

// cu_seqlens: as for launch_conv; state then holds one conv state per sequence.
cudaError_t launch_conv_state(const gdn_layer& L, const uint16_t* qkvz, int64_t ld, int64_t n, float* state,
                              cudaStream_t st, const int64_t* cu_seqlens, int n_seqs) {
    const int c_conv = 2 * L.n_qk_heads * L.dk + L.n_v_heads * L.dv;
    const SeqTable sq = cu_seqlens ? make_seq_table(cu_seqlens, n_seqs, 1) : one_seq_table(n, 1);
    conv_state_kernel<<<dim3((c_conv + 255) / 256, sq.n), 256, 0, st>>>(qkvz, ld, c_conv, state, sq);
    return cudaGetLastError();
}

// Conv-state snapshots of a prefill pass whose first token is number t0 of
// the prompt (t0 a multiple of 64): for every position p = k * every with t0 <
// p <= t0 + n (every a multiple of 64), snapshot k - 1 gets the raw inputs of
// tokens p-3, p-2, p-1 per channel, oldest first -- the conv state a prefill
// of the first p tokens leaves.  They lie in this pass (p - t0 >= 64).
__global__ void conv_ckpt_kernel(const uint16_t* __restrict__ qkvz, int64_t ld, int c_conv, int64_t t0, int64_t every,
                                 float* __restrict__ ckpt) {
    const int c = blockIdx.x * blockDim.x + threadIdx.x;
    if (c >= c_conv) return;
    const int64_t k = t0 / every + 1 + blockIdx.y, p = k * every;
    float* dst = ckpt + (k - 1) * c_conv * 3 + static_cast<int64_t>(c) * 3;
#pragma unroll
    for (int j = 0; j < 3; ++j) dst[j] = bf16_bits_to_float(qkvz[(p - 3 + j - t0) * ld + c]);
}

cudaError_t launch_conv_ckpt(const gdn_layer& L, const uint16_t* qkvz, int64_t ld, int64_t t0, int64_t n, int64_t every,
                             float* ckpt, cudaStream_t st) {
    const int c_conv = 2 * L.n_qk_heads * L.dk + L.n_v_heads * L.dv;
    const int64_t first = t0 / every + 1, last = (t0 + n) / every;   // snapshots k in [first, last]
    if (last < first) return cudaSuccess;
    conv_ckpt_kernel<<<dim3((c_conv + 255) / 256, static_cast<unsigned>(last - first + 1)), 256, 0, st>>>(
        qkvz, ld, c_conv, t0, every, ckpt);
    return cudaGetLastError();
}

int read_and_clear_conv_error() {
    int v = 0, z = 0;
    cudaMemcpyFromSymbol(&v, g_conv_error, sizeof(int));
    if (v) cudaMemcpyToSymbol(g_conv_error, &z, sizeof(int));
    return v;
}

}  // namespace gdn
