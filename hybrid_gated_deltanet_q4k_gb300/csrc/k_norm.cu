// Step 4 (+ the quantisation of step 5's input): gated RMSNorm per value head,
//     o_hat = o / sqrt(mean(o^2) + eps) * norm_w * SiLU(z),
// then, for Q4_K layers, the token row of o_hat (all Hv*dv values) quantised
// to int8 codes with one fp32 scale (amax/127, IEEE fp32) for the output
// projection.  The pages list the "gated-norm" kernel among a GDN layer's
// kernels ("CRUX parity spike" #4220, technique table row 2); the int8 rows
// feed the same integer product as step 1.
//
// One CTA per token; warp w normalises heads w, w+8, ...; the row stays in
// registers between the per-head norms, the row amax and the quantisation, so
// o and z are read once and the codes written once.
#include "common.cuh"
#include "tma.cuh"

namespace gdn {

static __device__ int g_norm_error;

constexpr int NORM_THREADS = 256;

// HPW heads per warp (Hv <= 8 HPW): the row's share of a thread lives in
// registers sized for exactly that many heads, which keeps the kernel small
// enough for 6 CTAs per SM and so enough loads in flight to cover HBM latency.
template <int CPL, bool QUANT, int HPW>
__global__ void __launch_bounds__(NORM_THREADS, HPW <= 4 ? 6 : 4)
gated_norm_kernel(const uint16_t* __restrict__ o, const uint16_t* __restrict__ z, int64_t ld_z, int hv, int64_t n,
                  const float* __restrict__ norm_w, float eps, uint16_t* __restrict__ codes,
                  float* __restrict__ scale, float* __restrict__ out_f32) {
    __shared__ float red[32];
    constexpr int D = CPL * 32;
    const int64_t t = blockIdx.x;
    if (!GDN_IN_RANGE(g_norm_error, t < n)) return;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int c_v = hv * D;
    float wv[CPL];
#pragma unroll
    for (int i = 0; i < CPL; ++i) wv[i] = norm_w[lane * CPL + i];
    // All of the warp's loads first (o as fp16 pairs, z as bf16 pairs), then the math:
    // a warp keeps its whole share of the row in flight.
    float v[HPW][CPL];
    uint32_t zb[HPW][CPL / 2];
#pragma unroll
    for (int hh = 0; hh < HPW; ++hh) {
        const int h = warp + 8 * hh;
        if (h < hv) {
            const int c0 = h * D + lane * CPL;
            if (CPL == 4) {
                const uint2 f = __ldg(reinterpret_cast<const uint2*>(o + t * c_v + c0));
                const float2 f0 = __half22float2(*reinterpret_cast<const __half2*>(&f.x));
                const float2 f1 = __half22float2(*reinterpret_cast<const __half2*>(&f.y));
                v[hh][0] = f0.x; v[hh][1 % CPL] = f0.y; v[hh][2 % CPL] = f1.x; v[hh][3 % CPL] = f1.y;
                const uint2 u = __ldg(reinterpret_cast<const uint2*>(z + t * ld_z + c0));
                zb[hh][0] = u.x; zb[hh][1 % (CPL / 2)] = u.y;
            } else {
                const uint32_t f = __ldg(reinterpret_cast<const uint32_t*>(o + t * c_v + c0));
                const float2 f0 = __half22float2(*reinterpret_cast<const __half2*>(&f));
                v[hh][0] = f0.x; v[hh][1 % CPL] = f0.y;
                zb[hh][0] = __ldg(reinterpret_cast<const uint32_t*>(z + t * ld_z + c0));
            }
        }
    }
    float amax = 0.0f;
#pragma unroll
    for (int hh = 0; hh < HPW; ++hh) {
        const int h = warp + 8 * hh;
        if (h < hv) {
            const int c0 = h * D + lane * CPL;
            float ss = 0.0f;
#pragma unroll
            for (int i = 0; i < CPL; ++i) ss = fmaf(v[hh][i], v[hh][i], ss);
            ss = warp_sum(ss);
            const float r = rsqrtf(ss / static_cast<float>(D) + eps);
#pragma unroll
            for (int i = 0; i < CPL; ++i) {
                const uint32_t zw = zb[hh][i >> 1];
                const float zv = __uint_as_float((i & 1) ? (zw & 0xffff0000u) : (zw << 16));
                v[hh][i] = v[hh][i] * r * wv[i] * silu_f(zv);
                amax = fmaxf(amax, fabsf(v[hh][i]));
            }
            if (!QUANT) {
#pragma unroll
                for (int i = 0; i < CPL; ++i) out_f32[t * c_v + c0 + i] = v[hh][i];
            }
        }
    }
    if (!QUANT) return;
    amax = block_max(amax, red);
    const QScale qsc = make_qscale(amax);
    if (threadIdx.x == 0) scale[t] = qsc.s;
#pragma unroll
    for (int hh = 0; hh < HPW; ++hh) {
        const int h = warp + 8 * hh;
        if (h < hv) {
            const int c0 = h * D + lane * CPL;
            float c[CPL];
            bool redo = !qsc.fast;
#pragma unroll
            for (int i = 0; i < CPL; ++i) c[i] = qcode_fast(v[hh][i], qsc, redo);
            if (redo) {
#pragma unroll
                for (int i = 0; i < CPL; ++i) c[i] = qcode_exact(v[hh][i], qsc.s);
            }
            uint32_t w[CPL / 2];
#pragma unroll
            for (int i = 0; i < CPL / 2; ++i) w[i] = codes_to_f16x2(c[2 * i], c[2 * i + 1]);
            if (CPL == 4)
                *reinterpret_cast<uint2*>(codes + t * c_v + c0) = make_uint2(w[0], w[1 % (CPL / 2)]);
            else
                *reinterpret_cast<uint32_t*>(codes + t * c_v + c0) = w[0];
        }
    }
}

// ------------------------------------------------------------ staged variant
// Q4_K layers with dv = 128: persistent CTAs walk a strided set of tokens;
// each token's o row and z row (2 x 2 C_v bytes) arrive in one of NORM_STAGES
// shared-memory stages by bulk copies issued NORM_STAGES - 1 tokens ahead, so
// loads stay in flight while the CTA normalises, reduces and quantises the
// current token.  Same arithmetic as gated_norm_kernel, element for element.
// Two stages (32 KB at Hv = 32): more CTAs share an SM than with a
// four-stage ring (64 KB), which keeps more tokens in flight per SM than a
// deeper ring per CTA.
constexpr int NORM_STAGES = 2;

template <int HPW>
__global__ void __launch_bounds__(NORM_THREADS)
gated_norm_staged_kernel(const uint16_t* __restrict__ o, const uint16_t* __restrict__ z, int64_t ld_z, int hv, int64_t n, const float* __restrict__ norm_w, float eps, uint16_t* __restrict__ codes,
                         float* __restrict__ scale) {
    constexpr int CPL = 4, D = 128;
    extern __shared__ __align__(16) unsigned char smem[];
    __shared__ float red[32];
    __shared__ __align__(8) uint64_t full[NORM_STAGES];
    const int c_v = hv * D;
    const uint32_t row_bytes = static_cast<uint32_t>(c_v) * 2;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    auto stage_o = [&](int s) { return reinterpret_cast<const uint16_t*>(smem + static_cast<size_t>(s) * 2 * row_bytes); };
    auto stage_z = [&](int s) { return reinterpret_cast<const uint16_t*>(smem + static_cast<size_t>(s) * 2 * row_bytes + row_bytes); };
    auto issue = [&](int s, int64_t t) {
        mbar_expect_tx(&full[s], 2 * row_bytes);
        bulk_load_1d(smem + static_cast<size_t>(s) * 2 * row_bytes, o + t * c_v, row_bytes, &full[s]);
        bulk_load_1d(smem + static_cast<size_t>(s) * 2 * row_bytes + row_bytes, z + t * ld_z, row_bytes, &full[s]);
    };
    if (threadIdx.x == 0) {
        for (int s = 0; s < NORM_STAGES; ++s) mbar_init_cta(&full[s], 1);
        mbar_init_fence();
        for (int s = 0; s < NORM_STAGES; ++s) {
            const int64_t t = blockIdx.x + static_cast<int64_t>(s) * gridDim.x;
            if (t < n) issue(s, t);
        }
    }
    __syncthreads();
    float wv[CPL];
#pragma unroll
    for (int i = 0; i < CPL; ++i) wv[i] = norm_w[lane * CPL + i];
    bool ok = true;
    for (int64_t it = 0;; ++it) {
        const int64_t t = blockIdx.x + it * gridDim.x;
        if (t >= n) break;
        const int s = static_cast<int>(it % NORM_STAGES);
        const uint32_t par = static_cast<uint32_t>((it / NORM_STAGES) & 1);
        if (ok && !mbar_wait_bounded(&full[s], par, &g_norm_error, ERR_WAIT_TIMEOUT)) ok = false;
        const uint16_t* os = stage_o(s);
        const uint16_t* zs = stage_z(s);
        float v[HPW][CPL];
        float amax = 0.0f;
#pragma unroll
        for (int hh = 0; hh < HPW; ++hh) {
            const int h = warp + 8 * hh;
            if (h < hv) {
                const int c0 = h * D + lane * CPL;
                const uint2 f = *reinterpret_cast<const uint2*>(os + c0);
                const uint2 u = *reinterpret_cast<const uint2*>(zs + c0);
                const float2 f0 = __half22float2(*reinterpret_cast<const __half2*>(&f.x));
                const float2 f1 = __half22float2(*reinterpret_cast<const __half2*>(&f.y));
                v[hh][0] = f0.x; v[hh][1] = f0.y; v[hh][2] = f1.x; v[hh][3] = f1.y;
                const uint32_t zb[2] = {u.x, u.y};
                float ss = 0.0f;
#pragma unroll
                for (int i = 0; i < CPL; ++i) ss = fmaf(v[hh][i], v[hh][i], ss);
                ss = warp_sum(ss);
                const float r = rsqrtf(ss / static_cast<float>(D) + eps);
#pragma unroll
                for (int i = 0; i < CPL; ++i) {
                    const uint32_t zw = zb[i >> 1];
                    const float zv = __uint_as_float((i & 1) ? (zw & 0xffff0000u) : (zw << 16));
                    v[hh][i] = v[hh][i] * r * wv[i] * silu_f(zv);
                    amax = fmaxf(amax, fabsf(v[hh][i]));
                }
            }
        }
        amax = block_max(amax, red);   // also: every warp is done with stage s
        if (threadIdx.x == 0 && t + NORM_STAGES * static_cast<int64_t>(gridDim.x) < n && ok)
            issue(s, t + NORM_STAGES * static_cast<int64_t>(gridDim.x));
        const QScale qsc = make_qscale(amax);
        if (threadIdx.x == 0) scale[t] = qsc.s;
#pragma unroll
        for (int hh = 0; hh < HPW; ++hh) {
            const int h = warp + 8 * hh;
            if (h < hv) {
                const int c0 = h * D + lane * CPL;
                float c[CPL];
                bool redo = !qsc.fast;
#pragma unroll
                for (int i = 0; i < CPL; ++i) c[i] = qcode_fast(v[hh][i], qsc, redo);
                if (redo) {
#pragma unroll
                    for (int i = 0; i < CPL; ++i) c[i] = qcode_exact(v[hh][i], qsc.s);
                }
                *reinterpret_cast<uint2*>(codes + t * c_v + c0) =
                    make_uint2(codes_to_f16x2(c[0], c[1]), codes_to_f16x2(c[2], c[3]));
            }
        }
    }
    // Every copy issued was waited for above unless a wait ran out; then let
    // the copies still in flight land (bounded) before the CTA exits.
    if (!__syncthreads_and(ok) && threadIdx.x == 0) {
        const int64_t total = (n - blockIdx.x + gridDim.x - 1) / gridDim.x;   // tokens of this CTA
        for (int64_t it = total > NORM_STAGES ? total - NORM_STAGES : 0; it < total; ++it)
            mbar_wait_bounded(&full[it % NORM_STAGES], static_cast<uint32_t>((it / NORM_STAGES) & 1), nullptr, 0,
                              20000000ull);
    }
}

// Staged kernel: dv = 128, Q4_K, z rows 16-byte aligned.  Returns false when
// those do not hold (the caller launches gated_norm_kernel).
static bool launch_norm_staged(const gdn_layer& L, const uint16_t* o, const uint16_t* z, int64_t ld_z, int64_t n,
                               uint16_t* codes, float* scale, cudaStream_t st, cudaError_t* err) {
    if (L.dv != 128 || L.wtype != GDN_W_Q4K || ld_z % 8 || (reinterpret_cast<uintptr_t>(z) & 15) ||
        (reinterpret_cast<uintptr_t>(o) & 15))
        return false;
    const int hv = L.n_v_heads;
    const size_t smem = static_cast<size_t>(NORM_STAGES) * 4 * hv * 128;
    int dev = 0, sms = 1;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int hpw = (hv + 7) / 8;
    auto go = [&](auto kernel) {
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        int per_sm = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, NORM_THREADS, smem) != cudaSuccess || per_sm < 1)
            per_sm = 1;
        const int64_t want = static_cast<int64_t>(per_sm) * sms;
        const unsigned grid = static_cast<unsigned>(n < want ? n : want);
        kernel<<<grid, NORM_THREADS, smem, st>>>(o, z, ld_z, hv, n, L.norm_w, L.eps_rms, codes, scale);
        *err = cudaGetLastError();
    };
    if (hpw <= 1) go(gated_norm_staged_kernel<1>);
    else if (hpw <= 2) go(gated_norm_staged_kernel<2>);
    else if (hpw <= 4) go(gated_norm_staged_kernel<4>);
    else go(gated_norm_staged_kernel<8>);
    return true;
}

int read_and_clear_norm_error() {
    int v = 0, zr = 0;
    cudaMemcpyFromSymbol(&v, g_norm_error, sizeof(int));
    if (v) cudaMemcpyToSymbol(g_norm_error, &zr, sizeof(int));
    return v;
}

template <int CPL, bool QUANT>
static void launch_norm_hpw(const gdn_layer& L, const uint16_t* o, const uint16_t* z, int64_t ld_z, unsigned grid,
                            uint16_t* codes, float* scale, float* out_f32, cudaStream_t st) {
    const int64_t n = grid;
    const int hpw = (L.n_v_heads + 7) / 8;
    if (hpw <= 1)
        gated_norm_kernel<CPL, QUANT, 1><<<grid, NORM_THREADS, 0, st>>>(o, z, ld_z, L.n_v_heads, n, L.norm_w, L.eps_rms, codes, scale, out_f32);
    else if (hpw <= 2)
        gated_norm_kernel<CPL, QUANT, 2><<<grid, NORM_THREADS, 0, st>>>(o, z, ld_z, L.n_v_heads, n, L.norm_w, L.eps_rms, codes, scale, out_f32);
    else if (hpw <= 4)
        gated_norm_kernel<CPL, QUANT, 4><<<grid, NORM_THREADS, 0, st>>>(o, z, ld_z, L.n_v_heads, n, L.norm_w, L.eps_rms, codes, scale, out_f32);
    else
        gated_norm_kernel<CPL, QUANT, 8><<<grid, NORM_THREADS, 0, st>>>(o, z, ld_z, L.n_v_heads, n, L.norm_w, L.eps_rms, codes, scale, out_f32);
}

cudaError_t launch_gated_norm(const gdn_layer& L, const uint16_t* o, const uint16_t* z, int64_t ld_z, int64_t n,
                              uint16_t* codes, float* scale, float* out_f32, cudaStream_t st) {
    cudaError_t serr = cudaSuccess;
    if (launch_norm_staged(L, o, z, ld_z, n, codes, scale, st, &serr)) return serr;
    const bool quant = L.wtype == GDN_W_Q4K;
    const unsigned grid = static_cast<unsigned>(n);
    if (L.dv == 128) {
        if (quant)
            launch_norm_hpw<4, true>(L, o, z, ld_z, grid, codes, scale, out_f32, st);
        else
            launch_norm_hpw<4, false>(L, o, z, ld_z, grid, codes, scale, out_f32, st);
    } else {
        if (quant)
            launch_norm_hpw<2, true>(L, o, z, ld_z, grid, codes, scale, out_f32, st);
        else
            launch_norm_hpw<2, false>(L, o, z, ld_z, grid, codes, scale, out_f32, st);
    }
    return cudaGetLastError();
}

}  // namespace gdn
