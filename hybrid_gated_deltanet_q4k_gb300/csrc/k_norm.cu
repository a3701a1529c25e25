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

namespace gdn {

constexpr int NORM_THREADS = 256;

// HPW heads per warp (Hv <= 8 HPW): the row's share of a thread lives in
// registers sized for exactly that many heads, which keeps the kernel small
// enough for 6 CTAs per SM and so enough loads in flight to cover HBM latency.
template <int CPL, bool QUANT, int HPW>
__global__ void __launch_bounds__(NORM_THREADS, HPW <= 4 ? 6 : 4)
gated_norm_kernel(const uint16_t* __restrict__ o, const uint16_t* __restrict__ z, int64_t ld_z, int hv,
                  const float* __restrict__ norm_w, float eps, uint16_t* __restrict__ codes,
                  float* __restrict__ scale, float* __restrict__ out_f32) {
    __shared__ float red[32];
    constexpr int D = CPL * 32;
    const int64_t t = blockIdx.x;
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

template <int CPL, bool QUANT>
static void launch_norm_hpw(const gdn_layer& L, const uint16_t* o, const uint16_t* z, int64_t ld_z, unsigned grid,
                            uint16_t* codes, float* scale, float* out_f32, cudaStream_t st) {
    const int hpw = (L.n_v_heads + 7) / 8;
    if (hpw <= 1)
        gated_norm_kernel<CPL, QUANT, 1><<<grid, NORM_THREADS, 0, st>>>(o, z, ld_z, L.n_v_heads, L.norm_w, L.eps_rms, codes, scale, out_f32);
    else if (hpw <= 2)
        gated_norm_kernel<CPL, QUANT, 2><<<grid, NORM_THREADS, 0, st>>>(o, z, ld_z, L.n_v_heads, L.norm_w, L.eps_rms, codes, scale, out_f32);
    else if (hpw <= 4)
        gated_norm_kernel<CPL, QUANT, 4><<<grid, NORM_THREADS, 0, st>>>(o, z, ld_z, L.n_v_heads, L.norm_w, L.eps_rms, codes, scale, out_f32);
    else
        gated_norm_kernel<CPL, QUANT, 8><<<grid, NORM_THREADS, 0, st>>>(o, z, ld_z, L.n_v_heads, L.norm_w, L.eps_rms, codes, scale, out_f32);
}

cudaError_t launch_gated_norm(const gdn_layer& L, const uint16_t* o, const uint16_t* z, int64_t ld_z, int64_t n,
                              uint16_t* codes, float* scale, float* out_f32, cudaStream_t st) {
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
