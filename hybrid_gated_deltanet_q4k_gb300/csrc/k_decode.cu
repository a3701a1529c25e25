// The decode step of the layer: one new token for each of B sequences, in
// five launches, each a programmatic dependent of the one before (it may be
// scheduled while that one runs; griddepcontrol.wait comes before anything it
// reads of that kernel's results):
//
// decode_pack_kernel -- the tokens' rows quantised once to int8 codes as the
//   prefill's step 1b does (scale s_x per token), packed four to a word with
//   the sums of every 16 codes; later the gated-norm output o_hat the same
//   way, after the RMS of each head.
//
// gemv_dot_kernel -- the projections for a few tokens.  Decoding a whole
//   weight matrix to int8 rows in HBM (step 1a of the prefill) would move 3.5x
//   the Q4_K bytes for one token, and re-quantising each weight costs more
//   instructions than reading it; a decode GEMV is bound by reading the
//   quantised weights once ("Qwen3.5 speed: prefill and decode parity with
//   llama.cpp" #5305, child ticket #5221: decode GEMV bandwidth against
//   llama.cpp's quantised GEMV, Q4_K and Q6_K).  So each weight sub-block
//   meets the tokens' codes as integers: for a Q4_K sub-block
//       sum_k w_k x_k = d*sc * sum q_k x_k - dmin*m * sum x_k,
//   for a Q6_K sub-block d*scale * (sum c_k x_k - 32 sum x_k), the integer
//   sums by dp4a on the packed 4-bit / 6-bit codes, the rest in fp32; the
//   token's total is then multiplied by s_x.  Weight tiles of 8 rows (one per
//   warp) arrive in shared memory by bulk copies through a ring of stages,
//   the first ones issued before the dependency wait, so each row is read
//   from HBM once with many bytes in flight.  Q4_K weights whose rows fit
//   shared memory beside 8 tokens' codes go to gemv_q4k_mma_kernel (below)
//   instead: the same sums on the fp16 tensor-core form.
//
// decode_mid_kernel -- per (value head, block of its state rows, sequence):
//   the conv, SiLU and L2 norms of the token's q, k, v, the gates, and one
//   token of the gated delta rule in fp32, the state read and written once:
//     S_i <- a S_i + b (v_i - a S_i.k) k^T,   o_i = S_i.q
//   for every row i (rows are independent).  One warp per row: each lane holds
//   D/32 consecutive entries; S_i.k, S_i.q and k.q are warp sums of the old
//   row, and o_i = a S_i.q + b (v_i - a S_i.k) (k.q) needs no second pass.
//   The pages measure this step per decode call (#5305, child ticket #5222:
//   the GDN recurrence at 44.7 us per call against llama.cpp's 2.5 us) and
//   name llama.cpp's form as prior art (a token loop with the state in
//   registers, "CRUX parity spike" #4220, technique table row 1).  It writes
//   the gated output o * norm_w * SiLU(z) and partial sums of o^2; the
//   output projection's kernel also shifts the conv tails (the readers of the
//   old tails are done).
#include "common.cuh"
#include "qk_decode.cuh"
#include "tma.cuh"

#include <mutex>

namespace gdn {

static __device__ int g_decode_error;

constexpr int GEMV_THREADS = 256;
constexpr int GEMV_WARPS = GEMV_THREADS / 32;          // = rows per tile: one row per warp
constexpr int GEMV_TOKENS = GDN_DECODE_GEMV_TOKENS;   // tokens per launch (codes in shared memory)
constexpr int GEMV_MAX_STAGES = 4;
constexpr int GEMV_SM_SMEM = 227 * 1024;              // shared memory of an SM for the CTAs it holds

struct GemvArgs {
    const uint8_t* blocks;   // [rows][cols/256] superblocks
    int rows, cols;
    int64_t row_bytes;       // cols/256 superblocks of the format's size
    int tile_rows;           // rows per tile: GEMV_WARPS, or 2 GEMV_WARPS for the one-token Q4_K form
    int ntiles, stages;      // tiles of tile_rows rows; shared-memory ring depth
    int64_t total_bytes;     // rows * row_bytes
    const uint16_t* xc;      // [g][cols] int8 codes as fp16 patterns
    const float* sx;         // [g]
    int g;                   // tokens of this launch, 1 .. GEMV_TOKENS
    uint16_t* out_bf16;      // out[t][r] for r < n_bf16, at t * ld_bf16 + r
    int64_t ld_bf16;
    int n_bf16;
    float* out_f32;          // r >= n_bf16: at t * ld_f32 + r - n_bf16
    int64_t ld_f32;
    // in_mode 0: xc holds the tokens' int8 codes as fp16 patterns; 1: xpack
    // holds them packed by decode_pack_kernel (per token stride_words words:
    // cols/4 words of 4 codes, then cols/16 sums of 16 codes).  sx: the scales.
    int in_mode;
    const uint32_t* xpack;
    int64_t xpack_stride;
    // optional (cs_state non-null): shift the conv tails of cs_n sequences by
    // one token, [x_{t-2}, x_{t-1}, x_t] from the raw projection row cs_qkvz
    float* cs_state;         // [cs_n][cs_c_conv][3]
    const uint16_t* cs_qkvz; // [cs_n][cs_ld] bf16
    int64_t cs_ld;
    int cs_c_conv, cs_n;
};

// Shared memory: the tokens' codes (g * cols bytes), their sums over blocks
// of 16 (g * cols/16 ints), then `stages` tiles of tile_rows weight rows,
// then one mbarrier per stage.  The one-token Q4_K form (mc) pads each
// superblock's 256 codes to 272 bytes and its 16 sums to 17 ints, so that 16
// lanes on 16 consecutive superblocks load from distinct banks at the same
// offset within a superblock.
__host__ __device__ inline int gemv_tile_rows(bool mc) { return mc ? 2 * GEMV_WARPS : GEMV_WARPS; }
__host__ __device__ inline int64_t gemv_tile_bytes(int64_t row_bytes, int tile_rows) { return tile_rows * row_bytes; }
__host__ __device__ inline int64_t gemv_xsum_offset(int g, int cols, bool mc) {
    const int64_t xs_bytes = mc ? cols + cols / 16 : static_cast<int64_t>(g) * cols;
    return (xs_bytes + 127) & ~127LL;
}
__host__ __device__ inline int64_t gemv_ring_offset(int g, int cols, bool mc) {
    const int64_t sums = mc ? cols / 16 + cols / 256 : static_cast<int64_t>(g) * (cols / 16);
    return (gemv_xsum_offset(g, cols, mc) + sums * 4 + 127) & ~127LL;
}
// ... then the barrier of the tokens' packed codes, per stage a count of the
// warps done with it, and an abort flag.
__host__ __device__ inline int64_t gemv_smem_bytes(int g, int cols, int64_t row_bytes, int stages, bool mc) {
    return gemv_ring_offset(g, cols, mc) + stages * gemv_tile_bytes(row_bytes, gemv_tile_rows(mc)) +
           8 * (GEMV_MAX_STAGES + 1) + 4 * GEMV_MAX_STAGES + 4;
}

// Copy tile `tile` into stage `s`: the whole bytes by one bulk copy (a tile
// starts on 16 bytes: 8 rows of 144 or 210 bytes per superblock are a multiple
// of 16), a ragged end of the last tile (< 16 bytes) by plain loads.  Thread 0.
__device__ __forceinline__ void gemv_issue(const GemvArgs& a, unsigned char* ring, uint64_t* full, int tile, int s) {
    if (tile >= a.ntiles) return;
    const int64_t tb = gemv_tile_bytes(a.row_bytes, a.tile_rows);
    const int64_t off = static_cast<int64_t>(tile) * tb;
    const int64_t bytes = (a.total_bytes - off) < tb ? (a.total_bytes - off) : tb;
    const int64_t b16 = bytes & ~15LL;
    unsigned char* dst = ring + s * tb;
    for (int64_t i = b16; i < bytes; ++i) dst[i] = a.blocks[off + i];
    mbar_expect_tx(full + s, static_cast<uint32_t>(b16));
    if (b16) bulk_load_1d(dst, a.blocks + off, static_cast<uint32_t>(b16), full + s);
}

// dot product of 4 unsigned bytes (a) with 4 signed bytes (b), plus c
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// One lane takes one 32-weight span of a superblock (a Q4_K sub-block; two
// 16-weight Q6_K sub-blocks): lane l of a warp step works on superblock
// step*4 + l/8, span l%8, so a warp covers 4 superblocks per step and each
// lane decodes its scales once per 32 weights.  Its codes come as 8 words of
// 4 packed bytes (weights 32j .. 32j+31 of the superblock, in order), and
//   sum_k w_k x_k = mul0 * dot(codes[0..15], x) + mul1 * dot(codes[16..31], x)
//                 + add0 * sum(x[0..15]) + add1 * sum(x[16..31]);
// for Q4_K one scale and one min cover the 32 weights (mul0 = mul1, add0 =
// add1), so the span takes a single dot product.
template <bool Q6>
__device__ __forceinline__ void span_codes(const uint8_t* blk, int j, uint32_t (&c)[8], float& mul0, float& mul1,
                                           float& add0, float& add1) {
    if constexpr (!Q6) {
        const uint4 hdr = *reinterpret_cast<const uint4*>(blk);
        const int k = j & 3;
        const uint32_t yk = __byte_perm(hdr.y, 0u, 0x4440 + k), zk = __byte_perm(hdr.z, 0u, 0x4440 + k);
        const uint32_t wk = __byte_perm(hdr.w, 0u, 0x4440 + k);
        const uint32_t sc = j < 4 ? (yk & 63u) : ((wk & 15u) | ((yk >> 2) & 0x30u));
        const uint32_t m = j < 4 ? (zk & 63u) : ((wk >> 4) | ((zk >> 2) & 0x30u));
        const float d = __half2float(__ushort_as_half(static_cast<uint16_t>(hdr.x & 0xffffu)));
        const float dmin = __half2float(__ushort_as_half(static_cast<uint16_t>(hdr.x >> 16)));
        const float ds = __fmul_rn(d, small_uint_to_float(sc)), dm = __fmul_rn(dmin, small_uint_to_float(m));
        // the span's codes in place: low nibbles (even j), or high nibbles
        // left at 16 q (odd j, their dot product 16 times too large: the
        // scale takes the 1/16, exactly)
        const uint4* q = reinterpret_cast<const uint4*>(blk + 16 + 32 * (j >> 1));
        const uint4 a = q[0], b = q[1];
        const uint32_t mask = (j & 1) ? 0xf0f0f0f0u : 0x0f0f0f0fu;
        c[0] = a.x & mask; c[1] = a.y & mask; c[2] = a.z & mask; c[3] = a.w & mask;
        c[4] = b.x & mask; c[5] = b.y & mask; c[6] = b.z & mask; c[7] = b.w & mask;
        mul0 = mul1 = (j & 1) ? __fmul_rn(ds, 0.0625f) : ds;
        add0 = add1 = -dm;
    } else {
        const int h = j >> 2, g = j & 3;
        const uint16_t* ql = reinterpret_cast<const uint16_t*>(blk + 64 * h + 32 * (g & 1));
        const uint16_t* qh = reinterpret_cast<const uint16_t*>(blk + 128 + 32 * h);
        const int nsh = 4 * (g >> 1), hsh = 2 * g;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const uint32_t lw = ql[2 * e] | (static_cast<uint32_t>(ql[2 * e + 1]) << 16);
            const uint32_t hw = qh[2 * e] | (static_cast<uint32_t>(qh[2 * e + 1]) << 16);
            c[e] = ((lw >> nsh) & 0x0f0f0f0fu) | (((hw >> hsh) & 0x03030303u) << 4);
        }
        const float d = __half2float(__ushort_as_half(*reinterpret_cast<const uint16_t*>(blk + 208)));
        const int8_t s0 = static_cast<int8_t>(blk[192 + 2 * j]), s1 = static_cast<int8_t>(blk[193 + 2 * j]);
        mul0 = __fmul_rn(d, static_cast<float>(s0));
        mul1 = __fmul_rn(d, static_cast<float>(s1));
        add0 = -32.0f * mul0;
        add1 = -32.0f * mul1;
    }
}

// The 6-bit scales and mins of a Q4_K superblock's 8 sub-blocks, one per
// byte: sl = sc[0..3], sh = sc[4..7], ml = m[0..3], mh = m[4..7] (sub-blocks
// 4..7 take their two high bits from the top bits of the bytes of 0..3).
__device__ __forceinline__ void q4k_unpack_scales(const uint4& h, uint32_t& sl, uint32_t& sh, uint32_t& ml,
                                                  uint32_t& mh) {
    sl = h.y & 0x3f3f3f3fu;
    ml = h.z & 0x3f3f3f3fu;
    sh = (h.w & 0x0f0f0f0fu) | ((h.y >> 2) & 0x30303030u);
    mh = ((h.w >> 4) & 0x0f0f0f0fu) | ((h.z >> 2) & 0x30303030u);
}

// One token's sums over two Q4_K rows in the fp32 operations of
// gemv_q4k_mma_kernel, so that a token decodes bit for bit the same alone as
// in a batch.  Per superblock i, the exact integer sums S = sum_j sc_j D_j and
// M = sum_j m_j X_j (D_j the sub-block's code-token dot product, X_j its token
// sum), then y_w = fma(-dmin, M, fma(d, S, y_w)) for the slice w = i mod 8,
// superblocks in increasing order; the eight slices are summed in order.  That
// kernel rounds the sum of S's two exact halves once, which is the conversion
// of the exact integer here.  Odd sub-blocks keep their codes at 16 q and even
// ones take 16 sc, so S arrives 16 times too large and d / 16 (exact) undoes
// it inside the same fma.
//
// The row at rb is summed in lanes 0-15, the row at rb + row_bytes in lanes
// 16-31, with the token's codes and sums in the padded layout (superblock i at
// 272 i bytes and 17 i ints).  Lane l of a half takes the whole superblocks l,
// l + 16, ...: their S and M by dp4a in one lane, with no shuffles; then slice
// w (lane w < 8) adds superblock w + 16 r (its own) and w + 8 + 16 r (from lane
// w + 8), in increasing order.  Every lane of a half returns its row's sum.
__device__ __forceinline__ float q4k_token_sum_mma_order(const uint8_t* rb, int64_t row_bytes, const uint32_t* xs,
                                                               const int* xsum, int nsb, int lane) {
    const int l = lane & 15, hb = lane & 16;
    const uint8_t* row = rb + (hb ? row_bytes : 0);
    float y = 0.0f;
    for (int r0 = 0; r0 < nsb; r0 += 16) {
        const int i = r0 + l;
        int S = 0, M = 0;
        float d16 = 0.0f, e = 0.0f;
        if (i < nsb) {
            const uint8_t* blk = row + i * 144;
            const uint4 hdr = *reinterpret_cast<const uint4*>(blk);
            uint32_t sl, sh, ml, mh;
            q4k_unpack_scales(hdr, sl, sh, ml, mh);
            const uint4* q = reinterpret_cast<const uint4*>(blk + 16);
            const uint4* xi = reinterpret_cast<const uint4*>(xs) + 17 * i;
            const int* si = xsum + 17 * i;
#pragma unroll
            for (int v = 0; v < 8; ++v) {
                // code bytes 16 v .. 16 v + 15: their low nibbles are weights 64 p + 16 qq
                // + (0..15), of sub-block 2 p (x unit 4 p + qq); the high nibbles weights
                // 64 p + 32 + 16 qq + (0..15), of sub-block 2 p + 1 (unit 4 p + 2 + qq)
                const int p = v >> 1, qq = v & 1, ul = 4 * p + qq, uh = 4 * p + 2 + qq;
                const uint4 c = q[v], xl = xi[ul], xh = xi[uh];
                int dl = dp4a_us(c.x & 0x0f0f0f0fu, xl.x, 0);
                dl = dp4a_us(c.y & 0x0f0f0f0fu, xl.y, dl);
                dl = dp4a_us(c.z & 0x0f0f0f0fu, xl.z, dl);
                dl = dp4a_us(c.w & 0x0f0f0f0fu, xl.w, dl);
                int dh = dp4a_us(c.x & 0xf0f0f0f0u, xh.x, 0);
                dh = dp4a_us(c.y & 0xf0f0f0f0u, xh.y, dh);
                dh = dp4a_us(c.z & 0xf0f0f0f0u, xh.z, dh);
                dh = dp4a_us(c.w & 0xf0f0f0f0u, xh.w, dh);
                const uint32_t sw = p < 2 ? sl : sh, mw = p < 2 ? ml : mh, k0 = (2 * p) & 3;
                const int sc0 = static_cast<int>(__byte_perm(sw, 0u, 0x4440u + k0));
                const int sc1 = static_cast<int>(__byte_perm(sw, 0u, 0x4441u + k0));
                const int m0 = static_cast<int>(__byte_perm(mw, 0u, 0x4440u + k0));
                const int m1 = static_cast<int>(__byte_perm(mw, 0u, 0x4441u + k0));
                // the even sub-block's codes count once and the odd one's 16 times: 16 sc D either way
                S += (sc0 << 4) * dl + sc1 * dh;
                M += m0 * si[ul] + m1 * si[uh];
            }
            d16 = __fmul_rn(__half2float(__ushort_as_half(static_cast<uint16_t>(hdr.x & 0xffffu))), 0.0625f);
            e = -__half2float(__ushort_as_half(static_cast<uint16_t>(hdr.x >> 16)));
        }
        const int src = hb + ((l + 8) & 15);
        const int S8 = __shfl_sync(0xffffffffu, S, src), M8 = __shfl_sync(0xffffffffu, M, src);
        const float d8 = __shfl_sync(0xffffffffu, d16, src), e8 = __shfl_sync(0xffffffffu, e, src);
        if (l < 8) {
            if (i < nsb) y = fmaf(e, static_cast<float>(M), fmaf(d16, static_cast<float>(S), y));
            if (i + 8 < nsb) y = fmaf(e8, static_cast<float>(M8), fmaf(d8, static_cast<float>(S8), y));
        }
    }
    float v = 0.0f;
#pragma unroll
    for (int w = 0; w < 8; ++w) v += __shfl_sync(0xffffffffu, y, hb + w);
    return v;
}

// One 16-code unit of a token's codes given as fp16 patterns of the integers
// (xc): the codes packed into 4 words of 4 int8, and their sum.
__device__ __forceinline__ void xc_unit(const uint16_t* src, uint4& w, int& sum) {
    const uint4 h0 = __ldg(reinterpret_cast<const uint4*>(src));
    const uint4 h1 = __ldg(reinterpret_cast<const uint4*>(src + 8));
    const uint32_t hw[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
    uint32_t pk[4];
    sum = 0;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const float2 f0 = __half22float2(*reinterpret_cast<const __half2*>(&hw[2 * q]));
        const float2 f1 = __half22float2(*reinterpret_cast<const __half2*>(&hw[2 * q + 1]));
        pk[q] = codes_to_i8x4(__fadd_rn(f0.x, QCODE_MAGIC), __fadd_rn(f0.y, QCODE_MAGIC), __fadd_rn(f1.x, QCODE_MAGIC),
                              __fadd_rn(f1.y, QCODE_MAGIC));
        sum = __dp4a(static_cast<int>(pk[q]), 0x01010101, sum);
    }
    w = make_uint4(pk[0], pk[1], pk[2], pk[3]);
}

// Bounded wait of one warp on a stage: gives up at once after any earlier
// wait of the CTA ran out.
__device__ __forceinline__ bool gemv_wait(uint64_t* bar, uint32_t parity, volatile int* abort) {
    if (*abort) return false;
    if (mbar_wait_bounded(bar, parity, &g_decode_error, ERR_WAIT_TIMEOUT)) return true;
    *abort = 1;
    return false;
}

// G: tokens the kernel computes (a power of two >= a.g; the codes of tokens
// a.g .. G-1 are zero and their sums are not stored).
// MC (Q4_K, one token): the sums in the fp32 operations of gemv_q4k_mma_kernel,
// two rows per warp (tiles of 2 GEMV_WARPS rows) and the token's codes padded.
template <bool Q6, int G, bool MC = false>
__global__ void __launch_bounds__(GEMV_THREADS, G <= 2 ? 4 : 2) gemv_dot_kernel(GemvArgs a) {
    static_assert(!MC || (!Q6 && G == 1), "the tensor-core order is for one token of Q4_K rows");
    constexpr int BYTES = Q6 ? 210 : 144;
    extern __shared__ __align__(128) unsigned char gsm[];
    uint32_t* xs = reinterpret_cast<uint32_t*>(gsm);                 // [G][cols / 4] packed int8
    int* xsum = reinterpret_cast<int*>(gsm + gemv_xsum_offset(G, a.cols, MC));   // [G][cols / 16] block sums
    unsigned char* ring = gsm + gemv_ring_offset(G, a.cols, MC);
    const int64_t tb = gemv_tile_bytes(a.row_bytes, a.tile_rows);
    uint64_t* full = reinterpret_cast<uint64_t*>(ring + a.stages * tb);
    uint64_t* xbar = full + GEMV_MAX_STAGES;                         // the packed codes (in_mode 1)
    int* done = reinterpret_cast<int*>(xbar + 1);                    // warps done with each stage
    volatile int* abort = reinterpret_cast<volatile int*>(done + GEMV_MAX_STAGES);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    if (tid == 0) {
        for (int i = 0; i < a.stages; ++i) {
            mbar_init_cta(full + i, 1);
            done[i] = 0;
        }
        mbar_init_cta(xbar, 1);
        *abort = 0;
        mbar_init_fence();
        for (int i = 0; i < a.stages; ++i) gemv_issue(a, ring, full, blockIdx.x + i * gridDim.x, i);
    }
    __shared__ float sxs[GEMV_TOKENS];
    // launched as a dependent of the previous kernel in the stream (programmatic
    // launch): the weight copies above read only the weights; everything the
    // previous kernels write (the inputs, the conv tails, the outputs' readers)
    // is touched only after that kernel has completed.  The next kernel may be
    // scheduled at once: it too waits for this one before it reads anything.
    pdl_trigger();
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int kw = a.cols >> 2, k16 = a.cols >> 4;
    if (!MC && a.in_mode == 1 && tid == 0) {
        // the tokens' packed codes and sums: two bulk copies per token
        const uint32_t bytes = static_cast<uint32_t>(a.cols + a.cols / 4);
        mbar_expect_tx(xbar, static_cast<uint32_t>(a.g) * bytes);
        for (int t = 0; t < a.g; ++t) {
            const uint32_t* src = a.xpack + t * a.xpack_stride;
            bulk_load_1d(xs + t * kw, src, static_cast<uint32_t>(a.cols), xbar);
            bulk_load_1d(xsum + t * k16, src + kw, static_cast<uint32_t>(a.cols / 4), xbar);
        }
    }
    if (tid < a.g) sxs[tid] = a.sx[tid];
    if (a.cs_state) {
        // conv tails move up by one token (the readers of the old tails have finished)
        const int64_t total = static_cast<int64_t>(a.cs_n) * a.cs_c_conv;
        for (int64_t i = static_cast<int64_t>(blockIdx.x) * GEMV_THREADS + tid; i < total;
             i += static_cast<int64_t>(gridDim.x) * GEMV_THREADS) {
            const int64_t sq = i / a.cs_c_conv, c = i - sq * a.cs_c_conv;
            float* t3 = a.cs_state + i * 3;
            const float x1 = t3[1], x2 = t3[2];
            t3[0] = x1;
            t3[1] = x2;
            t3[2] = bf16_bits_to_float(a.cs_qkvz[sq * a.cs_ld + c]);
        }
    }
    // tokens a.g .. G-1: zero codes (computed, not stored)
    for (int i = a.g * k16 + tid; i < G * k16; i += GEMV_THREADS) {
        const int t = i / k16, b = i - t * k16;
        *reinterpret_cast<uint4*>(xs + t * kw + 4 * b) = make_uint4(0u, 0u, 0u, 0u);
        xsum[i] = 0;
    }
    if constexpr (MC) {
        // one token: unit b of 16 codes (and its sum) to the padded place b + b / 16
        for (int b = tid; b < k16; b += GEMV_THREADS) {
            uint4 w;
            int sum;
            if (a.in_mode == 1) {
                w = __ldcg(reinterpret_cast<const uint4*>(a.xpack) + b);
                sum = __ldcg(reinterpret_cast<const int*>(a.xpack + kw) + b);
            } else {
                xc_unit(a.xc + 16 * b, w, sum);
            }
            reinterpret_cast<uint4*>(xs)[b + (b >> 4)] = w;
            xsum[b + (b >> 4)] = sum;
        }
    } else if (a.in_mode == 0) {
        for (int i = tid; i < a.g * k16; i += GEMV_THREADS) {
            const int t = i / k16, b = i - t * k16;
            uint4 w;
            xc_unit(a.xc + static_cast<int64_t>(t) * a.cols + 16 * b, w, xsum[i]);
            *reinterpret_cast<uint4*>(xs + t * kw + 4 * b) = w;
        }
    } else {
        gemv_wait(xbar, 0, abort);
    }
    __syncthreads();
    // Each warp takes its row of every tile the CTA walks, waiting on the
    // tile's stage by itself; the last warp done with a stage refills it with
    // the CTA's tile `stages` steps ahead (no CTA-wide barrier per tile).
    const int nsb = a.cols >> 8;
    const int j = lane & 7, sbl = lane >> 3;       // the lane's span and superblock within a step of 4
    int it = 0;
    for (int tile = blockIdx.x; tile < a.ntiles; tile += gridDim.x, ++it) {
        const int s = it % a.stages;
        if (!__all_sync(0xffffffffu, gemv_wait(full + s, (it / a.stages) & 1, abort))) break;
        const int wr = MC ? 2 * warp : warp;        // the warp's first row in the tile
        int row = tile * a.tile_rows + wr;
        if (row < a.rows) {
            const uint8_t* rb = ring + s * tb + static_cast<int64_t>(wr) * a.row_bytes;
            float mine = 0.0f;
            int t_out = lane;                          // the token whose sum this lane stores
            bool store = lane < a.g;
            if constexpr (MC) {
                mine = q4k_token_sum_mma_order(rb, a.row_bytes, xs, xsum, nsb, lane);
                row += lane >> 4;
                t_out = 0;
                store = (lane & 15) == 0 && row < a.rows;
            } else {
                float acc[G];
#pragma unroll
                for (int t = 0; t < G; ++t) acc[t] = 0.0f;
#pragma unroll 4
                for (int i = sbl; i < nsb; i += 4) {
                    uint32_t c[8];
                    float mul0, mul1, add0, add1;
                    span_codes<Q6>(rb + i * BYTES, j, c, mul0, mul1, add0, add1);
                    const int w0 = 64 * i + 8 * j;           // first x word of the span (256 i + 32 j bytes)
#pragma unroll
                    for (int t = 0; t < G; ++t) {
                        const uint4 xa = *reinterpret_cast<const uint4*>(xs + t * kw + w0);
                        const uint4 xb = *reinterpret_cast<const uint4*>(xs + t * kw + w0 + 4);
                        const int2 sx = *reinterpret_cast<const int2*>(xsum + t * k16 + 16 * i + 2 * j);
                        if constexpr (!Q6) {
                            // one scale for the 32 weights: one dot product
                            int d = dp4a_us(c[0], xa.x, 0);
                            d = dp4a_us(c[1], xa.y, d);
                            d = dp4a_us(c[2], xa.z, d);
                            d = dp4a_us(c[3], xa.w, d);
                            d = dp4a_us(c[4], xb.x, d);
                            d = dp4a_us(c[5], xb.y, d);
                            d = dp4a_us(c[6], xb.z, d);
                            d = dp4a_us(c[7], xb.w, d);
                            acc[t] = fmaf(mul0, static_cast<float>(d), fmaf(add0, static_cast<float>(sx.x + sx.y), acc[t]));
                        } else {
                            int d0 = dp4a_us(c[0], xa.x, 0);
                            d0 = dp4a_us(c[1], xa.y, d0);
                            d0 = dp4a_us(c[2], xa.z, d0);
                            d0 = dp4a_us(c[3], xa.w, d0);
                            int d1 = dp4a_us(c[4], xb.x, 0);
                            d1 = dp4a_us(c[5], xb.y, d1);
                            d1 = dp4a_us(c[6], xb.z, d1);
                            d1 = dp4a_us(c[7], xb.w, d1);
                            const float r = fmaf(mul0, static_cast<float>(d0), fmaf(add0, static_cast<float>(sx.x), acc[t]));
                            acc[t] = fmaf(mul1, static_cast<float>(d1), fmaf(add1, static_cast<float>(sx.y), r));
                        }
                    }
                }
#pragma unroll
                for (int t = 0; t < G; ++t) {
                    const float sum = warp_sum(acc[t]);
                    if (lane == t) mine = sum;
                }
            }
            if (store && GDN_IN_RANGE(g_decode_error, row < a.rows)) {
                const float y = mine * sxs[t_out];
                if (row < a.n_bf16)
                    a.out_bf16[t_out * a.ld_bf16 + row] = float_to_bf16_bits(y);
                else
                    a.out_f32[t_out * a.ld_f32 + (row - a.n_bf16)] = y;
            }
        }
        // this warp is done reading stage s (its loads have been consumed)
        __syncwarp();
        if (lane == 0) {
            __threadfence_block();
            if (atomicAdd(done + s, 1) == GEMV_WARPS - 1) {
                done[s] = 0;
                __threadfence_block();
                fence_proxy_async_smem();
                gemv_issue(a, ring, full, tile + a.stages * gridDim.x, s);
            }
        }
    }
    __syncthreads();
    if (*abort && tid == 0) {
        // a wait ran out: let copies already issued land (bounded) before the
        // shared memory is released
        for (int i = 0; i < a.stages; ++i)
            for (uint32_t par = 0; par < 2; ++par) mbar_wait_bounded(full + i, par, nullptr, 0, 20000000ull);
    }
}

template <bool Q6>
static void gemv_set_smem(int bytes) {
    cudaFuncSetAttribute(gemv_dot_kernel<Q6, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    cudaFuncSetAttribute(gemv_dot_kernel<Q6, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    cudaFuncSetAttribute(gemv_dot_kernel<Q6, 4>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    cudaFuncSetAttribute(gemv_dot_kernel<Q6, 8>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if constexpr (!Q6)
        cudaFuncSetAttribute(gemv_dot_kernel<false, 1, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

// A programmatic dependent launch: the CTAs may start while the previous
// kernel in the stream finishes (it signals when; see griddepcontrol in the
// kernel), so the weight copies start before the inputs exist.
template <bool Q6, int G, bool MC = false>
static cudaError_t gemv_launch_g(unsigned grid, size_t smem, cudaStream_t st, const GemvArgs& a) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(GEMV_THREADS, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute at;
    at.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, gemv_dot_kernel<Q6, G, MC>, a);
}

template <bool Q6>
static cudaError_t gemv_launch(int G, bool mc, unsigned grid, size_t smem, cudaStream_t st, const GemvArgs& a) {
    if constexpr (!Q6)
        if (G == 1 && mc) return gemv_launch_g<false, 1, true>(grid, smem, st, a);
    if (G == 1) return gemv_launch_g<Q6, 1>(grid, smem, st, a);
    if (G == 2) return gemv_launch_g<Q6, 2>(grid, smem, st, a);
    if (G == 4) return gemv_launch_g<Q6, 4>(grid, smem, st, a);
    return gemv_launch_g<Q6, 8>(grid, smem, st, a);
}

// gemv_q4k_mma_kernel -- the Q4_K projection with the per-sub-block dot
// products on the fp16 tensor-core form (mma.sync m16n8k16, fp32 sums): 16
// weight rows x 16 weights of a sub-block against 8 tokens' codes.  The same
// sum as gemv_dot_kernel,
//     sum_k w_k x_k = d*sc_j * sum_k q_k x_k - dmin*m_j * sum_k x_k,
// taken per superblock with every intermediate an exact integer:
//     y += d * (sum_j sum_k (sc_j q_k) x_k) - dmin * (sum_j sum_k m_j x_k).
// The A operand holds sc_j q_k (<= 63 * 15, exact in fp16: one fma on the
// fp16 pattern 1024 + q), or m_j repeated over the sub-block's positions; B
// holds the tokens' int8 codes as fp16 (exact).  Products are exact and the
// fp32 sums are integers, exact below 2^24 (a sub-block contributes at most
// 32 * 945 * 127 < 2^22, a superblock's min term < 2^21), so the superblock's
// two sums are, in practice, the exact integers.  Each token's result takes
// the same operations in the same order whatever the other tokens of the
// launch, so a batch gives each token's result bit for bit as that token
// alone.  (The int8 form of the instruction would take the codes as they are,
// but the int8 tensor rate of this part is far below its fp16 rate.)
//
// The contraction order within a sub-block is free: lane (g, q) of the
// instruction takes the weights and token codes 8q .. 8q+7 of the sub-block
// (its four fp16 pairs over the two k16 steps), which makes the weights one
// 8-byte load of consecutive Q4_K code bytes and the codes one 16-byte load.
//
// Work: tiles of 16 rows; the 8 warps of a CTA split a tile's superblocks
// (warp w takes superblocks w, w+8, ...) and their partial sums meet in
// shared memory in warp order.  Each tile's rows arrive by bulk copies (one
// per row, into rows padded to 32 mod 128 bytes so that the fragment loads
// are free of bank conflicts) through a ring of stages; the first stages are
// requested before the dependency wait.  Up to 16 tokens per launch (NT
// groups of 8), so the weights are read once for all of them.
constexpr int QM_WARPS = 8;
static_assert(QM_WARPS == 8, "q4k_token_sum_mma_order sums eight superblock slices, one per warp here");
constexpr int QM_THREADS = QM_WARPS * 32;
constexpr int QM_ROWS = 16;
constexpr int QM_MAX_STAGES = 6;
constexpr int QM_MAX_NT = 2;
constexpr int QM_CTAS_PER_SM = 1;

struct QmArgs {
    const uint8_t* blocks;   // [rows][cols/256] Q4_K superblocks
    int rows, cols;
    int64_t row_bytes;       // 144 * cols/256
    int row_stride;          // bytes of a row in a shared-memory stage
    int ntiles, stages;
    int in_mode;             // 0: xc fp16 patterns; 1: xpack (see GemvArgs)
    const uint16_t* xc;
    const uint32_t* xpack;
    int64_t xpack_stride;
    const float* sx;
    int g;                   // tokens of this launch, 1 .. 8 * NT
    uint16_t* out_bf16;
    int64_t ld_bf16;
    int n_bf16;
    float* out_f32;
    int64_t ld_f32;
    float* cs_state;
    const uint16_t* cs_qkvz;
    int64_t cs_ld;
    int cs_c_conv, cs_n;
};

// Shared memory: the tokens' codes as fp16 [8 NT][cols + 32] (rows 64 mod 128
// bytes apart: conflict-free 16-byte fragment loads), the warps' partial sums
// [QM_WARPS][NT][32 lanes] float4, the ring of stages [stages][16][row_stride],
// then one mbarrier per stage, the tokens' barrier and an abort flag.
__host__ __device__ inline int qm_row_stride(int64_t row_bytes) {
    const int rs = static_cast<int>((row_bytes + 15) & ~15LL);
    return rs + ((32 - rs % 128) + 128) % 128;
}
__host__ __device__ inline int64_t qm_x_stride(int cols) { return 2LL * cols + 64; }   // bytes
__host__ __device__ inline int64_t qm_red_offset(int nt, int cols) {
    return (8LL * nt * qm_x_stride(cols) + 127) & ~127LL;
}
__host__ __device__ inline int64_t qm_ring_offset(int nt, int cols) {
    return (qm_red_offset(nt, cols) + static_cast<int64_t>(QM_WARPS) * nt * 32 * 16 + 127) & ~127LL;
}
__host__ __device__ inline int64_t qm_smem_bytes(int nt, int cols, int64_t row_bytes, int stages) {
    return qm_ring_offset(nt, cols) + static_cast<int64_t>(stages) * QM_ROWS * qm_row_stride(row_bytes) +
           8 * (QM_MAX_STAGES + 1) + 4;
}

// Copy the valid rows of tile `tile` into stage `s`, one bulk copy per row
// (row_bytes is a multiple of 16: 144 bytes per superblock).  Thread 0.
__device__ __forceinline__ void qm_issue(const QmArgs& a, unsigned char* ring, uint64_t* full, int tile, int s) {
    if (tile >= a.ntiles) return;
    const int r0 = tile * QM_ROWS;
    const int nr = a.rows - r0 < QM_ROWS ? a.rows - r0 : QM_ROWS;
    mbar_expect_tx(full + s, static_cast<uint32_t>(nr * a.row_bytes));
    unsigned char* dst = ring + static_cast<int64_t>(s) * QM_ROWS * a.row_stride;
    for (int r = 0; r < nr; ++r)
        bulk_load_1d(dst + r * a.row_stride, a.blocks + static_cast<int64_t>(r0 + r) * a.row_bytes,
                     static_cast<uint32_t>(a.row_bytes), full + s);
}

// d += A (16 x 16 fp16) * B (16 x 8 fp16), fp32
__device__ __forceinline__ void mma_f16_m16n8k16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                                 uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t h2_bits(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ __half2 bits_h2(uint32_t b) { return *reinterpret_cast<__half2*>(&b); }

// Byte k of w (an integer < 1024) in both halves of an fp16 pair, exactly:
// the pattern 0x64nn is 1024 + nn.
__device__ __forceinline__ __half2 byte_h2(uint32_t w, int k) {
    const uint32_t m = __byte_perm(w, 0x64646464u, 0x4040u + 0x0101u * k);
    return __hsub2(bits_h2(m), __float2half2_rn(1024.0f));
}

// Bytes (0, 1) or (2, 3) of w as the fp16 pair (1024 + b0, 1024 + b1).
__device__ __forceinline__ uint32_t bytes_magic_h2(uint32_t w, int hi) {
    return __byte_perm(w, 0x64646464u, hi ? 0x7362u : 0x5140u);
}

template <int NT>
__global__ void __launch_bounds__(QM_THREADS, 1) gemv_q4k_mma_kernel(QmArgs a) {
    extern __shared__ __align__(128) unsigned char qsm[];
    unsigned char* xs = qsm;                                                      // [8 NT][cols + 32] fp16
    float4* red = reinterpret_cast<float4*>(qsm + qm_red_offset(NT, a.cols));     // [warps][NT][32]
    unsigned char* ring = qsm + qm_ring_offset(NT, a.cols);
    const int64_t tb = static_cast<int64_t>(QM_ROWS) * a.row_stride;
    uint64_t* full = reinterpret_cast<uint64_t*>(ring + a.stages * tb);
    uint64_t* xbar = full + QM_MAX_STAGES;
    volatile int* abort = reinterpret_cast<volatile int*>(xbar + 1);
    __shared__ float sxs[8 * QM_MAX_NT];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t xst = qm_x_stride(a.cols);

    if (tid == 0) {
        for (int i = 0; i < a.stages; ++i) mbar_init_cta(full + i, 1);
        mbar_init_cta(xbar, 1);
        *abort = 0;
        mbar_init_fence();
        for (int i = 0; i < a.stages; ++i) qm_issue(a, ring, full, blockIdx.x + i * gridDim.x, i);
    }
    // a programmatic dependent launch, as gemv_dot_kernel: only the weight
    // copies come before the wait
    pdl_trigger();
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (a.in_mode == 0 && tid == 0) {
        // fp16 patterns of the codes: one bulk copy per token
        mbar_expect_tx(xbar, static_cast<uint32_t>(a.g) * static_cast<uint32_t>(2 * a.cols));
        for (int t = 0; t < a.g; ++t)
            bulk_load_1d(xs + t * xst, a.xc + static_cast<int64_t>(t) * a.cols, static_cast<uint32_t>(2 * a.cols), xbar);
    }
    if (tid < a.g) sxs[tid] = a.sx[tid];
    if (a.cs_state) {
        const int64_t total = static_cast<int64_t>(a.cs_n) * a.cs_c_conv;
        for (int64_t i = static_cast<int64_t>(blockIdx.x) * QM_THREADS + tid; i < total;
             i += static_cast<int64_t>(gridDim.x) * QM_THREADS) {
            const int64_t sq = i / a.cs_c_conv, c = i - sq * a.cs_c_conv;
            float* t3 = a.cs_state + i * 3;
            const float x1 = t3[1], x2 = t3[2];
            t3[0] = x1;
            t3[1] = x2;
            t3[2] = bf16_bits_to_float(a.cs_qkvz[sq * a.cs_ld + c]);
        }
    }
    if (a.in_mode == 1) {
        // packed int8 codes to fp16: byte x + 128 under the pattern 0x64nn is
        // 1024 + x + 128, less 1152 exactly
        const int k16 = a.cols >> 4;
        const __half2 off = __float2half2_rn(1152.0f);
        for (int i = tid; i < a.g * k16; i += QM_THREADS) {
            const int t = i / k16, b = i - t * k16;
            const uint4 w = __ldg(reinterpret_cast<const uint4*>(a.xpack + t * a.xpack_stride + 4 * b));
            const uint32_t wv[4] = {w.x ^ 0x80808080u, w.y ^ 0x80808080u, w.z ^ 0x80808080u, w.w ^ 0x80808080u};
            uint32_t h[8];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                h[2 * e] = h2_bits(__hsub2(bits_h2(bytes_magic_h2(wv[e], 0)), off));
                h[2 * e + 1] = h2_bits(__hsub2(bits_h2(bytes_magic_h2(wv[e], 1)), off));
            }
            uint4* dst = reinterpret_cast<uint4*>(xs + t * xst + 32 * b);
            dst[0] = make_uint4(h[0], h[1], h[2], h[3]);
            dst[1] = make_uint4(h[4], h[5], h[6], h[7]);
        }
    }
    __syncthreads();
    if (a.in_mode == 0) gemv_wait(xbar, 0, abort);

    const int nsb = a.cols >> 8;
    const int gq = lane >> 2, q = lane & 3;
    const __half2 sixteenth = __float2half2_rn(0.0625f), m1024 = __float2half2_rn(-1024.0f);
    int it = 0;
    for (int tile = blockIdx.x; tile < a.ntiles; tile += gridDim.x, ++it) {
        const int s = it % a.stages;
        const bool ok = gemv_wait(full + s, (it / a.stages) & 1, abort);
        float y[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) y[nt][0] = y[nt][1] = y[nt][2] = y[nt][3] = 0.0f;
        if (ok) {
            const unsigned char* r0 = ring + s * tb + gq * a.row_stride;     // rows gq and gq + 8 of the tile
            const unsigned char* r1 = r0 + 8 * a.row_stride;
#pragma unroll 1
            for (int i = warp; i < nsb; i += QM_WARPS) {
                const unsigned char* p0 = r0 + i * 144;
                const unsigned char* p1 = r1 + i * 144;
                const uint4 h0 = *reinterpret_cast<const uint4*>(p0);
                const uint4 h1 = *reinterpret_cast<const uint4*>(p1);
                uint32_t sl0, sh0, ml0, mh0, sl1, sh1, ml1, mh1;
                q4k_unpack_scales(h0, sl0, sh0, ml0, mh0);
                q4k_unpack_scales(h1, sl1, sh1, ml1, mh1);
                // sums of sc_j q_k x_k and m_j x_k over the superblock, each
                // split over the two k16 steps of a sub-block (shorter chains)
                float sa[NT][4], sb[NT][4], ma[NT][4], mb[NT][4];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int c = 0; c < 4; ++c) sa[nt][c] = sb[nt][c] = ma[nt][c] = mb[nt][c] = 0.0f;
                const unsigned char* xb = xs + gq * xst + 16 * q + 512 * i;
#pragma unroll
                for (int p = 0; p < 4; ++p) {
                    // code bytes 32p + 8q .. +7 of both rows: sub-block 2p in
                    // the low nibbles, 2p + 1 in the high ones (as 16 q)
                    const uint2 c0 = *reinterpret_cast<const uint2*>(p0 + 16 + 32 * p + 8 * q);
                    const uint2 c1 = *reinterpret_cast<const uint2*>(p1 + 16 + 32 * p + 8 * q);
#pragma unroll
                    for (int hn = 0; hn < 2; ++hn) {
                        const int j = 2 * p + hn, k = j & 3;
                        const uint32_t msk = hn ? 0xf0f0f0f0u : 0x0f0f0f0fu;
                        __half2 s0 = byte_h2(j < 4 ? sl0 : sh0, k), s1 = byte_h2(j < 4 ? sl1 : sh1, k);
                        if (hn) {
                            s0 = __hmul2(s0, sixteenth);
                            s1 = __hmul2(s1, sixteenth);
                        }
                        const __half2 n0 = __hmul2(s0, m1024), n1 = __hmul2(s1, m1024);
                        // (1024 + q) s - 1024 s = q s, one rounding of an exact value
                        const uint32_t u0x = c0.x & msk, u0y = c0.y & msk, u1x = c1.x & msk, u1y = c1.y & msk;
                        const uint32_t a00 = h2_bits(__hfma2(bits_h2(bytes_magic_h2(u0x, 0)), s0, n0));
                        const uint32_t a02 = h2_bits(__hfma2(bits_h2(bytes_magic_h2(u0x, 1)), s0, n0));
                        const uint32_t a01 = h2_bits(__hfma2(bits_h2(bytes_magic_h2(u1x, 0)), s1, n1));
                        const uint32_t a03 = h2_bits(__hfma2(bits_h2(bytes_magic_h2(u1x, 1)), s1, n1));
                        const uint32_t a10 = h2_bits(__hfma2(bits_h2(bytes_magic_h2(u0y, 0)), s0, n0));
                        const uint32_t a12 = h2_bits(__hfma2(bits_h2(bytes_magic_h2(u0y, 1)), s0, n0));
                        const uint32_t a11 = h2_bits(__hfma2(bits_h2(bytes_magic_h2(u1y, 0)), s1, n1));
                        const uint32_t a13 = h2_bits(__hfma2(bits_h2(bytes_magic_h2(u1y, 1)), s1, n1));
                        const uint32_t m0 = h2_bits(byte_h2(j < 4 ? ml0 : mh0, k));
                        const uint32_t m1 = h2_bits(byte_h2(j < 4 ? ml1 : mh1, k));
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) {
                            const uint4 xv = *reinterpret_cast<const uint4*>(xb + nt * 8 * xst + 64 * j);
                            mma_f16_m16n8k16(sa[nt], a00, a01, a02, a03, xv.x, xv.y);
                            mma_f16_m16n8k16(sb[nt], a10, a11, a12, a13, xv.z, xv.w);
                            mma_f16_m16n8k16(ma[nt], m0, m1, m0, m1, xv.x, xv.y);
                            mma_f16_m16n8k16(mb[nt], m0, m1, m0, m1, xv.z, xv.w);
                        }
                    }
                }
                const float d0 = __half2float(__ushort_as_half(static_cast<uint16_t>(h0.x & 0xffffu)));
                const float e0 = -__half2float(__ushort_as_half(static_cast<uint16_t>(h0.x >> 16)));
                const float d1 = __half2float(__ushort_as_half(static_cast<uint16_t>(h1.x & 0xffffu)));
                const float e1 = -__half2float(__ushort_as_half(static_cast<uint16_t>(h1.x >> 16)));
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const float d = c < 2 ? d0 : d1, e = c < 2 ? e0 : e1;
                        y[nt][c] = fmaf(e, ma[nt][c] + mb[nt][c], fmaf(d, sa[nt][c] + sb[nt][c], y[nt][c]));
                    }
            }
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) red[(warp * NT + nt) * 32 + lane] = make_float4(y[nt][0], y[nt][1], y[nt][2], y[nt][3]);
        __syncthreads();   // every warp is done with stage s, and its partial sums are in place
        if (*abort) break;
        if (tid == 0) {
            fence_proxy_async_smem();
            qm_issue(a, ring, full, tile + a.stages * gridDim.x, s);
        }
        // output (row r, token t) sums the warps' partials in warp order;
        // lane (r % 8) * 4 + (t % 8) / 2 of each warp holds it in component
        // (r / 8) * 2 + t % 2 of its float4 for the token group t / 8
        const float* redf = reinterpret_cast<const float*>(red);
        for (int o = tid; o < QM_ROWS * 8 * NT; o += QM_THREADS) {
            const int r = o & (QM_ROWS - 1), t = o / QM_ROWS;
            const int row = tile * QM_ROWS + r;
            if (t < a.g && row < a.rows && GDN_IN_RANGE(g_decode_error, tile < a.ntiles)) {
                const int nt = t >> 3, tt = t & 7;
                const int li = (r & 7) * 4 + (tt >> 1), c = (r >> 3) * 2 + (tt & 1);
                float v = 0.0f;
#pragma unroll
                for (int w = 0; w < QM_WARPS; ++w) v += redf[((w * NT + nt) * 32 + li) * 4 + c];
                const float yv = v * sxs[t];
                if (row < a.n_bf16)
                    a.out_bf16[t * a.ld_bf16 + row] = float_to_bf16_bits(yv);
                else
                    a.out_f32[t * a.ld_f32 + (row - a.n_bf16)] = yv;
            }
        }
        __syncthreads();   // the partial sums are read
    }
    if (*abort && tid == 0) {
        // a wait ran out: let copies already issued land (bounded) before the
        // shared memory is released
        if (a.in_mode == 0) mbar_wait_bounded(xbar, 0, nullptr, 0, 20000000ull);
        for (int i = 0; i < a.stages; ++i)
            for (uint32_t par = 0; par < 2; ++par) mbar_wait_bounded(full + i, par, nullptr, 0, 20000000ull);
    }
}

template <int NT>
static cudaError_t qm_launch_nt(unsigned grid, size_t smem, cudaStream_t st, const QmArgs& a) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(QM_THREADS, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute at;
    at.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, gemv_q4k_mma_kernel<NT>, a);
}

// The Q4_K projection on gemv_q4k_mma_kernel: launches of up to 16 tokens
// (fewer when their codes and two stages would not fit shared memory),
// QM_CTAS_PER_SM CTAs per SM, as many stages as fit up to the tiles a CTA
// walks.  Only for rows where qm_fits holds.
// SM count and dynamic shared-memory budget of the tensor-core form, per device.
static int qm_sms[MAX_DEVICES] = {}, qm_budget[MAX_DEVICES] = {};
// The current device, its attributes set and figures queried (-1: none).
static int qm_init() {
    static PerDeviceOnce once;
    return once.run([](int dev) {
        int optin = 0;
        cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        cudaDeviceGetAttribute(&qm_sms[dev], cudaDevAttrMultiProcessorCount, dev);
        cudaFuncAttributes fa{};
        cudaFuncGetAttributes(&fa, gemv_q4k_mma_kernel<QM_MAX_NT>);
        const int stat = static_cast<int>(fa.sharedSizeBytes);
        const int per_cta = GEMV_SM_SMEM / QM_CTAS_PER_SM - 1024 - stat;
        qm_budget[dev] = optin - stat < per_cta ? optin - stat : per_cta;
        cudaFuncSetAttribute(gemv_q4k_mma_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, qm_budget[dev]);
        cudaFuncSetAttribute(gemv_q4k_mma_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, qm_budget[dev]);
    });
}

// Whether Q4_K rows of `cols` weights take the tensor-core form: 8 tokens'
// codes and two stages fit shared memory.
static bool qm_fits(int64_t cols) {
    const int dev = qm_init();
    return dev >= 0 && qm_smem_bytes(1, static_cast<int>(cols), (cols / 256) * 144, 2) <= qm_budget[dev];
}

static void launch_gemv_q4k_mma(const void* blocks, int64_t rows, int64_t cols, const uint16_t* xc,
                                const uint32_t* xpack, int64_t xpack_stride, const float* sx, int64_t n,
                                uint16_t* out_bf16, int64_t ld_bf16, int64_t n_bf16, float* out_f32, int64_t ld_f32,
                                cudaStream_t st, float* cs_state, const uint16_t* cs_qkvz, int64_t cs_ld,
                                int cs_c_conv, int cs_n, cudaError_t& err) {
    const int dev = qm_init();
    if (dev < 0) {
        err = cudaErrorInvalidDevice;
        return;
    }
    const int sms = qm_sms[dev], budget = qm_budget[dev];
    const int64_t row_bytes = (cols / 256) * 144;
    const int c = static_cast<int>(cols);
    int ntmax = QM_MAX_NT;
    while (ntmax > 1 && qm_smem_bytes(ntmax, c, row_bytes, 2) > budget) ntmax /= 2;
    const int ntiles = static_cast<int>((rows + QM_ROWS - 1) / QM_ROWS);
    const int ctas = QM_CTAS_PER_SM * sms;
    const unsigned grid = static_cast<unsigned>(ntiles < ctas ? ntiles : ctas);
    const int walk = (ntiles + static_cast<int>(grid) - 1) / static_cast<int>(grid);   // tiles of the busiest CTA
    err = cudaSuccess;
    for (int64_t t0 = 0; t0 < n; t0 += 8 * ntmax) {
        QmArgs a;
        a.blocks = static_cast<const uint8_t*>(blocks);
        a.rows = static_cast<int>(rows);
        a.cols = c;
        a.row_bytes = row_bytes;
        a.row_stride = qm_row_stride(row_bytes);
        a.ntiles = ntiles;
        a.in_mode = xpack ? 1 : 0;
        a.xc = xc ? xc + t0 * cols : nullptr;
        a.xpack = xpack ? xpack + t0 * xpack_stride : nullptr;
        a.xpack_stride = xpack_stride;
        a.sx = sx + t0;
        a.g = static_cast<int>(n - t0 < 8 * ntmax ? n - t0 : 8 * ntmax);
        a.out_bf16 = out_bf16 ? out_bf16 + t0 * ld_bf16 : nullptr;
        a.ld_bf16 = ld_bf16;
        a.n_bf16 = static_cast<int>(n_bf16);
        a.out_f32 = out_f32 ? out_f32 + t0 * ld_f32 : nullptr;
        a.ld_f32 = ld_f32;
        a.cs_state = t0 == 0 ? cs_state : nullptr;
        a.cs_qkvz = cs_qkvz;
        a.cs_ld = cs_ld;
        a.cs_c_conv = cs_c_conv;
        a.cs_n = cs_n;
        const int nt = a.g <= 8 ? 1 : 2;
        // no more stages than the busiest CTA has tiles: a small matrix
        // leaves the SMs' shared memory to the kernels beside it
        int stages = walk < QM_MAX_STAGES ? walk : QM_MAX_STAGES;
        while (stages > 1 && qm_smem_bytes(nt, c, row_bytes, stages) > budget) --stages;
        a.stages = stages;
        const size_t smem = static_cast<size_t>(qm_smem_bytes(nt, c, row_bytes, stages));
        err = nt == 1 ? qm_launch_nt<1>(grid, smem, st, a) : qm_launch_nt<2>(grid, smem, st, a);
        if (err == cudaSuccess) err = cudaGetLastError();
        if (err != cudaSuccess) return;
    }
}

// out[t][r] = s_x[t] * sum_k x[t][k] W[r][k] (W exactly decoded), for n tokens
// in launches of at most GEMV_TOKENS (fewer when a token's codes and the
// tiles would not fit shared memory); W in Q4_K (q6k false) or Q6_K.  The
// codes come as fp16 patterns xc [n][cols] or packed (xpack, stride
// xpack_stride words per token, written by launch_decode_pack); sx [n] the
// scales.  A persistent grid of up to four CTAs per SM walks the tiles.
// cs_state non-null: the first launch also shifts the conv tails of cs_n
// sequences (see GemvArgs).
cudaError_t launch_gemv_dot(const void* blocks, bool q6k, int64_t rows, int64_t cols, const uint16_t* xc,
                              const uint32_t* xpack, int64_t xpack_stride, const float* sx, int64_t n,
                              uint16_t* out_bf16, int64_t ld_bf16, int64_t n_bf16, float* out_f32, int64_t ld_f32,
                              cudaStream_t st, float* cs_state, const uint16_t* cs_qkvz, int64_t cs_ld, int cs_c_conv,
                              int cs_n) {
    // per device: SM count and the dynamic shared memory the kernels may take
    static int sms_of[MAX_DEVICES] = {}, optin_of[MAX_DEVICES] = {}, static_of[MAX_DEVICES] = {};
    static PerDeviceOnce once;
    const int dev = once.run([](int d) {
        int optin = 0;
        cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, d);
        // dynamic shared memory: the opt-in maximum less the kernels' static arrays
        cudaFuncAttributes fa{};
        cudaFuncGetAttributes(&fa, gemv_dot_kernel<true, 8>);
        static_of[d] = static_cast<int>(fa.sharedSizeBytes);
        optin -= static_of[d];
        gemv_set_smem<false>(optin);
        gemv_set_smem<true>(optin);
        optin_of[d] = optin;
        cudaDeviceGetAttribute(&sms_of[d], cudaDevAttrMultiProcessorCount, d);
    });
    if (dev < 0) return cudaErrorInvalidDevice;
    const int sms = sms_of[dev], max_optin = optin_of[dev], fa_static = static_of[dev];
    // Q4_K rows that fit the tensor-core form take it for several tokens; one
    // token takes the dp4a kernel in the same fp32 operations (a token's
    // result does not depend on the batch)
    const bool mma_q4k = !q6k && qm_fits(cols);
    if (mma_q4k && n > 1) {
        cudaError_t e = cudaSuccess;
        launch_gemv_q4k_mma(blocks, rows, cols, xc, xpack, xpack_stride, sx, n, out_bf16, ld_bf16, n_bf16, out_f32,
                            ld_f32, st, cs_state, cs_qkvz, cs_ld, cs_c_conv, cs_n, e);
        return e;
    }
    const int64_t row_bytes = (cols / 256) * (q6k ? 210 : 144);
    // tokens per launch (a power of two): what fits beside one stage
    int64_t gmax = GEMV_TOKENS;
    while (gmax > 1 && gemv_smem_bytes(static_cast<int>(gmax), static_cast<int>(cols), row_bytes, 1, false) > max_optin)
        gmax /= 2;
    // one Q4_K token (n == 1 here when mma_q4k): the tensor-core order, two rows per warp
    const bool mc = mma_q4k;
    if (gemv_smem_bytes(1, static_cast<int>(cols), row_bytes, 1, mc) > max_optin) return cudaErrorInvalidValue;
    const int tile_rows = gemv_tile_rows(mc);
    const int ntiles = static_cast<int>((rows + tile_rows - 1) / tile_rows);
    for (int64_t t0 = 0; t0 < n; t0 += gmax) {
        GemvArgs a;
        a.blocks = static_cast<const uint8_t*>(blocks);
        a.rows = static_cast<int>(rows);
        a.cols = static_cast<int>(cols);
        a.row_bytes = row_bytes;
        a.tile_rows = tile_rows;
        a.ntiles = ntiles;
        a.total_bytes = rows * row_bytes;
        a.xc = xc ? xc + t0 * cols : nullptr;
        a.xpack = xpack ? xpack + t0 * xpack_stride : nullptr;
        a.xpack_stride = xpack_stride;
        a.sx = sx + t0;
        a.in_mode = xpack ? 1 : 0;
        a.cs_state = t0 == 0 ? cs_state : nullptr;
        a.cs_qkvz = cs_qkvz;
        a.cs_ld = cs_ld;
        a.cs_c_conv = cs_c_conv;
        a.cs_n = cs_n;
        a.g = static_cast<int>(n - t0 < gmax ? n - t0 : gmax);
        a.out_bf16 = out_bf16 ? out_bf16 + t0 * ld_bf16 : nullptr;
        a.ld_bf16 = ld_bf16;
        a.n_bf16 = static_cast<int>(n_bf16);
        a.out_f32 = out_f32 ? out_f32 + t0 * ld_f32 : nullptr;
        a.ld_f32 = ld_f32;
        // tokens computed: a power of two >= g; CTAs per SM and ring depth:
        // the most CTAs (up to 4 at G <= 2, where registers allow them, else
        // 2) whose shared memory holds at least two stages each, then as many
        // stages as fit (one stage when nothing else fits)
        const int G = a.g <= 1 ? 1 : a.g <= 2 ? 2 : a.g <= 4 ? 4 : 8;
        int per_sm = G <= 2 ? 4 : 2, stages = 1;
        for (; per_sm >= 1; --per_sm) {
            const int64_t budget = GEMV_SM_SMEM / per_sm - 1024 - static_cast<int64_t>(fa_static);
            stages = GEMV_MAX_STAGES;
            while (stages > 1 && gemv_smem_bytes(G, a.cols, row_bytes, stages, mc) > budget) --stages;
            if (stages >= 2 || per_sm == 1) break;
        }
        if (per_sm < 1) per_sm = 1;
        a.stages = stages;
        const size_t smem = static_cast<size_t>(gemv_smem_bytes(G, a.cols, row_bytes, stages, mc));
        if (smem > static_cast<size_t>(max_optin)) return cudaErrorInvalidValue;
        const unsigned grid = static_cast<unsigned>(ntiles < per_sm * sms ? ntiles : per_sm * sms);
        cudaError_t e = q6k ? gemv_launch<true>(G, false, grid, smem, st, a) : gemv_launch<false>(G, mma_q4k, grid, smem, st, a);
        if (e == cudaSuccess) e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

// ------------------------------------------------------------ packed token rows

constexpr int PACK_THREADS = 256;

// Words per packed token row of `cols` codes (a multiple of 64, so every row
// starts on 16 bytes).
__host__ __device__ int64_t decode_pack_stride(int64_t cols) { return cols / 4 + cols / 16; }

// Elements off .. off+15 of a bf16 (f32 false) or fp32 row as floats, times sc.
__device__ __forceinline__ void pack_raw16(const void* src, bool f32, int64_t off, float sc, float (&w)[16]) {
    if (!f32) {
        const uint4* p = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(src) + off);
        const uint4 u0 = __ldg(p), u1 = __ldg(p + 1);
        const uint32_t u[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            w[2 * e] = __uint_as_float(u[e] << 16);
            w[2 * e + 1] = __uint_as_float(u[e] & 0xffff0000u);
        }
    } else {
        const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(src) + off);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float4 v = __ldg(p + e);
            w[4 * e] = v.x * sc; w[4 * e + 1] = v.y * sc; w[4 * e + 2] = v.z * sc; w[4 * e + 3] = v.w * sc;
        }
    }
}

// Token row t quantised once, by one CTA of PACK_THREADS threads, as the
// projection kernel takes it: scale amax/127 and the same codes as step 1b,
// written as cols/4 words of 4 int8 codes followed by cols/16 sums of 16
// codes (stride words per token), and the row's scale.  The row is bf16 (the
// decode input) or fp32 with head h multiplied first by rsqrt(sum_p
// psum[h][p] / d + eps) (the gated norm's RMS of o, from the partial sums of
// o^2 over the head's row blocks, added in order).  rh: hv floats, red:
// PACK_THREADS / 32 floats of shared memory.
__device__ void pack_row(const void* src, bool f32, int cols, const float* psum, int hv, int d, int split, float eps,
                         int t, uint32_t* pack, int64_t stride, float* scale, float* rh, float* red) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (psum) {
        for (int h = tid; h < hv; h += PACK_THREADS) {
            const float* ps = psum + (static_cast<int64_t>(t) * hv + h) * split;
            float sum = 0.0f;
            for (int p = 0; p < split; ++p) sum += ps[p];
            rh[h] = rsqrtf(sum / static_cast<float>(d) + eps);
        }
        __syncthreads();
    }
    const int k16 = cols >> 4;
    const int64_t row = static_cast<int64_t>(t) * cols;
    float amax = 0.0f;
    for (int b = tid; b < k16; b += PACK_THREADS) {
        float w[16];
        pack_raw16(src, f32, row + 16 * b, psum ? rh[(16 * b) / d] : 1.0f, w);
#pragma unroll
        for (int e = 0; e < 16; ++e) amax = fmaxf(amax, fabsf(w[e]));
    }
    amax = warp_max(amax);
    if (lane == 0) red[warp] = amax;
    __syncthreads();
    amax = red[0];
#pragma unroll
    for (int w = 1; w < PACK_THREADS / 32; ++w) amax = fmaxf(amax, red[w]);
    const QScale qsc = make_qscale(amax);
    if (tid == 0) scale[t] = qsc.s;
    uint32_t* words = pack + static_cast<int64_t>(t) * stride;
    int* sums = reinterpret_cast<int*>(words + (cols >> 2));
    for (int b = tid; b < k16; b += PACK_THREADS) {
        float w[16], c[16];
        pack_raw16(src, f32, row + 16 * b, psum ? rh[(16 * b) / d] : 1.0f, w);
        bool redo = !qsc.fast;
#pragma unroll
        for (int e = 0; e < 16; ++e) c[e] = qcode_fast(w[e], qsc, redo);
        if (redo) {
#pragma unroll
            for (int e = 0; e < 16; ++e) c[e] = qcode_exact(w[e], qsc.s);
        }
        uint32_t pk[4];
        int sum = 0;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            pk[q] = codes_to_i8x4(c[4 * q], c[4 * q + 1], c[4 * q + 2], c[4 * q + 3]);
            sum = __dp4a(static_cast<int>(pk[q]), 0x01010101, sum);
        }
        *reinterpret_cast<uint4*>(words + 4 * b) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        sums[b] = sum;
    }
}

// Rows packed one CTA per token (pack_row): bf16 x, or fp32 o_hat with
// psum / hv / d / split / eps for the RMS of each head.  A programmatic
// dependent: it lets the next kernel be scheduled, then waits for the
// previous one before it reads or writes anything.
__global__ void __launch_bounds__(PACK_THREADS) decode_pack_kernel(const void* src, int f32, int cols, const float* psum,
                                                                    int hv, int d, int split, float eps, uint32_t* pack,
                                                                    int64_t stride, float* scale) {
    pdl_trigger();
    asm volatile("griddepcontrol.wait;" ::: "memory");
    __shared__ float rh[64], red[PACK_THREADS / 32];
    pack_row(src, f32 != 0, cols, psum, hv, d, split, eps, blockIdx.x, pack, stride, scale, rh, red);
}

// n rows of src (bf16, or fp32 with psum / hv / d / split / eps for the RMS
// of each head) into pack [n][decode_pack_stride(cols)] and scale [n]; a
// programmatic dependent launch.
cudaError_t launch_decode_pack(const void* src, bool f32, int64_t n, int64_t cols, const float* psum, int hv, int d,
                               int split, float eps, uint32_t* pack, float* scale, cudaStream_t st) {
    if (cols % 256 != 0 || (psum && (hv > 64 || d < 16 || d % 16 != 0))) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(n), 1, 1);
    cfg.blockDim = dim3(PACK_THREADS, 1, 1);
    cfg.stream = st;
    cudaLaunchAttribute at;
    at.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, decode_pack_kernel, src, f32 ? 1 : 0, static_cast<int>(cols), psum, hv, d, split, eps,
                              pack, decode_pack_stride(cols), scale);
}

// ------------------------------------------------------------ conv, recurrence, gated norm

struct MidArgs {
    const uint16_t* qkvz;    // [B][ld] bf16 projection: q | k | v | z
    int64_t ld;
    const float* ba;         // [B][ld_ba] fp32 beta | alpha (gates from the projection)
    int64_t ld_ba;
    const float* gate_log_a; // [B][hv] drawn gates, or null
    const float* gate_b;
    const float* conv_w;     // [c_conv][4]
    const float* conv_state; // [B][c_conv][3], read only here
    const float* A_log;
    const float* dt_bias;
    const float* norm_w;     // [D]
    float* state;            // [B][hv][D][D], in place
    float* o_hat;            // [B][c_v] fp32 gated output, not yet RMS-normalised
    float* o_psum;           // [B][hv][MID_SPLIT] partial sums of o^2
    int hv, ratio, c_qk, c_conv, c_v;
    float eps_l2, eps_rms, q_scale;
};

constexpr int MID_THREADS = 256;
constexpr int MID_WARPS = MID_THREADS / 32;

// Block sum of one value per thread; every thread gets the total.
__device__ __forceinline__ float mid_block_sum(float v, float* red) {
    v = warp_sum(v);
    __syncthreads();
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    float r = 0.0f;
#pragma unroll
    for (int w = 0; w < MID_WARPS; ++w) r += red[w];
    return r;
}

// One CTA per (value head h, block of D / MID_SPLIT of its state rows,
// sequence): the conv of its key head's q and k channels and of its own v
// channels (SiLU, L2 norm of q and k, q scale), the gates, one token of the
// recurrence on its rows (a warp per row; S_i.k, S_i.q and k.q are warp sums
// of the old row, o_i = a S_i.q + u k.q with u = b (v_i - a S_i.k)), and the
// gated output o_i * norm_w_i * SiLU(z_i) with the block's partial sum of o^2
// (the RMS of the head is applied by the output projection, which adds the
// partial sums in order); everything in fp32.
constexpr int MID_SPLIT = 4;

template <int D>
__global__ void __launch_bounds__(MID_THREADS) decode_mid_kernel(MidArgs a) {
    constexpr int E = D / 32;                        // state entries per lane
    constexpr int NR = D / MID_SPLIT;                // rows of this CTA
    constexpr int R = NR / MID_WARPS;                // rows per warp
    __shared__ float qs[D], ks[D], vs[NR], gz[NR], red[MID_WARPS];
    __shared__ float gate[2];
    // a programmatic dependent of the input projection: the next kernel may be
    // scheduled at once; nothing is read before the projection has completed
    pdl_trigger();
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int h = blockIdx.x / MID_SPLIT, part = blockIdx.x % MID_SPLIT, sq = blockIdx.y, hk = h / a.ratio;
    const int i0 = part * NR;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint16_t* row = a.qkvz + static_cast<int64_t>(sq) * a.ld;
    const float* tail = a.conv_state + static_cast<int64_t>(sq) * a.c_conv * 3;
    // conv + SiLU: q and k of the key head (all D), v of this CTA's rows
    for (int i = tid; i < 2 * D + NR; i += MID_THREADS) {
        const int part2 = i < D ? 0 : (i < 2 * D ? 1 : 2);
        const int e = i - part2 * D;
        const int c = part2 == 0 ? hk * D + e : (part2 == 1 ? a.c_qk + hk * D + e : 2 * a.c_qk + h * D + i0 + e);
        const float4 w = *reinterpret_cast<const float4*>(a.conv_w + static_cast<int64_t>(c) * 4);
        const float y = conv4_silu(w, tail[c * 3 + 0], tail[c * 3 + 1], tail[c * 3 + 2], bf16_bits_to_float(row[c]));
        (part2 == 0 ? qs : (part2 == 1 ? ks : vs))[e] = y;
    }
    for (int e = tid; e < NR; e += MID_THREADS) {
        const float z = bf16_bits_to_float(row[a.c_conv + h * D + i0 + e]);
        gz[e] = silu_f(z) * a.norm_w[i0 + e];
    }
    if (tid == 0) {
        const int64_t gi = static_cast<int64_t>(sq) * a.hv + h;
        float la, b;
        if (a.gate_log_a) {
            la = a.gate_log_a[gi];
            b = a.gate_b[gi];
        } else {
            const float* bar = a.ba + static_cast<int64_t>(sq) * a.ld_ba;
            gate_values(bar[h], bar[a.hv + h], a.A_log[h], a.dt_bias[h], la, b);
        }
        gate[0] = expf(la);
        gate[1] = b;
    }
    __syncthreads();
    // L2 norms of q and k (q then scaled)
    float q2 = 0.0f, k2 = 0.0f;
    for (int e = tid; e < D; e += MID_THREADS) {
        q2 = fmaf(qs[e], qs[e], q2);
        k2 = fmaf(ks[e], ks[e], k2);
    }
    q2 = mid_block_sum(q2, red);
    k2 = mid_block_sum(k2, red);
    const float rq = rsqrtf(q2 + a.eps_l2) * a.q_scale, rk = rsqrtf(k2 + a.eps_l2);
    float q[E], k[E];
    float kq = 0.0f;
#pragma unroll
    for (int e = 0; e < E; ++e) {
        q[e] = qs[E * lane + e] * rq;
        k[e] = ks[E * lane + e] * rk;
        kq = fmaf(k[e], q[e], kq);
    }
    kq = warp_sum(kq);
    const float dec = gate[0], beta = gate[1];
    float* sbase = a.state + (static_cast<int64_t>(sq) * a.hv + h) * D * D + E * lane;
    float* ohat = a.o_hat + static_cast<int64_t>(sq) * a.c_v + h * D + i0;
    // the warp's rows i0 + warp + MID_WARPS * r, all loaded before the first is used
    float sr[R][E];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const float* sp = sbase + static_cast<int64_t>(i0 + warp + MID_WARPS * r) * D;
        if (E == 4) {
            const float4 v4 = *reinterpret_cast<const float4*>(sp);
            sr[r][0] = v4.x; sr[r][1 % E] = v4.y; sr[r][2 % E] = v4.z; sr[r][3 % E] = v4.w;
        } else {
            const float2 v2 = *reinterpret_cast<const float2*>(sp);
            sr[r][0] = v2.x; sr[r][1 % E] = v2.y;
        }
    }
    float o2 = 0.0f;   // lane 0: this warp's share of the sum of o^2
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const int il = warp + MID_WARPS * r;      // row within the CTA's block
        float* sp = sbase + static_cast<int64_t>(i0 + il) * D;
        float (&s)[E] = sr[r];
        float sk = 0.0f, sqv = 0.0f;
#pragma unroll
        for (int e = 0; e < E; ++e) {
            sk = fmaf(s[e], k[e], sk);
            sqv = fmaf(s[e], q[e], sqv);
        }
        sk = warp_sum(sk);
        sqv = warp_sum(sqv);
        const float u = beta * (vs[il] - dec * sk);   // b (v_i - a S_i.k)
#pragma unroll
        for (int e = 0; e < E; ++e) s[e] = fmaf(u, k[e], dec * s[e]);
        if (E == 4)
            *reinterpret_cast<float4*>(sp) = make_float4(s[0], s[1 % E], s[2 % E], s[3 % E]);
        else
            *reinterpret_cast<float2*>(sp) = make_float2(s[0], s[1 % E]);
        if (lane == 0) {
            const float o = fmaf(u, kq, dec * sqv);   // S_new . q
            o2 = fmaf(o, o, o2);
            ohat[il] = o * gz[il];
        }
    }
    o2 = mid_block_sum(lane == 0 ? o2 : 0.0f, red);
    if (tid == 0) a.o_psum[(static_cast<int64_t>(sq) * a.hv + h) * MID_SPLIT + part] = o2;
}

// o_hat *= rsqrt(mean o^2 + eps) per token and head, from the partial sums
// (the decode step's path for more tokens than one projection launch takes).
__global__ void decode_rms_apply_kernel(float* o_hat, const float* psum, int hv, int d, int c_v, float eps) {
    pdl_trigger();
    const int sq = blockIdx.y;
    for (int e = blockIdx.x * blockDim.x + threadIdx.x; e < c_v; e += gridDim.x * blockDim.x) {
        const int h = e / d;
        const float* ps = psum + (static_cast<int64_t>(sq) * hv + h) * MID_SPLIT;
        float sum = 0.0f;
        for (int p = 0; p < MID_SPLIT; ++p) sum += ps[p];
        o_hat[static_cast<int64_t>(sq) * c_v + e] *= rsqrtf(sum / static_cast<float>(d) + eps);
    }
}

cudaError_t launch_decode_rms_apply(const gdn_layer& L, float* o_hat, const float* psum, int64_t n_seqs, cudaStream_t st) {
    const int c_v = L.n_v_heads * L.dv;
    decode_rms_apply_kernel<<<dim3(static_cast<unsigned>((c_v + 255) / 256), static_cast<unsigned>(n_seqs)), 256, 0, st>>>(
        o_hat, psum, L.n_v_heads, L.dv, c_v, L.eps_rms);
    return cudaGetLastError();
}

cudaError_t launch_decode_mid(const gdn_layer& L, const uint16_t* qkvz, int64_t ld, const float* ba, int64_t ld_ba,
                              const float* conv_state, int64_t n_seqs, float* state, float* o_hat, float* o_psum,
                              cudaStream_t st) {
    MidArgs a;
    const int d = L.dk;
    a.qkvz = qkvz;
    a.ld = ld;
    a.ba = ba;
    a.ld_ba = ld_ba;
    a.gate_log_a = L.gate_log_a;
    a.gate_b = L.gate_b;
    a.conv_w = L.conv_w;
    a.conv_state = conv_state;
    a.A_log = L.A_log;
    a.dt_bias = L.dt_bias;
    a.norm_w = L.norm_w;
    a.state = state;
    a.o_hat = o_hat;
    a.o_psum = o_psum;
    a.hv = L.n_v_heads;
    a.ratio = L.n_v_heads / L.n_qk_heads;
    a.c_qk = L.n_qk_heads * d;
    a.c_v = L.n_v_heads * d;
    a.c_conv = 2 * a.c_qk + a.c_v;
    a.eps_l2 = L.eps_l2;
    a.eps_rms = L.eps_rms;
    a.q_scale = L.q_scale;
    // a programmatic dependent launch (the kernel waits for the projection first)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(a.hv * MID_SPLIT), static_cast<unsigned>(n_seqs), 1);
    cfg.blockDim = dim3(MID_THREADS, 1, 1);
    cfg.stream = st;
    cudaLaunchAttribute at;
    at.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &at;
    cfg.numAttrs = 1;
    const cudaError_t e = d == 128 ? cudaLaunchKernelEx(&cfg, decode_mid_kernel<128>, a)
                                   : cudaLaunchKernelEx(&cfg, decode_mid_kernel<64>, a);
    return e != cudaSuccess ? e : cudaGetLastError();
}

int read_and_clear_decode_error() {
    int v = 0, z = 0;
    cudaMemcpyFromSymbol(&v, g_decode_error, sizeof(int));
    if (v) cudaMemcpyToSymbol(g_decode_error, &z, sizeof(int));
    return v;
}

}  // namespace gdn
