// Step 1a for Q6_K weights: superblocks -> int8 rows with one fp32 scale per row.
//
// sparkinfer PR #464 ("fused Q4K/Q6K->int8 dequant + token-parallel GDN conv
// ..."), Summary, "Fused Q4_K/Q6_K -> int8-row dequant": the same fused
// decode-and-quantise as for Q4_K, for the Q6_K tensors that Q4_K_M files
// carry; the quantisation starts from the exact fp32 decode.
//
// Layout of one 210-byte superblock (GGUF Q6_K): ql[128] | qh[64] | int8
// scales[16] | fp16 d.  Weight v (half h = v / 128, group g = (v % 128) / 32,
// lane l = v % 32) has the 6-bit code c = low | high << 4 with low = nibble
// g / 2 of ql[64h + 32(g % 2) + l] and high = bits 2g, 2g+1 of qh[32h + l];
// it decodes to d * scales[v / 16] * (c - 32).  |d| has 11 significant bits,
// |scale| <= 128 and |c - 32| <= 32, so the product is exact in fp32 in any
// order of evaluation.
//
// One warp per weight row.  In iteration i the warp decodes superblock i,
// lane L the 8 consecutive weights 8L .. 8L+7: they share h, g and one scale,
// and their codes sit in 8 consecutive ql bytes (one nibble each) and 8
// consecutive qh bytes (one bit pair each).  Superblocks are only 2-byte
// aligned (210 = 2 * 105), so the lane reads 16-bit words.  Pass 1 finds the
// row amax from each lane's largest |c - 32| (one multiply per lane and
// superblock); pass 2 decodes, quantises with the row scale and writes the 8
// codes as one vector (int8: 8 bytes, fp16 carriers: 16 bytes).
#include "common.cuh"
#include "qk_decode.cuh"

namespace gdn {

static __device__ int g_q6k_error;   // index checks of the debug build

constexpr int Q6_THREADS = 256;
constexpr int Q6_BLOCK = 210;

template <typename OutT>
struct Q6Job {
    const uint8_t* blocks;
    int64_t rows;
    int cols;
    OutT* codes;
    float* scale;
};

template <typename OutT>
__global__ void __launch_bounds__(Q6_THREADS, 4) q6k_deq_rows_warp_kernel(Q6Job<OutT> j) {
    const int lane = threadIdx.x & 31;
    const int64_t row = static_cast<int64_t>(blockIdx.x) * (Q6_THREADS / 32) + (threadIdx.x >> 5);
    if (row >= j.rows) return;
    const int nsb = j.cols >> 8;
    const uint8_t* rb = j.blocks + row * static_cast<int64_t>(nsb) * Q6_BLOCK;

    float amax = 0.0f;
#pragma unroll 4
    for (int i = 0; i < nsb; ++i) amax = fmaxf(amax, Q6KLane::amax(rb + i * Q6_BLOCK, lane));
    amax = warp_max(amax);
    const QScale qsc = make_qscale(amax);
    if (lane == 0 && GDN_IN_RANGE(g_q6k_error, row < j.rows)) j.scale[row] = qsc.s;
    OutT* out = j.codes + row * static_cast<int64_t>(j.cols) + lane * 8;
#pragma unroll 4
    for (int i = 0; i < nsb; ++i) {
        float w[8], c[8];
        Q6KLane::decode(rb + i * Q6_BLOCK, lane, w);
        quantise8(w, qsc, c);
        if (GDN_IN_RANGE(g_q6k_error, i * 256 + lane * 8 + 8 <= j.cols)) store_codes8<OutT>(out + i * 256, c);
    }
}

template <typename OutT>
static cudaError_t launch_q6k(const void* blocks, int64_t rows, int64_t cols, OutT* q, float* s, cudaStream_t st) {
    const Q6Job<OutT> j{static_cast<const uint8_t*>(blocks), rows, static_cast<int>(cols), q, s};
    const int64_t wpb = Q6_THREADS / 32;
    q6k_deq_rows_warp_kernel<OutT><<<static_cast<unsigned>((rows + wpb - 1) / wpb), Q6_THREADS, 0, st>>>(j);
    return cudaGetLastError();
}

cudaError_t launch_q6k_deq_i8(const void* blocks, int64_t rows, int64_t cols, int8_t* q, float* s, cudaStream_t st) {
    return launch_q6k<int8_t>(blocks, rows, cols, q, s, st);
}

cudaError_t launch_q6k_deq_codes(const void* blocks, int64_t rows, int64_t cols, uint16_t* q, float* s,
                                 cudaStream_t st) {
    return launch_q6k<uint16_t>(blocks, rows, cols, q, s, st);
}

int read_and_clear_q6k_error() {
    int v = 0, z = 0;
    cudaMemcpyFromSymbol(&v, g_q6k_error, sizeof(int));
    if (v) cudaMemcpyToSymbol(g_q6k_error, &z, sizeof(int));
    return v;
}

}  // namespace gdn
