// Step 1a: Q4_K superblocks -> int8 rows with one fp32 scale per row.
//
// sparkinfer PR #464 ("fused Q4K/Q6K->int8 dequant + token-parallel GDN conv
// ..."), Summary, "Fused Q4_K/Q6_K -> int8-row dequant": one block per weight
// row decodes the superblocks in registers and writes int8 + a per-row scale
// directly, with no bf16 scratch; the quantisation starts from the exact fp32
// decode (same page, Correctness paragraph).
//
// Layout of one 144-byte superblock (GGUF Q4_K): fp16 d, fp16 dmin, 12 bytes of
// 6-bit scales/mins, 128 bytes of 4-bit codes; sub-block j of 32 weights
// decodes as d*sc_j*q - dmin*m_j.  Weight 64p+l (l<32) is the low nibble of
// code byte 32p+l, weight 64p+32+l its high nibble.
//
// The row's codes are written as soon as its amax is known: HBM traffic is
// the 144 B / 256 weights read plus the codes written, nothing else.
#include "common.cuh"
#include "qk_decode.cuh"

namespace gdn {

static __device__ int g_q4k_error;   // index checks of the debug build

// One warp per weight row: in iteration i the warp decodes superblock i, lane
// l the 8 weights 8l .. 8l+7 (sub-block l/4, the low or high nibbles of 8 code
// bytes).  Pass 1 finds the row amax without decoding every weight: d*sc*q -
// dmin*m, rounded once, is monotonic in q, so the largest magnitude of a
// lane's 8 weights is at its smallest or largest 4-bit code (byte-wise SIMD
// min/max).  The amax is a warp reduction (no block barrier).  Pass 2 reloads
// the lane's 16-byte header and 8 code bytes (L1 hits), decodes, quantises and
// writes its 8 codes as one vector: consecutive lanes write consecutive bytes.
// Nothing is held across the passes, so the kernel runs at full occupancy, and
// no instruction converts between integer and float (byte permutes build the
// codes' floats and take the stored codes from the quantiser's magic floats).
// One launch covers two matrices (the rows of the second follow those of the
// first), so a layer's two weight matrices share one grid and one tail.
constexpr int DEQ_WARP_THREADS = 256;

template <typename OutT>
struct DeqJob {
    const uint8_t* blocks;
    int64_t rows;
    int cols;
    OutT* codes;
    float* scale;
};

template <typename OutT>
__global__ void __launch_bounds__(DEQ_WARP_THREADS, 4)
q4k_deq_rows_warp_kernel(DeqJob<OutT> j0, DeqJob<OutT> j1) {
    const int lane = threadIdx.x & 31;
    int64_t row = static_cast<int64_t>(blockIdx.x) * (DEQ_WARP_THREADS / 32) + (threadIdx.x >> 5);
    const bool second = row >= j0.rows;
    const DeqJob<OutT> j = second ? j1 : j0;
    if (second) row -= j0.rows;
    if (row >= j.rows) return;
    const int nsb = j.cols >> 8;
    const uint8_t* rb = j.blocks + row * static_cast<int64_t>(nsb) * 144;

    float amax = 0.0f;
#pragma unroll 8
    for (int i = 0; i < nsb; ++i) amax = fmaxf(amax, Q4KLane::amax(rb + i * 144, lane));
    amax = warp_max(amax);
    const QScale qsc = make_qscale(amax);
    if (lane == 0 && GDN_IN_RANGE(g_q4k_error, row < j.rows)) j.scale[row] = qsc.s;
    OutT* out = j.codes + row * static_cast<int64_t>(j.cols) + lane * 8;
#pragma unroll 4
    for (int i = 0; i < nsb; ++i) {
        float w[8], c[8];
        Q4KLane::decode(rb + i * 144, lane, w);
        quantise8(w, qsc, c);
        if (GDN_IN_RANGE(g_q4k_error, i * 256 + lane * 8 + 8 <= j.cols)) store_codes8<OutT>(out + i * 256, c);
    }
}

template <typename OutT>
static cudaError_t launch_deq(const DeqJob<OutT>& j0, const DeqJob<OutT>& j1, cudaStream_t st) {
    const int64_t wpb = DEQ_WARP_THREADS / 32;
    q4k_deq_rows_warp_kernel<OutT><<<static_cast<unsigned>((j0.rows + j1.rows + wpb - 1) / wpb), DEQ_WARP_THREADS, 0, st>>>(
        j0, j1);
    return cudaGetLastError();
}

cudaError_t launch_q4k_deq_i8(const void* blocks, int64_t rows, int64_t cols, int8_t* q, float* s,
                              cudaStream_t st) {
    const DeqJob<int8_t> j0{static_cast<const uint8_t*>(blocks), rows, static_cast<int>(cols), q, s};
    return launch_deq<int8_t>(j0, DeqJob<int8_t>{nullptr, 0, 256, nullptr, nullptr}, st);
}

cudaError_t launch_q4k_deq_codes(const void* blocks, int64_t rows, int64_t cols, uint16_t* q, float* s,
                                 cudaStream_t st) {
    const DeqJob<uint16_t> j0{static_cast<const uint8_t*>(blocks), rows, static_cast<int>(cols), q, s};
    return launch_deq<uint16_t>(j0, DeqJob<uint16_t>{nullptr, 0, 256, nullptr, nullptr}, st);
}

// Both weight matrices of a layer in one launch.
cudaError_t launch_q4k_deq_codes2(const void* b0, int64_t rows0, int64_t cols0, uint16_t* q0, float* s0,
                                  const void* b1, int64_t rows1, int64_t cols1, uint16_t* q1, float* s1,
                                  cudaStream_t st) {
    const DeqJob<uint16_t> j0{static_cast<const uint8_t*>(b0), rows0, static_cast<int>(cols0), q0, s0};
    const DeqJob<uint16_t> j1{static_cast<const uint8_t*>(b1), rows1, static_cast<int>(cols1), q1, s1};
    return launch_deq<uint16_t>(j0, j1, st);
}

int read_and_clear_q4k_error() {
    int v = 0, z = 0;
    cudaMemcpyFromSymbol(&v, g_q4k_error, sizeof(int));
    if (v) cudaMemcpyToSymbol(g_q4k_error, &z, sizeof(int));
    return v;
}

}  // namespace gdn
