// Causal grouped-query attention for the prefill of the hybrid model's
// full-attention layers, on the fifth-generation tensor cores.
//
// The pages' second prefill workload: "qwen35 batched prefill: flash attention
// for the full-attention layers" (#5305, sub-ticket #4442); at 32k tokens the
// prefill rate falls because those layers run "cuBLAS f32 with a materialised
// score matrix" ("CRUX parity spike" #4220, long-context finding 2), and the
// flash path the same page traces takes "f16 inputs, f32 accumulation".  Here
// the score matrix never leaves the SM: bf16 inputs, fp32 accumulation in
// TMEM, softmax in fp32.
//
// For query head h (key/value head h / (Hq/Hkv)) and query i at position
// p_i = nk - nq + i:  o_i = sum_{j <= p_i} softmax_j(scale q_i.k_j) v_j.
//
// One CTA per (tile of 128 queries, query head), the tiles with the most keys
// first.  Keys come in blocks of 128.  Per block j:
//   S_j = Q K_j^T            tcgen05.mma kind::f16 (bf16), M = 128, N = 128,
//                            K = D, A and B from shared memory, into TMEM
//   softmax warps            two threads per query row, 64 scores each from
//                            TMEM (once read, S_{j+1} may overwrite them),
//                            causal mask on diagonal blocks, the running
//                            maximum m (the halves swap their block maxima),
//                            P_j = 2^(s scale log2e - m) in bf16 back into
//                            TMEM (two buffers), l += sum P
//   O += P_j V_j             M = 128, K = 128, N = D, A (P) from TMEM, B (V^T)
//                            from shared memory, O accumulated in TMEM
// An M = 128, N = 128 instruction with both operands in shared memory reads
// about as many bytes per cycle as shared memory delivers, so shared-memory
// traffic (operand reads, TMA writes of K and V^T) bounds the kernel with the
// tensor math: P kept in TMEM takes its writes and the second product's A
// reads off shared memory.
// The maximum is raised only when a row's block maximum exceeds it by more
// than 2^8 (so P <= 256, fine for bf16); then the warp's O columns are scaled
// by 2^(m_old - m_new) in TMEM (tcgen05.ld / st) after the previous product
// has finished.  O / l at the end is the softmax exactly, whatever maxima were
// used.  V is read through its transpose V^T [Hkv][D][nk], written by a
// transpose kernel first, so the B operands of both products are K-major.
// Warps: 0 TMA for Q and K, 10 TMA for V^T (one block each at D = 256, two
// below), 1 TMEM owner and MMA issuer (it issues S_j and P_j V_j in whichever
// order they become ready), 2-9 softmax (warp w reads TMEM lanes 32 (w % 4)
// .. +31; warps 2-5 and 6-9 take the two halves of those rows).  Every wait is
// bounded; after a wait runs out the CTA stops issuing, lets its copies and
// products finish and returns with an error word set (GDN_ETIMEOUT).
#include "common.cuh"
#include "tma.cuh"
#include "tcgen05.cuh"

#include <mutex>

namespace gdn {

static __device__ int g_attn_error;

constexpr int ATT_BM = 128;   // queries per CTA
constexpr int ATT_BN = 128;   // keys per block
constexpr int ATT_SM_WARPS = 8;   // softmax warps: two per row quadrant, each half of a row's scores
constexpr int ATT_THREADS = 96 + 32 * ATT_SM_WARPS;
constexpr int ATT_VWARP = 2 + ATT_SM_WARPS;
constexpr float ATT_RESCALE_LOG2 = 8.0f;   // raise the maximum only past this margin

// Shared memory.  K and V^T hold one key block each at D = 256 (no room for
// two), two at smaller D.  P lives in TMEM, not here.
template <int D>
struct AttSmem {
    static constexpr int NS = D / 64;                    // 64-element slabs of a row
    static constexpr int ST = D == 256 ? 1 : 2;          // key blocks held at once
    static constexpr int Q0 = 0;                         // Q: NS slabs of [128 rows][64] bf16 (16 KB)
    static constexpr int QSLAB = ATT_BM * 128;
    static constexpr int K0 = Q0 + NS * QSLAB;           // K: ST blocks x NS slabs of [128 keys][64] (16 KB)
    static constexpr int KSLAB = ATT_BN * 128;
    static constexpr int KSTAGE = NS * KSLAB;
    static constexpr int V0 = K0 + ST * KSTAGE;          // V^T: ST blocks x 2 slabs of [D rows][64 keys]
    static constexpr int VSLAB = D * 128;
    static constexpr int VSTAGE = 2 * VSLAB;
    static constexpr int B0 = V0 + ST * VSTAGE;          // mbarriers
    // barrier indices: Q full; K and V^T full / empty per block slot; S full;
    // S consumed (the softmax has read it); P full and P V done per P buffer
    static constexpr int QF = 0, KF = 1, KE = 3, VF = 5, VE = 7, SF = 9, SC = 10, PF = 11, PV = 13, FIN = 15,
                         NBAR = 16;
    static constexpr int X0 = (B0 + 8 * NBAR + 15) & ~15;    // row maxima: [2 rounds][2 halves][128] fp32
    static constexpr int LS0 = X0 + 4 * ATT_BM * 4;          // row sums of each half: [2][128] fp32
    static constexpr int MISC0 = LS0 + 2 * ATT_BM * 4;       // TMEM base, abort flag
    static constexpr int BYTES = MISC0 + 16;
};

static_assert(AttSmem<256>::BYTES + 1024 <= 227 * 1024, "d = 256 tiles must fit the shared memory of a CTA");

struct AttArgs {
    int nq, nk, hq, hkv, ratio;
    float sl2;          // scale * log2(e)
    uint16_t* o;        // [nq][hq][D] bf16
    int ntiles;         // query tiles of ATT_BM
};

// Bounded wait that gives up at once after any earlier wait of the CTA ran out.
__device__ __forceinline__ bool att_wait(uint64_t* bar, uint32_t parity, volatile int* abort) {
    if (*abort) return false;
    if (mbar_wait_bounded(bar, parity, &g_attn_error, ERR_WAIT_TIMEOUT)) return true;
    *abort = 1;
    return false;
}

__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t bf16x2_bits(float lo, float hi) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
}

// Non-blocking test of a phase (the MMA issuer polls two kinds of work and
// must not be suspended on one while the other is ready).
__device__ __forceinline__ bool att_ready(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ void att_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

template <int D>
__global__ void __launch_bounds__(ATT_THREADS, 1)
attn_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
            const __grid_constant__ CUtensorMap mv, AttArgs a) {
    using L = AttSmem<D>;
    constexpr int ST = L::ST;
    extern __shared__ __align__(1024) unsigned char smb[];
    unsigned char* base = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smb) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(base + L::B0);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(base + L::MISC0);
    volatile int* abort = reinterpret_cast<volatile int*>(base + L::MISC0 + 4);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    // the tiles with the most keys first
    const int tile = a.ntiles - 1 - static_cast<int>(blockIdx.x) / a.hq;
    const int h = static_cast<int>(blockIdx.x) % a.hq, g = h / a.ratio;
    const int q0 = tile * ATT_BM, off = a.nk - a.nq;
    const int last_pos = off + min(q0 + ATT_BM, a.nq) - 1;   // the tile's largest query position
    const int nb = last_pos / ATT_BN + 1;                     // key blocks it needs

    if (tid == 0) {
        for (int i = 0; i < L::NBAR; ++i)
            mbar_init_cta(bars + i, (i == L::SC || i == L::PF || i == L::PF + 1) ? 32 * ATT_SM_WARPS : 1);
        mbar_init_fence();
        *abort = 0;
    }
    if (warp == 1) t5::alloc(tslot, 512);
    t5::fence_before();
    __syncthreads();
    t5::fence_after();
    const uint32_t tmem = *tslot;
    const uint32_t sbase = smem_addr(base);
    // TMEM columns: S 0-127 (fp32), P_j 128 + 64 (j & 1) .. +63 (bf16 pairs), O from 256
    constexpr uint32_t PCOL = ATT_BN, OCOL = 2 * ATT_BN;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA: Q, K
        if (lane == 0) {
            mbar_expect_tx(bars + L::QF, L::NS * L::QSLAB);
            for (int s = 0; s < L::NS; ++s)
                tma_load_2d_tile(base + L::Q0 + s * L::QSLAB, &mq, bars + L::QF, h * D + 64 * s, q0);
            for (int j = 0; j < nb; ++j) {
                const int sl = j % ST, use = j / ST;
                if (j >= ST && !att_wait(bars + L::KE + sl, (use - 1) & 1, abort)) break;
                mbar_expect_tx(bars + L::KF + sl, L::KSTAGE);
                for (int s = 0; s < L::NS; ++s)
                    tma_load_2d_tile(base + L::K0 + sl * L::KSTAGE + s * L::KSLAB, &mk, bars + L::KF + sl, g * D + 64 * s,
                                     j * ATT_BN);
            }
        }
    } else if (warp == ATT_VWARP) {
        // ------------------------------------------------------------ TMA: V^T
        if (lane == 0) {
            for (int j = 0; j < nb; ++j) {
                const int sl = j % ST, use = j / ST;
                if (j >= ST && !att_wait(bars + L::VE + sl, (use - 1) & 1, abort)) break;
                mbar_expect_tx(bars + L::VF + sl, L::VSTAGE);
                for (int s = 0; s < 2; ++s)
                    tma_load_2d_tile(base + L::V0 + sl * L::VSTAGE + s * L::VSLAB, &mv, bars + L::VF + sl,
                                     j * ATT_BN + 64 * s, g * D);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        // Two kinds of work, issued in whichever order they become ready: S_j
        // (its K block has landed and the softmax has read S_{j-1}; S_j may
        // run ahead of P_{j-1} V_{j-1} by one block) and P_j V_j (the softmax
        // has written P_j, its V^T block has landed).  One thread polls both;
        // a stall past 2 s sets the error word.
        if (lane == 0) {
            constexpr uint32_t IDS = t5::idesc_bf16(ATT_BM, ATT_BN), IDO = t5::idesc_bf16(ATT_BM, D);
            bool ok = att_wait(bars + L::QF, 0, abort);
            if (ok) t5::fence_after();
            int ns = 0, np = 0;   // the next S and PV to issue
            uint64_t t_last = globaltimer_ns();
            while (ok && np < nb) {
                bool did = false;
                if (ns < nb && ns <= np + 1 && (ns == 0 || att_ready(bars + L::SC, (ns - 1) & 1)) &&
                    att_ready(bars + L::KF + ns % ST, (ns / ST) & 1)) {
                    // S_ns = Q K_ns^T into TMEM columns 0-127
                    t5::fence_after();
                    const int sl = ns % ST;
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const int s = kk >> 2, w = kk & 3;
                        const uint64_t da = t5::desc_sw128(sbase + L::Q0 + s * L::QSLAB + w * 32);
                        const uint64_t db = t5::desc_sw128(sbase + L::K0 + sl * L::KSTAGE + s * L::KSLAB + w * 32);
                        t5::mma_f16(tmem, da, db, IDS, kk > 0 ? 1u : 0u);
                    }
                    t5::commit(bars + L::SF);
                    t5::commit(bars + L::KE + sl);
                    ++ns;
                    did = true;
                } else if (np < ns && att_ready(bars + L::PF + (np & 1), (np >> 1) & 1) &&
                           att_ready(bars + L::VF + np % ST, (np / ST) & 1)) {
                    // O += P_np V_np over 8 key steps of 16, P from TMEM, N = D
                    t5::fence_after();
                    const int sl = np % ST;
                    const uint32_t pa = tmem + PCOL + (np & 1) * (ATT_BN / 2);
#pragma unroll
                    for (int kk = 0; kk < ATT_BN / 16; ++kk) {
                        const int s = kk >> 2, w = kk & 3;
                        const uint64_t db = t5::desc_sw128(sbase + L::V0 + sl * L::VSTAGE + s * L::VSLAB + w * 32);
                        t5::mma_f16_ts(tmem + OCOL, pa + kk * 8, db, IDO, (np > 0 || kk > 0) ? 1u : 0u);
                    }
                    t5::commit(bars + L::PV + (np & 1));
                    t5::commit(bars + L::VE + sl);
                    ++np;
                    did = true;
                }
                if (did) {
                    t_last = globaltimer_ns();
                } else if (*abort || globaltimer_ns() - t_last > 2000000000ull) {
                    if (!*abort) atomicCAS(&g_attn_error, 0, ERR_WAIT_TIMEOUT);
                    *abort = 1;
                    ok = false;
                }
            }
            // every product issued has completed before TMEM is released
            t5::commit(bars + L::FIN);
            mbar_wait_bounded(bars + L::FIN, 0, nullptr, 0, 200000000ull);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ softmax
        // Warp w reads TMEM lanes 32 (w % 4) .. +31 (rows r); warps 2-5 take the
        // scores 0-63 of their rows' block and the O columns 0 .. D/2-1, warps
        // 6-9 the scores 64-127 and O columns D/2 .. D-1; the two halves of a
        // row swap their block maxima through shared memory (two rounds of
        // buffers) and keep partial sums, added at the end.
        const int quad = warp & 3, half = (warp - 2) >> 2, r = 32 * quad + lane, pos = off + q0 + r;
        const uint32_t trow = tmem + (static_cast<uint32_t>(32 * quad) << 16);
        float* xmax = reinterpret_cast<float*>(base + L::X0);
        float* lsum = reinterpret_cast<float*>(base + L::LS0);
        const int pos_min = off + q0;   // every query of the tile sees keys <= pos_min
        float m = 0.0f, l = 0.0f;
        bool ok = true;
        for (int j = 0; j < nb; ++j) {
            ok = __all_sync(0xffffffffu, ok && att_wait(bars + L::SF, j & 1, abort));
            float x[64];
            float bm = -INFINITY;
            if (ok) {
                t5::fence_after();
                float s0[32], s1[32];
                t5::ld32(trow + 64 * half, s0);
                t5::ld32(trow + 64 * half + 32, s1);
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    x[c] = s0[c];
                    x[32 + c] = s1[c];
                }
            }
            // S_j is in registers: S_{j+1} may overwrite it
            t5::fence_before();
            att_arrive(bars + L::SC);
            if (ok) {
                const int key0 = j * ATT_BN + 64 * half;
                if (key0 + 63 > pos_min || key0 + 63 >= a.nk) {   // a block on the diagonal or past the keys
#pragma unroll
                    for (int c = 0; c < 64; ++c)
                        if (!(key0 + c <= pos && key0 + c < a.nk)) x[c] = -INFINITY;
                }
#pragma unroll
                for (int c = 0; c < 64; ++c) bm = fmaxf(bm, x[c]);
            }
            // the row's maximum over both halves (raw scores; the scale is positive)
            xmax[((j & 1) * 2 + half) * ATT_BM + r] = bm;
            asm volatile("bar.sync 1, %0;" ::"n"(32 * ATT_SM_WARPS) : "memory");
            bm = fmaxf(bm, xmax[((j & 1) * 2 + (half ^ 1)) * ATT_BM + r]) * a.sl2;
            // P buffer j & 1 is free once P_{j-2} V_{j-2} has finished
            if (j >= 2) ok = __all_sync(0xffffffffu, ok && att_wait(bars + L::PV + (j & 1), ((j - 2) >> 1) & 1, abort));
            if (!ok) {
                att_arrive(bars + L::PF + (j & 1));
                continue;
            }
            if (j == 0) {
                m = bm;   // finite: key 0 is visible to every query
            } else if (__any_sync(0xffffffffu, bm > m + ATT_RESCALE_LOG2)) {
                // O is rescaled once P_{j-1} V_{j-1} has finished
                ok = __all_sync(0xffffffffu, att_wait(bars + L::PV + ((j - 1) & 1), ((j - 1) >> 1) & 1, abort));
                if (!ok) {
                    att_arrive(bars + L::PF + (j & 1));
                    continue;
                }
                const float mn = fmaxf(m, bm), alpha = ex2_approx(m - mn);
                m = mn;
                l *= alpha;
                t5::fence_after();
#pragma unroll 1
                for (int c0 = half * (D / 2); c0 < (half + 1) * (D / 2); c0 += 32) {
                    float ov[32];
                    t5::ld32(trow + OCOL + c0, ov);
#pragma unroll
                    for (int e = 0; e < 32; ++e) ov[e] *= alpha;
                    t5::st32(trow + OCOL + c0, ov);
                }
            }
            // P = 2^(s scale log2e - m) in bf16 pairs, this half's 64 keys into
            // 32 TMEM columns of P buffer j & 1
            float sum = 0.0f;
            uint32_t pk[32];
#pragma unroll
            for (int c = 0; c < 32; ++c) {
                const float p0 = ex2_approx(fmaf(x[2 * c], a.sl2, -m));
                const float p1 = ex2_approx(fmaf(x[2 * c + 1], a.sl2, -m));
                sum += p0 + p1;
                pk[c] = bf16x2_bits(p0, p1);
            }
            l += sum;
            t5::fence_after();   // after the wait for P_{j-2} V_{j-2}
            t5::st32u(trow + PCOL + (j & 1) * (ATT_BN / 2) + 32 * half, pk);
            t5::fence_before();
            att_arrive(bars + L::PF + (j & 1));
        }
        ok = __all_sync(0xffffffffu, ok && att_wait(bars + L::PV + ((nb - 1) & 1), ((nb - 1) >> 1) & 1, abort));
        lsum[half * ATT_BM + r] = l;
        asm volatile("bar.sync 1, %0;" ::"n"(32 * ATT_SM_WARPS) : "memory");
        if (ok) {
            t5::fence_after();
            const float inv = 1.0f / (lsum[r] + lsum[ATT_BM + r]);
            const bool store = q0 + r < a.nq && GDN_IN_RANGE(g_attn_error, h < a.hq);
            uint16_t* orow = a.o + (static_cast<int64_t>(q0 + r) * a.hq + h) * D;
#pragma unroll 1
            for (int c0 = half * (D / 2); c0 < (half + 1) * (D / 2); c0 += 32) {
                float ov[32];
                t5::ld32(trow + OCOL + c0, ov);
                if (store) {
#pragma unroll
                    for (int e = 0; e < 32; e += 8)
                        *reinterpret_cast<uint4*>(orow + c0 + e) =
                            make_uint4(bf16x2_bits(ov[e] * inv, ov[e + 1] * inv), bf16x2_bits(ov[e + 2] * inv, ov[e + 3] * inv),
                                       bf16x2_bits(ov[e + 4] * inv, ov[e + 5] * inv), bf16x2_bits(ov[e + 6] * inv, ov[e + 7] * inv));
                }
            }
        }
    }

    if (*abort && tid == 0) {
        // a wait ran out: let copies already issued land (bounded) before the
        // shared memory is released
        for (int i = L::QF; i < L::VE + 2; ++i)
            for (uint32_t par = 0; par < 2; ++par) mbar_wait_bounded(bars + i, par, nullptr, 0, 20000000ull);
    }
    t5::fence_before();
    __syncthreads();
    if (warp == 1) {
        t5::fence_after();
        t5::dealloc(tmem, 512);
    }
}

// V [nk][hkv][D] -> V^T [hkv][D][nkp] (bf16), through 64 x 64 tiles in shared memory.
__global__ void __launch_bounds__(256) attn_vt_kernel(const uint16_t* __restrict__ v, uint16_t* __restrict__ vt, int nk,
                                                      int hkv, int d, int64_t nkp) {
    __shared__ uint16_t t[64][66];
    const int k0 = blockIdx.x * 64, e0 = blockIdx.y * 64, g = blockIdx.z;
    for (int i = threadIdx.x; i < 64 * 64; i += 256) {
        const int key = i >> 6, e = i & 63;
        t[e][key] = k0 + key < nk ? v[(static_cast<int64_t>(k0 + key) * hkv + g) * d + e0 + e] : 0;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < 64 * 64; i += 256) {
        const int e = i >> 6, key = i & 63;
        if (k0 + key < nk && GDN_IN_RANGE(g_attn_error, g < hkv && e0 + e < d && k0 + key < nkp))
            vt[(static_cast<int64_t>(g) * d + e0 + e) * nkp + k0 + key] = t[e][key];
    }
}

static PFN_cuTensorMapEncodeTiled_v12000 attn_map_encoder() {
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

// bf16 matrix [rows][cols] (row stride ld elements), boxes of 64 columns x box_rows, 128-byte swizzle, zero fill.
static bool attn_map(CUtensorMap* map, const uint16_t* ptr, int64_t rows, int64_t cols, int64_t ld, int box_rows) {
    auto enc = attn_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2};
    cuuint32_t box[2] = {64, static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(ptr), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int64_t attn_vt_ld(int64_t nk) { return (nk + 7) & ~int64_t(7); }

size_t attn_workspace_bytes(int64_t nk, int hkv, int d) {
    return static_cast<size_t>(hkv) * d * attn_vt_ld(nk) * 2;
}

template <int D>
static cudaError_t launch_attn_d(const uint16_t* q, const uint16_t* k, const uint16_t* vt, int64_t nq, int64_t nk, int hq,
                                 int hkv, float scale, uint16_t* o, cudaStream_t st) {
    static PerDeviceOnce attr_once;
    // at least 120 KB, so that one CTA holds an SM (it allocates all 512 TMEM columns)
    constexpr int smem = AttSmem<D>::BYTES + 1024 > 120 * 1024 ? AttSmem<D>::BYTES + 1024 : 120 * 1024;
    if (attr_once.run([](int) { cudaFuncSetAttribute(attn_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem); }) < 0)
        return cudaErrorInvalidDevice;
    CUtensorMap mq, mk, mv;
    if (!attn_map(&mq, q, nq, static_cast<int64_t>(hq) * D, static_cast<int64_t>(hq) * D, ATT_BM) ||
        !attn_map(&mk, k, nk, static_cast<int64_t>(hkv) * D, static_cast<int64_t>(hkv) * D, ATT_BN) ||
        !attn_map(&mv, vt, static_cast<int64_t>(hkv) * D, nk, attn_vt_ld(nk), D))
        return cudaErrorInvalidValue;
    AttArgs a;
    a.nq = static_cast<int>(nq);
    a.nk = static_cast<int>(nk);
    a.hq = hq;
    a.hkv = hkv;
    a.ratio = hq / hkv;
    a.sl2 = scale * 1.4426950408889634f;
    a.o = o;
    a.ntiles = static_cast<int>((nq + ATT_BM - 1) / ATT_BM);
    attn_kernel<D><<<static_cast<unsigned>(a.ntiles * hq), ATT_THREADS, smem, st>>>(mq, mk, mv, a);
    return cudaGetLastError();
}

cudaError_t launch_attn(const uint16_t* q, const uint16_t* k, const uint16_t* v, int64_t nq, int64_t nk, int hq, int hkv,
                        int d, float scale, uint16_t* o, void* workspace, cudaStream_t st) {
    uint16_t* vt = static_cast<uint16_t*>(workspace);
    const dim3 tg(static_cast<unsigned>((nk + 63) / 64), static_cast<unsigned>(d / 64), static_cast<unsigned>(hkv));
    attn_vt_kernel<<<tg, 256, 0, st>>>(v, vt, static_cast<int>(nk), hkv, d, attn_vt_ld(nk));
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (d == 64) return launch_attn_d<64>(q, k, vt, nq, nk, hq, hkv, scale, o, st);
    if (d == 128) return launch_attn_d<128>(q, k, vt, nq, nk, hq, hkv, scale, o, st);
    return launch_attn_d<256>(q, k, vt, nq, nk, hq, hkv, scale, o, st);
}

int read_and_clear_attn_error() {
    int v = 0, z = 0;
    cudaMemcpyFromSymbol(&v, g_attn_error, sizeof(int));
    if (v) cudaMemcpyToSymbol(g_attn_error, &z, sizeof(int));
    return v;
}

}  // namespace gdn
