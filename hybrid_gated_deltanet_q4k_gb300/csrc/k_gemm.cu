// Steps 1c and 5: the quantised projections, out = ((float)(A . B^T) * sa) * sb.
//
// The pages feed int8 weight rows and int8 activations to an int8 tensor-core
// GEMM (sparkinfer PR #464, Summary: "int8 tensor-core GEMM"; its follow-up
// "int8-native prefill GEMM (mma.sync m16n8k32)").  sm_103a's fifth-generation
// tensor cores have no int8 MMA kind (ptxas rejects tcgen05.mma .kind::i8 for
// sm_103a), so the same integer product is taken on fp16 operands: every int8
// code is exact in fp16, every product (|q| <= 127, so < 2^14) is exact, and an
// fp32 accumulator holds every partial sum of up to 1024 such products exactly
// (1024 * 127^2 < 2^24).  The K loop therefore runs in segments of 1024: each
// segment accumulates in its own TMEM buffer, the epilogue converts the
// segment to int32 and sums the segments in registers.  The result is the
// exact integer product whatever the data.
//
// Kernel structure: persistent pairs of CTAs (thread-block clusters of 2, one
// CTA per SM, 320 threads each) on the fifth-generation tensor cores' two-SM
// mode (tcgen05 .cta_group::2).  A pair computes 256 x 256 output tiles: each
// CTA stages its 128 rows of A and its half (128 rows) of B, and one
// instruction of the even CTA multiplies M = 256 (both CTAs' A rows) by
// N = 256 (both B halves), each CTA's TMEM receiving its own 128 rows.  Per
// output element a CTA stages and reads a third less shared memory than a
// one-SM M = 128, N = 256 product, whose operand traffic (TMA writes plus
// tensor reads) is what bounds it.
//   warp 0      TMA producer (both CTAs): 128x64 A tile + 128x64 B half per
//               stage, 6 stages of 32 KB, 128-byte swizzle; every copy of the
//               pair completes on the even CTA's stage barrier;
//   warp 1      TMEM allocator (both CTAs, one collective pair allocation of
//               512 columns) and, in the even CTA, the MMA issuer:
//               tcgen05.mma.cta_group::2 kind::f16 M=256 N=256 K=16, fp32
//               accumulators in two 256-column buffers (one per K segment,
//               ping-pong); its commits signal both CTAs' barriers;
//   warps 2-9   epilogue (both CTAs): tcgen05.ld of each finished segment of
//               the CTA's 128 rows (warp w reads TMEM lanes 32*(w%4).., half
//               (w-2)/4 of the 256 columns), int32 running sums in registers,
//               then the fp32 rescale and the stores.  Each warp releases the
//               buffer right after reading it (to the even CTA's barrier), so
//               the next segment's MMAs overlap the conversion and stores.
// Every wait is bounded (about two seconds); a wait that runs out records
// ERR_WAIT_TIMEOUT in this unit's error word and the CTA winds down: it waits
// (bounded) for the copies and MMAs in flight, meets its peer at the closing
// cluster barrier, frees the TMEM and returns.
#include "common.cuh"
#include "tcgen05.cuh"

#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

namespace gdn {

static __device__ int g_gemm_error;

namespace tc {
constexpr int BM = 128;              // A rows per CTA (a pair covers 2 * BM)
constexpr int BN = 256;              // output columns per tile (each CTA stages BN / 2 rows of B)
constexpr int BK = 64;               // fp16 elements = 128 bytes = one swizzle row
constexpr int STAGES = 6;
constexpr int SEG_KB = 16;           // k-blocks per exact fp32 segment (16 * 64 = 1024)
constexpr int A_BYTES = BM * BK * 2; // 16 KB
constexpr int B_BYTES = BN / 2 * BK * 2; // 16 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int NUM_EPI_WARPS = 8;
constexpr int THREADS = 64 + NUM_EPI_WARPS * 32;
constexpr uint32_t TMEM_COLS = 512;  // two accumulator buffers of BN columns
constexpr int BAR_BYTES = 256;
// epilogue staging: one 32-row x 64-column bf16 tile (4 KB, 128-byte swizzle) per epilogue warp
constexpr int EPI_TILE_BYTES = 32 * 64 * 2;
constexpr int EPI_BYTES = NUM_EPI_WARPS * EPI_TILE_BYTES;
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + EPI_BYTES + BAR_BYTES + 1024;  // + alignment slack
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;
constexpr uint64_t DRAIN_LIMIT_NS = 20000000ull;

// Instruction descriptor, kind::f16: D fp32 (bits 4-5 = 1), A and B fp16
// (bits 7-9, 10-12 = 0), both K-major (bits 15, 16 = 0), N>>3 at bits 17-22,
// M>>4 at bits 24-28.
// The pair instruction: M = 2 * BM.
constexpr uint32_t IDESC = (1u << 4) | (static_cast<uint32_t>(BN >> 3) << 17) | (static_cast<uint32_t>((2 * BM) >> 4) << 24);
}  // namespace tc

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for the phase of `bar` with the given parity to complete.  Gives up
// when another role has aborted, or after `limit` ns (recording the timeout).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          uint64_t limit = tc::WAIT_LIMIT_NS) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 64; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (global_ns() - t0 > limit) {
            atomicCAS(&g_gemm_error, 0, ERR_WAIT_TIMEOUT);
            *abort_flag = 1;
            return false;
        }
    }
}

// Tensor store of a shared-memory tile (bulk async group of this thread).
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, const void* src, int x, int y) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y), "r"(smem_u32(src))
                 : "memory");
}
__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_group_read0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_group0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor, K-major, 128-byte swizzle: start address
// >> 4 (bits 0-13), stride between 8-row groups 1024 B >> 4 (bits 32-45),
// descriptor version 1 (bit 46), swizzle mode 2 = 128 B (bits 61-63).  The
// leading-dimension offset is unused for swizzled K-major operands whose K
// extent per MMA (32 B) stays inside one 128-byte swizzle row.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    return static_cast<uint64_t>((saddr >> 4) & 0x3FFFu) | (static_cast<uint64_t>(1) << 16) |
           (static_cast<uint64_t>(1024 >> 4) << 32) | (static_cast<uint64_t>(1) << 46) |
           (static_cast<uint64_t>(2) << 61);
}

// The pair product: descriptors address this (even) CTA's tiles; the odd CTA's
// tiles sit at the same offsets of its shared memory.
__device__ __forceinline__ void mma_f16_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t accumulate) {
    t5::mma_f16_pair(d_tmem, adesc, bdesc, tc::IDESC, accumulate);
}

// Arrive on the mbarrier at this offset in both CTAs of the pair once the MMAs
// issued so far have completed.
__device__ __forceinline__ void mma_commit_pair(uint64_t* bar) { t5::commit_pair(bar); }

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

struct GemmArgs {
    const float* sa;
    const float* sb;
    int M, N, K;
    uint16_t* out_bf16;
    int64_t ld_bf16;
    int n_bf16;
    float* out_f32;
    int64_t ld_f32;
    int vec_ok;     // 16-byte vector stores are aligned
    int tma_store;  // bf16 output through shared memory and TMA tensor stores (the third tensor map)
};

__device__ __forceinline__ void store_group8(const GemmArgs& g, int row, int n, const float* y) {
    if (!GDN_IN_RANGE(g_gemm_error, row < g.M && n < g.N)) return;
    if (g.vec_ok && n + 8 <= g.N && n + 8 <= g.n_bf16) {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
            w[i] = static_cast<uint32_t>(float_to_bf16_bits(y[2 * i])) |
                   (static_cast<uint32_t>(float_to_bf16_bits(y[2 * i + 1])) << 16);
        *reinterpret_cast<uint4*>(g.out_bf16 + row * g.ld_bf16 + n) = make_uint4(w[0], w[1], w[2], w[3]);
    } else if (g.vec_ok && n >= g.n_bf16 && n + 8 <= g.N) {
        float4* p = reinterpret_cast<float4*>(g.out_f32 + row * g.ld_f32 + (n - g.n_bf16));
        p[0] = make_float4(y[0], y[1], y[2], y[3]);
        p[1] = make_float4(y[4], y[5], y[6], y[7]);
    } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int c = n + j;
            if (c < g.N) {
                if (c < g.n_bf16)
                    g.out_bf16[row * g.ld_bf16 + c] = float_to_bf16_bits(y[j]);
                else
                    g.out_f32[row * g.ld_f32 + (c - g.n_bf16)] = y[j];
            }
        }
    }
}

// Tile order: groups of GROUP_N column tiles, and within a group the ~76 pair
// tiles in flight at a time span ~GROUP_N columns x ~5 row blocks of 256.  The
// group's B columns (GROUP_N * 256 rows of K codes, 32 MB at K = 4096) stay in
// L2 while A streams through once per group; in plain row-major order every
// row block sweeps all of B, which for a large B (the input projection's is
// ~100 MB) falls out of L2 and is re-read from DRAM.
constexpr int GROUP_N = 16;
__device__ __forceinline__ void tile_origin(int tile, int num_m, int num_n, int& m0, int& n0) {
    const int group = tile / (GROUP_N * num_m);
    const int first = group * GROUP_N;
    const int width = min(GROUP_N, num_n - first);
    const int r = tile - group * GROUP_N * num_m;
    m0 = (r / width) * (2 * tc::BM);
    n0 = (first + r % width) * tc::BN;
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(tc::THREADS, 1)
gemm_codes_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                  const __grid_constant__ CUtensorMap tmC, GemmArgs g) {
    using namespace tc;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* epi = smem + STAGES * STAGE_BYTES;   // epilogue staging, 1024-byte aligned
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES + EPI_BYTES);
    uint64_t* empty = full + STAGES;
    uint64_t* acc_full = empty + STAGES;
    uint64_t* acc_empty = acc_full + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_empty + 2);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();
    const bool leader = rank == 0;
    const int pair = blockIdx.x >> 1, num_pairs = gridDim.x >> 1;
    const int num_m = (g.M + 2 * BM - 1) / (2 * BM), num_n = (g.N + BN - 1) / BN;
    const int num_tiles = num_m * num_n;
    const int nkb = g.K / BK;
    const int nseg = (nkb + SEG_KB - 1) / SEG_KB;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);     // even CTA: its producer's arrive (+ both CTAs' bytes)
            mbar_init(&empty[s], 1);    // the pair's commit
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&acc_full[b], 1);                     // the pair's commit
            mbar_init(&acc_empty[b], 2 * NUM_EPI_WARPS);    // even CTA: one arrival per epilogue warp of the pair
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        t5::alloc_pair(tmem_slot, TMEM_COLS);
    }
    tc_fence_before();
    // both CTAs' barriers are initialised before either signals the other's
    cluster_sync();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer (both CTAs)
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmA)) : "memory");
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmB)) : "memory");
            const uint32_t full0 = cluster_addr(&full[0], 0);   // the even CTA's stage barriers
            uint32_t stage = 0, phase = 0;
            uint32_t armed = 0;              // bit s: stage s has been filled at least once (even CTA)
            uint32_t armed_parity = 0;       // bit s: parity of its last fill
            bool ok = true;
            for (int tile = pair; ok && tile < num_tiles; tile += num_pairs) {
                int m0, n0;
                tile_origin(tile, num_m, num_n, m0, n0);
                for (int kb = 0; kb < nkb; ++kb) {
                    if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag)) { ok = false; break; }
                    uint8_t* sA = smem + stage * STAGE_BYTES;
                    if (leader) mbar_arrive_expect_tx(&full[stage], 2 * STAGE_BYTES);
                    tma_load_2d_pair(sA, &tmA, full0 + 8 * stage, kb * BK, m0 + static_cast<int>(rank) * BM);
                    tma_load_2d_pair(sA + A_BYTES, &tmB, full0 + 8 * stage, kb * BK, n0 + static_cast<int>(rank) * (BN / 2));
                    armed |= 1u << stage;
                    armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
            }
            // Let every copy of the pair land before the CTAs exit (the even CTA's
            // barriers count the odd CTA's copies too).
            if (leader)
                for (int s = 0; s < STAGES; ++s)
                    if (armed & (1u << s)) {
                        int dummy = 0;
                        mbar_wait(&full[s], (armed_parity >> s) & 1u, reinterpret_cast<volatile int*>(&dummy), DRAIN_LIMIT_NS);
                    }
        }
    } else if (warp == 1) {
        if (lane == 0 && leader) {
            // ------------------------------------------------ MMA issuer (even CTA)
            uint32_t stage = 0, phase = 0, acc_ctr = 0;
            bool ok = true, committed = false;
            uint32_t last_buf = 0, last_par = 0;
            for (int tile = pair; ok && tile < num_tiles; tile += num_pairs) {
                for (int seg = 0; ok && seg < nseg; ++seg) {
                    const uint32_t buf = acc_ctr & 1u, par = (acc_ctr >> 1) & 1u;
                    if (!mbar_wait(&acc_empty[buf], par ^ 1u, abort_flag)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t d_tmem = tmem_base + buf * BN;
                    const int kb0 = seg * SEG_KB, kb1 = min(nkb, kb0 + SEG_KB);
                    for (int kb = kb0; kb < kb1; ++kb) {
                        if (!mbar_wait(&full[stage], phase, abort_flag)) { ok = false; break; }
                        tc_fence_after();
                        const uint32_t sa_addr = smem_u32(smem + stage * STAGE_BYTES);
                        const uint64_t adesc = sw128_desc(sa_addr);
                        const uint64_t bdesc = sw128_desc(sa_addr + A_BYTES);
#pragma unroll
                        for (int kk = 0; kk < BK / 16; ++kk)
                            mma_f16_pair(d_tmem, adesc + 2 * kk, bdesc + 2 * kk, (kb > kb0 || kk > 0) ? 1u : 0u);
                        mma_commit_pair(&empty[stage]);
                        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                    }
                    mma_commit_pair(&acc_full[buf]);
                    committed = true;
                    last_buf = buf;
                    last_par = par;
                    ++acc_ctr;
                }
            }
            // Let the last MMAs finish before TMEM is freed.
            if (committed) {
                int dummy = 0;
                mbar_wait(&acc_full[last_buf], last_par, reinterpret_cast<volatile int*>(&dummy), DRAIN_LIMIT_NS);
            }
        }
    } else {
        // ---------------------------------------------------- epilogue (both CTAs)
        const int quarter = warp & 3;
        const int half = (warp - 2) >> 2;
        const uint32_t acc_empty0 = cluster_addr(&acc_empty[0], 0);
        uint32_t acc_ctr = 0;
        bool ok = true;
        for (int tile = pair; ok && tile < num_tiles; tile += num_pairs) {
            int m0, n0;
            tile_origin(tile, num_m, num_n, m0, n0);
            m0 += static_cast<int>(rank) * BM;
            int32_t acc[128];
#pragma unroll
            for (int i = 0; i < 128; ++i) acc[i] = 0;
            for (int seg = 0; seg < nseg; ++seg) {
                const uint32_t buf = acc_ctr & 1u, par = (acc_ctr >> 1) & 1u;
                bool w = mbar_wait(&acc_full[buf], par, abort_flag);
                if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
                tc_fence_after();
                const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + buf * BN + half * 128;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint32_t r[32];
                    tmem_ld32(taddr + c * 32, r);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 32; ++j) acc[c * 32 + j] += __float2int_rn(__uint_as_float(r[j]));
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(acc_empty0 + 8 * buf);
                ++acc_ctr;
            }
            if (!ok) break;
            const int row = m0 + quarter * 32 + lane;
            const bool valid = row < g.M;
            const float srow = valid ? g.sa[row] : 0.0f;
            const int nbase = n0 + half * 128;
            uint8_t* ebuf = epi + (warp - 2) * EPI_TILE_BYTES;
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                const int n = nbase + 64 * c;
                if (g.tma_store && n + 64 <= g.n_bf16) {
                    if (m0 + quarter * 32 >= g.M) continue;   // every row of this warp's box is past M
                    // bf16 rows of 64 columns into this warp's staging tile (lane = row,
                    // 128-byte swizzle), then one tensor store; the TMA clips rows past M
                    uint32_t w[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const float y0 = __fmul_rn(__fmul_rn(__int2float_rn(acc[64 * c + 2 * j]), srow), __ldg(g.sb + n + 2 * j));
                        const float y1 =
                            __fmul_rn(__fmul_rn(__int2float_rn(acc[64 * c + 2 * j + 1]), srow), __ldg(g.sb + n + 2 * j + 1));
                        w[j] = static_cast<uint32_t>(float_to_bf16_bits(y0)) |
                               (static_cast<uint32_t>(float_to_bf16_bits(y1)) << 16);
                    }
                    if (lane == 0) bulk_wait_group_read0();   // the previous store has read the tile
                    __syncwarp();
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        *reinterpret_cast<uint4*>(ebuf + lane * 128 + ((q ^ (lane & 7)) << 4)) =
                            make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(&tmC, ebuf, n, m0 + quarter * 32);
                        bulk_commit_group();
                    }
                } else if (valid) {
#pragma unroll
                    for (int grp = 0; grp < 8; ++grp) {
                        const int nn = n + grp * 8;
                        if (nn < g.N) {
                            float y[8];
#pragma unroll
                            for (int j = 0; j < 8; ++j) {
                                const float scol = (nn + j < g.N) ? __ldg(g.sb + nn + j) : 0.0f;
                                y[j] = __fmul_rn(__fmul_rn(__int2float_rn(acc[64 * c + grp * 8 + j]), srow), scol);
                            }
                            store_group8(g, row, nn, y);
                        }
                    }
                }
            }
        }
    }

    // this warp's tensor stores have completed before the shared memory goes
    if (warp >= 2 && lane == 0) bulk_wait_group0();
    tc_fence_before();
    __syncthreads();
    // neither CTA frees its shared memory or TMEM while the pair's MMAs may
    // still read the one or write the other
    cluster_sync();
    if (warp == 1) {
        tc_fence_after();
        t5::dealloc_pair(tmem_base, TMEM_COLS);
    }
}

// ---------------------------------------------------------------- host side

static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
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

// 2-D fp16 tensor [rows][K], box of box_rows x 64 elements, 128-byte swizzle,
// zero fill outside the tensor.
static bool make_map(CUtensorMap* map, const void* base, int64_t rows, int64_t K, int box_rows) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(tc::BK), static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

static int sm_count() {
    int dev = 0, n = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    return n > 0 ? n : 1;
}

// bf16 output [rows][n_cols] with row pitch ld (elements): boxes of 32 rows x
// 64 columns, 128-byte swizzle, for the epilogue's tensor stores.
static bool make_store_map(CUtensorMap* map, const void* base, int64_t rows, int64_t n_cols, int64_t ld) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(n_cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2};
    cuuint32_t box[2] = {64, 32};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Clusters of 2 CTAs of the projection kernel that fit on device `dev` (the
// current one) at once; the kernel's shared-memory attribute is set first.
static int resident_pairs(int dev) {
    static int cached[MAX_DEVICES] = {};
    static PerDeviceOnce once;
    once.run([](int d) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(sm_count()), 1, 1);
        cfg.blockDim = dim3(tc::THREADS, 1, 1);
        cfg.dynamicSmemBytes = tc::SMEM_BYTES;
        cudaLaunchAttribute attr;
        attr.id = cudaLaunchAttributeClusterDimension;
        attr.val.clusterDim.x = 2;
        attr.val.clusterDim.y = 1;
        attr.val.clusterDim.z = 1;
        cfg.attrs = &attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, gemm_codes_kernel, &cfg) != cudaSuccess || n < 1) {
            cudaGetLastError();
            n = sm_count() / 2;
        }
        cached[d] = n;
    });
    return cached[dev];
}

// Returns cudaErrorInvalidValue when a tensor map cannot be built (caller
// validated shapes and alignment first).
cudaError_t launch_gemm_codes(const uint16_t* a, const float* sa, const uint16_t* b, const float* sb, int64_t M,
                              int64_t N, int64_t K, uint16_t* out_bf16, int64_t ld_bf16, int64_t n_bf16,
                              float* out_f32, int64_t ld_f32, cudaStream_t st) {
    CUtensorMap ma, mb;
    if (!make_map(&ma, a, M, K, tc::BM) || !make_map(&mb, b, N, K, tc::BN / 2)) return cudaErrorInvalidValue;
    static PerDeviceOnce attr_once;
    const int dev = attr_once.run([](int) {
        cudaFuncSetAttribute(gemm_codes_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, tc::SMEM_BYTES);
    });
    if (dev < 0) return cudaErrorInvalidDevice;
    GemmArgs g;
    g.sa = sa;
    g.sb = sb;
    g.M = static_cast<int>(M);
    g.N = static_cast<int>(N);
    g.K = static_cast<int>(K);
    g.out_bf16 = out_bf16;
    g.ld_bf16 = ld_bf16;
    g.n_bf16 = static_cast<int>(n_bf16);
    g.out_f32 = out_f32;
    g.ld_f32 = ld_f32;
    const bool bf_ok = out_bf16 == nullptr || ((reinterpret_cast<uintptr_t>(out_bf16) & 15) == 0 && ld_bf16 % 8 == 0);
    const bool f_ok = out_f32 == nullptr ||
                      ((reinterpret_cast<uintptr_t>(out_f32) & 15) == 0 && ld_f32 % 4 == 0 && n_bf16 % 4 == 0);
    g.vec_ok = (bf_ok && f_ok) ? 1 : 0;
    // bf16 output through TMA tensor stores when it is 16-byte aligned with a
    // row pitch of a multiple of 8 elements
    CUtensorMap mc = ma;
    g.tma_store = (out_bf16 != nullptr && bf_ok && n_bf16 >= 64 && make_store_map(&mc, out_bf16, M, n_bf16, ld_bf16)) ? 1 : 0;
    // pairs of CTAs (clusters of 2): as many as can be resident at once (a
    // cluster stays within one GPC), at most one per tile
    const int64_t tiles = ((M + 2 * tc::BM - 1) / (2 * tc::BM)) * ((N + tc::BN - 1) / tc::BN);
    const int max_pairs = resident_pairs(dev);
    const int pairs = static_cast<int>(tiles < max_pairs ? tiles : max_pairs);
    const int grid = 2 * (pairs > 0 ? pairs : 1);
    gemm_codes_kernel<<<grid, tc::THREADS, tc::SMEM_BYTES, st>>>(ma, mb, mc, g);
    return cudaGetLastError();
}

int read_and_clear_gemm_error() {
    int v = 0, z = 0;
    cudaMemcpyFromSymbol(&v, g_gemm_error, sizeof(int));
    if (v) cudaMemcpyToSymbol(g_gemm_error, &z, sizeof(int));
    return v;
}

// ------------------------------------------------------------ fp32 projection
// F32 layers only (no quantisation): a plain shared-memory tiled fp32 product
// on the CUDA cores, 64x64 tiles, 4x4 outputs per thread.
__global__ void __launch_bounds__(256) gemm_f32_kernel(const float* __restrict__ A, const float* __restrict__ B, int M,
                                                       int N, int K, uint16_t* out_bf16, int64_t ld_bf16, int n_bf16,
                                                       float* out_f32, int64_t ld_f32) {
    __shared__ float As[16][64 + 4];
    __shared__ float Bs[16][64 + 4];
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    const int m0 = blockIdx.y * 64, n0 = blockIdx.x * 64;
    float acc[4][4] = {};
    for (int k0 = 0; k0 < K; k0 += 16) {
        for (int i = threadIdx.x; i < 64 * 16; i += 256) {
            const int r = i / 16, c = i % 16;
            As[c][r] = (m0 + r < M && k0 + c < K) ? A[static_cast<int64_t>(m0 + r) * K + k0 + c] : 0.0f;
            Bs[c][r] = (n0 + r < N && k0 + c < K) ? B[static_cast<int64_t>(n0 + r) * K + k0 + c] : 0.0f;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < 16; ++kk) {
            float av[4], bv[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                av[i] = As[kk][ty * 4 + i];
                bv[i] = Bs[kk][tx * 4 + i];
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int m = m0 + ty * 4 + i;
        if (m >= M) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int n = n0 + tx * 4 + j;
            if (n >= N) continue;
            if (n < n_bf16)
                out_bf16[m * ld_bf16 + n] = float_to_bf16_bits(acc[i][j]);
            else
                out_f32[m * ld_f32 + (n - n_bf16)] = acc[i][j];
        }
    }
}

cudaError_t launch_gemm_f32(const float* a, const float* b, int64_t M, int64_t N, int64_t K, uint16_t* out_bf16,
                            int64_t ld_bf16, int64_t n_bf16, float* out_f32, int64_t ld_f32, cudaStream_t st) {
    dim3 grid(static_cast<unsigned>((N + 63) / 64), static_cast<unsigned>((M + 63) / 64));
    gemm_f32_kernel<<<grid, 256, 0, st>>>(a, b, static_cast<int>(M), static_cast<int>(N), static_cast<int>(K), out_bf16,
                                          ld_bf16, static_cast<int>(n_bf16), out_f32, ld_f32);
    return cudaGetLastError();
}

}  // namespace gdn
