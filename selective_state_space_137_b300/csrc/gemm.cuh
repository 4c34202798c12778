// gemm.cuh -- C = A B^T on the fifth-generation tensor cores (tcgen05), for
// the selection projections of S6 ("Mamba的三大创新", the selection
// mechanism: Delta, B, C are linear functions of the input):
//   x_proj : (tokens x dim) . (R + 2N x dim)^T  -> dt_low | B | C
//   dt_proj: (tokens x R)   . (dim x R)^T        -> delta_raw
// Both operands are K-major bf16 (rows of A and of B run along K); the
// accumulator is fp32 in tensor memory; the result is rounded to bf16.
//
// One CTA computes a 128 x BN tile with 4 warps:
//   warp 0 lane 0: TMA producer -- a STAGES-deep ring of 64-wide K slabs of A
//     (128 rows) and B (BN rows), 128-byte swizzle (the tcgen05 canonical
//     K-major layout: 8-row, 1024-byte swizzle atoms);
//   warp 1 lane 0: MMA issuer -- four tcgen05.mma (K = 16 each) per slab into
//     one TMEM accumulator, and tcgen05.commit to release each stage back to
//     the producer and, at the end, to signal the epilogue;
//   warps 0..3: epilogue -- warp w reads TMEM lanes 32w .. 32w + 31 (tile
//     rows) with tcgen05.ld, converts to bf16 and writes each column into one
//     of up to three output segments (column ranges with their own base
//     pointer and row stride).
// Warp 0 allocates the TMEM columns and frees them after the epilogue.  Every
// wait is bounded (2 s of %globaltimer); on a timeout the CTA latches the
// error word, lets its in-flight copies and MMAs finish (bounded), frees TMEM
// and exits.
#pragma once
#include "common.cuh"
#include "tile_io.cuh"   // softplus_tiled
#include "tma.cuh"

namespace ssm {

constexpr int kGemmBM = 128, kGemmBK = 64, kGemmThreads = 128;

struct GemmSeg {
    void* ptr;        // bf16 output, row-major
    int64_t ld;       // row stride (elements)
    int col0, ncol;   // global column range [col0, col0 + ncol) of C written here
};

struct GemmParams {
    int64_t M;        // rows of A and C
    int N, K;         // columns of C (rows of B), reduction length
    GemmSeg seg[3];
    int nseg;
    // epilogue of the persistent kernel: c = act(c + col_bias[col])
    const float* col_bias = nullptr;   // (N) or NULL
    int act = 0;                        // 0: none, 1: softplus
};

template <int BN, int S_>
struct GemmCfg {
    static constexpr int S = S_;   // TMA ring depth
    static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "tcgen05 M=128 needs N % 16 == 0, N <= 256");
    static constexpr int A_BYTES = kGemmBM * kGemmBK * 2;       // 16 KB
    static constexpr int B_BYTES = BN * kGemmBK * 2;
    static constexpr int STAGE = (A_BYTES + B_BYTES + 1023) / 1024 * 1024;
    static constexpr int OFF_BAR = S * STAGE;
    // full[S], empty[S], acc; then the TMEM address word
    static constexpr int OFF_TMEM = OFF_BAR + (2 * S + 1) * 8;
    static constexpr int SMEM = OFF_TMEM + 16 + 1024;            // + alignment slack
    static constexpr int TMEM_COLS = BN <= 32 ? 32 : BN <= 64 ? 64 : BN <= 128 ? 128 : 256;
};

// ---- tcgen05 wrappers (inline PTX) ------------------------------------------

__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(dst_smem)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// D[tmem] (+)= A[smem desc] . B[smem desc]^T, kind::f16 (bf16 in, fp32 accumulate)
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                       uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// arrive once on `bar` when every tcgen05.mma issued so far by this thread is done
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_addr(bar))
        : "memory");
}
// 16 consecutive 32-bit columns of this thread's TMEM lane
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float* v) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Shared-memory matrix descriptor of a K-major tile written by TMA with
// 128-byte swizzle: start address >> 4 (bits 0-13), leading-dimension offset
// (unused for swizzled K-major, encoded 1; bits 16-29), stride between 8-row
// atoms 1024 B (bits 32-45), descriptor version 1 (bits 46-47), base offset 0
// (1024-byte aligned atoms), swizzle mode 2 = 128-byte (bits 61-63).
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Instruction descriptor, kind::f16: fp32 accumulator (bits 4-5 = 1), bf16 A
// and B (bits 7-9, 10-12 = 1), both K-major (bits 15, 16 = 0), N >> 3 (bits
// 17-22), M >> 4 (bits 24-28).
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar, int c0,
                                            int c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_addr(bar)), "r"(c0), "r"(c1)
        : "memory");
}

struct GemmMaps {
    CUtensorMap a, b;   // A: (M, K), box 64 x 128; B: (N, K), box 64 x BN; 128-byte swizzle
};

template <int BN, int STAGES>
__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_bf16_tn_kernel(const __grid_constant__ GemmMaps maps, const GemmParams p) {
    using Cfg = GemmCfg<BN, STAGES>;
    constexpr int S = Cfg::S;
    extern __shared__ unsigned char smem_raw[];
    // 1024-byte alignment for the swizzle atoms
    unsigned char* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + Cfg::OFF_BAR);
    uint64_t* empty = full + S;
    uint64_t* acc = empty + S;
    uint32_t* tmem_word = reinterpret_cast<uint32_t*>(smem + Cfg::OFF_TMEM);
    volatile uint32_t* fail = tmem_word + 1;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t m0 = (int64_t)blockIdx.x * kGemmBM;
    const int n0 = blockIdx.y * BN;
    const int nk = (p.K + kGemmBK - 1) / kGemmBK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(acc, 1);
        *fail = 0;
        fence_barrier_init();
    }
    if (warp == 0) {   // the whole warp allocates (converged: .sync.aligned)
        __syncwarp();
        tmem_alloc(tmem_word, Cfg::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_word;

    int issued = 0;       // producer: slabs issued
    int committed = 0;    // MMA thread: slabs whose MMAs were committed
    if (warp == 0 && lane == 0) {
        // ---- TMA producer
        prefetch_tmap(&maps.a);
        prefetch_tmap(&maps.b);
        for (int i = 0; i < nk; ++i) {
            const int s = i % S;
            if (i >= S && !mbar_wait_bounded(&empty[s], (uint32_t)(((i / S) - 1) & 1))) {
                *fail = 1;
                break;
            }
            unsigned char* st = smem + s * Cfg::STAGE;
            mbar_arrive_expect_tx(&full[s], (uint32_t)(Cfg::A_BYTES + Cfg::B_BYTES));
            tma_load_2d(st, &maps.a, &full[s], i * kGemmBK, (int)m0);
            tma_load_2d(st + Cfg::A_BYTES, &maps.b, &full[s], i * kGemmBK, n0);
            issued = i + 1;
        }
    } else if (warp == 1 && lane == 0) {
        // ---- MMA issuer
        constexpr uint32_t idesc = idesc_bf16_f32(kGemmBM, BN);
        for (int i = 0; i < nk; ++i) {
            const int s = i % S;
            if (!mbar_wait_bounded(&full[s], (uint32_t)((i / S) & 1))) {
                *fail = 1;
                break;
            }
            tc_fence_after();
            const uint32_t a0 = smem_addr(smem + s * Cfg::STAGE);
            const uint32_t b0 = a0 + Cfg::A_BYTES;
#pragma unroll
            for (int kk = 0; kk < kGemmBK / 16; ++kk) {
                // K advances 16 elements = 32 bytes inside the 128-byte swizzle row
                tc_mma(tmem, smem_desc_sw128(a0 + kk * 32), smem_desc_sw128(b0 + kk * 32), idesc,
                       (i > 0 || kk > 0) ? 1u : 0u);
            }
            tc_commit(&empty[s]);   // the stage is free once these MMAs have read it
            committed = i + 1;
        }
        tc_commit(acc);             // the accumulator is complete (or as far as it got)
    }

    // ---- epilogue: TMEM -> registers -> bf16 -> global
    const bool acc_ok = mbar_wait_bounded(acc, 0u);
    if (!acc_ok) *fail = 1;
    __syncwarp();          // the producer and MMA lanes rejoin their warps
    tc_fence_after();
    if (acc_ok && *fail == 0) {
        const int64_t row = m0 + warp * 32 + lane;
        const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
#pragma unroll 1
        for (int c = 0; c < BN; c += 16) {
            float v[16];
            tmem_ld16(lane_base + (uint32_t)c, v);   // every lane of the warp takes part
            if (row >= p.M) continue;
            const int col = n0 + c;
            // the segment holding this 16-column chunk, when it holds all of it
            __nv_bfloat16* o = nullptr;
#pragma unroll
            for (int q = 0; q < 3; ++q)   // static indices: the parameters stay in place
                if (q < p.nseg && col >= p.seg[q].col0 && col + 16 <= p.seg[q].col0 + p.seg[q].ncol)
                    o = static_cast<__nv_bfloat16*>(p.seg[q].ptr) + row * p.seg[q].ld + (col - p.seg[q].col0);
            if (o != nullptr && col + 16 <= p.N) {
                if ((reinterpret_cast<uintptr_t>(o) & 15) == 0) {   // two 16-byte stores
                    uint32_t w[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        __nv_bfloat162 pr = __floats2bfloat162_rn(v[2 * j], v[2 * j + 1]);
                        w[j] = *reinterpret_cast<uint32_t*>(&pr);
                    }
                    reinterpret_cast<uint4*>(o)[0] = make_uint4(w[0], w[1], w[2], w[3]);
                    reinterpret_cast<uint4*>(o)[1] = make_uint4(w[4], w[5], w[6], w[7]);
                    continue;
                }
            }
#pragma unroll
            for (int j = 0; j < 16; ++j) {   // column by column
                if (col + j >= p.N) break;
#pragma unroll
                for (int q = 0; q < 3; ++q) {
                    if (q >= p.nseg) break;
                    if (col + j >= p.seg[q].col0 && col + j < p.seg[q].col0 + p.seg[q].ncol) {
                        __nv_bfloat16* o = static_cast<__nv_bfloat16*>(p.seg[q].ptr);
                        o[row * p.seg[q].ld + (col + j - p.seg[q].col0)] = __float2bfloat16_rn(v[j]);
                    }
                }
            }
        }
    }
    if (*fail && threadIdx.x == 0) atomicExch(&g_ssm_device_error, kDevErrTimeout);
    // in-flight copies of a failed CTA land before its shared memory is released
    if (warp == 0 && lane == 0 && *fail) {
        for (int i = issued - S > 0 ? issued - S : 0; i < issued; ++i)
            mbar_wait_bounded(&full[i % S], (uint32_t)((i / S) & 1), 100000000ull);
    }
    (void)committed;
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        __syncwarp();
        tmem_dealloc(tmem, Cfg::TMEM_COLS);
    }
}

// ---------------------------------------------------------------------------
// Persistent form for output-heavy products with a short K loop (dt_proj:
// K = dt_rank, C = tokens x dim): a CTA keeps one N tile, whose B rows (all
// of K) it loads into shared memory once, and walks M tiles, so only the A
// tiles stream through the ring (half the operand bytes of re-reading both
// per tile, and a ring twice as deep in tiles).  The grid is a multiple of
// the N tiles: CTA c takes N tile c % ntn and M tiles c / ntn, c / ntn + g,
// ... (g CTAs per N tile).  Two TMEM accumulators: while the epilogue warps
// drain tile j, the producer and the MMA thread are already on tile j + 1.
//   warp 0 lane 0: TMA producer (B once, then the A ring across tiles)
//   warp 1 lane 0: MMA issuer; acc_full[a] <- commit, waits acc_empty[a]
//   warps 2..9   : epilogue; warp w reads TMEM lanes 32 (w % 4) .. and half
//                  of the tile's columns (two warps per lane quarter: the
//                  epilogue, not the MMA, bounds this output-heavy GEMM, and
//                  8 warps beat 4 and 16, measured); rows go through a
//                  padded shared-memory tile and leave as whole row pieces
//                  (coalesced), then acc_empty[a] is released.
#ifndef SSM_GP_EPI
#define SSM_GP_EPI 8
#endif
constexpr int kGemmPEpi = SSM_GP_EPI;
static_assert(kGemmPEpi % 4 == 0, "whole lane quarters");
constexpr int kGemmPThreads = 64 + 32 * kGemmPEpi;

template <int BN, int STAGES>
struct GemmPCfg {
    static_assert(BN % 16 == 0 && BN >= 16 && BN <= 128, "two accumulators of BN columns in 256");
    static constexpr int S = STAGES;
    static constexpr int A_BYTES = kGemmBM * kGemmBK * 2;
    static constexpr int B_BYTES = BN * kGemmBK * 2;                // one K slab of the N tile
    static constexpr int STAGE = (A_BYTES + 1023) / 1024 * 1024;    // the ring holds A slabs
    static constexpr int B_SLAB = (B_BYTES + 1023) / 1024 * 1024;
    static constexpr int ROWB = BN * 2 + 16;                        // padded output row (bytes)
    static constexpr int OFF_B = S * STAGE;                         // nk resident B slabs
    // after the B slabs (nk of them): the output rows, then full[S], empty[S],
    // acc_full[2], acc_empty[2], bfull; the TMEM address word; the fail word
    __host__ __device__ static constexpr int off_out(int nk) { return OFF_B + nk * B_SLAB; }
    __host__ __device__ static constexpr int off_bar(int nk) { return off_out(nk) + kGemmBM * ROWB; }
    __host__ __device__ static constexpr int off_tmem(int nk) { return off_bar(nk) + (2 * S + 5) * 8; }
    __host__ __device__ static constexpr int smem(int nk) { return off_tmem(nk) + 16 + 1024; }
    static constexpr int ACC_COLS = BN <= 32 ? 32 : BN <= 64 ? 64 : 128;
    static constexpr int TMEM_COLS = 2 * ACC_COLS;
};

template <int BN, int STAGES>
__global__ void __launch_bounds__(kGemmPThreads, 1)
    gemm_bf16_tn_persistent_kernel(const __grid_constant__ GemmMaps maps, const GemmParams p) {
    using Cfg = GemmPCfg<BN, STAGES>;
    constexpr int S = Cfg::S;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    const int nk = (p.K + kGemmBK - 1) / kGemmBK;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + Cfg::off_bar(nk));
    uint64_t* empty = full + S;
    uint64_t* acc_full = empty + S;
    uint64_t* acc_empty = acc_full + 2;
    uint64_t* bfull = acc_empty + 2;
    uint32_t* tmem_word = reinterpret_cast<uint32_t*>(smem + Cfg::off_tmem(nk));
    volatile uint32_t* fail = tmem_word + 1;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int mtiles = (int)((p.M + kGemmBM - 1) / kGemmBM);
    const int ntn = (p.N + BN - 1) / BN;
    // this CTA's N tile and M tiles mt0, mt0 + g, ... (no work past ntn * g)
    const int g = (int)gridDim.x / ntn;
    const int nt = (int)blockIdx.x % ntn;
    const int mt0 = (int)blockIdx.x < ntn * g ? (int)blockIdx.x / ntn : mtiles;
    const int n0 = nt * BN;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&acc_full[a], 1);
            mbar_init(&acc_empty[a], 32 * kGemmPEpi);
        }
        mbar_init(bfull, 1);
        *fail = 0;
        fence_barrier_init();
    }
    if (warp == 0) {
        __syncwarp();
        tmem_alloc(tmem_word, Cfg::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_word;

    int issued = 0;
    bool b_issued = false;
    if (warp == 0 && lane == 0) {
        // ---- TMA producer: the N tile's B slabs once, then the A slabs of each tile
        prefetch_tmap(&maps.a);
        prefetch_tmap(&maps.b);
        if (mt0 < mtiles) {
            mbar_arrive_expect_tx(bfull, (uint32_t)(nk * Cfg::B_BYTES));
            for (int i = 0; i < nk; ++i)
                tma_load_2d(smem + Cfg::OFF_B + i * Cfg::B_SLAB, &maps.b, bfull, i * kGemmBK, n0);
            b_issued = true;
        }
        int it = 0;   // slab counter across tiles
        for (int mt = mt0; mt < mtiles && !*fail; mt += g) {
            const int64_t m0 = (int64_t)mt * kGemmBM;
            for (int i = 0; i < nk; ++i, ++it) {
                const int s = it % S;
                if (it >= S && !mbar_wait_bounded(&empty[s], (uint32_t)(((it / S) - 1) & 1))) {
                    *fail = 1;
                    break;
                }
                unsigned char* st = smem + s * Cfg::STAGE;
                mbar_arrive_expect_tx(&full[s], (uint32_t)Cfg::A_BYTES);
                tma_load_2d(st, &maps.a, &full[s], i * kGemmBK, (int)m0);
                issued = it + 1;
            }
        }
    } else if (warp == 1 && lane == 0) {
        // ---- MMA issuer
        constexpr uint32_t idesc = idesc_bf16_f32(kGemmBM, BN);
        if (mt0 < mtiles && !mbar_wait_bounded(bfull, 0u)) *fail = 1;
        int it = 0, j = 0;
        for (int mt = mt0; mt < mtiles && !*fail; mt += g, ++j) {
            const int a = j & 1;
            const int use = j >> 1;
            if (use >= 1 && !mbar_wait_bounded(&acc_empty[a], (uint32_t)((use - 1) & 1))) {
                *fail = 1;
                break;
            }
            tc_fence_after();
            const uint32_t d = tmem + (uint32_t)(a * Cfg::ACC_COLS);
            for (int i = 0; i < nk; ++i, ++it) {
                const int s = it % S;
                if (!mbar_wait_bounded(&full[s], (uint32_t)((it / S) & 1))) {
                    *fail = 1;
                    break;
                }
                tc_fence_after();
                const uint32_t a0 = smem_addr(smem + s * Cfg::STAGE);
                const uint32_t b0 = smem_addr(smem + Cfg::OFF_B + i * Cfg::B_SLAB);
#pragma unroll
                for (int kk = 0; kk < kGemmBK / 16; ++kk)
                    tc_mma(d, smem_desc_sw128(a0 + kk * 32), smem_desc_sw128(b0 + kk * 32), idesc,
                           (i > 0 || kk > 0) ? 1u : 0u);
                tc_commit(&empty[s]);
            }
            tc_commit(&acc_full[a]);
            if (*fail) break;
        }
    } else if (warp >= 2) {
        // ---- epilogue
        const int q = warp & 3;                               // TMEM lane quarter of this warp
        constexpr int HALVES = kGemmPEpi / 4;                 // warps per lane quarter
        constexpr int CW = BN / HALVES;                       // columns of this warp
        const int c0 = ((warp - 2) / 4) * CW;
        unsigned char* const out_tile = smem + Cfg::off_out(nk);
        unsigned char* outrow = out_tile + (q * 32 + lane) * Cfg::ROWB;
        __nv_bfloat16* C = static_cast<__nv_bfloat16*>(p.seg[0].ptr);
        const int64_t ld = p.seg[0].ld;
        int j = 0;
        for (int mt = mt0; mt < mtiles; mt += g, ++j) {
            const int a = j & 1;
            if (!mbar_wait_bounded(&acc_full[a], (uint32_t)((j >> 1) & 1))) {
                *fail = 1;
                break;
            }
            __syncwarp();
            tc_fence_after();
            const uint32_t base = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(a * Cfg::ACC_COLS);
            const int n0e = n0;
#pragma unroll 1
            for (int c = c0; c < c0 + CW; c += 16) {
                float vv[16];
                tmem_ld16(base + (uint32_t)c, vv);
                if (p.col_bias || p.act) {   // the step Delta = softplus(c + bias), finished here
#pragma unroll
                    for (int k2 = 0; k2 < 16; ++k2) {
                        const int col = n0e + c + k2;
                        float u = vv[k2] + ((p.col_bias && col < p.N) ? __ldg(p.col_bias + col) : 0.f);
                        vv[k2] = p.act ? softplus_tiled<__nv_bfloat16>(u) : u;
                    }
                }
                uint32_t w[8];
#pragma unroll
                for (int k2 = 0; k2 < 8; ++k2) {
                    __nv_bfloat162 pr = __floats2bfloat162_rn(vv[2 * k2], vv[2 * k2 + 1]);
                    w[k2] = *reinterpret_cast<uint32_t*>(&pr);
                }
                reinterpret_cast<uint4*>(outrow + c * 2)[0] = make_uint4(w[0], w[1], w[2], w[3]);
                reinterpret_cast<uint4*>(outrow + c * 2)[1] = make_uint4(w[4], w[5], w[6], w[7]);
            }
            tc_fence_before();
            mbar_arrive(&acc_empty[a]);   // TMEM buffer a may be overwritten now
            __syncwarp();
            // the warp's 32 rows leave as whole pieces of CW columns: lane l writes 16 bytes
            const int64_t m0 = (int64_t)mt * kGemmBM;
            constexpr int CH16 = CW * 2 / 16;                 // 16-byte chunks per row piece
            constexpr int RPI = 32 / CH16 > 0 ? 32 / CH16 : 1;   // rows per warp instruction
#pragma unroll 4
            for (int r0 = 0; r0 < 32; r0 += RPI) {
                const int r = r0 + lane / CH16;
                const int ch = lane % CH16;
                if (lane / CH16 >= RPI) continue;
                const int64_t row = m0 + q * 32 + r;
                const int col = n0 + c0 + ch * 8;
                if (row >= p.M || col >= p.N) continue;
                const uint4 val = *reinterpret_cast<const uint4*>(
                    out_tile + (q * 32 + r) * Cfg::ROWB + (c0 + ch * 8) * 2);
                __nv_bfloat16* dst = C + row * ld + col;
                if (col + 8 <= p.N && (reinterpret_cast<uintptr_t>(dst) & 15) == 0) {
                    *reinterpret_cast<uint4*>(dst) = val;
                } else {
                    const __nv_bfloat16* e = reinterpret_cast<const __nv_bfloat16*>(&val);
                    for (int k2 = 0; k2 < 8 && col + k2 < p.N; ++k2) dst[k2] = e[k2];
                }
            }
            __syncwarp();   // the staging rows are rewritten by the next tile
        }
    }
    if (*fail && threadIdx.x == 0) atomicExch(&g_ssm_device_error, kDevErrTimeout);
    if (warp == 0 && lane == 0 && *fail) {
        // after a timeout, let the loads still in flight land before the CTA's
        // shared memory is released
        if (b_issued) mbar_wait_bounded(bfull, 0u, 100000000ull);
        for (int i = issued - S > 0 ? issued - S : 0; i < issued; ++i)
            mbar_wait_bounded(&full[i % S], (uint32_t)((i / S) & 1), 100000000ull);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        __syncwarp();
        tmem_dealloc(tmem, Cfg::TMEM_COLS);
    }
}

}  // namespace ssm
