// scan_warp.cuh -- single-warp selective scan (path 3; bf16 or fp32 I/O,
// dstate 8, 16, 32 or 64).
//
// A CTA is one warp and owns 16 channels of one sequence over a range of
// time steps, walked in tiles of 16 steps.  TMA brings the x, delta, z tiles
// [16 steps][16 channels] and the B, C tiles [16][N] into a ring of shared
// stages.  Lane (p, s) = (lane & 7, lane >> 3) owns the channel pair
// (2p, 2p + 1) and the states [K s, K (s + 1)), K = N / 4, of both channels;
// the pair's two channels ride in the two halves of every f32x2 register, so
// one B[n] or C[n] value read from shared memory serves two channels.
//
// Per tile the warp does three things:
//   pre-pass  (lane p, steps s, s + 4, s + 8, s + 12): Delta' = softplus(delta +
//             bias) log2 e and Delta x = (Delta' ln 2) x for its channel pair,
//             once per token; B and C widened to fp32;
//   scan      per step, for each of its states
//               dA = 2^(Delta' A[n])   h = dA h + (Delta x) B[n]
//               y_s += C[n] h
//             (Delta' A = Delta A log2 e),
//             leaving one partial readout per state quarter;
//   post-pass (same lanes as the pre-pass): y = (sum of the four partial
//             readouts + D x) silu(z), cast, and one TMA store of the tile.
// Iteration j runs the scan of tile j, the pre-pass of tile j + 1 and the
// post-pass of tile j - 1 as one block of independent work, with every shared
// load before every shared store, so the compiler can interleave the three.
// There is no other warp and no block barrier: the warps of an SM are
// independent CTAs.
//
// MODE_AGG gives a chunk's end state from a zero start and its sum of Delta
// (no z, C, readout or output), for the cross-chunk carry.  MODE_STATES runs
// a chunk from its start state and writes the state before every tile (the
// checkpoints the backward reads), with no readout or output either.
//
// This is the recurrent mode of the selective SSM (stage 2 in
// "Mamba的三大创新") with the Mamba block's gate and skip fused in; the
// expanded state (B, L, D, N) is never materialised.
#pragma once
#include "common.cuh"
#include "scan_generic.cuh"
#include "tile_io.cuh"
#include "tma.cuh"

#ifndef SSM_WARP_STAGES
#define SSM_WARP_STAGES 8   // TMA ring depth for dstate <= 16 (tiles in flight ahead of the compute)
#endif

namespace ssm {

// Larger states take longer per tile, so fewer tiles in flight cover the same
// memory latency, and the stages are larger: 8 stages up to dstate 16, 4 at
// 32 and 3 at 64 keep the CTA's shared memory near 24-32 KB (power-of-two
// counts make the stage index a mask).
template <typename IO, int N_, int S_ = (N_ <= 16 ? SSM_WARP_STAGES : N_ == 32 ? 4 : 3)>
struct WarpCfg {
    static constexpr int N = N_, K = N / 4, DC = 16, NP = 8, T = 16, S = S_;
    // resident CTAs per SM the register budget must allow (255 registers a thread)
    static constexpr int MINB = 8;
    static_assert(N == 8 || N == 16 || N == 32 || N == 64, "dstate 8, 16, 32 or 64");
    static constexpr int ESZ = (int)sizeof(IO);
    static constexpr int TOK_BYTES = T * DC * ESZ;   // one x / delta / z / out tile
    static constexpr int BC_BYTES = T * N * ESZ;     // one B / C tile
    static constexpr int OFF_X = 0;
    static constexpr int OFF_DL = OFF_X + TOK_BYTES;
    static constexpr int OFF_Z = OFF_DL + TOK_BYTES;
    static constexpr int OFF_B = OFF_Z + TOK_BYTES;
    static constexpr int OFF_C = OFF_B + BC_BYTES;
    static constexpr int STAGE = round_up(OFF_C + BC_BYTES, 128);
    static constexpr int OFF_DD = S * STAGE;                  // float4 [T][NP]
    static constexpr int OFF_BC = OFF_DD + T * NP * 16;       // float [T][2N]: ln2 B | C
    static constexpr int OFF_Y = OFF_BC + T * 2 * N * 4;      // float2 [T][4][NP]
    static constexpr int OFF_OB = round_up(OFF_Y + T * 4 * NP * 8, 128);   // IO [2][T][DC]
    static constexpr int OFF_BAR = OFF_OB + 2 * TOK_BYTES;
    static constexpr int SMEM = OFF_BAR + S * 8;
    static constexpr int BC_CHUNKS = T * 2 * N / 4;           // 16-byte chunks of one fp32 B|C tile
    static constexpr int BC_PER_LANE = (BC_CHUNKS + 31) / 32;
    static_assert(TOK_BYTES % 128 == 0 && BC_BYTES % 128 == 0, "TMA boxes stay 128-byte aligned");
};

// Delta' = softplus(u) log2 e for a channel pair.  bf16 I/O: log2(1 + 2^(u log2 e))
// on the SFU (exact to fp32 below the clamp; above it log2(1 + 2^v) = v to fp32
// and the max returns v itself).  fp32 I/O: the libm form.
template <typename IO>
__device__ __forceinline__ float2 softplus_log2e(float2 u);
template <>
__device__ __forceinline__ float2 softplus_log2e<__nv_bfloat16>(float2 u) {
    const float2 v = __fmul2_rn(u, make_float2(kLog2e, kLog2e));
    const float2 w = make_float2(ex2_sfu(fminf(v.x, 64.f)), ex2_sfu(fminf(v.y, 64.f)));
    const float2 q = __fadd2_rn(w, make_float2(1.f, 1.f));
    float l0, l1;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(l0) : "f"(q.x));
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(l1) : "f"(q.y));
    return make_float2(fmaxf(v.x, l0), fmaxf(v.y, l1));
}
template <>
__device__ __forceinline__ float2 softplus_log2e<float>(float2 u) {
    return make_float2(softplus_accurate(u.x) * kLog2e, softplus_accurate(u.y) * kLog2e);
}

// silu of a pair: bf16 I/O v / (1 + 2^(-v log2 e)) on the SFU, fp32 I/O libm.
template <typename IO>
__device__ __forceinline__ float2 silu2(float2 v);
template <>
__device__ __forceinline__ float2 silu2<__nv_bfloat16>(float2 v) {
    const float2 m = __fmul2_rn(v, make_float2(-kLog2e, -kLog2e));
    const float2 q = __fadd2_rn(make_float2(ex2_sfu(m.x), ex2_sfu(m.y)), make_float2(1.f, 1.f));
    float r0, r1;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r0) : "f"(q.x));
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r1) : "f"(q.y));
    return __fmul2_rn(v, make_float2(r0, r1));
}
template <>
__device__ __forceinline__ float2 silu2<float>(float2 v) {
    return make_float2(silu_accurate(v.x), silu_accurate(v.y));
}

// Packs two fp32 values as two io elements (one 32-bit word for bf16).
__device__ __forceinline__ void store_pair(float* p, float2 v) { *reinterpret_cast<float2*>(p) = v; }
__device__ __forceinline__ void store_pair(__nv_bfloat16* p, float2 v) {
    *reinterpret_cast<__nv_bfloat162*>(p) = __floats2bfloat162_rn(v.x, v.y);
}

// SP: Delta = softplus(delta + bias) (else delta + bias); ZG: the silu(z) gate;
// PJR: 0, or the rank R of dt_proj fused in front (delta = dt_low W_dt^T formed
// in the kernel, see below).
template <typename IO, typename Cfg, int MODE, bool SP, bool ZG, int PJR = 0>
struct WarpScan {
    static constexpr int N = Cfg::N, K = Cfg::K, DC = Cfg::DC, NP = Cfg::NP, T = Cfg::T, S = Cfg::S;
    static constexpr bool FULL = (MODE == MODE_FULL);

    // pre-pass results of one tile, stored after the loads of the iteration
    struct Pre {
        float4 dd[T / 4];                  // (Delta'_c0, Delta'_c1, Delta'x_c0, Delta'x_c1)
        float4 bc[Cfg::BC_PER_LANE];       // B | C widened
    };

    unsigned char* smem;
    const ScanParams* p;
    int lane, pp, s, d0, b;
    float2 bias2, dsk2;

    __device__ __forceinline__ const unsigned char* stage(int j) const {
        return smem + ((unsigned)j % (unsigned)S) * Cfg::STAGE;
    }
    __device__ __forceinline__ float4* dd() const { return reinterpret_cast<float4*>(smem + Cfg::OFF_DD); }
    __device__ __forceinline__ float* bc() const { return reinterpret_cast<float*>(smem + Cfg::OFF_BC); }
    __device__ __forceinline__ float2* ys() const { return reinterpret_cast<float2*>(smem + Cfg::OFF_Y); }
    // fused dt_proj: the raw step of tile j, fp32 [T][16], two buffers after the CTA's other storage
    __device__ __forceinline__ float* dtile(int j) const {
        return reinterpret_cast<float*>(smem + Cfg::SMEM + (j & 1) * T * DC * 4);
    }

    // ---- pre-pass of tile j: loads and arithmetic only, one token pair (steps
    // 4 i + s of this lane's channel pair) or one 16-byte chunk of B | C at a time
    __device__ __forceinline__ void pre_token(int j, int i, int steps, Pre& r, float2& dsum2) const {
        const unsigned char* stg = stage(j);
        const IO* xs = reinterpret_cast<const IO*>(stg + Cfg::OFF_X);
        const IO* ds = reinterpret_cast<const IO*>(stg + Cfg::OFF_DL);
        const int t = 4 * i + s;
        const float2 xv = load2(xs + t * DC + 2 * pp);
        float2 draw;
        if constexpr (PJR > 0) draw = *reinterpret_cast<const float2*>(dtile(j) + t * DC + 2 * pp);
        else draw = load2(ds + t * DC + 2 * pp);
        const float2 u = __fadd2_rn(draw, bias2);
        const float2 dl = SP ? softplus_log2e<IO>(u) : __fmul2_rn(u, make_float2(kLog2e, kLog2e));
        // Delta x = (Delta' ln 2) x: the input term of the scan
        const float2 dx = __fmul2_rn(__fmul2_rn(dl, make_float2(kLn2, kLn2)), xv);
        r.dd[i] = make_float4(dl.x, dl.y, dx.x, dx.y);
        if (MODE == MODE_AGG && t < steps) dsum2 = __fadd2_rn(dsum2, dl);
    }
    // 16-byte chunks of fp32 B | C per row (the aggregate pass widens B only)
    static constexpr int CHN = FULL ? 2 * N / 4 : N / 4;
    static constexpr int NCHUNK = T * CHN;
    static constexpr int CHUNKS_PER_LANE = (NCHUNK + 31) / 32;
    __device__ __forceinline__ void pre_bc(int j, int r2, Pre& r) const {
        const unsigned char* stg = stage(j);
        const IO* Bs = reinterpret_cast<const IO*>(stg + Cfg::OFF_B);
        const IO* Cs = reinterpret_cast<const IO*>(stg + Cfg::OFF_C);
        const int u = lane + 32 * r2;
        if (u >= NCHUNK) return;
        const int t = u / CHN;
        const int kk = (u % CHN) * 4;
        const IO* src = (kk < N ? Bs : Cs) + t * N + (kk % N);
        float f[4];
        if (sizeof(IO) == 2) {
            const uint2 v = *reinterpret_cast<const uint2*>(src);
            f[0] = __uint_as_float(v.x << 16); f[1] = __uint_as_float(v.x & 0xffff0000u);
            f[2] = __uint_as_float(v.y << 16); f[3] = __uint_as_float(v.y & 0xffff0000u);
        } else {
            const float4 v = *reinterpret_cast<const float4*>(src);
            f[0] = v.x; f[1] = v.y; f[2] = v.z; f[3] = v.w;
        }
        r.bc[r2] = make_float4(f[0], f[1], f[2], f[3]);
    }
    __device__ __forceinline__ void pre_compute(int j, int steps, Pre& r, float2& dsum2) const {
#pragma unroll
        for (int i = 0; i < T / 4; ++i) pre_token(j, i, steps, r, dsum2);
#pragma unroll
        for (int r2 = 0; r2 < CHUNKS_PER_LANE; ++r2) pre_bc(j, r2, r);
    }
    __device__ __forceinline__ void pre_store(const Pre& r) const {
#pragma unroll
        for (int i = 0; i < T / 4; ++i) dd()[(4 * i + s) * NP + pp] = r.dd[i];
#pragma unroll
        for (int r2 = 0; r2 < CHUNKS_PER_LANE; ++r2) {
            const int u = lane + 32 * r2;
            if (u < NCHUNK)   // row u / CHN, chunk u % CHN of the [T][2N] fp32 tile
                reinterpret_cast<float4*>(bc())[(u / CHN) * (2 * N / 4) + u % CHN] = r.bc[r2];
        }
    }

    // ---- one step of the recurrence for this lane's K states of both channels
    __device__ __forceinline__ float2 step(int t, float2 (&h)[K], const float2 (&a2)[K]) const {
        const float4 dq = dd()[t * NP + pp];
        const float* row = bc() + t * 2 * N + K * s;
        const float2 dl2 = make_float2(dq.x, dq.y);
        const float2 dx2 = make_float2(dq.z, dq.w);
        float2 y2 = make_float2(0.f, 0.f);
#pragma unroll
        for (int q4 = 0; q4 < K; q4 += 4) {
            float bv[4] = {0.f, 0.f, 0.f, 0.f}, cv[4] = {0.f, 0.f, 0.f, 0.f};
            if constexpr (K >= 4) {
                const float4 b4 = *reinterpret_cast<const float4*>(row + q4);
                bv[0] = b4.x; bv[1] = b4.y; bv[2] = b4.z; bv[3] = b4.w;
                if (FULL) {
                    const float4 c4 = *reinterpret_cast<const float4*>(row + N + q4);
                    cv[0] = c4.x; cv[1] = c4.y; cv[2] = c4.z; cv[3] = c4.w;
                }
            } else {   // dstate 8: two states per lane
                const float2 b2 = *reinterpret_cast<const float2*>(row);
                bv[0] = b2.x; bv[1] = b2.y;
                if (FULL) {
                    const float2 c2 = *reinterpret_cast<const float2*>(row + N);
                    cv[0] = c2.x; cv[1] = c2.y;
                }
            }
#pragma unroll
            for (int r = 0; r < 4 && q4 + r < K; ++r) {
                const int q = q4 + r;
                const float2 arg = __fmul2_rn(dl2, a2[q]);
                const float2 dA = make_float2(ex2_sfu(arg.x), ex2_sfu(arg.y));
                h[q] = __ffma2_rn(dA, h[q], __fmul2_rn(dx2, make_float2(bv[r], bv[r])));
                if (FULL) y2 = __ffma2_rn(make_float2(cv[r], cv[r]), h[q], y2);
            }
        }
        return y2;
    }

    // ---- post-pass of tile j: loads and arithmetic only, one token pair at a time
    __device__ __forceinline__ void post_token(int j, int i, float2 (&yo)[T / 4]) const {
        const unsigned char* stg = stage(j);
        const IO* xs = reinterpret_cast<const IO*>(stg + Cfg::OFF_X);
        const IO* zs = reinterpret_cast<const IO*>(stg + Cfg::OFF_Z);
        const int t = 4 * i + s;
        // the four partial readouts, rotated so a quarter-warp's reads spread over the banks
        const float2* yr = ys() + t * 4 * NP + pp;
        float2 y = __fadd2_rn(__fadd2_rn(yr[(s & 3) * NP], yr[((s + 1) & 3) * NP]),
                              __fadd2_rn(yr[((s + 2) & 3) * NP], yr[((s + 3) & 3) * NP]));
        y = __ffma2_rn(dsk2, load2(xs + t * DC + 2 * pp), y);
        if (ZG) y = __fmul2_rn(y, silu2<IO>(load2(zs + t * DC + 2 * pp)));
        yo[i] = y;
    }
    __device__ __forceinline__ void post_compute(int j, float2 (&yo)[T / 4]) const {
#pragma unroll
        for (int i = 0; i < T / 4; ++i) post_token(j, i, yo);
    }
    __device__ __forceinline__ void post_store(int j, const float2 (&yo)[T / 4]) const {
        IO* ob = reinterpret_cast<IO*>(smem + Cfg::OFF_OB + (j & 1) * Cfg::TOK_BYTES);
#pragma unroll
        for (int i = 0; i < T / 4; ++i) store_pair(ob + (4 * i + s) * DC + 2 * pp, yo[i]);
    }
};

// PJR > 0 (bf16 I/O): dt_proj fused in front.  The raw step of tile m,
// delta_raw[t][c] = sum_r dt_low[t][r] W_dt[d0 + c][r] over the tile's 16 steps
// and 16 channels, is a [16 x R] x [R x 16] product: R / 16 k-steps of two
// m16n8k16 tensor-core products (channels 0-7 and 8-15), fp32 accumulation.
// The reduction index is permuted so that every lane's operands are contiguous:
// lane (g, q) = (lane / 4, lane % 4) covers r in [q R/4, (q + 1) R/4), and
// k-step kk takes r = q R/4 + 4 kk + {0, 1} for the fragment's k = 2q, 2q + 1
// and + {2, 3} for k = 2q + 8, 2q + 9 (the same permutation on both operands
// leaves the sum unchanged).  W_dt's fragments stay in registers; the dt_low
// rows g and g + 8 of a tile are loaded from global memory (L2: one sequence's
// dt_low is read by all its channel blocks) right before their product, two
// tiles ahead of their use, and the product lands in a double-buffered fp32
// tile that the pre-pass reads in place of the delta tile.
// CK: the kernel writes checkpoints (p.ckpt) -- the training forward and
// MODE_STATES; the plain forward is compiled without that code (its mere
// presence costs the plain forward 5%: measured 0.751 against 0.711 ms on the
// Mamba-1.4B layer).
template <typename IO, typename Cfg, int MODE, bool SP, bool ZG, int PJR = 0, bool CK = false>
__global__ void __launch_bounds__(32, Cfg::MINB)
    scan_warp_kernel(const __grid_constant__ TiledMaps maps, const ScanParams p) {
    using W = WarpScan<IO, Cfg, MODE, SP, ZG, PJR>;
    constexpr bool PJ = PJR > 0;
    static_assert(!PJ || (PJR % 32 == 0 && PJR <= 128 && sizeof(IO) == 2), "fused dt_proj: bf16, R = 32 .. 128");
    constexpr int N = Cfg::N, K = Cfg::K, DC = Cfg::DC, NP = Cfg::NP, T = Cfg::T, S = Cfg::S;
    constexpr bool FULL = (MODE == MODE_FULL);
    extern __shared__ __align__(1024) unsigned char smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + Cfg::OFF_BAR);

    W w;
    w.smem = smem;
    w.p = &p;
    w.lane = threadIdx.x;
    w.pp = w.lane & 7;
    w.s = w.lane >> 3;
    w.d0 = blockIdx.x * DC;
    w.b = blockIdx.y;
    const int lane = w.lane, pp = w.pp, s = w.s, d0 = w.d0, b = w.b;
    const int k = blockIdx.z;
    const int64_t t_begin = (int64_t)k * p.chunk_len;
    int64_t t_end = t_begin + p.chunk_len;
    if (t_end > p.seqlen) t_end = p.seqlen;
    const int ntiles = t_end > t_begin ? (int)((t_end - t_begin + T - 1) / T) : 0;
    constexpr bool z_on = FULL && ZG;
    const uint32_t stage_tx = (uint32_t)(Cfg::TOK_BYTES * ((z_on ? 3 : 2) - (PJ ? 1 : 0)) +
                                         Cfg::BC_BYTES * (FULL ? 2 : 1));
    auto issue = [&](int j) {   // TMA loads of tile j into stage j % S (lane 0)
        const unsigned sj = (unsigned)j % S;
        unsigned char* st = smem + sj * Cfg::STAGE;
        const int t0 = (int)(t_begin + (int64_t)j * T);
        mbar_arrive_expect_tx(&full[sj], stage_tx);
        tma_load_3d(st + Cfg::OFF_X, &maps.x, &full[sj], d0, t0, b);
        if (!PJ) tma_load_3d(st + Cfg::OFF_DL, &maps.delta, &full[sj], d0, t0, b);
        if (z_on) tma_load_3d(st + Cfg::OFF_Z, &maps.z, &full[sj], d0, t0, b);
        tma_load_3d(st + Cfg::OFF_B, &maps.B, &full[sj], 0, t0, b);
        if (FULL) tma_load_3d(st + Cfg::OFF_C, &maps.C, &full[sj], 0, t0, b);
    };
    auto steps_of = [&](int j) {
        const int64_t left = t_end - (t_begin + (int64_t)j * T);
        return (int)(left < T ? left : T);
    };

    if (lane == 0) {
        for (int q = 0; q < S; ++q) mbar_init(&full[q], 1);
        fence_barrier_init();
        prefetch_tmap(&maps.x);
        if (!PJ) prefetch_tmap(&maps.delta);
        prefetch_tmap(&maps.B);
        if (FULL) {
            prefetch_tmap(&maps.C);
            prefetch_tmap(&maps.out);
            if (z_on) prefetch_tmap(&maps.z);
        }
        for (int j = 0; j < S && j < ntiles; ++j) issue(j);
    }
    __syncwarp();

    // channel pair (c0, c0 + 1) of this lane
    const int c0 = 2 * pp;
    const bool v0 = d0 + c0 < p.dim, v1 = d0 + c0 + 1 < p.dim;
    w.bias2 = make_float2((p.delta_bias && v0) ? __ldg(p.delta_bias + d0 + c0) : 0.f,
                          (p.delta_bias && v1) ? __ldg(p.delta_bias + d0 + c0 + 1) : 0.f);
    w.dsk2 = make_float2((FULL && p.D && v0) ? __ldg(p.D + d0 + c0) : 0.f,
                         (FULL && p.D && v1) ? __ldg(p.D + d0 + c0 + 1) : 0.f);
    // states [K s, K s + K) of both channels, the pair in the halves of an f32x2
    float2 a2[K], h[K];
    {
        const int64_t ch0 = (int64_t)b * p.dim + d0 + c0;
        const float* src = nullptr;
        if (MODE != MODE_AGG) {
            if (p.nchunk > 1) src = p.carry + (((int64_t)b * p.nchunk + k) * p.dim + d0 + c0) * N;
            else if (p.initial_state) src = p.initial_state + ch0 * N;
        }
#pragma unroll
        for (int q = 0; q < K; ++q) {
            const int n = K * s + q;
            a2[q] = make_float2(v0 ? __ldg(p.A + (int64_t)(d0 + c0) * N + n) : 0.f,
                                v1 ? __ldg(p.A + (int64_t)(d0 + c0 + 1) * N + n) : 0.f);
            h[q] = make_float2((src && v0) ? src[n] : 0.f, (src && v1) ? src[N + n] : 0.f);
        }
    }

    // ---- fused dt_proj (PJ): W_dt fragments in registers, dt_low rows one tile ahead
    constexpr int RW = PJ ? PJR / 8 : 1;   // 32-bit words (bf16 pairs) of a lane's R/4 slice of a row
    uint32_t wf[2][RW], ad[2][RW];
    const int pg = lane >> 2, pq = lane & 3;
    if constexpr (PJ) {
        const __nv_bfloat16* Wd = static_cast<const __nv_bfloat16*>(p.W_dt);
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            const int64_t c = (int64_t)d0 + 8 * nt + pg;
            const uint4* src = reinterpret_cast<const uint4*>(Wd + c * PJR + (PJR / 4) * pq);
#pragma unroll
            for (int v = 0; v < RW / 4; ++v) {
                const uint4 u4 = c < p.dim ? __ldg(src + v) : make_uint4(0u, 0u, 0u, 0u);
                wf[nt][4 * v] = u4.x; wf[nt][4 * v + 1] = u4.y;
                wf[nt][4 * v + 2] = u4.z; wf[nt][4 * v + 3] = u4.w;
            }
        }
    }
    auto pj_load = [&](int m) {   // dt_low rows g, g + 8 of tile m (zeros past the sequence)
        if constexpr (PJ) {
            const __nv_bfloat16* dl = static_cast<const __nv_bfloat16*>(p.dt_low);
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
                const int64_t t = t_begin + (int64_t)m * T + pg + 8 * rr;
                const bool in = m < ntiles && t < p.seqlen;
                const uint4* src = reinterpret_cast<const uint4*>(
                    dl + (((int64_t)b * p.seqlen + (in ? t : 0)) * PJR + (PJR / 4) * pq));
#pragma unroll
                for (int v = 0; v < RW / 4; ++v) {
                    const uint4 u4 = in ? __ldg(src + v) : make_uint4(0u, 0u, 0u, 0u);
                    ad[rr][4 * v] = u4.x; ad[rr][4 * v + 1] = u4.y;
                    ad[rr][4 * v + 2] = u4.z; ad[rr][4 * v + 3] = u4.w;
                }
            }
        }
    };
    auto pj_product = [&](int m) {   // the raw step of tile m into its fp32 tile
        if constexpr (PJ) {
            float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
            for (int kk = 0; kk < PJR / 16; ++kk)
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
                    mma_bf16_16816(acc[nt], ad[0][2 * kk], ad[1][2 * kk], ad[0][2 * kk + 1],
                                   ad[1][2 * kk + 1], wf[nt][2 * kk], wf[nt][2 * kk + 1]);
            float* dt = w.dtile(m);
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                *reinterpret_cast<float2*>(dt + pg * DC + 8 * nt + 2 * pq) = make_float2(acc[nt][0], acc[nt][1]);
                *reinterpret_cast<float2*>(dt + (pg + 8) * DC + 8 * nt + 2 * pq) =
                    make_float2(acc[nt][2], acc[nt][3]);
            }
        }
    };
    if constexpr (PJ) {   // the raw steps of tiles 0 and 1 before the prologue
        pj_load(0);
        pj_product(0);
        pj_load(1);
        pj_product(1);
        __syncwarp();
    }

    float2 dsum2 = make_float2(0.f, 0.f);   // AGG: sum of Delta' over this lane's tokens
    bool ok = true;
    int issued = ntiles < S ? ntiles : S;   // tiles whose TMA loads were issued
    int waited = 0;                         // tiles whose loads were seen to land
    auto wait_stage = [&](int j) {
        const bool landed = __all_sync(0xffffffffu, mbar_wait_bounded(&full[(unsigned)j % S],
                                                                      (uint32_t)(((unsigned)j / S) & 1)));
        if (landed) waited = j + 1;
        return landed;
    };
    auto issue_next = [&]() {   // the stage of tile issued - S is read by no one now
        if (issued < ntiles) {
            if (lane == 0) issue(issued);
            ++issued;
        }
    };
    auto ckpt_store = [&](int j) {   // training forward: the state before tile j (T = 16 steps)
        if constexpr (CK && MODE != MODE_AGG) {
            if (!p.ckpt) return;
            const int64_t tile = t_begin / T + j;
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                if (!(c ? v1 : v0)) continue;
                float* ck = p.ckpt + ((((int64_t)b * p.ckpt_tiles + tile) * p.dim + d0 + c0 + c) * N) + K * s;
                if constexpr (K % 4 == 0) {   // 16-byte stores (K s floats from a 16-byte aligned row)
#pragma unroll
                    for (int q = 0; q < K; q += 4)
                        *reinterpret_cast<float4*>(ck + q) =
                            c ? make_float4(h[q].y, h[q + 1].y, h[q + 2].y, h[q + 3].y)
                              : make_float4(h[q].x, h[q + 1].x, h[q + 2].x, h[q + 3].x);
                } else {
#pragma unroll
                    for (int q = 0; q < K; ++q) ck[q] = c ? h[q].y : h[q].x;
                }
            }
        }
    };
    // output tile jp leaves by TMA store from ob[jp & 1]
    auto finish_post = [&](int jp, const float2 (&yo)[T / 4]) {
        w.post_store(jp, yo);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            tma_store_3d(&maps.out, smem + Cfg::OFF_OB + (jp & 1) * Cfg::TOK_BYTES, d0,
                         (int)(t_begin + (int64_t)jp * T), b);
            bulk_commit();
        }
    };

    // prologue: the pre-pass of tile 0
    if (ntiles > 0) {
        ok = wait_stage(0);
        if (ok) {
            typename W::Pre pr;
            w.pre_compute(0, steps_of(0), pr, dsum2);
            __syncwarp();
            w.pre_store(pr);
            if (!FULL) issue_next();   // the aggregate pass has no post-pass: stage 0 is free
            __syncwarp();
        }
    }
    for (int j = 0; ok && j < ntiles; ++j) {
        const int steps = steps_of(j);
        const bool has_pre = j + 1 < ntiles;
        const bool has_post = FULL && j >= 1;
        if (has_pre && !wait_stage(j + 1)) { ok = false; break; }
        ckpt_store(j);
        if (has_post && lane == 0) bulk_wait_read<1>();   // the store that last read ob[(j - 1) & 1]
        typename W::Pre pr;
        float2 yo[T / 4];
        if (steps == T && has_pre && (has_post || !FULL)) {
            // ---- the steady state: loads and arithmetic of the three parts as one block
            // the per-token work of the neighbouring tiles is spread over the
            // steps in source order, so the scheduler starts from an interleaving
            float2 yp[T];
            const int steps_next = steps_of(j + 1);
#pragma unroll
            for (int t = 0; t < T; ++t) {
                yp[t] = w.step(t, h, a2);
                if (t % 4 == 0) w.pre_token(j + 1, t / 4, steps_next, pr, dsum2);
                if (FULL && t % 4 == 2) w.post_token(j - 1, t / 4, yo);
#pragma unroll
                for (int r2 = t * W::CHUNKS_PER_LANE / T; r2 < (t + 1) * W::CHUNKS_PER_LANE / T; ++r2)
                    w.pre_bc(j + 1, r2, pr);
            }
            __syncwarp();
            // ---- then the stores
            w.pre_store(pr);
            if (FULL) {
#pragma unroll
                for (int t = 0; t < T; ++t) w.ys()[(t * 4 + s) * NP + pp] = yp[t];
            }
        } else {
            // first, last or partial tile
            if (has_post) w.post_compute(j - 1, yo);
            if (has_pre) w.pre_compute(j + 1, steps_of(j + 1), pr, dsum2);
            __syncwarp();
            for (int t = 0; t < steps; ++t) {
                const float2 y2 = w.step(t, h, a2);
                if (FULL) w.ys()[(t * 4 + s) * NP + pp] = y2;
            }
            __syncwarp();
            if (has_pre) w.pre_store(pr);
        }
        // the raw step of tile j + 2 (read by its pre-pass in the next iteration);
        // dtile((j + 2) & 1) was last read by the pre-pass of tile j
        pj_load(j + 2);
        pj_product(j + 2);
        if (has_post) finish_post(j - 1, yo);
        if (has_post || (!FULL && has_pre)) issue_next();
        __syncwarp();
    }
    // epilogue: the post-pass of the last tile
    if (ok && FULL && ntiles > 0) {
        float2 yo[T / 4];
        if (lane == 0) bulk_wait_read<1>();
        w.post_compute(ntiles - 1, yo);
        __syncwarp();
        finish_post(ntiles - 1, yo);
    }
    if (lane == 0) {
        bulk_wait<0>();
        // after a timeout, let the loads already issued land before the CTA's
        // shared memory is released
        if (!ok)
            for (int jj = waited; jj < issued; ++jj)
                mbar_wait_bounded(&full[jj % S], (uint32_t)((jj / S) & 1), 100000000ull);
    }
    if (!ok) return;

    if (MODE == MODE_STATES) return;
    if (!FULL) {
        // the chunk's sum of Delta: lanes s = 0..3 of a channel pair hold partial sums
        dsum2.x += __shfl_xor_sync(0xffffffffu, dsum2.x, 8);
        dsum2.y += __shfl_xor_sync(0xffffffffu, dsum2.y, 8);
        dsum2.x += __shfl_xor_sync(0xffffffffu, dsum2.x, 16);
        dsum2.y += __shfl_xor_sync(0xffffffffu, dsum2.y, 16);
        if (s == 0) {
            float* dst = p.dsum + ((int64_t)b * p.nchunk + k) * p.dim + d0 + c0;
            if (v0) dst[0] = dsum2.x * kLn2;
            if (v1) dst[1] = dsum2.y * kLn2;
        }
    }
#pragma unroll
    for (int c = 0; c < 2; ++c) {
        if (!(c ? v1 : v0)) continue;
        float* dst = nullptr;
        const int64_t ch = (int64_t)b * p.dim + d0 + c0 + c;
        if (FULL) {
            if (p.last_state && k == p.nchunk - 1) dst = p.last_state + ch * N + K * s;
        } else {
            dst = p.carry + (((int64_t)b * p.nchunk + k) * p.dim + d0 + c0 + c) * N + K * s;
        }
        if (dst) {
            if constexpr (K >= 4) {
#pragma unroll
                for (int q = 0; q < K; q += 4)
                    *reinterpret_cast<float4*>(dst + q) =
                        c ? make_float4(h[q].y, h[q + 1].y, h[q + 2].y, h[q + 3].y)
                          : make_float4(h[q].x, h[q + 1].x, h[q + 2].x, h[q + 3].x);
            } else {
#pragma unroll
                for (int q = 0; q < K; ++q) dst[q] = c ? h[q].y : h[q].x;
            }
        }
    }
}

}  // namespace ssm
