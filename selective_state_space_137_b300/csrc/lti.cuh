// lti.cuh -- the time-invariant (LTI, S4) model in its convolution mode
// ("Mamba的三大创新", stage 3): with a constant step and input-independent
// B, C the recurrence unrolls into a causal convolution with the kernel
//   K[d][k] = sum_n C[d][n] exp(k Delta[d] A[d][n]) Bbar[d][n],  k = 0 .. L-1
// (Bbar = Delta B, or ((exp(Delta A) - 1) / A) B for the exact zero-order hold),
// and y[b][t][d] = sum_{k<=t} K[d][k] x[b][t-k][d] + D[d] x[b][t][d], gated by
// silu(z) when z is given.
//
// lti_kernel_kernel: one thread per (d, k), the N terms in a loop; K rows
//   are written along k, coalesced.
// lti_conv_kernel: a CTA owns 32 channels x 64 output steps of one sequence;
//   thread (c, g) accumulates the 8 outputs t = t0 + 8g .. t0 + 8g + 7 of
//   channel c.  Inputs come in chunks of 64 steps (x chunk and the matching
//   K segment staged in shared memory, zero below k = 0); for each input step
//   the 8 needed taps are a sliding register window, so every multiply-add
//   costs about one instruction.  The work is L^2/2 multiply-adds per
//   (sequence, channel): the recurrence (ssm_scan_fwd) reaches the same
//   result in L N operations, which is what this part favours for long L.
//
// lti_conv_mma_kernel (bf16 I/O, dim a multiple of 8): the same sum on the
//   tensor cores.  For channel d the outputs of 8 sequences are Y = T X,
//   T[t][s] = K[d][t - s] (s <= t), a lower-triangular Toeplitz matrix times
//   the (L x 8) inputs.  A warp owns one channel, a CTA 8 channels and 8
//   sequences; a work item is a group of 128 output steps (8 blocks of 16),
//   walked over the input chunks of 128 steps up to it.  Block (i, j) of T
//   depends on i - j only, so a chunk needs the A fragments of 15 block
//   diagonals, all inside a 256-tap window of K that the warp rebuilds per
//   chunk from global memory, for up to 64 mma.sync m16n8k16 products.
//   K enters as two bf16 terms, hi = bf16(K) and lo = bf16(K - hi), so a tap
//   is carried to about 2^-17 of its value (bf16 alone, 2^-9 a tap, drifts
//   past the bf16 output bound when a slowly decaying K is summed over
//   hundreds of steps); x is bf16 already, so both products are exact and
//   accumulate in fp32.  x chunks arrive by TMA and are transposed once into
//   per-channel rows of step pairs; the outputs (+ D x, times silu(z)) leave
//   by TMA store.
#pragma once
#include "common.cuh"
#include "tile_io.cuh"   // silu_tiled
#include "tma.cuh"

namespace ssm {

struct LtiKernelParams {
    const float* delta;   // (dim)
    const float* A;       // (dim, N)
    const float* B;       // (dim, N)
    const float* C;       // (dim, N)
    float* K;             // (dim, L)
    int64_t dim, seqlen;
    int N;
    int zoh;
};

// Grid: one block per (channel, 256-step block of k), flattened.
__global__ void __launch_bounds__(256) lti_kernel_kernel(LtiKernelParams p) {
    const int64_t kblocks = (p.seqlen + 255) / 256;
    const int64_t d = (int64_t)blockIdx.x / kblocks;
    const int64_t k = ((int64_t)blockIdx.x % kblocks) * 256 + threadIdx.x;
    if (k >= p.seqlen) return;
    const float dt = __ldg(p.delta + d);
    float acc = 0.f;
    for (int n = 0; n < p.N; ++n) {
        const float a = __ldg(p.A + d * p.N + n);
        const float gain = p.zoh ? (a != 0.f ? expm1f(dt * a) / a : dt) : dt;
        // exp(k Delta a) through exp2 of a product formed in one rounding
        const float decay = exp2f((float)k * (dt * a * kLog2e));
        acc = fmaf(__ldg(p.C + d * p.N + n) * gain * __ldg(p.B + d * p.N + n), decay, acc);
    }
    p.K[d * p.seqlen + k] = acc;
}

struct LtiConvParams {
    const float* K;   // (dim, L)
    const void* x;    // (batch, L, dim)
    const float* D;   // (dim) or NULL
    const void* z;    // (batch, L, dim) or NULL
    void* out;        // (batch, L, dim)
    int64_t batch, seqlen, dim;
};

constexpr int kLtiCh = 32, kLtiTo = 64, kLtiTs = 64, kLtiR = 8;

template <typename IO>
__global__ void __launch_bounds__(256) lti_conv_kernel(LtiConvParams p) {
    __shared__ float xs[kLtiTs][kLtiCh + 1];                // x chunk, [step][channel]
    __shared__ float ks[kLtiCh][kLtiTo + kLtiTs + 1];       // K segment per channel
    const int c = threadIdx.x % kLtiCh;
    const int g = threadIdx.x / kLtiCh;                      // 0..7: outputs 8g .. 8g+7
    const int64_t d0 = (int64_t)blockIdx.x * kLtiCh;
    const int64_t t0 = (int64_t)blockIdx.y * kLtiTo;
    const int64_t b = blockIdx.z;
    const int64_t d = d0 + c;
    const IO* x = static_cast<const IO*>(p.x);
    float acc[kLtiR];
#pragma unroll
    for (int r = 0; r < kLtiR; ++r) acc[r] = 0.f;

    // inputs s0 .. s0 + 63 feed outputs t0 .. t0 + 63 through k = t - s in
    // [t0 - s0 - 63, t0 - s0 + 63]; ks[c][j] holds K[t0 - s0 - 63 + j]
    for (int64_t s0 = 0; s0 < t0 + kLtiTo && s0 < p.seqlen; s0 += kLtiTs) {
        __syncthreads();
        for (int e = threadIdx.x; e < kLtiTs * kLtiCh; e += blockDim.x) {
            const int si = e / kLtiCh, cc = e % kLtiCh;
            const int64_t s = s0 + si;
            xs[si][cc] = (s < p.seqlen && d0 + cc < p.dim)
                             ? load_f32(x + (b * p.seqlen + s) * p.dim + d0 + cc) : 0.f;
        }
        const int64_t kb = t0 - s0 - (kLtiTs - 1);
        for (int e = threadIdx.x; e < kLtiCh * (kLtiTo + kLtiTs); e += blockDim.x) {
            const int cc = e / (kLtiTo + kLtiTs), j = e % (kLtiTo + kLtiTs);
            const int64_t kk = kb + j;
            ks[cc][j] = (kk >= 0 && kk < p.seqlen && d0 + cc < p.dim)
                            ? __ldg(p.K + (d0 + cc) * p.seqlen + kk) : 0.f;
        }
        __syncthreads();
        // output t = t0 + 8g + r, input s = s0 + si: k = t - s, at ks index
        // (t - s) - kb = 8g + r - si + 63
        const int base = kLtiR * g + (kLtiTs - 1);
        float win[kLtiR];
#pragma unroll
        for (int r = 0; r < kLtiR; ++r) win[r] = ks[c][base + r];   // si = 0
#pragma unroll 8
        for (int si = 0; si < kLtiTs; ++si) {
            const float xv = xs[si][c];
#pragma unroll
            for (int r = 0; r < kLtiR; ++r) acc[r] = fmaf(win[r], xv, acc[r]);
            // next input step: every tap index moves down by one
#pragma unroll
            for (int r = kLtiR - 1; r > 0; --r) win[r] = win[r - 1];
            win[0] = si + 1 < kLtiTs ? ks[c][base - si - 1] : 0.f;
        }
    }
    if (d >= p.dim) return;
    const IO* z = static_cast<const IO*>(p.z);
    IO* out = static_cast<IO*>(p.out);
    const float Dd = p.D ? __ldg(p.D + d) : 0.f;
#pragma unroll
    for (int r = 0; r < kLtiR; ++r) {
        const int64_t t = t0 + kLtiR * g + r;
        if (t >= p.seqlen) break;
        const int64_t tok = (b * p.seqlen + t) * p.dim + d;
        float y = fmaf(Dd, load_f32(x + tok), acc[r]);
        if (z) y *= silu_accurate(load_f32(z + tok));
        store_io(out + tok, y);
    }
}

// ---------------------------------------------------------------------------
constexpr int kLtiMmaCh = 8, kLtiMmaB = 8, kLtiMmaChunk = 128;

struct LtiMmaMaps {
    CUtensorMap x, z, out;   // (dim, L, batch) bf16, box 8 x 128 x 8
};

struct LtiMmaCfg {
    static constexpr int TILE = kLtiMmaB * kLtiMmaChunk * kLtiMmaCh * 2;   // one [8][128][8] bf16 box
    // the chunk transposed per channel: bf16 pairs (x[t], x[t+1]) as words,
    // [channel][sequence][64 words], word w of sequence n stored at w ^ 4 (n & 7)
    // so that the 8 sequences of one B-fragment load fall on different banks
    static constexpr int XTW = kLtiMmaChunk / 2;
    // the K window of one chunk: words u = 0 .. 255 hold the pairs
    // (K[k], K[k - 1]), k = 128 (Dc - 1) + u for the chunk distance Dc,
    // as hi and lo terms: uint32 [8 channels][2][256]
    static constexpr int WIN = 256;
    static constexpr int OFF_X = 0;                                     // the x chunk [n][t][ch]
    static constexpr int OFF_Z = TILE;                                  // z, then the output
    static constexpr int OFF_XT = 2 * TILE;                             // uint32 [8][8][XTW]
    static constexpr int OFF_W = OFF_XT + kLtiMmaCh * kLtiMmaB * XTW * 4;
    static constexpr int OFF_BAR = OFF_W + kLtiMmaCh * 2 * WIN * 4;     // x, z
    static constexpr int SMEM = OFF_BAR + 2 * 8;
};

// The (hi, lo) bf16 pair words of one K window (per warp; lane j holds taps
// k0 + j + 32 i in v[i], vm1 = K[k0 - 1]).
__device__ __forceinline__ void lti_window_store(uint32_t* wh, uint32_t* wl, const float (&v)[8], float vm1,
                                                 int lane) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        float prev = __shfl_up_sync(0xffffffffu, v[i], 1);   // K[k - 1]
        if (i > 0) {
            const float wrap = __shfl_sync(0xffffffffu, v[i - 1], 31);
            if (lane == 0) prev = wrap;
        } else if (lane == 0) {
            prev = vm1;
        }
        const __nv_bfloat162 hi = __floats2bfloat162_rn(v[i], prev);   // low half K[k]
        const float2 hf = __bfloat1622float2(hi);
        const __nv_bfloat162 lo = __floats2bfloat162_rn(v[i] - hf.x, prev - hf.y);
        wh[lane + 32 * i] = *reinterpret_cast<const uint32_t*>(&hi);
        wl[lane + 32 * i] = *reinterpret_cast<const uint32_t*>(&lo);
    }
}

template <bool ZG>
__global__ void __launch_bounds__(256, 2)
    lti_conv_mma_kernel(const __grid_constant__ LtiMmaMaps maps, LtiConvParams p) {
    using Cfg = LtiMmaCfg;
    constexpr int CH = kLtiMmaCh, NB = kLtiMmaB, TC = kLtiMmaChunk;
    extern __shared__ __align__(1024) unsigned char smem[];
    __nv_bfloat16* zs = reinterpret_cast<__nv_bfloat16*>(smem + Cfg::OFF_Z);   // z, then out
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + Cfg::OFF_BAR);   // [0]: x, [1]: z
    uint32_t* xt = reinterpret_cast<uint32_t*>(smem + Cfg::OFF_XT);
    const __nv_bfloat16* xs = reinterpret_cast<const __nv_bfloat16*>(smem + Cfg::OFF_X);   // [n][t][ch]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, q = lane & 3;
    uint32_t* wh = reinterpret_cast<uint32_t*>(smem + Cfg::OFF_W) + warp * 2 * Cfg::WIN;   // this channel's
    uint32_t* wl = wh + Cfg::WIN;
    const int nb0 = blockIdx.y * NB;
    const int64_t L = p.seqlen;

    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; ++i) mbar_init(&bar[i], 1);
        fence_barrier_init();
        prefetch_tmap(&maps.x);
        prefetch_tmap(&maps.out);
        if (ZG) prefetch_tmap(&maps.z);
    }
    __syncthreads();

    // Work items are (block of 8 channels, group of 128 output steps); group G
    // takes G + 1 chunk products.  The grid is persistent: items are taken
    // heaviest first, CTA j taking position j of even rounds and P - 1 - j of
    // odd ones (P CTAs), which evens out the sum of weights per CTA.
    // Every wait is bounded and every decision to stop is made by the whole CTA
    // (__syncthreads_or), so no warp is left at a barrier the others skipped.
    const int ngroups = (int)((L + TC - 1) / TC);
    const int ncb = (int)(p.dim / CH);
    const int64_t nitems = (int64_t)ncb * ngroups;
    const int P = gridDim.x;
    bool ok = true;
    int xphase = 0, zphase = 0;
    bool x_pending = false, z_pending = false;   // thread 0: TMA loads not yet seen to land
    for (int64_t r = 0; ok; ++r) {
        const int64_t idx = r * P + ((r & 1) ? P - 1 - (int)blockIdx.x : (int)blockIdx.x);
        if (idx >= nitems) break;
        const int G = ngroups - 1 - (int)(idx / ncb);
        const int d0 = (int)(idx % ncb) * CH;
        const int64_t d = d0 + warp;
        const float Dd = p.D ? __ldg(p.D + d) : 0.f;
        const float* Kd = p.K + d * L;
        if (ZG && threadIdx.x == 0) {   // the gate of this group (zs is free: the last store has read it)
            bulk_wait_read<0>();
            mbar_arrive_expect_tx(&bar[1], (uint32_t)Cfg::TILE);
            tma_load_3d(zs, &maps.z, &bar[1], d0, G * TC, nb0);
            z_pending = true;
        }
        float acc[8][4];
#pragma unroll
        for (int ob = 0; ob < 8; ++ob)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[ob][e] = 0.f;
        // chunk c + 1 is loaded into xs as soon as chunk c has been transposed out
        // of it, so its load runs under chunk c's products
        for (int c = 0; c <= G; ++c) {
            // the K window of chunk distance Dc = G - c: taps k0 .. k0 + 255 and
            // k0 - 1, k0 = 128 (Dc - 1), zero outside [0, L) (loaded here, stored
            // once the chunk has landed)
            const int Dc = G - c;
            const int64_t k0 = 128 * (int64_t)(Dc - 1);
            float kv[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int64_t k = k0 + lane + 32 * i;
                kv[i] = (k >= 0 && k < L) ? __ldg(Kd + k) : 0.f;
            }
            const float kvm1 = (k0 - 1 >= 0 && k0 - 1 < L) ? __ldg(Kd + k0 - 1) : 0.f;
            if (threadIdx.x == 0 && c == 0) {
                mbar_arrive_expect_tx(&bar[0], (uint32_t)Cfg::TILE);
                tma_load_3d(smem + Cfg::OFF_X, &maps.x, &bar[0], d0, 0, nb0);
                x_pending = true;
            }
            const bool got = mbar_wait_bounded(&bar[0], (uint32_t)xphase);
            if (__syncthreads_or(!got)) {
                ok = false;
                break;
            }
            x_pending = false;
            xphase ^= 1;
            {   // transpose: thread i takes the step pairs (t, t + 1) of entries i and
                // i + 256 of [8 sequences][64 pairs], all 8 channels (two 16-byte loads)
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const int e = threadIdx.x + 256 * r;
                    const int n = e >> 6, tp = (e & 63) * 2;
                    const uint4 v0 = *reinterpret_cast<const uint4*>(xs + (n * TC + tp) * CH);
                    const uint4 v1 = *reinterpret_cast<const uint4*>(xs + (n * TC + tp + 1) * CH);
                    const uint32_t w0[4] = {v0.x, v0.y, v0.z, v0.w}, w1[4] = {v1.x, v1.y, v1.z, v1.w};
#pragma unroll
                    for (int ch = 0; ch < CH; ++ch) {
                        const uint32_t lo = (ch & 1) ? (w0[ch >> 1] >> 16) : (w0[ch >> 1] & 0xffffu);
                        const uint32_t hi = (ch & 1) ? (w1[ch >> 1] & 0xffff0000u) : (w1[ch >> 1] << 16);
                        xt[(ch * NB + n) * Cfg::XTW + ((e & 63) ^ (4 * n))] = lo | hi;
                    }
                }
            }
            __syncthreads();
            if (threadIdx.x == 0 && c < G) {   // xs is free: every thread has transposed it
                mbar_arrive_expect_tx(&bar[0], (uint32_t)Cfg::TILE);
                tma_load_3d(smem + Cfg::OFF_X, &maps.x, &bar[0], d0, (c + 1) * TC, nb0);
                x_pending = true;
            }
            __syncwarp();   // this warp's reads of the previous window are done
            lti_window_store(wh, wl, kv, kvm1, lane);
            __syncwarp();
            // B fragments of the chunk's 8 input blocks: (X[s][g], X[s + 1][g]) with
            // s = 16 ib + 2 q and + 8: the word s / 2 of row g of this channel
            uint32_t bq[8][2];
            const uint32_t* xw = xt + (warp * NB + g) * Cfg::XTW;
#pragma unroll
            for (int ib = 0; ib < 8; ++ib) {
                bq[ib][0] = xw[(8 * ib + q) ^ (4 * g)];
                bq[ib][1] = xw[(8 * ib + q + 4) ^ (4 * g)];
            }
            // the 15 block diagonals ob - ib = e - 7: block diagonal D = 8 Dc + e - 7
            // has A fragments pair(m), pair(m + 8), pair(m - 8), pair(m) with
            // m = 16 D + g - 2 q, window words u = 16 e + 16 + g - 2 q (+ 8, - 8);
            // blocks above the diagonal (D < 0) are zero and skipped
#pragma unroll
            for (int e = 0; e < 15; ++e) {
                if (Dc == 0 && e < 7) continue;
                const int u = 16 * e + 16 + g - 2 * q;
                const uint32_t h0 = wh[u], h1 = wh[u + 8], h2 = wh[u - 8];
                const uint32_t l0 = wl[u], l1 = wl[u + 8], l2 = wl[u - 8];
#pragma unroll
                for (int ib = 0; ib < 8; ++ib) {
                    const int ob = ib + e - 7;
                    if (ob >= 0 && ob < 8) {
                        mma_bf16_16816(acc[ob], h0, h1, h2, h0, bq[ib][0], bq[ib][1]);
                        mma_bf16_16816(acc[ob], l0, l1, l2, l0, bq[ib][0], bq[ib][1]);
                    }
                }
            }
        }
        if (!ok) break;
        // epilogue: y = acc + D x, times silu(z); acc[ob] = Y[16 ob + g (+8)][2 q (+1)].
        // xs still holds the last chunk (c = G), x of this group's steps; zs holds z
        // (ZG) or is free once the previous group's store has read it.
        if (ZG) {
            const bool got = mbar_wait_bounded(&bar[1], (uint32_t)zphase);
            if (__syncthreads_or(!got)) {
                ok = false;
                break;
            }
            z_pending = false;
            zphase ^= 1;
        } else {
            if (threadIdx.x == 0) bulk_wait_read<0>();
            __syncthreads();
        }
        unsigned short* zr = reinterpret_cast<unsigned short*>(zs);
        const unsigned short* xr2 = reinterpret_cast<const unsigned short*>(xs);
#pragma unroll
        for (int ob = 0; ob < 8; ++ob) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int t = 16 * ob + g + 8 * (e >> 1);
                const int n = 2 * q + (e & 1);
                const int idx = (n * TC + t) * CH + warp;
                float y = fmaf(Dd, __uint_as_float((uint32_t)xr2[idx] << 16), acc[ob][e]);
                if (ZG) y *= silu_tiled<__nv_bfloat16>(__uint_as_float((uint32_t)zr[idx] << 16));
                __nv_bfloat16 yb = __float2bfloat16_rn(y);
                zr[idx] = *reinterpret_cast<unsigned short*>(&yb);
            }
        }
        fence_proxy_async_smem();
        __syncthreads();
        if (threadIdx.x == 0) {
            tma_store_3d(&maps.out, zs, d0, G * TC, nb0);
            bulk_commit();
        }
    }
    if (threadIdx.x == 0) {
        bulk_wait<0>();
        // after a timeout, let the loads still in flight land before the CTA's
        // shared memory is released
        if (x_pending) mbar_wait_bounded(&bar[0], (uint32_t)xphase, 100000000ull);
        if (z_pending) mbar_wait_bounded(&bar[1], (uint32_t)zphase, 100000000ull);
    }
}

}  // namespace ssm
