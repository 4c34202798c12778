// conv.cuh -- causal depthwise conv1d (+ SiLU) over time, standalone.
//
// The local-context convolution the Mamba block applies to x before the
// selective SSM ("Mamba的三大创新", simplified-architecture section; a causal
// Conv1d layer in the unite.ai overview):
//   x_conv[t, d] = act(bias[d] + sum_{k<K} w[d][k] * x[t - (K-1) + k, d]).
// Memory-bound: each thread owns VEC consecutive channels of one sequence
// over a chunk of time steps and slides a (K-1)-row window of raw inputs in
// registers, so every input is loaded once (plus K-1 rows per chunk, mostly
// from L2) and every output stored once, with 16-byte accesses when VEC > 1.
#pragma once
#include "common.cuh"
#include "scan_generic.cuh"   // kMaxConvWidth
#include "tile_io.cuh"     // silu_tiled, unpack / pack
#include "tma.cuh"

#ifndef SSM_CONV_UNROLL
#define SSM_CONV_UNROLL 4    // rows loaded ahead per thread
#endif
#ifndef SSM_CONV_MINBLOCKS
#define SSM_CONV_MINBLOCKS 1 // resident 128-thread blocks per SM the registers must allow
#endif

namespace ssm {

struct ConvParams {
    const void* x;
    const float* w;
    const float* bias;
    const float* state_in;
    void* out;
    float* state_out;
    int64_t batch, seqlen, dim;
    int64_t chunk;      // time steps per thread
    int width;
    int act;
};

// VEC consecutive io elements as fp32: one 16- or 8-byte load when the
// vector has that size, else element by element; and back.
template <typename IO, int VEC>
__device__ __forceinline__ void load_row(const IO* p, float* f) {
    constexpr int BYTES = VEC * (int)sizeof(IO);
    if constexpr (BYTES == 16) {
        unpack<IO>(__ldg(reinterpret_cast<const uint4*>(p)), f);
    } else if constexpr (BYTES == 8 || BYTES == 4) {
        uint4 w = make_uint4(0u, 0u, 0u, 0u);
        if constexpr (BYTES == 8) {
            const uint2 v = __ldg(reinterpret_cast<const uint2*>(p));
            w.x = v.x; w.y = v.y;
        } else {
            w.x = __ldg(reinterpret_cast<const unsigned*>(p));
        }
        float g[8];
        unpack<IO>(w, g);
#pragma unroll
        for (int v2 = 0; v2 < VEC; ++v2) f[v2] = g[v2];
    } else {
#pragma unroll
        for (int v2 = 0; v2 < VEC; ++v2) f[v2] = load_f32(p + v2);
    }
}

template <typename IO, int VEC>
__device__ __forceinline__ void store_row(IO* p, const float* f) {
    constexpr int BYTES = VEC * (int)sizeof(IO);
    if constexpr (BYTES == 16) {
        *reinterpret_cast<uint4*>(p) = pack<IO>(f);
    } else if constexpr (BYTES == 8 || BYTES == 4) {
        float g[8] = {};
#pragma unroll
        for (int v2 = 0; v2 < VEC; ++v2) g[v2] = f[v2];
        const uint4 v = pack<IO>(g);
        if constexpr (BYTES == 8) *reinterpret_cast<uint2*>(p) = make_uint2(v.x, v.y);
        else *reinterpret_cast<unsigned*>(p) = v.x;
    } else {
#pragma unroll
        for (int v2 = 0; v2 < VEC; ++v2) store_io(p + v2, f[v2]);
    }
}

// Width K is a template parameter so that the taps and the window are plain
// registers; the time loop is unrolled by U with the U row loads issued before
// the arithmetic, so each thread keeps U 16-byte loads in flight.
template <typename IO, int VEC, int K>
__global__ void __launch_bounds__(128, SSM_CONV_MINBLOCKS) conv1d_kernel(ConvParams p) {
    constexpr int H = K - 1;
    constexpr int HW = H > 0 ? H : 1;   // window array extent
    constexpr int U = SSM_CONV_UNROLL;
    const int64_t dv = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;   // channel vector
    const int64_t d0 = dv * VEC;
    if (d0 >= p.dim) return;
    const int64_t b = blockIdx.z;
    const int64_t t0 = (int64_t)blockIdx.y * p.chunk;
    int64_t t1 = t0 + p.chunk;
    if (t1 > p.seqlen) t1 = p.seqlen;
    if (t0 >= t1) return;
    const IO* x = static_cast<const IO*>(p.x) + b * p.seqlen * p.dim + d0;
    IO* out = static_cast<IO*>(p.out) + b * p.seqlen * p.dim + d0;

    float w[VEC][K], bias[VEC], wnd[HW][VEC];
#pragma unroll
    for (int v = 0; v < VEC; ++v) {
        bias[v] = p.bias ? __ldg(p.bias + d0 + v) : 0.f;
#pragma unroll
        for (int q = 0; q < K; ++q) w[v][q] = __ldg(p.w + (d0 + v) * K + q);
    }
    // the H raw inputs before t0: from x, or the conv state before t = 0
#pragma unroll
    for (int q = 0; q < H; ++q) {
        const int64_t tt = t0 - H + q;
        if (tt >= 0) {
            load_row<IO, VEC>(x + tt * p.dim, wnd[q]);
        } else {
#pragma unroll
            for (int v = 0; v < VEC; ++v)
                wnd[q][v] = p.state_in ? __ldg(p.state_in + ((b * p.dim + d0 + v) * H + (H + tt))) : 0.f;
        }
    }
    for (int64_t t = t0; t < t1; t += U) {
        float raw[U][VEC];
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (t + u < t1) load_row<IO, VEC>(x + (t + u) * p.dim, raw[u]);
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (t + u >= t1) break;
            float y[VEC];
#pragma unroll
            for (int v = 0; v < VEC; ++v) {
                float acc = bias[v];
#pragma unroll
                for (int q = 0; q < H; ++q) acc = fmaf(w[v][q], wnd[q][v], acc);
                acc = fmaf(w[v][H], raw[u][v], acc);
                y[v] = p.act ? silu_tiled<IO>(acc) : acc;
            }
            store_row<IO, VEC>(out + (t + u) * p.dim, y);
#pragma unroll
            for (int q = 0; q < H; ++q)
#pragma unroll
                for (int v = 0; v < VEC; ++v) wnd[q][v] = q + 1 < H ? wnd[q + 1][v] : raw[u][v];
        }
    }
    if (p.state_out && t1 == p.seqlen) {
#pragma unroll
        for (int q = 0; q < H; ++q)
#pragma unroll
            for (int v = 0; v < VEC; ++v) p.state_out[(b * p.dim + d0 + v) * H + q] = wnd[q][v];
    }
}

}  // namespace ssm

// ---------------------------------------------------------------------------
// The same convolution streamed through shared memory by TMA: a CTA owns
// kConvCC channels of one sequence over a chunk of time and walks it in
// kConvTT-step tiles.  Each tile's x box starts H = K-1 rows early (the
// history; rows before t = 0 read as zeros and are replaced by the conv
// state), lands in an S-stage mbarrier ring, and thread c slides the K-tap
// window of channel c down the tile; the output tile leaves by TMA store
// (two buffers).  Every byte of x is read once from DRAM (the halo rows of a
// tile were the previous tile's rows, from L2), every output written once.
namespace ssm {

// 16-step tiles in a 2-stage ring: about 18 KB of shared memory per CTA, so
// 16 CTAs (64 warps) fit an SM and hide the latency of the per-token chain
// (measured on the bench shape: 104 us, against 133 us for 32 x 4 and 107 us
// for 16 x 3).
#ifndef SSM_CONV_TT
#define SSM_CONV_TT 16
#endif
#ifndef SSM_CONV_STAGES
#define SSM_CONV_STAGES 2
#endif
constexpr int kConvCC = 128, kConvTT = SSM_CONV_TT, kConvStages = SSM_CONV_STAGES;

struct ConvMaps {
    CUtensorMap x, out;   // (dim, seqlen, batch); boxes [TT + H][CC] and [TT][CC]
};

template <typename IO, int K>
struct ConvTmaCfg {
    static constexpr int H = K - 1, ESZ = (int)sizeof(IO);
    static constexpr int IN_ROWS = kConvTT + H;
    static constexpr int STAGE = round_up(IN_ROWS * kConvCC * ESZ, 128);
    static constexpr int OUT = kConvTT * kConvCC * ESZ;
    static constexpr int OFF_OUT = kConvStages * STAGE;
    static constexpr int OFF_BAR = round_up(OFF_OUT + 2 * OUT, 128);
    static constexpr int SMEM = OFF_BAR + kConvStages * 8;
};

template <typename IO, int K>
__global__ void __launch_bounds__(kConvCC) conv1d_tma_kernel(const __grid_constant__ ConvMaps maps,
                                                             ConvParams p) {
    using Cfg = ConvTmaCfg<IO, K>;
    constexpr int H = Cfg::H, S = kConvStages, TT = kConvTT, CC = kConvCC;
    extern __shared__ __align__(1024) unsigned char smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + Cfg::OFF_BAR);
    const int c = threadIdx.x;
    const int d0 = blockIdx.x * CC;
    const int64_t d = (int64_t)d0 + c;
    const bool dval = d < p.dim;
    const int b = blockIdx.z;
    const int64_t c0 = (int64_t)blockIdx.y * p.chunk;
    int64_t c1 = c0 + p.chunk;
    if (c1 > p.seqlen) c1 = p.seqlen;
    const int ntiles = c1 > c0 ? (int)((c1 - c0 + TT - 1) / TT) : 0;

    int issued = 0;   // thread 0's count of tiles whose loads went out
    auto issue = [&](int j) {
        issued = j + 1;
        const int t0 = (int)(c0 + (int64_t)j * TT);
        mbar_arrive_expect_tx(&full[j % S], (uint32_t)(Cfg::IN_ROWS * CC * Cfg::ESZ));
        tma_load_3d(smem + (j % S) * Cfg::STAGE, &maps.x, &full[j % S], d0, t0 - H, b);
    };
    if (c == 0) {
        for (int s = 0; s < S; ++s) mbar_init(&full[s], 1);
        fence_barrier_init();
    }
    __syncthreads();
    if (c == 0) {
        prefetch_tmap(&maps.x);
        prefetch_tmap(&maps.out);
        for (int j = 0; j < S && j < ntiles; ++j) issue(j);
    }
    float w[K], bias = 0.f;
#pragma unroll
    for (int q = 0; q < K; ++q) w[q] = dval ? __ldg(p.w + d * K + q) : 0.f;
    if (p.bias && dval) bias = __ldg(p.bias + d);
    bool ok = true;
    for (int j = 0; j < ntiles; ++j) {
        const bool landed = mbar_wait_bounded(&full[j % S], (uint32_t)((j / S) & 1));
        if (c == 0) bulk_wait_read<1>();   // the store that last read this tile's output buffer
        // one decision for the whole block: a timed-out wait ends every thread's loop
        if (!__syncthreads_and(landed)) { ok = false; break; }
        const IO* xs = reinterpret_cast<const IO*>(smem + (j % S) * Cfg::STAGE);
        IO* os = reinterpret_cast<IO*>(smem + Cfg::OFF_OUT + (j & 1) * Cfg::OUT);
        const int64_t t0 = c0 + (int64_t)j * TT;
        // the window: raw inputs at times t0 - H .. t0 - 1 (stage rows 0 .. H-1)
        float win[H > 0 ? H : 1];
#pragma unroll
        for (int q = 0; q < H; ++q) {
            const int64_t tt = t0 - H + q;
            win[q] = tt >= 0 ? load1(xs + q * CC + c)
                             : ((p.state_in && dval) ? __ldg(p.state_in + ((int64_t)b * p.dim + d) * H + H + tt) : 0.f);
        }
#pragma unroll 8
        for (int r = 0; r < TT; ++r) {
            const float xv = load1(xs + (H + r) * CC + c);
            float acc = bias;
#pragma unroll
            for (int q = 0; q < H; ++q) acc = fmaf(w[q], win[q], acc);
            acc = fmaf(w[H], xv, acc);
            store_io(os + r * CC + c, p.act ? silu_tiled<IO>(acc) : acc);
#pragma unroll
            for (int q = 0; q < H; ++q) win[q] = q + 1 < H ? win[q + 1] : xv;
        }
        // the final conv state: the last H raw inputs of the sequence
        if (p.state_out && dval && c1 == p.seqlen && j == ntiles - 1) {
            const int last = (int)(c1 - t0);   // rows of this tile that exist
#pragma unroll
            for (int q = 0; q < H; ++q) {
                const int64_t tt = p.seqlen - H + q;
                const float v = tt >= 0 ? load1(xs + (last + q) * CC + c)
                                        : (p.state_in ? __ldg(p.state_in + ((int64_t)b * p.dim + d) * H + H + tt) : 0.f);
                p.state_out[((int64_t)b * p.dim + d) * H + q] = v;
            }
        }
        fence_proxy_async_smem();
        __syncthreads();   // the tile's inputs are read and its outputs written
        if (c == 0) {
            tma_store_3d(&maps.out, os, d0, (int)t0, b);
            bulk_commit();
            if (j + S < ntiles) issue(j + S);
        }
    }
    if (c == 0) {
        bulk_wait<0>();
        if (!ok) {   // the loads still in flight land before the CTA exits
            for (int j = issued - S > 0 ? issued - S : 0; j < issued; ++j)
                mbar_wait_bounded(&full[j % S], (uint32_t)((j / S) & 1), 100000000ull);
        }
    }
}

}  // namespace ssm
