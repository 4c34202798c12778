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
#include "scan_tiled.cuh"     // silu_tiled, unpack / pack

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
