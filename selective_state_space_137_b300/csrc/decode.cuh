// decode.cuh -- one recurrent step for one new token per sequence (decode).
//
// Recurrent inference with a fixed-size state and constant work per token
// ("Mamba的三大创新", model comparison table, RNN / SSM / Mamba rows): the
// state (batch, dim, N) fp32 is read once, advanced by one token and written
// back in place.  The step is bound by HBM traffic on that state, so the
// layout puts LPC consecutive lanes on one channel, each lane owning SPL
// consecutive states, which makes every warp load and store one contiguous
// run of the state with 128-bit accesses (SPL = 4).
#pragma once
#include "common.cuh"
#include "scan_generic.cuh"   // kMaxConvWidth
#include "tile_io.cuh"     // softplus_tiled / silu_tiled

namespace ssm {

struct DecodeParams {
    float* state;
    const void* x;
    const void* delta;
    const float* A;
    const void* B;
    const void* C;
    const float* D;
    const void* z;
    const float* delta_bias;
    void* out;
    int64_t batch, dim;
    int softplus;
    bool vec = false;   // A 16-byte and B, C (4 x element)-byte aligned: the VEC kernel
    // causal conv in front (read only by kernels instantiated with CONV)
    float* conv_state = nullptr;            // (batch, dim, conv_width - 1), shifted in place
    const float* conv_w = nullptr;          // (dim, conv_width)
    const float* conv_bias = nullptr;       // (dim) or NULL
    int conv_width = 1;
    int conv_act = 0;
};

template <int N>
struct DecodeShape {
    static constexpr int LPC = N >= 4 ? (N / 4 > 32 ? 32 : N / 4) : 1;  // lanes per channel
    static constexpr int SPL = N / LPC;                               // states per lane
};

// SPL consecutive io elements as fp32: 16- or 8-byte loads when SPL allows
// and the caller's pointers are aligned for them (VEC, chosen at launch),
// element loads otherwise.
template <int SPL, bool VEC>
__device__ __forceinline__ void load_vec(const float* p, float* f) {
    if (SPL % 4 == 0 && VEC) {
#pragma unroll
        for (int j = 0; j < SPL; j += 4) {
            const float4 v = __ldg(reinterpret_cast<const float4*>(p + j));
            f[j] = v.x; f[j + 1] = v.y; f[j + 2] = v.z; f[j + 3] = v.w;
        }
    } else {
#pragma unroll
        for (int j = 0; j < SPL; ++j) f[j] = __ldg(p + j);
    }
}
template <int SPL, bool VEC>
__device__ __forceinline__ void load_vec(const __nv_bfloat16* p, float* f) {
    if (SPL % 4 == 0 && VEC) {
#pragma unroll
        for (int j = 0; j < SPL; j += 4) {
            const uint2 v = __ldg(reinterpret_cast<const uint2*>(p + j));
            f[j] = __uint_as_float(v.x << 16); f[j + 1] = __uint_as_float(v.x & 0xffff0000u);
            f[j + 2] = __uint_as_float(v.y << 16); f[j + 3] = __uint_as_float(v.y & 0xffff0000u);
        }
    } else {
#pragma unroll
        for (int j = 0; j < SPL; ++j) f[j] = load_f32(p + j);
    }
}

// Grid: x covers the channels of one sequence (LPC lanes per channel, 256
// threads per block), y is the sequence.  Each thread loads its 16-byte slice
// of the state, the matching A row slice and B/C slices with vector loads, and
// the channel's x, delta, z; no integer division is needed to locate them.
// KW: the conv width as a compile-time constant (0: read from p.conv_width,
// up to kMaxConvWidth); a fixed width keeps the conv step within 32 registers.
template <typename IO, int N, bool CONV = false, bool ZOH = false, bool VEC = true, int KW = 0>
__global__ void __launch_bounds__(256, CONV ? (KW > 0 ? (sizeof(IO) == 2 ? 8 : 6) : 5) : (ZOH ? 4 : 8))
state_update_kernel(DecodeParams p) {
    constexpr int LPC = DecodeShape<N>::LPC;
    constexpr int SPL = DecodeShape<N>::SPL;
    const int lin = blockIdx.x * blockDim.x + threadIdx.x;    // lane index within the sequence
    const int64_t b = blockIdx.y;
    const int d_raw = lin / LPC;                                // LPC is a power of two
    const int sub = lin % LPC;
    const bool valid = d_raw < p.dim;
    const int d = valid ? d_raw : 0;                            // whole lane groups stay for the shuffles
    const int64_t ch = b * p.dim + d;

    const IO* x = static_cast<const IO*>(p.x);
    const IO* dl = static_cast<const IO*>(p.delta);
    const IO* Bm = static_cast<const IO*>(p.B);
    const IO* Cm = static_cast<const IO*>(p.C);
    const IO* z = static_cast<const IO*>(p.z);

    float h[SPL], a[SPL], bv[SPL], cv[SPL];
    float* st = p.state + ch * N + sub * SPL;
    if (SPL % 4 == 0) {
#pragma unroll
        for (int j = 0; j < SPL; j += 4) {
            const float4 v = *reinterpret_cast<const float4*>(st + j);
            h[j] = v.x; h[j + 1] = v.y; h[j + 2] = v.z; h[j + 3] = v.w;
        }
    } else {
#pragma unroll
        for (int j = 0; j < SPL; ++j) h[j] = st[j];
    }
    load_vec<SPL, VEC>(p.A + (int64_t)d * N + sub * SPL, a);
    load_vec<SPL, VEC>(Bm + b * N + sub * SPL, bv);
    load_vec<SPL, VEC>(Cm + b * N + sub * SPL, cv);
    float xv = load_f32(x + ch);
    // every input is loaded before the conv history is rewritten in place, so
    // all loads of the step go out together
    const float u = load_f32(dl + ch) + (p.delta_bias ? __ldg(p.delta_bias + d) : 0.f);
    const float zv = z ? load_f32(z + ch) : 0.f;
    const float dsk = p.D ? __ldg(p.D + d) : 0.f;
    if (CONV) {
        // x_conv from the K-1 stored inputs and the new one.
        constexpr int KM = KW > 0 ? KW : kMaxConvWidth;
        constexpr int HM = KM - 1;
        const int H = KW > 0 ? KW - 1 : p.conv_width - 1;
        const float raw = xv;
        float cw[KM];
#pragma unroll
        for (int q = 0; q < KM; ++q)
            cw[q] = q <= H ? __ldg(p.conv_w + (int64_t)d * (H + 1) + q) : 0.f;
        float acc = p.conv_bias ? __ldg(p.conv_bias + d) : 0.f;
        if (H <= LPC) {
            // lane `sub` of the channel holds history slot `sub`: one load and
            // one store per lane, the other slots by shuffle
            const int base = (threadIdx.x & 31) - sub;
            const float v = sub < H ? p.conv_state[ch * H + sub] : 0.f;
#pragma unroll
            for (int q = 0; q < HM; ++q) {
                const float cq = __shfl_sync(0xffffffffu, v, (base + (q < LPC ? q : 0)) & 31);
                if (q < H) acc = fmaf(cw[q], cq, acc);
            }
            const float nxt = __shfl_sync(0xffffffffu, v, (base + (sub + 1 < LPC ? sub + 1 : 0)) & 31);
            if (valid && sub < H) p.conv_state[ch * H + sub] = sub + 1 < H ? nxt : raw;
        } else {
            // longer histories: every lane reads them (one batch of loads), the
            // channel's first lane writes the shifted state after a warp sync
            float cs[HM];
#pragma unroll
            for (int q = 0; q < HM; ++q) cs[q] = q < H ? p.conv_state[ch * H + q] : 0.f;
#pragma unroll
            for (int q = 0; q < HM; ++q)
                if (q < H) acc = fmaf(cw[q], cs[q], acc);
            __syncwarp();
            if (valid && sub == 0) {
#pragma unroll
                for (int q = 0; q < HM; ++q)
                    if (q < H) p.conv_state[ch * H + q] = q + 1 < H ? cs[q + 1] : raw;
            }
        }
#pragma unroll
        for (int q = 0; q < KM; ++q)
            if (q == H) acc = fmaf(cw[q], xv, acc);
        xv = p.conv_act ? silu_tiled<IO>(acc) : acc;
    }

    const float dt = p.softplus ? softplus_tiled<IO>(u) : u;
    const float dx = dt * xv;
    float y = 0.f;
#pragma unroll
    for (int j = 0; j < SPL; ++j) {
        const float dA = ex2_sfu(dt * (a[j] * kLog2e));
        if (ZOH) {   // exact zero-order hold: ((exp(Delta A) - 1) / A) B x
            const float gain = a[j] != 0.f ? expm1f(dt * a[j]) / a[j] : dt;
            h[j] = fmaf(dA, h[j], gain * xv * bv[j]);
        } else {
            h[j] = fmaf(dA, h[j], dx * bv[j]);
        }
        y = fmaf(cv[j], h[j], y);
    }
#pragma unroll
    for (int off = LPC / 2; off > 0; off >>= 1) y += __shfl_xor_sync(0xffffffffu, y, off);
    if (!valid) return;
    if (SPL % 4 == 0) {
#pragma unroll
        for (int j = 0; j < SPL; j += 4)
            *reinterpret_cast<float4*>(st + j) = make_float4(h[j], h[j + 1], h[j + 2], h[j + 3]);
    } else {
#pragma unroll
        for (int j = 0; j < SPL; ++j) st[j] = h[j];
    }
    if (sub == 0) {
        y = fmaf(dsk, xv, y);
        if (z) y *= silu_tiled<IO>(zv);
        store_io(static_cast<IO*>(p.out) + ch, y);
    }
}

}  // namespace ssm
