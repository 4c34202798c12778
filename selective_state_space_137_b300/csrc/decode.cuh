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
};

template <int N>
struct DecodeShape {
    static constexpr int LPC = N >= 4 ? (N / 4 > 32 ? 32 : N / 4) : 1;  // lanes per channel
    static constexpr int SPL = N / LPC;                               // states per lane
};

template <typename IO, int N>
__global__ void __launch_bounds__(256) state_update_kernel(DecodeParams p) {
    constexpr int LPC = DecodeShape<N>::LPC;
    constexpr int SPL = DecodeShape<N>::SPL;
    const int64_t gid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t chan = gid / LPC;            // (b, d) flattened
    const int sub = (int)(gid % LPC);
    const bool valid = chan < p.batch * p.dim;
    const int64_t c = valid ? chan : 0;         // keep whole lane groups alive for the shuffles
    const int64_t b = c / p.dim;
    const int64_t d = c % p.dim;

    const IO* x = static_cast<const IO*>(p.x);
    const IO* dl = static_cast<const IO*>(p.delta);
    const IO* Bm = static_cast<const IO*>(p.B);
    const IO* Cm = static_cast<const IO*>(p.C);
    const IO* z = static_cast<const IO*>(p.z);

    float* st = p.state + c * N + sub * SPL;
    float h[SPL];
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

    const float xv = load_f32(x + c);
    const float u = load_f32(dl + c) + (p.delta_bias ? __ldg(p.delta_bias + d) : 0.f);
    const float dt = p.softplus ? softplus_accurate(u) : u;
    const float dx = dt * xv;
    float y = 0.f;
#pragma unroll
    for (int j = 0; j < SPL; ++j) {
        const int n = sub * SPL + j;
        const float dA = ex2_sfu(dt * (__ldg(p.A + d * N + n) * kLog2e));
        h[j] = fmaf(dA, h[j], dx * load_f32(Bm + b * N + n));
        y = fmaf(load_f32(Cm + b * N + n), h[j], y);
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
        y = fmaf(p.D ? __ldg(p.D + d) : 0.f, xv, y);
        if (z) y *= silu_accurate(load_f32(z + c));
        store_io(static_cast<IO*>(p.out) + c, y);
    }
}

}  // namespace ssm
