// scan_generic.cuh -- general selective-scan kernels: one thread per
// (batch, channel), the whole N-wide state in registers, any io dtype, any
// supported N, any alignment.  Long sequences are cut into chunks that run
// in parallel, joined by a carry pass (see the three-launch scheme in
// ssm_api.cu).
//
// The recurrence is the recurrent mode (stage 2) of the selective SSM:
// h_t = exp(Delta_t A) h_{t-1} + Delta_t B_t x_t, read out as
// y_t = C_t . h_t + D x_t and gated by silu(z_t) ("Mamba的三大创新",
// section on the hardware-aware parallel scan).
#pragma once
#include "common.cuh"

namespace ssm {

struct ScanParams {
    const void* x;
    const void* delta;
    const float* A;
    const void* B;
    const void* C;
    const float* D;
    const void* z;
    const float* delta_bias;
    void* out;
    float* last_state;
    const float* initial_state;
    float* carry;      // (batch, nchunk, dim, N): chunk end-states, then chunk start-states
    float* dsum;       // (batch, nchunk, dim): sum of Delta over each chunk
    int64_t batch, seqlen, dim;
    int64_t chunk_len;
    int nchunk;
    int softplus;
    // causal conv in front of the scan (read only by kernels instantiated with CONV)
    const float* conv_w = nullptr;          // (dim, conv_width)
    const float* conv_bias = nullptr;       // (dim) or NULL
    const float* conv_state_in = nullptr;   // (batch, dim, conv_width - 1) or NULL
    float* conv_state_out = nullptr;        // (batch, dim, conv_width - 1) or NULL
    int conv_width = 1;
    int conv_act = 0;
    // training forward: the state before every 16th token, (batch, ceil(L/16), dim, N)
    float* ckpt = nullptr;
    int64_t ckpt_tiles = 0;
    // dt_proj fused in front (read only by kernels instantiated with it):
    // delta_raw = dt_low W_dt^T, dt_low (batch, seqlen, R) and W_dt (dim, R) bf16
    const void* dt_low = nullptr;
    const void* W_dt = nullptr;
};

constexpr int kCkptSteps = 16;

constexpr int kMaxConvWidth = 8;

// MODE_FULL  : outputs for tokens of one chunk, from its start state.
// MODE_AGG   : chunk end-state from a zero start, plus the chunk's sum of Delta.
// MODE_STATES: the state before every 16th token of one chunk, from its start
//              state, and nothing else (the backward's recompute; the one-warp
//              scan only).
enum { MODE_FULL = 0, MODE_AGG = 1, MODE_STATES = 2 };

// ZOH: the exact zero-order-hold input term ((exp(Delta A) - 1) / A) B x in
// place of Delta B x (expm1f keeps it accurate for small Delta A).
template <typename IO, int N, int MODE, bool CONV = false, bool ZOH = false>
__global__ void __launch_bounds__(128) scan_generic_kernel(ScanParams p) {
    const int64_t d = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t b = blockIdx.y;
    const int k = blockIdx.z;
    if (d >= p.dim) return;
    const int64_t t0 = (int64_t)k * p.chunk_len;
    int64_t t1 = t0 + p.chunk_len;
    if (t1 > p.seqlen) t1 = p.seqlen;

    const IO* __restrict__ x = static_cast<const IO*>(p.x);
    const IO* __restrict__ dl = static_cast<const IO*>(p.delta);
    const IO* __restrict__ Bm = static_cast<const IO*>(p.B);
    const IO* __restrict__ Cm = static_cast<const IO*>(p.C);
    const IO* __restrict__ z = static_cast<const IO*>(p.z);
    IO* __restrict__ out = static_cast<IO*>(p.out);

    float a2[N], h[N];
#pragma unroll
    for (int n = 0; n < N; ++n) a2[n] = __ldg(p.A + d * N + n) * kLog2e;

    const int64_t chan = b * p.dim + d;
    if (MODE == MODE_AGG) {
#pragma unroll
        for (int n = 0; n < N; ++n) h[n] = 0.f;
    } else if (p.nchunk > 1) {
        const float* cin = p.carry + ((b * p.nchunk + k) * p.dim + d) * N;
#pragma unroll
        for (int n = 0; n < N; ++n) h[n] = cin[n];
    } else if (p.initial_state) {
#pragma unroll
        for (int n = 0; n < N; ++n) h[n] = __ldg(p.initial_state + chan * N + n);
    } else {
#pragma unroll
        for (int n = 0; n < N; ++n) h[n] = 0.f;
    }
    const float bias = p.delta_bias ? __ldg(p.delta_bias + d) : 0.f;
    const float dskip = p.D ? __ldg(p.D + d) : 0.f;

    // conv: window of the K-1 raw inputs before t0 (state or zeros before t = 0)
    const int H = CONV ? p.conv_width - 1 : 0;
    float cw[kMaxConvWidth], wnd[kMaxConvWidth];
    const float cbias = (CONV && p.conv_bias) ? __ldg(p.conv_bias + d) : 0.f;
    if (CONV) {
#pragma unroll
        for (int q = 0; q < kMaxConvWidth; ++q) {
            cw[q] = q < p.conv_width ? __ldg(p.conv_w + d * p.conv_width + q) : 0.f;
            wnd[q] = 0.f;
            if (q < H) {
                const int64_t tt = t0 - H + q;
                if (tt >= 0) wnd[q] = load_f32(x + (b * p.seqlen + tt) * p.dim + d);
                else if (p.conv_state_in) wnd[q] = __ldg(p.conv_state_in + chan * H + (H + tt));
            }
        }
    }

    float dsum = 0.f;
    for (int64_t t = t0; t < t1; ++t) {
        if (MODE == MODE_FULL && p.ckpt && t % kCkptSteps == 0) {
            float* ck = p.ckpt + ((b * p.ckpt_tiles + t / kCkptSteps) * p.dim + d) * N;
#pragma unroll
            for (int n = 0; n < N; ++n) ck[n] = h[n];
        }
        const int64_t tok = (b * p.seqlen + t) * p.dim + d;
        const int64_t row = (b * p.seqlen + t) * N;
        float xv = load_f32(x + tok);
        if (CONV) {
            // taps 0..H-1 on the window, tap H on the current input (static
            // register indices only: H is a runtime width)
            const float raw = xv;
            float acc = cbias;
#pragma unroll
            for (int q = 0; q < kMaxConvWidth; ++q) {
                if (q < H) acc = fmaf(cw[q], wnd[q], acc);
                else if (q == H) acc = fmaf(cw[q], raw, acc);
            }
#pragma unroll
            for (int q = 0; q < kMaxConvWidth - 1; ++q)
                wnd[q] = (q + 1 < H) ? wnd[q + 1] : ((q + 1 == H) ? raw : wnd[q]);
            xv = p.conv_act ? silu_accurate(acc) : acc;
        }
        const float u = load_f32(dl + tok) + bias;
        const float dt = p.softplus ? softplus_accurate(u) : u;
        const float dx = dt * xv;
        float y = 0.f;
#pragma unroll
        for (int n = 0; n < N; ++n) {
            const float dA = ex2_sfu(dt * a2[n]);
            if (ZOH) {
                const float an = a2[n] * kLn2;
                const float gain = an != 0.f ? expm1f(dt * an) / an : dt;
                h[n] = fmaf(dA, h[n], gain * xv * load_f32(Bm + row + n));
            } else {
                h[n] = fmaf(dA, h[n], dx * load_f32(Bm + row + n));
            }
            if (MODE == MODE_FULL) y = fmaf(load_f32(Cm + row + n), h[n], y);
        }
        if (MODE == MODE_FULL) {
            y = fmaf(dskip, xv, y);
            if (z) y *= silu_accurate(load_f32(z + tok));
            store_io(out + tok, y);
        } else {
            dsum += dt;
        }
    }

    if (MODE == MODE_AGG) {
        float* cend = p.carry + ((b * p.nchunk + k) * p.dim + d) * N;
#pragma unroll
        for (int n = 0; n < N; ++n) cend[n] = h[n];
        p.dsum[(b * p.nchunk + k) * p.dim + d] = dsum;
    } else if (k == p.nchunk - 1) {
        if (p.last_state) {
#pragma unroll
            for (int n = 0; n < N; ++n) p.last_state[chan * N + n] = h[n];
        }
        if (CONV && p.conv_state_out) {
#pragma unroll
            for (int q = 0; q < kMaxConvWidth - 1; ++q)
                if (q < H) p.conv_state_out[chan * H + q] = wnd[q];
        }
    }
}

// Carry pass: turns the chunk end-states (from a zero start) into the true
// start state of every chunk.  For one (b, d, n):
//   s_0 = h_init;  s_{k+1} = exp(A * sum_k Delta) * s_k + e_k
// which is the associative combine (a1, b1) o (a2, b2) = (a1 a2, a2 b1 + b2)
// of the parallel scan, applied left to right over the chunks.  The decay of a
// whole chunk is exp(A * sum Delta) because A does not depend on time.
__global__ void carry_kernel(const float* __restrict__ A, const float* __restrict__ initial_state,
                             float* carry, const float* __restrict__ dsum, int64_t batch,
                             int64_t dim, int N, int nchunk) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;  // over (b, d, n)
    if (i >= batch * dim * N) return;
    const int n = (int)(i % N);
    const int64_t d = (i / N) % dim;
    const int64_t b = i / (N * dim);
    const float a2 = A[d * N + n] * kLog2e;
    float s = initial_state ? initial_state[i] : 0.f;
    for (int k = 0; k < nchunk; ++k) {
        float* slot = carry + ((b * nchunk + k) * dim + d) * N + n;
        // end state of chunk k from zero; the last chunk has none (its slot
        // only receives the start state)
        const float e = k + 1 < nchunk ? *slot : 0.f;
        *slot = s;                                 // start state of chunk k
        if (k + 1 < nchunk) {
            const float decay = exp2f(a2 * dsum[(b * nchunk + k) * dim + d]);
            s = fmaf(decay, s, e);
        }
    }
}

}  // namespace ssm
