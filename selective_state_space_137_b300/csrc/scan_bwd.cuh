// scan_bwd.cuh -- gradients of the selective scan (the backward half of
// training), recomputing the states instead of storing them.
//
// Forward, per (b, d) and time t (the recurrent mode of "Mamba的三大创新",
// stage 2):  Delta_t = softplus(delta_t + bias),  dA_t = exp(Delta_t A),
//   h_t = dA_t h_{t-1} + Delta_t B_t x_t,  yc_t = C_t . h_t + D x_t,
//   out_t = yc_t silu(z_t).
// Backward, time reversed, with g_t = dL/dh_t and G = dA_{t+1} g_{t+1}:
//   dyc = dout silu(z),  g_t = dyc C_t + G,   dz = dout yc silu'(z)
//   dC_t += dyc h_t,  dB_t += g_t Delta_t x_t                  (sums over d)
//   dx_t = dyc D + Delta_t sum_n g B,  dDelta_t = x_t sum_n g B + sum_n A g dA_t h_{t-1}
//   dA += Delta_t g dA_t h_{t-1},  dD += dyc x,  dbias += ddelta  (sums over b, t)
//   ddelta_t = dDelta_t sigmoid(delta_t + bias)  (softplus' = sigmoid)
//
// Launches (K time chunks; K = 1 needs only the last two):
//   1. forward aggregate + carry (scan_generic.cuh): the state at every chunk start;
//   2. scan_bwd_agg_kernel: per chunk k >= 1, E_k = dA_{t0} g_{t0} computed with
//      nothing coming from the right, and the chunk's sum of Delta;
//   3. scan_bwd_carry_kernel: right to left, the term e_k that chunk k receives
//      from chunk k+1:  e_{K-1} = dlast,  e_{k-1} = E_k + exp(A sum_k Delta) e_k;
//   4. scan_bwd_kernel: per chunk, a forward sweep that stores the state at every
//      16-step tile start, then tiles in reverse: the tile's 16 states are
//      recomputed into registers and the reverse step runs over them;
//   5. scan_bwd_reduce_kernel: dB, dC (sums of the per-CTA partials over the
//      channel blocks) and dA, dD, dbias (sums over sequences and chunks).
// Every sum is formed in a fixed order: the result does not depend on timing.
//
// Thread layout of the sweeps: LPC lanes per channel, SPL states per lane
// (N = 16: 4 x 4), CPW channels per warp, W warps (CH channels) per CTA, W
// chosen by the host per shape (8 on the register path).  The per-step dB/dC
// contributions are summed over the warp's channels -- by recursive halving
// of shuffles on the register path (each round a lane keeps half of its values
// and adds the partner's half), through a per-warp shared-memory block in the
// TMA-staged sweep -- then over the CTA's warps through shared memory at the
// end of each tile.
#pragma once
#include "common.cuh"
#include "tile_io.cuh"   // softplus_tiled, silu_tiled, round_up, load1
#include "tma.cuh"

namespace ssm {

struct BwdParams {
    const void* x;
    const void* delta;
    const float* A;
    const void* B;
    const void* C;
    const float* D;
    const void* z;
    const float* delta_bias;
    const float* initial_state;
    const void* dout;
    const float* dlast;
    void* dx;
    void* ddelta;
    void* dz;
    float* dinit;
    // workspace
    const float* fstart;   // (batch, K, dim, N): state at each chunk start (K > 1)
    float* ebuf;           // (batch, K, dim, N): E_k, then the incoming term e_k
    float* bdsum;          // (batch, K, dim): sum of Delta over chunk k
    float* ckpt;           // (batch, ntiles, dim, N): state at each tile start
    int ckpt_given;        // 1: ckpt was written by the training forward (no forward sweep)
    float* pBC;            // (nblk, batch, seqlen, 2N): per-CTA dB | dC
    float* pA;             // (batch * K, dim, N)
    float* pD;             // (batch * K, dim)
    float* pbias;          // (batch * K, dim)
    int64_t batch, seqlen, dim, chunk_len, ntiles;
    int nchunk;
    int softplus;
    bool vec;              // B and C bases aligned for SPL-element vector loads
};

constexpr int kBwdT = 16;       // steps per tile (checkpoint spacing)
constexpr int kBwdWarps = 8;    // warps per CTA of the register-path sweep

// W: warps per CTA (the host picks it so that the CTAs spread evenly over the SMs)
template <int N, int W_ = kBwdWarps>
struct BwdShape {
    static constexpr int LPC = N >= 4 ? (N / 4 > 32 ? 32 : N / 4) : 1;   // lanes per channel
    static constexpr int SPL = N / LPC;                                  // states per lane
    static constexpr int CPW = 32 / LPC;                                 // channels per warp
    static constexpr int W = W_;                                         // warps per CTA
    static constexpr int CH = CPW * W;                                   // channels per CTA
    static constexpr int MINB = 65536 / (W * 32 * 128);                  // CTAs per SM at 128 registers
    static constexpr int V = 2 * SPL;                                    // dB | dC values per lane
    static constexpr int SMEM = W * kBwdT * 2 * N * 4;
};

template <int SPL, typename IO>
__device__ __forceinline__ void bwd_load(const IO* p, float* f, bool vec) {
    if (SPL % 4 == 0 && vec) {
#pragma unroll
        for (int j = 0; j < SPL; j += 4) {
            if (sizeof(IO) == 4) {
                const float4 v = __ldg(reinterpret_cast<const float4*>(p + j));
                f[j] = v.x; f[j + 1] = v.y; f[j + 2] = v.z; f[j + 3] = v.w;
            } else {
                const uint2 v = __ldg(reinterpret_cast<const uint2*>(p + j));
                f[j] = __uint_as_float(v.x << 16); f[j + 1] = __uint_as_float(v.x & 0xffff0000u);
                f[j + 2] = __uint_as_float(v.y << 16); f[j + 3] = __uint_as_float(v.y & 0xffff0000u);
            }
        }
    } else {
#pragma unroll
        for (int j = 0; j < SPL; ++j) f[j] = load_f32(p + j);
    }
}

// The same from shared memory (plain loads; __ldg is for global memory only).
template <int SPL, typename IO>
__device__ __forceinline__ void bwd_load_smem(const IO* p, float* f) {
    if (SPL % 4 == 0) {
#pragma unroll
        for (int j = 0; j < SPL; j += 4) {
            if (sizeof(IO) == 4) {
                const float4 v = *reinterpret_cast<const float4*>(p + j);
                f[j] = v.x; f[j + 1] = v.y; f[j + 2] = v.z; f[j + 3] = v.w;
            } else {
                const uint2 v = *reinterpret_cast<const uint2*>(p + j);
                f[j] = __uint_as_float(v.x << 16); f[j + 1] = __uint_as_float(v.x & 0xffff0000u);
                f[j + 2] = __uint_as_float(v.y << 16); f[j + 3] = __uint_as_float(v.y & 0xffff0000u);
            }
        }
    } else {
#pragma unroll
        for (int j = 0; j < SPL; ++j) f[j] = load1(p + j);
    }
}

// Sum over the lanes of a warp that hold the same state slice (the channel
// bits of the lane index, xor offsets LPC .. 16).  On return lane holds
// `held` = V >> r values at v[0 .. held), the sums of the original values
// base + i, where base is returned; when the channel bits outnumber the
// halving rounds, the extra rounds add whole arrays (results replicated).
template <int V, int LPC>
__device__ __forceinline__ int reduce_channels(float (&v)[V], int lane) {
    int base = 0;
    int cnt = V;
#pragma unroll
    for (int o = 16; o >= LPC; o >>= 1) {
        if (cnt > 1) {
            const bool up = (lane & o) != 0;
            const int half = cnt / 2;
#pragma unroll
            for (int i = 0; i < V / 2; ++i) {
                if (i < half) {
                    const float send = up ? v[i] : v[half + i];
                    const float keep = up ? v[half + i] : v[i];
                    v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
                }
            }
            if (up) base += half;
            cnt = half;
        } else {
            v[0] += __shfl_xor_sync(0xffffffffu, v[0], o);
        }
    }
    return base;
}

// Sum of a per-lane value over the LPC lanes of one channel.
template <int LPC>
__device__ __forceinline__ float reduce_slices(float v) {
#pragma unroll
    for (int o = LPC / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// sigmoid(u) = 1 / (1 + 2^(-u log2 e)) with the SFU exponential and the
// approximate reciprocal (saturates to 0 and 1 at the ends).
__device__ __forceinline__ float sigmoid_fast(float u) {
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(1.f + ex2_sfu(-u * kLog2e)));
    return r;
}

// ---------------------------------------------------------------------------
// 2. Backward aggregate of chunk k >= 1: E_k with nothing from the right.
// LPC lanes per channel, SPL states per lane (the sweep's layout).  The chunk
// is walked from its end in groups of kAggGS steps: the CTA stages the
// group's C rows (shared by its channels) in fp32 shared memory (two
// buffers, one barrier per group), and lane j of a channel evaluates the
// per-token values (Delta, dyc) of steps t - j, t - j - LPC, ..., all loads
// of the group issued together; the values reach the channel's other lanes by
// shuffle.  Delta and dyc use the sweep's formulas.
constexpr int kAggGS = 32;
constexpr int kAggThreads = 128;

template <typename IO, int N>
__global__ void __launch_bounds__(kAggThreads) scan_bwd_agg_kernel(BwdParams p) {
    using S = BwdShape<N>;
    constexpr int LPC = S::LPC, SPL = S::SPL, GS = kAggGS, R = GS / LPC;
    __shared__ __align__(16) float cs[2][GS][N];
    const int64_t lin = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t d_raw = lin / LPC;
    const int sub = (int)(lin % LPC);
    const bool valid = d_raw < p.dim;
    const int64_t d = valid ? d_raw : 0;        // idle lanes stay for the shuffles and barriers
    const int base = (int)(threadIdx.x & 31) - sub;
    const int n0 = sub * SPL;
    const int64_t b = blockIdx.y;
    const int k = blockIdx.z + 1;
    const int64_t t0 = (int64_t)k * p.chunk_len;
    int64_t t1 = t0 + p.chunk_len;
    if (t1 > p.seqlen) t1 = p.seqlen;
    const IO* delta = static_cast<const IO*>(p.delta);
    const IO* Cm = static_cast<const IO*>(p.C);
    const IO* z = static_cast<const IO*>(p.z);
    const IO* dout = static_cast<const IO*>(p.dout);
    float a2[SPL], G[SPL];
#pragma unroll
    for (int q = 0; q < SPL; ++q) {
        a2[q] = __ldg(p.A + d * N + n0 + q) * kLog2e;
        G[q] = 0.f;
    }
    const float bias = p.delta_bias ? __ldg(p.delta_bias + d) : 0.f;
    float dsum = 0.f;
    int buf = 0;
    for (int64_t tg = t1 - 1; tg >= t0; tg -= GS, buf ^= 1) {
        // the group's C rows, row j = step tg - j (zero before the chunk)
        for (int e = threadIdx.x; e < GS * N; e += kAggThreads) {
            const int64_t t = tg - e / N;
            cs[buf][e / N][e % N] = t >= t0 ? load_f32(Cm + (b * p.seqlen + t) * N + e % N) : 0.f;
        }
        // this lane's steps of the group: raw loads first, then the formulas
        float u[R], dy[R], zz[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int64_t tm = tg - sub - LPC * r;
            const int64_t tok = (b * p.seqlen + (tm >= t0 ? tm : t0)) * p.dim + d;
            u[r] = load_f32(delta + tok);
            dy[r] = load_f32(dout + tok);
            zz[r] = z ? load_f32(z + tok) : 0.f;
        }
        float dt_m[R], dyc_m[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const bool in = tg - sub - LPC * r >= t0;
            const float uu = u[r] + bias;
            dt_m[r] = in ? (p.softplus ? softplus_tiled<IO>(uu) : uu) : 0.f;
            dyc_m[r] = in ? (z ? dy[r] * (zz[r] * sigmoid_fast(zz[r])) : dy[r]) : 0.f;
            dsum += dt_m[r];
        }
        __syncthreads();   // cs[buf] is complete (and cs[buf ^ 1] is no longer read)
#pragma unroll
        for (int j = 0; j < GS; ++j) {
            const float dt = __shfl_sync(0xffffffffu, dt_m[j / LPC], base + j % LPC);
            const float dyc = __shfl_sync(0xffffffffu, dyc_m[j / LPC], base + j % LPC);
            if (tg - j >= t0) {   // the same for every thread of the CTA
                float cv[SPL];
#pragma unroll
                for (int q = 0; q < SPL; ++q) cv[q] = cs[buf][j][n0 + q];
#pragma unroll
                for (int q = 0; q < SPL; ++q) {
                    const float g = fmaf(dyc, cv[q], G[q]);
                    G[q] = ex2_sfu(dt * a2[q]) * g;
                }
            }
        }
    }
    dsum = reduce_slices<LPC>(dsum);
    if (!valid) return;
    float* e = p.ebuf + ((b * p.nchunk + k) * p.dim + d) * N + n0;
#pragma unroll
    for (int q = 0; q < SPL; ++q) e[q] = G[q];
    if (sub == 0) p.bdsum[(b * p.nchunk + k) * p.dim + d] = dsum;
}

// 3. Right-to-left combine of the chunk terms, per (b, d, n).
__global__ void scan_bwd_carry_kernel(const float* __restrict__ A, const float* __restrict__ dlast,
                                      float* ebuf, const float* __restrict__ bdsum, int64_t batch,
                                      int64_t dim, int N, int nchunk) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= batch * dim * N) return;
    const int n = (int)(i % N);
    const int64_t d = (i / N) % dim;
    const int64_t b = i / (N * dim);
    const float a2 = A[d * N + n] * kLog2e;
    float e = dlast ? dlast[i] : 0.f;
    for (int k = nchunk - 1; k >= 0; --k) {
        float* slot = ebuf + ((b * nchunk + k) * dim + d) * N + n;
        const float Ek = k > 0 ? *slot : 0.f;
        *slot = e;                                  // what chunk k receives from the right
        if (k > 0) e = fmaf(exp2f(a2 * bdsum[(b * nchunk + k) * dim + d]), e, Ek);
    }
}

// 4. The reverse sweep of one chunk for CH channels of one sequence.
template <typename IO, int N, int W = kBwdWarps>
__global__ void __launch_bounds__(W * 32, BwdShape<N, W>::MINB) scan_bwd_kernel(BwdParams p) {
    using S = BwdShape<N, W>;
    constexpr int LPC = S::LPC, SPL = S::SPL, CPW = S::CPW, CH = S::CH, V = S::V, T = kBwdT;
    extern __shared__ float red[];   // [W][T][2N]
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int sub = lane % LPC;
    const int64_t d_raw = (int64_t)blockIdx.x * CH + warp * CPW + lane / LPC;
    const bool valid = d_raw < p.dim;
    const int64_t d = valid ? d_raw : 0;   // idle lanes stay for the shuffles
    const int64_t b = blockIdx.y;
    const int k = blockIdx.z;
    const int64_t t0 = (int64_t)k * p.chunk_len;
    int64_t t1 = t0 + p.chunk_len;
    if (t1 > p.seqlen) t1 = p.seqlen;
    const int n0 = sub * SPL;

    const IO* x = static_cast<const IO*>(p.x);
    const IO* delta = static_cast<const IO*>(p.delta);
    const IO* Bm = static_cast<const IO*>(p.B);
    const IO* Cm = static_cast<const IO*>(p.C);
    const IO* z = static_cast<const IO*>(p.z);
    const IO* dout = static_cast<const IO*>(p.dout);

    float an[SPL], a2[SPL], h[SPL], G[SPL], dAacc[SPL];
#pragma unroll
    for (int j = 0; j < SPL; ++j) {
        an[j] = __ldg(p.A + d * N + n0 + j);
        a2[j] = an[j] * kLog2e;
        dAacc[j] = 0.f;
        const int64_t si = (b * p.dim + d) * N + n0 + j;
        const int64_t ci = ((b * p.nchunk + k) * p.dim + d) * N + n0 + j;
        h[j] = p.ckpt_given ? 0.f   // the tile states come from the checkpoints
             : p.nchunk > 1 ? p.fstart[ci] : (p.initial_state ? __ldg(p.initial_state + si) : 0.f);
        G[j] = p.nchunk > 1 ? p.ebuf[ci] : (p.dlast ? __ldg(p.dlast + si) : 0.f);
    }
    const float bias = p.delta_bias ? __ldg(p.delta_bias + d) : 0.f;
    const float Dd = p.D ? __ldg(p.D + d) : 0.f;
    const int ntile = (int)((t1 - t0 + T - 1) / T);
    const int64_t tile0 = t0 / T;
    auto ckpt_at = [&](int j) { return p.ckpt + ((b * p.ntiles + tile0 + j) * p.dim + d) * N + n0; };
    auto dt_of = [&](int64_t tok) {
        const float u = load_f32(delta + tok) + bias;
        return p.softplus ? softplus_tiled<IO>(u) : u;
    };

    // ---- forward sweep: the state at every tile start (unless the forward kept them)
    for (int j = 0; j < ntile && !p.ckpt_given; ++j) {
        const int64_t ts = t0 + (int64_t)j * T;
        if (valid) {
            float* ck = ckpt_at(j);
#pragma unroll
            for (int q = 0; q < SPL; ++q) ck[q] = h[q];
        }
        const int steps = (int)((t1 - ts) < T ? (t1 - ts) : T);
        for (int s = 0; s < steps; ++s) {
            const int64_t t = ts + s;
            const int64_t tok = (b * p.seqlen + t) * p.dim + d;
            const float dt = dt_of(tok);
            const float dx = dt * load_f32(x + tok);
            float bv[SPL];
            bwd_load<SPL>(Bm + (b * p.seqlen + t) * N + n0, bv, p.vec);
#pragma unroll
            for (int q = 0; q < SPL; ++q) h[q] = fmaf(ex2_sfu(dt * a2[q]), h[q], dx * bv[q]);
        }
    }

    // ---- reverse sweep over the tiles
    float dD = 0.f, dbias = 0.f;
    float* myred = red + warp * (T * 2 * N);
    for (int j = ntile - 1; j >= 0; --j) {
        const int64_t ts = t0 + (int64_t)j * T;
        const int steps = (int)((t1 - ts) < T ? (t1 - ts) : T);
        float hs[SPL];
        {
            const float* ck = ckpt_at(j);
#pragma unroll
            for (int q = 0; q < SPL; ++q) hs[q] = valid ? ck[q] : 0.f;
        }
        // recompute the tile's states (registers, static indices)
        float hist[T][SPL], dth[T];
        {
            float hc[SPL];
#pragma unroll
            for (int q = 0; q < SPL; ++q) hc[q] = hs[q];
#pragma unroll
            for (int s = 0; s < T; ++s) {
                if (s < steps) {
                    const int64_t t = ts + s;
                    const int64_t tok = (b * p.seqlen + t) * p.dim + d;
                    const float dt = dt_of(tok);
                    dth[s] = dt;
                    const float dx = dt * load_f32(x + tok);
                    float bv[SPL];
                    bwd_load<SPL>(Bm + (b * p.seqlen + t) * N + n0, bv, p.vec);
#pragma unroll
                    for (int q = 0; q < SPL; ++q) {
                        hc[q] = fmaf(ex2_sfu(dt * a2[q]), hc[q], dx * bv[q]);
                        hist[s][q] = hc[q];
                    }
                }
            }
        }
#pragma unroll
        for (int s = T - 1; s >= 0; --s) {
            if (s < steps) {
                const int64_t t = ts + s;
                const int64_t tok = (b * p.seqlen + t) * p.dim + d;
                const float dt = dth[s];
                const float xv = load_f32(x + tok);
                float bv[SPL], cv[SPL];
                bwd_load<SPL>(Bm + (b * p.seqlen + t) * N + n0, bv, p.vec);
                bwd_load<SPL>(Cm + (b * p.seqlen + t) * N + n0, cv, p.vec);
                // yc = C . h_t + D x (needed for dz only)
                float yp = 0.f;
#pragma unroll
                for (int q = 0; q < SPL; ++q) yp = fmaf(cv[q], hist[s][q], yp);
                const float dov = load_f32(dout + tok);
                float dyc = dov, dzv = 0.f;
                if (z) {
                    const float zv = load_f32(z + tok);
                    const float sg = sigmoid_fast(zv);
                    dyc = dov * zv * sg;
                    const float yc = reduce_slices<LPC>(yp) + Dd * xv;
                    dzv = dov * yc * sg * (1.f + zv * (1.f - sg));
                }
                float vals[V];
                float s1 = 0.f, s2 = 0.f;
#pragma unroll
                for (int q = 0; q < SPL; ++q) {
                    const float hprev = s > 0 ? hist[s > 0 ? s - 1 : 0][q] : hs[q];
                    const float g = fmaf(dyc, cv[q], G[q]);
                    const float dA = ex2_sfu(dt * a2[q]);
                    const float qv = g * dA * hprev;
                    s1 = fmaf(g, bv[q], s1);
                    s2 = fmaf(an[q], qv, s2);
                    dAacc[q] = fmaf(dt, qv, dAacc[q]);
                    vals[q] = g * dt * xv;                // dB
                    vals[SPL + q] = dyc * hist[s][q];     // dC
                    G[q] = dA * g;
                }
                s1 = reduce_slices<LPC>(s1);
                s2 = reduce_slices<LPC>(s2);
                const float ddt = fmaf(xv, s1, s2);
                const float du = p.softplus ? ddt * sigmoid_fast(load_f32(delta + tok) + bias) : ddt;
                dD = fmaf(dyc, xv, dD);
                dbias += du;
                if (valid && sub == 0) {
                    store_io(static_cast<IO*>(p.dx) + tok, fmaf(dt, s1, dyc * Dd));
                    store_io(static_cast<IO*>(p.ddelta) + tok, du);
                    if (p.dz) store_io(static_cast<IO*>(p.dz) + tok, dzv);
                }
                // dB | dC summed over the warp's channels (idle lanes add zeros)
                if (!valid) {
#pragma unroll
                    for (int i = 0; i < V; ++i) vals[i] = 0.f;
                }
                const int base = reduce_channels<V, LPC>(vals, lane);
                constexpr int HOLD = V / CPW > 0 ? V / CPW : 1;   // values a lane holds
                // lanes whose leftover channel bits are zero write (replicas skip)
                const bool writer = CPW <= V || ((lane / LPC) % (CPW / (V < CPW ? V : CPW))) == 0;
                if (writer) {
#pragma unroll
                    for (int i = 0; i < HOLD; ++i) {
                        const int vi = base + i;               // original value index
                        const int kind = vi / SPL, jj = vi % SPL;
                        myred[s * 2 * N + kind * N + n0 + jj] = vals[i];
                    }
                }
            }
        }
        __syncthreads();
        // sum over the CTA's warps and store this tile's partials
        for (int e = threadIdx.x; e < steps * 2 * N; e += blockDim.x) {
            float acc = 0.f;
#pragma unroll
            for (int w = 0; w < S::W; ++w) acc += red[w * T * 2 * N + e];
            const int s = e / (2 * N), v = e % (2 * N);
            p.pBC[(((int64_t)blockIdx.x * p.batch + b) * p.seqlen + ts + s) * 2 * N + v] = acc;
        }
        __syncthreads();
    }

    // ---- per-(sequence, chunk) partial sums over time; the initial state's gradient
    if (!valid) return;
    const int64_t bk = b * p.nchunk + k;
#pragma unroll
    for (int q = 0; q < SPL; ++q) p.pA[(bk * p.dim + d) * N + n0 + q] = dAacc[q];
    if (sub == 0) {   // every lane of the channel holds the whole dD and dbias
        p.pD[bk * p.dim + d] = dD;
        p.pbias[bk * p.dim + d] = dbias;
    }
    if (k == 0 && p.dinit) {
#pragma unroll
        for (int q = 0; q < SPL; ++q) p.dinit[(b * p.dim + d) * N + n0 + q] = G[q];
    }
}

// ---------------------------------------------------------------------------
// 4'. The same reverse sweep with every tile's inputs staged in shared memory
// by TMA (two-stage ring, the next tile in flight while this one computes) and
// the per-token gradients written back a tile at a time by TMA stores.  Used
// when the rows are 16-byte multiples and the tensors 16-byte aligned; the
// arithmetic is that of scan_bwd_kernel.
//
// Load sequence u = 0 .. nfwd + ntile - 1: u < nfwd is forward-sweep tile u
// (x, delta, B); u >= nfwd is reverse tile nfwd + ntile - 1 - u (x, delta,
// dout, z, B, C); nfwd = 0 when the training forward kept the checkpoints.
// Stage u % 2, parity (u / 2) & 1.
struct BwdMaps {
    CUtensorMap x, delta, dout, z, B, C, dx, ddelta, dz;
};

template <typename IO, int N, int W>
struct BwdTmaCfg {
    using S = BwdShape<N, W>;
    static constexpr int CH = S::CH, T = kBwdT, ESZ = (int)sizeof(IO), NST = 2;
    static constexpr int TOK = T * CH * ESZ;                 // one [T][CH] tile
    static constexpr int ROW = T * N * ESZ;                  // one [T][N] tile
    static constexpr int OFF_X = 0, OFF_DL = TOK, OFF_DO = 2 * TOK, OFF_Z = 3 * TOK;
    static constexpr int OFF_B = 4 * TOK, OFF_C = 4 * TOK + ROW;
    static constexpr int STAGE = round_up(4 * TOK + 2 * ROW, 128);
    static constexpr int OFF_OUT = NST * STAGE;              // [2][3][T][CH] io
    static constexpr int OFF_RED = round_up(OFF_OUT + 2 * 3 * TOK, 128);
    // per-token values of the tile, computed once per (step, channel) by the
    // channel's lanes together: [NSCR][T][SROW] fp32 (padded rows: the lanes
    // of a channel write different steps without bank conflicts)
    static constexpr int SROW = CH + 8, NSCR = 6;
    enum { S_DT = 0, S_DX, S_X, S_DYC, S_ZF, S_SGU };
    static constexpr int OFF_SCR = OFF_RED + S::W * T * 2 * N * 4;
    // per warp, two buffers of [CPW][RS] fp32: the step's dB | dC terms of the
    // warp's channels, summed over the channels by lane o = output o.  RS = N
    // mod 32 puts the rows that a quarter-warp writes on disjoint banks.
    static constexpr int RS = 2 * N + (32 - N % 32) % 32;
    static constexpr int WSUM = S::CPW * RS;
    static constexpr int OFF_WSUM = OFF_SCR + NSCR * T * SROW * 4;
    static constexpr int OFF_BAR = OFF_WSUM + S::W * 2 * WSUM * 4;
    static constexpr int OFF_FLAG = OFF_BAR + NST * 8;
    static constexpr int SMEM = OFF_FLAG + 16;
    static_assert((CH * ESZ) % 16 == 0 && (N * ESZ) % 16 == 0, "TMA rows are 16-byte multiples");
};

template <typename IO, int N, int W>
__global__ void __launch_bounds__(W * 32, BwdShape<N, W>::MINB)
    scan_bwd_tma_kernel(const __grid_constant__ BwdMaps maps, BwdParams p) {
    using Cfg = BwdTmaCfg<IO, N, W>;
    using S = BwdShape<N, W>;
    constexpr int LPC = S::LPC, SPL = S::SPL, CPW = S::CPW, CH = S::CH, V = S::V, T = kBwdT;
    constexpr int NST = Cfg::NST;
    extern __shared__ __align__(1024) unsigned char smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + Cfg::OFF_BAR);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Cfg::OFF_FLAG);
    float* red = reinterpret_cast<float*>(smem + Cfg::OFF_RED);
    float* scr = reinterpret_cast<float*>(smem + Cfg::OFF_SCR) + 0;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    float* wsum = reinterpret_cast<float*>(smem + Cfg::OFF_WSUM) + warp * 2 * Cfg::WSUM;
    const int sub = lane % LPC;
    const int cl = warp * CPW + lane / LPC;                 // channel within the CTA
    const int d0 = blockIdx.x * CH;
    const int64_t d_raw = (int64_t)d0 + cl;
    const bool valid = d_raw < p.dim;
    const int64_t d = valid ? d_raw : 0;
    const int b = blockIdx.y;
    const int k = blockIdx.z;
    const int64_t t0 = (int64_t)k * p.chunk_len;
    int64_t t1 = t0 + p.chunk_len;
    if (t1 > p.seqlen) t1 = p.seqlen;
    const int n0 = sub * SPL;
    const int ntile = (int)((t1 - t0 + T - 1) / T);
    const int nfwd = p.ckpt_given ? 0 : ntile;   // forward-sweep loads
    const int nload = nfwd + ntile;
    const bool z_on = p.z != nullptr;
    const bool dz_on = p.dz != nullptr;

    int issued = 0;             // loads issued so far (thread 0's count)
    auto issue = [&](int u) {   // one thread
        issued = u + 1;
        unsigned char* st = smem + (u % NST) * Cfg::STAGE;
        const bool fwd = u < nfwd;
        const int j = fwd ? u : nfwd + ntile - 1 - u;
        const int r = (int)(t0 + (int64_t)j * T);
        uint64_t* bar = &full[u % NST];
        const uint32_t tx = fwd ? (uint32_t)(2 * Cfg::TOK + Cfg::ROW)
                                : (uint32_t)((z_on ? 4 : 3) * Cfg::TOK + 2 * Cfg::ROW);
        mbar_arrive_expect_tx(bar, tx);
        tma_load_3d(st + Cfg::OFF_X, &maps.x, bar, d0, r, b);
        tma_load_3d(st + Cfg::OFF_DL, &maps.delta, bar, d0, r, b);
        tma_load_3d(st + Cfg::OFF_B, &maps.B, bar, 0, r, b);
        if (!fwd) {
            tma_load_3d(st + Cfg::OFF_DO, &maps.dout, bar, d0, r, b);
            if (z_on) tma_load_3d(st + Cfg::OFF_Z, &maps.z, bar, d0, r, b);
            tma_load_3d(st + Cfg::OFF_C, &maps.C, bar, 0, r, b);
        }
    };

    if (threadIdx.x == 0) {
        for (int i = 0; i < NST; ++i) mbar_init(&full[i], 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        prefetch_tmap(&maps.x);
        prefetch_tmap(&maps.delta);
        prefetch_tmap(&maps.B);
        for (int u = 0; u < NST && u < nload; ++u) issue(u);
    }

    float an[SPL], a2[SPL], h[SPL], G[SPL], dAacc[SPL];
#pragma unroll
    for (int j = 0; j < SPL; ++j) {
        an[j] = __ldg(p.A + d * N + n0 + j);
        a2[j] = an[j] * kLog2e;
        dAacc[j] = 0.f;
        const int64_t si = ((int64_t)b * p.dim + d) * N + n0 + j;
        const int64_t ci = (((int64_t)b * p.nchunk + k) * p.dim + d) * N + n0 + j;
        h[j] = p.ckpt_given ? 0.f   // the tile states come from the checkpoints
             : p.nchunk > 1 ? p.fstart[ci] : (p.initial_state ? __ldg(p.initial_state + si) : 0.f);
        G[j] = p.nchunk > 1 ? p.ebuf[ci] : (p.dlast ? __ldg(p.dlast + si) : 0.f);
    }
    const float bias = p.delta_bias ? __ldg(p.delta_bias + d) : 0.f;
    const float Dd = p.D ? __ldg(p.D + d) : 0.f;
    const int64_t tile0 = t0 / T;
    auto ckpt_at = [&](int j) {
        return p.ckpt + (((int64_t)b * p.ntiles + tile0 + j) * p.dim + d) * N + n0;
    };
    auto wait_stage = [&](int u) {
        if (!mbar_wait_bounded(&full[u % NST], (uint32_t)((u / NST) & 1))) *abort_flag = 1;
    };
    // after a block barrier: every thread sees the same flag
    auto aborted = [&]() { return *abort_flag != 0; };
    auto refill = [&](int u) {   // after the barrier that follows the last read of stage u
        if (threadIdx.x == 0 && u + NST < nload) issue(u + NST);
    };

    // ---- forward sweep: the state at every tile start (unless the forward kept them)
    for (int j = 0; j < nfwd; ++j) {
        const int u = j;
        wait_stage(u);
        if (valid) {
            float* ck = ckpt_at(j);
#pragma unroll
            for (int q = 0; q < SPL; ++q) ck[q] = h[q];
        }
        const unsigned char* st = smem + (u % NST) * Cfg::STAGE;
        const IO* xs = reinterpret_cast<const IO*>(st + Cfg::OFF_X);
        const IO* ds = reinterpret_cast<const IO*>(st + Cfg::OFF_DL);
        const IO* Bs = reinterpret_cast<const IO*>(st + Cfg::OFF_B);
        const int steps = (int)((t1 - (t0 + (int64_t)j * T)) < T ? (t1 - (t0 + (int64_t)j * T)) : T);
        if (!aborted()) {
            // Delta and Delta*x once per (step, channel): lane sub takes steps sub, sub + LPC, ...
#pragma unroll
            for (int m = 0; m < T / LPC; ++m) {
                const int sl = sub + LPC * m;
                const float u_ = load1(ds + sl * CH + cl) + bias;
                const float dt = p.softplus ? softplus_tiled<IO>(u_) : u_;
                scr[Cfg::S_DT * T * Cfg::SROW + sl * Cfg::SROW + cl] = dt;
                scr[Cfg::S_DX * T * Cfg::SROW + sl * Cfg::SROW + cl] = dt * load1(xs + sl * CH + cl);
            }
            __syncwarp();
#pragma unroll 4
            for (int s = 0; s < steps; ++s) {
                const float dt = scr[Cfg::S_DT * T * Cfg::SROW + s * Cfg::SROW + cl];
                const float dx = scr[Cfg::S_DX * T * Cfg::SROW + s * Cfg::SROW + cl];
                float bv[SPL];
                bwd_load_smem<SPL>(Bs + s * N + n0, bv);
#pragma unroll
                for (int q = 0; q < SPL; ++q) h[q] = fmaf(ex2_sfu(dt * a2[q]), h[q], dx * bv[q]);
            }
        }
        __syncthreads();
        if (aborted()) break;
        refill(u);
    }

    // ---- reverse sweep
    float dD = 0.f, dbias = 0.f;
    float* myred = red + warp * (T * 2 * N);
    float hs_next[SPL];
    if (ntile > 0 && !aborted()) {
        const float* ck = ckpt_at(ntile - 1);
#pragma unroll
        for (int q = 0; q < SPL; ++q) hs_next[q] = valid ? ck[q] : 0.f;
    }
    for (int jj = 0; jj < ntile && !aborted(); ++jj) {
        const int j = ntile - 1 - jj;
        const int u = nfwd + jj;
        const int64_t ts = t0 + (int64_t)j * T;
        const int steps = (int)((t1 - ts) < T ? (t1 - ts) : T);
        float hs[SPL];
#pragma unroll
        for (int q = 0; q < SPL; ++q) hs[q] = hs_next[q];
        if (j > 0) {   // the next tile's checkpoint, in flight during this tile
            const float* ck = ckpt_at(j - 1);
#pragma unroll
            for (int q = 0; q < SPL; ++q) hs_next[q] = valid ? ck[q] : 0.f;
        }
        wait_stage(u);
        const unsigned char* st = smem + (u % NST) * Cfg::STAGE;
        const IO* xs = reinterpret_cast<const IO*>(st + Cfg::OFF_X);
        const IO* ds = reinterpret_cast<const IO*>(st + Cfg::OFF_DL);
        const IO* dos = reinterpret_cast<const IO*>(st + Cfg::OFF_DO);
        const IO* zs = reinterpret_cast<const IO*>(st + Cfg::OFF_Z);
        const IO* Bs = reinterpret_cast<const IO*>(st + Cfg::OFF_B);
        const IO* Cs = reinterpret_cast<const IO*>(st + Cfg::OFF_C);
        IO* ob = reinterpret_cast<IO*>(smem + Cfg::OFF_OUT + (jj & 1) * 3 * Cfg::TOK);
        if (!aborted()) {
            // per-token values once per (step, channel), split over the channel's lanes
#pragma unroll
            for (int m = 0; m < T / LPC; ++m) {
                const int sl = sub + LPC * m;
                const float u_ = load1(ds + sl * CH + cl) + bias;
                const float dt = p.softplus ? softplus_tiled<IO>(u_) : u_;
                const float xv = load1(xs + sl * CH + cl);
                const float dov = load1(dos + sl * CH + cl);
                float dyc = dov, zf = 0.f;
                if (z_on) {
                    const float zv = load1(zs + sl * CH + cl);
                    const float sg = sigmoid_fast(zv);
                    dyc = dov * zv * sg;
                    zf = dov * sg * (1.f + zv * (1.f - sg));
                }
                // a channel past the last one: Delta x = dyc = 0 makes its dB and dC
                // terms exactly 0 (its inputs are channel 0's, finite), so the
                // per-step channel sums need no masking
                if (!valid) dyc = 0.f;
                const float dxs = valid ? dt * xv : 0.f;
                float* sc = scr + sl * Cfg::SROW + cl;
                sc[Cfg::S_DT * T * Cfg::SROW] = dt;
                sc[Cfg::S_DX * T * Cfg::SROW] = dxs;
                sc[Cfg::S_X * T * Cfg::SROW] = xv;
                sc[Cfg::S_DYC * T * Cfg::SROW] = dyc;
                sc[Cfg::S_ZF * T * Cfg::SROW] = zf;
                sc[Cfg::S_SGU * T * Cfg::SROW] = p.softplus ? sigmoid_fast(u_) : 1.f;
                if (sl < steps) dD = fmaf(dyc, xv, dD);
            }
            __syncwarp();
            auto sv = [&](int which, int s_) { return scr[which * T * Cfg::SROW + s_ * Cfg::SROW + cl]; };
            float hist[T][SPL];
            {
                float hc[SPL];
#pragma unroll
                for (int q = 0; q < SPL; ++q) hc[q] = hs[q];
#pragma unroll
                for (int s = 0; s < T; ++s) {
                    if (s < steps) {
                        const float dt = sv(Cfg::S_DT, s);
                        const float dx = sv(Cfg::S_DX, s);
                        float bv[SPL];
                        bwd_load_smem<SPL>(Bs + s * N + n0, bv);
                        const f32x2 dt2 = pk2(dt, dt), dx2 = pk2(dx, dx);
#pragma unroll
                        for (int q = 0; q < SPL; q += 2) {
                            float e0, e1;
                            upk2(mul2(dt2, pk2(a2[q], a2[q + 1])), e0, e1);
                            const f32x2 hn = fma2(pk2(ex2_sfu(e0), ex2_sfu(e1)), pk2(hc[q], hc[q + 1]),
                                                  mul2(dx2, pk2(bv[q], bv[q + 1])));
                            upk2(hn, hc[q], hc[q + 1]);
                            hist[s][q] = hc[q];
                            hist[s][q + 1] = hc[q + 1];
                        }
                    }
                }
            }
#pragma unroll
            for (int s = T - 1; s >= 0; --s) {
                if (s < steps) {
                    const float dt = sv(Cfg::S_DT, s);
                    const float dx = sv(Cfg::S_DX, s);
                    const float xv = sv(Cfg::S_X, s);
                    const float dyc = sv(Cfg::S_DYC, s);
                    float bv[SPL], cv[SPL];
                    bwd_load_smem<SPL>(Bs + s * N + n0, bv);
                    bwd_load_smem<SPL>(Cs + s * N + n0, cv);
                    float dzv = 0.f;
                    if (z_on) {
                        float yp = 0.f;
#pragma unroll
                        for (int q = 0; q < SPL; ++q) yp = fmaf(cv[q], hist[s][q], yp);
                        dzv = sv(Cfg::S_ZF, s) * (reduce_slices<LPC>(yp) + Dd * xv);
                    }
                    float vals[V];
                    float s1 = 0.f, s2 = 0.f;
                    {   // the same per-state terms on pairs of states (f32x2)
                        const f32x2 dyc2 = pk2(dyc, dyc), dt2 = pk2(dt, dt), dx2 = pk2(dx, dx);
                        f32x2 s1v = pk2(0.f, 0.f), s2v = pk2(0.f, 0.f);
#pragma unroll
                        for (int q = 0; q < SPL; q += 2) {
                            const int sp = s > 0 ? s - 1 : 0;
                            const f32x2 hprev = s > 0 ? pk2(hist[sp][q], hist[sp][q + 1]) : pk2(hs[q], hs[q + 1]);
                            const f32x2 g = fma2(dyc2, pk2(cv[q], cv[q + 1]), pk2(G[q], G[q + 1]));
                            float e0, e1;
                            upk2(mul2(dt2, pk2(a2[q], a2[q + 1])), e0, e1);
                            const f32x2 gd = mul2(g, pk2(ex2_sfu(e0), ex2_sfu(e1)));
                            const f32x2 qv = mul2(gd, hprev);
                            s1v = fma2(g, pk2(bv[q], bv[q + 1]), s1v);
                            s2v = fma2(pk2(an[q], an[q + 1]), qv, s2v);
                            upk2(fma2(dt2, qv, pk2(dAacc[q], dAacc[q + 1])), dAacc[q], dAacc[q + 1]);
                            upk2(mul2(g, dx2), vals[q], vals[q + 1]);                       // dB
                            upk2(mul2(dyc2, pk2(hist[s][q], hist[s][q + 1])), vals[SPL + q],
                                 vals[SPL + q + 1]);                                      // dC
                            upk2(gd, G[q], G[q + 1]);
                        }
                        float a_, b_;
                        upk2(s1v, a_, b_);
                        s1 = a_ + b_;
                        upk2(s2v, a_, b_);
                        s2 = a_ + b_;
                    }
                    s1 = reduce_slices<LPC>(s1);
                    s2 = reduce_slices<LPC>(s2);
                    const float du = fmaf(xv, s1, s2) * sv(Cfg::S_SGU, s);
                    dbias += du;
                    if (sub == 0) {
                        store_io(ob + s * CH + cl, fmaf(dt, s1, dyc * Dd));
                        store_io(ob + Cfg::TOK / Cfg::ESZ + s * CH + cl, du);
                        store_io(ob + 2 * (Cfg::TOK / Cfg::ESZ) + s * CH + cl, dzv);
                    }
                    {   // sums over the warp's channels through shared memory: lane
                        // (channel c, slice sub) writes its terms to row c, then lane o
                        // adds output o down the CPW rows (one conflict-free load each)
                        float* wb = wsum + (s & 1) * Cfg::WSUM;
                        static_assert(SPL % 4 == 0, "float4 rows");
                        float* row = wb + (lane / LPC) * Cfg::RS + n0;
#pragma unroll
                        for (int q = 0; q < SPL; q += 4) {
                            *reinterpret_cast<float4*>(row + q) =
                                make_float4(vals[q], vals[q + 1], vals[q + 2], vals[q + 3]);
                            *reinterpret_cast<float4*>(row + N + q) =
                                make_float4(vals[SPL + q], vals[SPL + q + 1], vals[SPL + q + 2],
                                            vals[SPL + q + 3]);
                        }
                        __syncwarp();
#pragma unroll
                        for (int o0 = 0; o0 < 2 * N; o0 += 32) {
                            const int o = o0 + lane;
                            if (o < 2 * N) {
                                float acc = wb[o];
#pragma unroll
                                for (int c = 1; c < CPW; ++c) acc += wb[c * Cfg::RS + o];
                                myred[s * 2 * N + o] = acc;
                            }
                        }
                    }
                }
            }
            __syncwarp();   // the scratch rows are rewritten by the next tile's prologue
        }
        fence_proxy_async_smem();   // the output tile is read by the TMA store below
        __syncthreads();
        if (aborted()) break;
        for (int e = threadIdx.x; e < steps * 2 * N; e += blockDim.x) {
            float acc = 0.f;
#pragma unroll
            for (int w = 0; w < S::W; ++w) acc += red[w * T * 2 * N + e];
            const int s = e / (2 * N), v = e % (2 * N);
            p.pBC[(((int64_t)blockIdx.x * p.batch + b) * p.seqlen + ts + s) * 2 * N + v] = acc;
        }
        if (threadIdx.x == 0) {
            tma_store_3d(&maps.dx, ob, d0, (int)ts, b);
            tma_store_3d(&maps.ddelta, ob + Cfg::TOK / Cfg::ESZ, d0, (int)ts, b);
            if (dz_on) tma_store_3d(&maps.dz, ob + 2 * (Cfg::TOK / Cfg::ESZ), d0, (int)ts, b);
            bulk_commit();
            bulk_wait_read<1>();     // the output buffer written next is free again
        }
        __syncthreads();             // red and the stage are free; ob[(jj + 1) & 1] too
        refill(u);
    }
    if (threadIdx.x == 0) {
        bulk_wait<0>();
        if (aborted()) {
            // let the loads still in flight land before the CTA exits
            for (int u = issued - NST > 0 ? issued - NST : 0; u < issued; ++u)
                mbar_wait_bounded(&full[u % NST], (uint32_t)((u / NST) & 1), 100000000ull);
        }
    }
    if (aborted()) return;
    dD = reduce_slices<LPC>(dD);   // each lane summed the steps of its prologue share
    if (!valid) return;
    const int64_t bk = (int64_t)b * p.nchunk + k;
#pragma unroll
    for (int q = 0; q < SPL; ++q) p.pA[(bk * p.dim + d) * N + n0 + q] = dAacc[q];
    if (sub == 0) {
        p.pD[bk * p.dim + d] = dD;
        p.pbias[bk * p.dim + d] = dbias;
    }
    if (k == 0 && p.dinit) {
#pragma unroll
        for (int q = 0; q < SPL; ++q) p.dinit[((int64_t)b * p.dim + d) * N + n0 + q] = G[q];
    }
}

// 5. Final sums: dB, dC over the channel blocks; dA, dD, dbias over (b, k).
template <int N>
__global__ void scan_bwd_reduce_kernel(BwdParams p, int nblk, float* __restrict__ dB,
                                       float* __restrict__ dC, float* __restrict__ dA,
                                       float* __restrict__ dD, float* __restrict__ dbias) {
    const int64_t nbc = p.batch * p.seqlen * 2 * N;
    const int64_t npar = p.dim * N + 2 * p.dim;
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i < nbc) {
        float acc = 0.f;
        for (int c = 0; c < nblk; ++c) acc += p.pBC[(int64_t)c * nbc + i];
        const int v = (int)(i % (2 * N));
        const int64_t row = i / (2 * N);                 // (b, t)
        if (v < N) dB[row * N + v] = acc;
        else dC[row * N + v - N] = acc;
        return;
    }
    const int64_t j = i - nbc;
    if (j >= npar) return;
    const int64_t nbk = p.batch * p.nchunk;
    if (j < p.dim * N) {
        float acc = 0.f;
        for (int64_t c = 0; c < nbk; ++c) acc += p.pA[c * p.dim * N + j];
        dA[j] = acc;
    } else if (j < p.dim * N + p.dim) {
        const int64_t dd = j - p.dim * N;
        float acc = 0.f;
        for (int64_t c = 0; c < nbk; ++c) acc += p.pD[c * p.dim + dd];
        if (dD) dD[dd] = acc;
    } else {
        const int64_t dd = j - p.dim * N - p.dim;
        float acc = 0.f;
        for (int64_t c = 0; c < nbk; ++c) acc += p.pbias[c * p.dim + dd];
        if (dbias) dbias[dd] = acc;
    }
}

}  // namespace ssm
