// scan_tiled.cuh -- the B300 selective-scan kernel (path 1).
//
// One CTA owns DC consecutive channels of one sequence and walks a range of
// time steps in tiles of T steps.  Per tile:
//   * TMA brings the x, delta, z tiles [T][DC] and the B, C tiles [T][N] of
//     the sequence into a ring of S shared-memory stages (mbarrier-completed),
//     up to S tiles ahead of the compute;
//   * pre-pass (all threads, 16-byte vectors): Delta = softplus(delta + bias)
//     and Delta*x once per token into smem as (Delta, Delta*x) pairs, and B, C
//     widened to fp32 -- the per-token work is done once, not once per state;
//   * scan: thread (c, s) holds states [s*NS, s*NS+NS) of channel c in
//     registers (NS = N/KS) and runs the recurrence over the tile:
//       dA = 2^(Delta * A[n]*log2 e)   (ex2 on the special-function unit)
//       h  = dA*h + (Delta*x)*B[n]     y += C[n]*h
//     leaving one partial sum of y per state slice in smem;
//   * post-pass (16-byte vectors): y = (sum of slices + D*x) * silu(z), cast
//     to the I/O type into an smem tile that one TMA store writes back.
// The state never leaves registers except at the chunk end.  This is the
// recurrent mode (stage 2) of the selective SSM computed without
// materialising the expanded state ("Mamba的三大创新", hardware-aware scan
// section), with the gate and skip of the Mamba block fused in.
//
// The same kernel in MODE_AGG produces a chunk's end state from a zero start
// and its sum of Delta (no z, no C, no output), for the cross-chunk carry.
#pragma once
#include "common.cuh"
#include "scan_generic.cuh"
#include "tma.cuh"

namespace ssm {

struct TiledMaps {
    CUtensorMap x, delta, z, B, C, out;
};

__host__ __device__ constexpr int round_up(int v, int a) { return (v + a - 1) / a * a; }

template <typename IO, int N_, int KS_, int DC_, int T_, int S_>
struct TiledCfg {
    static constexpr int N = N_, KS = KS_, DC = DC_, T = T_, S = S_;
    static constexpr int NS = N / KS;                 // states per thread
    static constexpr int THREADS = DC * KS;
    static constexpr int ESZ = (int)sizeof(IO);
    static constexpr int V = 16 / ESZ;                // elements per 16-byte vector
    static constexpr int TOK_BYTES = T * DC * ESZ;    // one x / delta / z / out tile
    static constexpr int BC_BYTES = T * N * ESZ;      // one B / C tile
    static constexpr int OFF_X = 0;
    static constexpr int OFF_DL = round_up(OFF_X + TOK_BYTES, 128);
    static constexpr int OFF_Z = round_up(OFF_DL + TOK_BYTES, 128);
    static constexpr int OFF_B = round_up(OFF_Z + TOK_BYTES, 128);
    static constexpr int OFF_C = round_up(OFF_B + BC_BYTES, 128);
    static constexpr int STAGE = round_up(OFF_C + BC_BYTES, 128);
    static constexpr int YP_STRIDE = T * DC + 16;     // floats; +16 staggers the slices' banks
    static constexpr int OFF_DD = S * STAGE;                                   // float2 [T][DC]
    static constexpr int OFF_BC = round_up(OFF_DD + T * DC * 8, 128);         // float [T][2N]
    static constexpr int OFF_YP = round_up(OFF_BC + T * 2 * N * 4, 128);      // float [KS][YP_STRIDE]
    static constexpr int OFF_OB = round_up(OFF_YP + KS * YP_STRIDE * 4, 128); // IO [2][T][DC]
    static constexpr int OFF_BAR = round_up(OFF_OB + 2 * TOK_BYTES, 128);
    static constexpr int SMEM = OFF_BAR + S * 8;
    static_assert(N % KS == 0 && NS % 4 == 0, "each thread owns a multiple of 4 states");
    static_assert((DC * ESZ) % 16 == 0 && (N * ESZ) % 16 == 0, "TMA rows are 16-byte multiples");
    static_assert(DC % V == 0 && N % V == 0, "16-byte vectors tile the rows");
    static_assert(THREADS % (DC / V) == 0, "each thread keeps the same channel vector");
};

template <typename IO>
__device__ __forceinline__ void unpack(const uint4& v, float* f);
template <>
__device__ __forceinline__ void unpack<float>(const uint4& v, float* f) {
    f[0] = __uint_as_float(v.x); f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z); f[3] = __uint_as_float(v.w);
}
template <>
__device__ __forceinline__ void unpack<__nv_bfloat16>(const uint4& v, float* f) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}
template <typename IO>
__device__ __forceinline__ uint4 pack(const float* f);
template <>
__device__ __forceinline__ uint4 pack<float>(const float* f) {
    return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                      __float_as_uint(f[3]));
}
template <>
__device__ __forceinline__ uint4 pack<__nv_bfloat16>(const float* f) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        __nv_bfloat162 p = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
        w[i] = *reinterpret_cast<uint32_t*>(&p);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// softplus for the tiled path.  fp32 I/O keeps the accurate libm form; for
// bf16 I/O: log(1 + e^u) = ln2 * log2(1 + 2^(u log2 e)) on the SFU (relative
// error of Delta below 1e-3 even where 1 + e^u rounds, far inside the bf16
// output tolerance), and u itself above 20.
template <typename IO>
__device__ __forceinline__ float softplus_tiled(float u);
template <>
__device__ __forceinline__ float softplus_tiled<float>(float u) { return softplus_accurate(u); }
template <>
__device__ __forceinline__ float softplus_tiled<__nv_bfloat16>(float u) {
    float l;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(l) : "f"(1.f + ex2_sfu(u * kLog2e)));
    return u > 20.f ? u : l * kLn2;
}

template <typename IO>
__device__ __forceinline__ float silu_tiled(float v);
template <>
__device__ __forceinline__ float silu_tiled<float>(float v) { return silu_accurate(v); }
template <>
__device__ __forceinline__ float silu_tiled<__nv_bfloat16>(float v) {
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(1.f + ex2_sfu(-v * kLog2e)));
    return v * r;
}

template <typename IO, typename Cfg, int MODE>
__global__ void __launch_bounds__(Cfg::THREADS)
    scan_tiled_kernel(const __grid_constant__ TiledMaps maps, const ScanParams p) {
    constexpr int N = Cfg::N, NS = Cfg::NS, DC = Cfg::DC, T = Cfg::T, S = Cfg::S, V = Cfg::V;
    constexpr int KS = Cfg::KS, THREADS = Cfg::THREADS;
    constexpr bool FULL = (MODE == MODE_FULL);
    extern __shared__ __align__(1024) unsigned char smem[];
    float2* dd = reinterpret_cast<float2*>(smem + Cfg::OFF_DD);
    float* bc = reinterpret_cast<float*>(smem + Cfg::OFF_BC);
    float* yp = reinterpret_cast<float*>(smem + Cfg::OFF_YP);
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + Cfg::OFF_BAR);

    const int tid = threadIdx.x;
    const int d0 = blockIdx.x * DC;
    const int b = blockIdx.y;
    const int k = blockIdx.z;
    const int64_t t_begin = (int64_t)k * p.chunk_len;
    int64_t t_end = t_begin + p.chunk_len;
    if (t_end > p.seqlen) t_end = p.seqlen;
    const int ntiles = t_end > t_begin ? (int)((t_end - t_begin + T - 1) / T) : 0;
    const bool z_on = FULL && p.z != nullptr;
    const uint32_t stage_tx = (uint32_t)(Cfg::TOK_BYTES * (z_on ? 3 : 2) +
                                         Cfg::BC_BYTES * (FULL ? 2 : 1));

    auto issue = [&](int j) {  // TMA loads of tile j into stage j % S (thread 0)
        unsigned char* st = smem + (j % S) * Cfg::STAGE;
        const int t0 = (int)(t_begin + (int64_t)j * T);
        mbar_arrive_expect_tx(&bar[j % S], stage_tx);
        tma_load_3d(st + Cfg::OFF_X, &maps.x, &bar[j % S], d0, t0, b);
        tma_load_3d(st + Cfg::OFF_DL, &maps.delta, &bar[j % S], d0, t0, b);
        if (z_on) tma_load_3d(st + Cfg::OFF_Z, &maps.z, &bar[j % S], d0, t0, b);
        tma_load_3d(st + Cfg::OFF_B, &maps.B, &bar[j % S], 0, t0, b);
        if (FULL) tma_load_3d(st + Cfg::OFF_C, &maps.C, &bar[j % S], 0, t0, b);
    };

    if (tid == 0) {
        for (int s = 0; s < S; ++s) mbar_init(&bar[s], 1);
        fence_barrier_init();
    }
    __syncthreads();
    if (tid == 0) {
        prefetch_tmap(&maps.x);
        prefetch_tmap(&maps.delta);
        prefetch_tmap(&maps.B);
        if (FULL) {
            prefetch_tmap(&maps.C);
            prefetch_tmap(&maps.out);
            if (z_on) prefetch_tmap(&maps.z);
        }
        for (int j = 0; j < S && j < ntiles; ++j) issue(j);
    }

    // ---- per-thread constants
    const int c = tid % DC;              // scan: channel within the block
    const int s = tid / DC;              // scan: state slice
    const int d = d0 + c;
    const bool dval = d < p.dim;
    float a2[NS], h[NS];
#pragma unroll
    for (int j = 0; j < NS; ++j)
        a2[j] = dval ? __ldg(p.A + (int64_t)d * N + s * NS + j) * kLog2e : 0.f;
    const int64_t chan = (int64_t)b * p.dim + d;
    if (!FULL || !dval) {
#pragma unroll
        for (int j = 0; j < NS; ++j) h[j] = 0.f;
    } else if (p.nchunk > 1) {
        const float* cin = p.carry + (((int64_t)b * p.nchunk + k) * p.dim + d) * N + s * NS;
#pragma unroll
        for (int j = 0; j < NS; ++j) h[j] = cin[j];
    } else if (p.initial_state) {
#pragma unroll
        for (int j = 0; j < NS; ++j) h[j] = __ldg(p.initial_state + chan * N + s * NS + j);
    } else {
#pragma unroll
        for (int j = 0; j < NS; ++j) h[j] = 0.f;
    }
    // pre/post-pass: this thread always handles the same V channels
    const int vc = (tid % (DC / V)) * V;
    float bias[V], dsk[V];
#pragma unroll
    for (int i = 0; i < V; ++i) {
        const int dd_ = d0 + vc + i;
        bias[i] = (p.delta_bias && dd_ < p.dim) ? __ldg(p.delta_bias + dd_) : 0.f;
        dsk[i] = (FULL && p.D && dd_ < p.dim) ? __ldg(p.D + dd_) : 0.f;
    }
    float dsum = 0.f;
    int failed = -1;   // tile whose wait gave up

    for (int j = 0; j < ntiles; ++j) {
        const int st = j % S;
        const unsigned char* stg = smem + st * Cfg::STAGE;
        const int t0 = (int)(t_begin + (int64_t)j * T);
        const int steps = (int)((t_end - t0) < T ? (t_end - t0) : T);
        // wait for tile j (bounded); all threads agree on giving up
        const bool got = mbar_wait_bounded(&bar[st], (uint32_t)((j / S) & 1));
        if (__syncthreads_or(!got)) { failed = j; break; }

        // ---- pre-pass: (Delta, Delta*x) per token, B and C to fp32
        const IO* xs = reinterpret_cast<const IO*>(stg + Cfg::OFF_X);
        const IO* ds = reinterpret_cast<const IO*>(stg + Cfg::OFF_DL);
        for (int g = tid; g < T * DC / V; g += THREADS) {
            const int t = g / (DC / V);
            float xv[V], dv[V];
            unpack<IO>(*reinterpret_cast<const uint4*>(xs + t * DC + vc), xv);
            unpack<IO>(*reinterpret_cast<const uint4*>(ds + t * DC + vc), dv);
            float4* out2 = reinterpret_cast<float4*>(dd + t * DC + vc);
#pragma unroll
            for (int i = 0; i < V; i += 2) {
                const float u0 = dv[i] + bias[i], u1 = dv[i + 1] + bias[i + 1];
                const float t0v = p.softplus ? softplus_tiled<IO>(u0) : u0;
                const float t1v = p.softplus ? softplus_tiled<IO>(u1) : u1;
                out2[i / 2] = make_float4(t0v, t0v * xv[i], t1v, t1v * xv[i + 1]);
            }
        }
        {
            const IO* Bs = reinterpret_cast<const IO*>(stg + Cfg::OFF_B);
            const IO* Cs = reinterpret_cast<const IO*>(stg + Cfg::OFF_C);
            for (int g = tid; g < T * N / V * (FULL ? 2 : 1); g += THREADS) {
                const int which = g / (T * N / V);             // 0 = B, 1 = C
                const int e = (g % (T * N / V)) * V;           // element within [T][N]
                const int t = e / N, n = e % N;
                float f[V];
                unpack<IO>(*reinterpret_cast<const uint4*>((which ? Cs : Bs) + e), f);
                float4* o = reinterpret_cast<float4*>(bc + t * 2 * N + which * N + n);
#pragma unroll
                for (int i = 0; i < V; i += 4) o[i / 4] = make_float4(f[i], f[i + 1], f[i + 2], f[i + 3]);
            }
        }
        __syncthreads();

        // ---- scan over the tile
        float* ys = yp + s * Cfg::YP_STRIDE;
#pragma unroll 2
        for (int t = 0; t < steps; ++t) {
            const float2 dv = dd[t * DC + c];
            const float* row = bc + t * 2 * N;
            float Bv[NS], Cv[NS];
#pragma unroll
            for (int q = 0; q < NS; q += 4) {
                const float4 b4 = *reinterpret_cast<const float4*>(row + s * NS + q);
                Bv[q] = b4.x; Bv[q + 1] = b4.y; Bv[q + 2] = b4.z; Bv[q + 3] = b4.w;
                if (FULL) {
                    const float4 c4 = *reinterpret_cast<const float4*>(row + N + s * NS + q);
                    Cv[q] = c4.x; Cv[q + 1] = c4.y; Cv[q + 2] = c4.z; Cv[q + 3] = c4.w;
                }
            }
            float y0 = 0.f, y1 = 0.f;
#pragma unroll
            for (int q = 0; q < NS; ++q) {
                const float dA = ex2_sfu(dv.x * a2[q]);
                h[q] = fmaf(dA, h[q], dv.y * Bv[q]);
                if (FULL) {
                    if (q & 1) y1 = fmaf(Cv[q], h[q], y1);
                    else y0 = fmaf(Cv[q], h[q], y0);
                }
            }
            if (FULL) ys[t * DC + c] = y0 + y1;
            else dsum += dv.x;
        }

        if (FULL) {
            if (tid == 0) bulk_wait_read<1>();   // the store that last used ob[j & 1] has read it
            __syncthreads();
            // ---- post-pass: skip, gate, cast, into the out tile
            const IO* zs = reinterpret_cast<const IO*>(stg + Cfg::OFF_Z);
            IO* ob = reinterpret_cast<IO*>(smem + Cfg::OFF_OB + (j & 1) * Cfg::TOK_BYTES);
            for (int g = tid; g < T * DC / V; g += THREADS) {
                const int t = g / (DC / V);
                float xv[V], yv[V], zv[V];
                unpack<IO>(*reinterpret_cast<const uint4*>(xs + t * DC + vc), xv);
                if (z_on) unpack<IO>(*reinterpret_cast<const uint4*>(zs + t * DC + vc), zv);
#pragma unroll
                for (int i = 0; i < V; i += 4) {
                    float4 acc = *reinterpret_cast<const float4*>(yp + t * DC + vc + i);
#pragma unroll
                    for (int q = 1; q < KS; ++q) {
                        const float4 o = *reinterpret_cast<const float4*>(
                            yp + q * Cfg::YP_STRIDE + t * DC + vc + i);
                        acc.x += o.x; acc.y += o.y; acc.z += o.z; acc.w += o.w;
                    }
                    yv[i] = acc.x; yv[i + 1] = acc.y; yv[i + 2] = acc.z; yv[i + 3] = acc.w;
                }
#pragma unroll
                for (int i = 0; i < V; ++i) {
                    float y = fmaf(dsk[i], xv[i], yv[i]);
                    if (z_on) y *= silu_tiled<IO>(zv[i]);
                    yv[i] = y;
                }
                *reinterpret_cast<uint4*>(ob + t * DC + vc) = pack<IO>(yv);
            }
            fence_proxy_async_smem();
        }
        __syncthreads();   // pre/post reads of stage st and the out tile writes are done
        if (tid == 0) {
            if (FULL) {
                tma_store_3d(&maps.out,
                             smem + Cfg::OFF_OB + (j & 1) * Cfg::TOK_BYTES, d0, t0, b);
                bulk_commit();
            }
            if (j + S < ntiles) issue(j + S);   // stage st is free again
        }
    }
    if (tid == 0) bulk_wait<0>();
    if (failed >= 0) {
        // A wait gave up: let the loads this CTA issued and did not consume
        // (tiles failed .. failed+S-1) land before its shared memory is released.
        if (tid == 0)
            for (int j = failed; j < failed + S && j < ntiles; ++j)
                mbar_wait_bounded(&bar[j % S], (uint32_t)((j / S) & 1), 100000000ull);
        return;
    }

    if (!dval) return;
    if (FULL) {
        if (p.last_state && k == p.nchunk - 1) {
#pragma unroll
            for (int q = 0; q < NS; q += 4)
                *reinterpret_cast<float4*>(p.last_state + chan * N + s * NS + q) =
                    make_float4(h[q], h[q + 1], h[q + 2], h[q + 3]);
        }
    } else {
        float* cend = p.carry + (((int64_t)b * p.nchunk + k) * p.dim + d) * N + s * NS;
#pragma unroll
        for (int q = 0; q < NS; q += 4)
            *reinterpret_cast<float4*>(cend + q) = make_float4(h[q], h[q + 1], h[q + 2], h[q + 3]);
        if (s == 0) p.dsum[((int64_t)b * p.nchunk + k) * p.dim + d] = dsum;
    }
}

}  // namespace ssm
