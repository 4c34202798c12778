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

#ifndef SSM_SCAN_PACKED
#define SSM_SCAN_PACKED 0     // 1: state pairs in f32x2 registers; 0: scalar fp32
#endif
#ifndef SSM_SCAN_UNROLL
#define SSM_SCAN_UNROLL 2     // time steps unrolled in the scan loop
#endif

namespace ssm {

constexpr int kScanUnroll = SSM_SCAN_UNROLL;

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
    static_assert(THREADS % (DC / 2) == 0, "fixed channel pair per thread");
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

// Two adjacent io elements as fp32 (one 4- or 8-byte shared load), and back.
__device__ __forceinline__ float2 load2(const float* p) { return *reinterpret_cast<const float2*>(p); }
__device__ __forceinline__ float2 load2(const __nv_bfloat16* p) {
    const uint32_t w = *reinterpret_cast<const uint32_t*>(p);
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}
__device__ __forceinline__ float load1(const float* p) { return *p; }
__device__ __forceinline__ float load1(const __nv_bfloat16* p) {
    return __uint_as_float((uint32_t)(*reinterpret_cast<const unsigned short*>(p)) << 16);
}
__device__ __forceinline__ void store2(float* p, float lo, float hi) {
    *reinterpret_cast<float2*>(p) = make_float2(lo, hi);
}
__device__ __forceinline__ void store2(__nv_bfloat16* p, float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    *reinterpret_cast<__nv_bfloat162*>(p) = v;
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
    // softplus(u) >= u, and the formula is exact to fp32 for u <= 80 (the
    // clamp keeps 2^(u log2 e) finite); above, max() returns u itself.
    float l;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(l) : "f"(1.f + ex2_sfu(fminf(u, 80.f) * kLog2e)));
    return fmaxf(u, l * kLn2);
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
    // pre- and post-pass: this thread always handles the channel pair `qc`, `qc+1`
    const int qc = (tid % (DC / 2)) * 2;
    const float2 bias2 =
        make_float2((p.delta_bias && d0 + qc < p.dim) ? __ldg(p.delta_bias + d0 + qc) : 0.f,
                    (p.delta_bias && d0 + qc + 1 < p.dim) ? __ldg(p.delta_bias + d0 + qc + 1) : 0.f);
    const float2 dsk2 =
        make_float2((FULL && p.D && d0 + qc < p.dim) ? __ldg(p.D + d0 + qc) : 0.f,
                    (FULL && p.D && d0 + qc + 1 < p.dim) ? __ldg(p.D + d0 + qc + 1) : 0.f);
    float2 a2p[NS / 2], hp[NS / 2];
#pragma unroll
    for (int q = 0; q < NS / 2; ++q) {
        a2p[q] = make_float2(a2[2 * q], a2[2 * q + 1]);
        hp[q] = make_float2(h[2 * q], h[2 * q + 1]);
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

        // ---- pre-pass: (Delta, Delta*x) per token, B and C to fp32.  Lanes take
        // consecutive channel pairs of a row: conflict-free 16-byte stores.
        const IO* xs = reinterpret_cast<const IO*>(stg + Cfg::OFF_X);
        const IO* ds = reinterpret_cast<const IO*>(stg + Cfg::OFF_DL);
#pragma unroll 4
        for (int g = tid; g < T * DC / 2; g += THREADS) {
            const int o = (g / (DC / 2)) * DC + qc;
            const float2 xv = load2(xs + o);
            const float2 u = __fadd2_rn(load2(ds + o), bias2);
            float d0v = u.x, d1v = u.y;
            if (p.softplus) {
                d0v = softplus_tiled<IO>(d0v);
                d1v = softplus_tiled<IO>(d1v);
            }
            const float2 dx = __fmul2_rn(make_float2(d0v, d1v), xv);
            *reinterpret_cast<float4*>(dd + o) = make_float4(d0v, dx.x, d1v, dx.y);
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
#pragma unroll kScanUnroll
        for (int t = 0; t < steps; ++t) {
            const float2 dq = dd[t * DC + c];             // (Delta, Delta*x)
            const float* row = bc + t * 2 * N + s * NS;
#if SSM_SCAN_PACKED
            // pairs of states in float2 registers (f32x2 FMA/MUL)
            const float2 dl2 = make_float2(dq.x, dq.x);
            const float2 dx2 = make_float2(dq.y, dq.y);
            float2 y2 = make_float2(0.f, 0.f);
#pragma unroll
            for (int q = 0; q < NS / 2; q += 2) {
                const float4 b4 = *reinterpret_cast<const float4*>(row + 2 * q);
                float4 c4;
                if (FULL) c4 = *reinterpret_cast<const float4*>(row + N + 2 * q);
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const float2 arg = __fmul2_rn(dl2, a2p[q + r]);
                    const float2 dA = make_float2(ex2_sfu(arg.x), ex2_sfu(arg.y));
                    const float2 bb = r ? make_float2(b4.z, b4.w) : make_float2(b4.x, b4.y);
                    hp[q + r] = __ffma2_rn(dA, hp[q + r], __fmul2_rn(dx2, bb));
                    if (FULL) {
                        const float2 cc = r ? make_float2(c4.z, c4.w) : make_float2(c4.x, c4.y);
                        y2 = __ffma2_rn(cc, hp[q + r], y2);
                    }
                }
            }
            const float yv = y2.x + y2.y;
#else
            float Bv[NS], Cv[NS];
#pragma unroll
            for (int q = 0; q < NS; q += 4) {
                const float4 b4 = *reinterpret_cast<const float4*>(row + q);
                Bv[q] = b4.x; Bv[q + 1] = b4.y; Bv[q + 2] = b4.z; Bv[q + 3] = b4.w;
                if (FULL) {
                    const float4 c4 = *reinterpret_cast<const float4*>(row + N + q);
                    Cv[q] = c4.x; Cv[q + 1] = c4.y; Cv[q + 2] = c4.z; Cv[q + 3] = c4.w;
                }
            }
            float ya = 0.f, yb = 0.f;
#pragma unroll
            for (int q = 0; q < NS; ++q) {
                float& hq = (q & 1) ? hp[q / 2].y : hp[q / 2].x;
                const float a = (q & 1) ? a2p[q / 2].y : a2p[q / 2].x;
                const float dA = ex2_sfu(dq.x * a);
                hq = fmaf(dA, hq, dq.y * Bv[q]);
                if (FULL) {
                    if (q & 1) yb = fmaf(Cv[q], hq, yb);
                    else ya = fmaf(Cv[q], hq, ya);
                }
            }
            const float yv = ya + yb;
#endif
            if (FULL) ys[t * DC + c] = yv;
            else dsum += dq.x;
        }

        if (FULL) {
            if (tid == 0) bulk_wait_read<1>();   // the store that last used ob[j & 1] has read it
            __syncthreads();
            // ---- post-pass: skip, gate, cast, into the out tile (channel pairs)
            const IO* zs = reinterpret_cast<const IO*>(stg + Cfg::OFF_Z);
            IO* ob = reinterpret_cast<IO*>(smem + Cfg::OFF_OB + (j & 1) * Cfg::TOK_BYTES);
#pragma unroll 2
            for (int g = tid; g < T * DC / 2; g += THREADS) {
                const int t = g / (DC / 2);
                const int o = t * DC + qc;
                float2 y = *reinterpret_cast<const float2*>(yp + o);
#pragma unroll
                for (int q = 1; q < KS; ++q)
                    y = __fadd2_rn(y, *reinterpret_cast<const float2*>(yp + q * Cfg::YP_STRIDE + o));
                y = __ffma2_rn(dsk2, load2(xs + o), y);
                float y0 = y.x, y1 = y.y;
                if (z_on) {
                    const float2 zv = load2(zs + o);
                    y0 *= silu_tiled<IO>(zv.x);
                    y1 *= silu_tiled<IO>(zv.y);
                }
                store2(ob + o, y0, y1);
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
    float* dst = nullptr;
    if (FULL) {
        if (p.last_state && k == p.nchunk - 1) dst = p.last_state + chan * N + s * NS;
    } else {
        dst = p.carry + (((int64_t)b * p.nchunk + k) * p.dim + d) * N + s * NS;
        if (s == 0) p.dsum[((int64_t)b * p.nchunk + k) * p.dim + d] = dsum;
    }
    if (dst) {
#pragma unroll
        for (int q = 0; q < NS / 2; q += 2)
            *reinterpret_cast<float4*>(dst + 2 * q) = make_float4(hp[q].x, hp[q].y, hp[q + 1].x, hp[q + 1].y);
    }
}

}  // namespace ssm
