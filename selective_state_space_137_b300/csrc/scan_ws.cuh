// scan_ws.cuh -- warp-specialised selective scan (path 2; bf16 or fp32 I/O,
// dstate 16).
//
// A CTA owns 16 channels of one sequence and two warps:
//   helper warp: issues the TMA loads of x, delta, z, B, C tiles (T steps),
//     computes per token (Delta, Delta*x) and widens B, C to fp32 (pre-pass),
//     then, once the scan has produced a tile's partial readouts, applies
//     skip + silu gate, casts, and TMA-stores the output tile (post-pass);
//   scan warp: lane (c, s) = (lane % 16, lane / 16) keeps states
//     [8s, 8s+8) of channel c in registers and runs, step after step,
//       dA = 2^(Delta * A[n] log2 e)   h = dA h + (Delta x) B[n]   y_s = sum C[n] h
//     with no block-wide barrier: it only waits for "tile ready" and
//     signals "readout written" on shared-memory mbarriers.
// The two warps hand tiles over through a ring of R slots (per slot: the
// (Delta, Delta*x) tile, the fp32 B/C tile, and the two partial readouts).
// The per-token work (softplus, skip, gate, conversions) thereby runs beside
// the recurrence instead of between its tiles.
//
// Ordering of the ring (slot i = j % R for tile j):
//   helper: pre(j) -> arrive ready[i] ... wait done[i'] (tile j-1) -> post(j-1)
//   scan:   wait ready[i] -> scan tile j -> arrive done[i]
// The helper writes slot i for tile j only after its own post(j-R), which
// waited for done of tile j-R, so the scan has finished with the slot.
//
// This is the recurrent mode of the selective SSM (stage 2 in
// "Mamba的三大创新") with the gate and skip of the Mamba block fused in; the
// expanded state is never materialised.
#pragma once
#include "common.cuh"
#include "scan_generic.cuh"
#include "scan_tiled.cuh"
#include "tma.cuh"

#ifndef SSM_WS_UNROLL
#define SSM_WS_UNROLL 4      // time steps unrolled in the scan warp's loop
#endif
#ifndef SSM_WS_PIPE
#define SSM_WS_PIPE 1        // 1: software-pipelined scan loop (decays one step ahead)
#endif
#ifndef SSM_WS_FULLUNROLL
#define SSM_WS_FULLUNROLL 1  // 1: full tiles run a fully unrolled scan (constant offsets)
#endif
#ifndef SSM_WS_MINBLOCKS
#define SSM_WS_MINBLOCKS 7   // resident CTAs per SM the register budget must allow
#endif

namespace ssm {

constexpr int kWsUnroll = SSM_WS_UNROLL;

template <typename IO, int T_, int S_, int R_>
struct WsCfg {
    static constexpr int N = 16, DC = 16, KS = 2, NS = 8, T = T_, S = S_, R = R_;
    static constexpr int THREADS = 64;
    static constexpr int ESZ = (int)sizeof(IO);
    static constexpr int TOK_BYTES = T * DC * ESZ;
    static constexpr int BC_BYTES = T * N * ESZ;
    static constexpr int OFF_X = 0;
    static constexpr int OFF_DL = round_up(OFF_X + TOK_BYTES, 128);
    static constexpr int OFF_Z = round_up(OFF_DL + TOK_BYTES, 128);
    static constexpr int OFF_B = round_up(OFF_Z + TOK_BYTES, 128);
    static constexpr int OFF_C = round_up(OFF_B + BC_BYTES, 128);
    static constexpr int STAGE = round_up(OFF_C + BC_BYTES, 128);
    // ring slot: dd float2 [T][16] | bc float [T][32] | yp float [2][T*16 + 16]
    static constexpr int YP_STRIDE = T * DC + 16;
    static constexpr int SL_DD = 0;
    static constexpr int SL_BC = round_up(SL_DD + T * DC * 8, 128);
    static constexpr int SL_YP = round_up(SL_BC + T * 2 * N * 4, 128);
    static constexpr int SLOT = round_up(SL_YP + KS * YP_STRIDE * 4, 128);
    static constexpr int OFF_RING = S * STAGE;
    static constexpr int OFF_OB = round_up(OFF_RING + R * SLOT, 128);
    static constexpr int OFF_BAR = round_up(OFF_OB + 2 * TOK_BYTES, 128);
    // barriers: full[S] (TMA), ready[R] (pre-pass done), done[R] (scan done)
    static constexpr int SMEM = OFF_BAR + (S + 2 * R) * 8;
};

template <typename IO, typename Cfg, int MODE>
__global__ void __launch_bounds__(64, SSM_WS_MINBLOCKS)
    scan_ws_kernel(const __grid_constant__ TiledMaps maps, const ScanParams p) {
    constexpr int N = Cfg::N, NS = Cfg::NS, DC = Cfg::DC, T = Cfg::T, S = Cfg::S, R = Cfg::R;
    constexpr bool FULL = (MODE == MODE_FULL);
    extern __shared__ __align__(1024) unsigned char smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + Cfg::OFF_BAR);
    uint64_t* ready = full + S;
    uint64_t* done = ready + R;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int d0 = blockIdx.x * DC;
    const int b = blockIdx.y;
    const int k = blockIdx.z;
    const int64_t t_begin = (int64_t)k * p.chunk_len;
    int64_t t_end = t_begin + p.chunk_len;
    if (t_end > p.seqlen) t_end = p.seqlen;
    const int ntiles = t_end > t_begin ? (int)((t_end - t_begin + T - 1) / T) : 0;
    const bool z_on = FULL && p.z != nullptr;

    // Role choice.  An SM issues from four sub-partitions, and a warp's
    // sub-partition follows its hardware slot (%warpid mod 4).  A two-warp CTA
    // gets two consecutive slots, so a fixed "warp 1 scans" would put every
    // scan warp of the SM on two of the four sub-partitions.  Instead the CTA
    // picks its scan warp from warp 0's slot so that successive CTAs alternate
    // between the sub-partitions (slot pairs 0-1, 2-3, 4-5, 6-7 scan on 0, 2,
    // 1, 3).  The rule names exactly one warp whatever the slots are; only the
    // speed depends on the slot layout.
    __shared__ unsigned slot_of[2];
    if (lane == 0) {
        unsigned wid;
        asm volatile("mov.u32 %0, %%warpid;" : "=r"(wid));
        slot_of[warp] = wid;
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) mbar_init(&full[s], 1);
        for (int r = 0; r < R; ++r) {
            mbar_init(&ready[r], 32);
            mbar_init(&done[r], 32);
        }
        fence_barrier_init();
    }
    __syncthreads();
    const unsigned w0 = slot_of[0];
    const int scan_warp = ((w0 & 1u) == ((w0 >> 2) & 1u)) ? 0 : 1;

    if (warp != scan_warp) {
        // ================= helper warp =================
        const uint32_t stage_tx = (uint32_t)(Cfg::TOK_BYTES * (z_on ? 3 : 2) +
                                             Cfg::BC_BYTES * (FULL ? 2 : 1));
        auto issue = [&](int j) {
            unsigned char* st = smem + (j % S) * Cfg::STAGE;
            const int t0 = (int)(t_begin + (int64_t)j * T);
            mbar_arrive_expect_tx(&full[j % S], stage_tx);
            tma_load_3d(st + Cfg::OFF_X, &maps.x, &full[j % S], d0, t0, b);
            tma_load_3d(st + Cfg::OFF_DL, &maps.delta, &full[j % S], d0, t0, b);
            if (z_on) tma_load_3d(st + Cfg::OFF_Z, &maps.z, &full[j % S], d0, t0, b);
            tma_load_3d(st + Cfg::OFF_B, &maps.B, &full[j % S], 0, t0, b);
            if (FULL) tma_load_3d(st + Cfg::OFF_C, &maps.C, &full[j % S], 0, t0, b);
        };
        if (lane == 0) {
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
        const int qc = (lane % (DC / 2)) * 2;
        const float2 bias2 = make_float2(
            (p.delta_bias && d0 + qc < p.dim) ? __ldg(p.delta_bias + d0 + qc) : 0.f,
            (p.delta_bias && d0 + qc + 1 < p.dim) ? __ldg(p.delta_bias + d0 + qc + 1) : 0.f);
        const float2 dsk2 =
            make_float2((FULL && p.D && d0 + qc < p.dim) ? __ldg(p.D + d0 + qc) : 0.f,
                        (FULL && p.D && d0 + qc + 1 < p.dim) ? __ldg(p.D + d0 + qc + 1) : 0.f);
        bool ok = true;

        // post-pass of tile j: skip + gate + cast + TMA store; frees stage j % S
        auto post = [&](int j) {
            const int i = j % R;
            ok = ok && mbar_wait_bounded(&done[i], (uint32_t)((j / R) & 1));
            const unsigned char* stg = smem + (j % S) * Cfg::STAGE;
            const int t0 = (int)(t_begin + (int64_t)j * T);
            if (FULL && ok) {
                const float* yp = reinterpret_cast<const float*>(smem + Cfg::OFF_RING + i * Cfg::SLOT + Cfg::SL_YP);
                const IO* xs = reinterpret_cast<const IO*>(stg + Cfg::OFF_X);
                const IO* zs = reinterpret_cast<const IO*>(stg + Cfg::OFF_Z);
                IO* ob = reinterpret_cast<IO*>(smem + Cfg::OFF_OB + (j & 1) * Cfg::TOK_BYTES);
                if (lane == 0) bulk_wait_read<1>();   // the store that last used ob[j & 1]
                __syncwarp();
#pragma unroll 4
                for (int gi = lane; gi < T * DC / 2; gi += 32) {
                    const int o = (gi / (DC / 2)) * DC + qc;
                    float2 y = __fadd2_rn(*reinterpret_cast<const float2*>(yp + o),
                                          *reinterpret_cast<const float2*>(yp + Cfg::YP_STRIDE + o));
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
                __syncwarp();
                if (lane == 0) {
                    tma_store_3d(&maps.out, ob, d0, t0, b);
                    bulk_commit();
                }
            }
            __syncwarp();
            if (lane == 0 && ok && j + S < ntiles) issue(j + S);   // stage j % S is free again
        };

        for (int j = 0; j < ntiles && ok; ++j) {
            const int i = j % R;
            // the slot's previous tile (j - R) was posted before this point
            ok = ok && mbar_wait_bounded(&full[j % S], (uint32_t)((j / S) & 1));
            if (!ok) break;
            const unsigned char* stg = smem + (j % S) * Cfg::STAGE;
            unsigned char* slot = smem + Cfg::OFF_RING + i * Cfg::SLOT;
            float2* dd = reinterpret_cast<float2*>(slot + Cfg::SL_DD);
            float* bc = reinterpret_cast<float*>(slot + Cfg::SL_BC);
            const IO* xs = reinterpret_cast<const IO*>(stg + Cfg::OFF_X);
            const IO* ds = reinterpret_cast<const IO*>(stg + Cfg::OFF_DL);
#pragma unroll 4
            for (int gi = lane; gi < T * DC / 2; gi += 32) {
                const int o = (gi / (DC / 2)) * DC + qc;
                const float2 xv = load2(xs + o);
                const float2 u = __fadd2_rn(load2(ds + o), bias2);
                float e0 = u.x, e1 = u.y;
                if (p.softplus) {
                    e0 = softplus_tiled<IO>(e0);
                    e1 = softplus_tiled<IO>(e1);
                }
                const float2 dx = __fmul2_rn(make_float2(e0, e1), xv);
                *reinterpret_cast<float4*>(dd + o) = make_float4(e0, dx.x, e1, dx.y);
            }
            {
                const IO* Bs = reinterpret_cast<const IO*>(stg + Cfg::OFF_B);
                const IO* Cs = reinterpret_cast<const IO*>(stg + Cfg::OFF_C);
                constexpr int V = 16 / Cfg::ESZ;
#pragma unroll
                for (int g = lane; g < T * N / V * (FULL ? 2 : 1); g += 32) {
                    const int which = g / (T * N / V);
                    const int e = (g % (T * N / V)) * V;
                    float f[V];
                    unpack<IO>(*reinterpret_cast<const uint4*>((which ? Cs : Bs) + e), f);
                    float4* o4 = reinterpret_cast<float4*>(bc + (e / N) * 2 * N + which * N + e % N);
#pragma unroll
                    for (int v = 0; v < V; v += 4) o4[v / 4] = make_float4(f[v], f[v + 1], f[v + 2], f[v + 3]);
                }
            }
            mbar_arrive(&ready[i]);          // every helper lane: its writes are published
            if (j >= 1) post(j - 1);
        }
        if (ok && ntiles > 0) post(ntiles - 1);
        if (lane == 0) bulk_wait<0>();
        if (!ok) {
            // let the loads that were issued land before the CTA's smem goes away
            if (lane == 0)
                for (int j = 0; j < ntiles; ++j) mbar_wait_bounded(&full[j % S], (uint32_t)((j / S) & 1), 50000000ull);
        }
        return;
    }

    // ================= scan warp =================
    const int c = lane & 15;
    const int s = lane >> 4;
    const int d = d0 + c;
    const bool dval = d < p.dim;
    float2 a2[NS / 2], h[NS / 2];
#pragma unroll
    for (int q = 0; q < NS / 2; ++q) {
        const int n = s * NS + 2 * q;
        a2[q] = dval ? make_float2(__ldg(p.A + (int64_t)d * N + n) * kLog2e,
                                   __ldg(p.A + (int64_t)d * N + n + 1) * kLog2e)
                     : make_float2(0.f, 0.f);
        float2 h0 = make_float2(0.f, 0.f);
        if (FULL && dval) {
            const float* src = nullptr;
            if (p.nchunk > 1) src = p.carry + (((int64_t)b * p.nchunk + k) * p.dim + d) * N;
            else if (p.initial_state) src = p.initial_state + ((int64_t)b * p.dim + d) * N;
            if (src) h0 = make_float2(src[n], src[n + 1]);
        }
        h[q] = h0;
    }
    float dsum = 0.f;
    bool ok = true;
    for (int j = 0; j < ntiles; ++j) {
        const int i = j % R;
        if (!mbar_wait_bounded(&ready[i], (uint32_t)((j / R) & 1))) { ok = false; break; }
        const unsigned char* slot = smem + Cfg::OFF_RING + i * Cfg::SLOT;
        const float2* dd = reinterpret_cast<const float2*>(slot + Cfg::SL_DD);
        const float* bc = reinterpret_cast<const float*>(slot + Cfg::SL_BC);
        float* ys = reinterpret_cast<float*>(const_cast<unsigned char*>(slot) + Cfg::SL_YP) + s * Cfg::YP_STRIDE;
        const int t0 = (int)(t_begin + (int64_t)j * T);
        const int steps = (int)((t_end - t0) < T ? (t_end - t0) : T);
        // One time step of the recurrence for this lane's 8 states.
        auto step = [&](int t) {
            const float2 dq = dd[t * DC + c];
            const float* row = bc + t * 2 * N + s * NS;
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
                    const float2 arg = __fmul2_rn(dl2, a2[q + r]);
                    const float2 dA = make_float2(ex2_sfu(arg.x), ex2_sfu(arg.y));
                    const float2 bb = r ? make_float2(b4.z, b4.w) : make_float2(b4.x, b4.y);
                    h[q + r] = __ffma2_rn(dA, h[q + r], __fmul2_rn(dx2, bb));
                    if (FULL) {
                        const float2 cc = r ? make_float2(c4.z, c4.w) : make_float2(c4.x, c4.y);
                        y2 = __ffma2_rn(cc, h[q + r], y2);
                    }
                }
            }
            if (FULL) ys[t * DC + c] = y2.x + y2.y;
            else dsum += dq.x;
        };
#if SSM_WS_FULLUNROLL
        if (steps == T) {
            // full tile: every offset is a compile-time constant
#pragma unroll
            for (int t = 0; t < T; ++t) step(t);
        } else {
            for (int t = 0; t < steps; ++t) step(t);
        }
#else
#if SSM_WS_PIPE
        // Software-pipelined: the operands and decays of step t+1 are loaded
        // and computed (SFU) while step t's state update and readout run.
        float2 cur_dq = dd[c];
        float4 cur_b[2], cur_c[2];
        float2 cur_dA[NS / 2];
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            cur_b[q] = *reinterpret_cast<const float4*>(bc + s * NS + 4 * q);
            if (FULL) cur_c[q] = *reinterpret_cast<const float4*>(bc + N + s * NS + 4 * q);
        }
#pragma unroll
        for (int q = 0; q < NS / 2; ++q) {
            const float2 arg = __fmul2_rn(make_float2(cur_dq.x, cur_dq.x), a2[q]);
            cur_dA[q] = make_float2(ex2_sfu(arg.x), ex2_sfu(arg.y));
        }
#pragma unroll 2
        for (int t = 0; t < steps; ++t) {
            const int tn = t + 1 < steps ? t + 1 : t;
            const float2 nxt_dq = dd[tn * DC + c];
            float4 nxt_b[2], nxt_c[2];
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                nxt_b[q] = *reinterpret_cast<const float4*>(bc + tn * 2 * N + s * NS + 4 * q);
                if (FULL) nxt_c[q] = *reinterpret_cast<const float4*>(bc + tn * 2 * N + N + s * NS + 4 * q);
            }
            float2 nxt_dA[NS / 2];
#pragma unroll
            for (int q = 0; q < NS / 2; ++q) {
                const float2 arg = __fmul2_rn(make_float2(nxt_dq.x, nxt_dq.x), a2[q]);
                nxt_dA[q] = make_float2(ex2_sfu(arg.x), ex2_sfu(arg.y));
            }
            const float2 dx2 = make_float2(cur_dq.y, cur_dq.y);
            float2 y2 = make_float2(0.f, 0.f);
#pragma unroll
            for (int q = 0; q < NS / 2; ++q) {
                const float4 b4 = cur_b[q / 2];
                const float2 bb = (q & 1) ? make_float2(b4.z, b4.w) : make_float2(b4.x, b4.y);
                h[q] = __ffma2_rn(cur_dA[q], h[q], __fmul2_rn(dx2, bb));
                if (FULL) {
                    const float4 c4 = cur_c[q / 2];
                    const float2 cc = (q & 1) ? make_float2(c4.z, c4.w) : make_float2(c4.x, c4.y);
                    y2 = __ffma2_rn(cc, h[q], y2);
                }
            }
            if (FULL) ys[t * DC + c] = y2.x + y2.y;
            else dsum += cur_dq.x;
            cur_dq = nxt_dq;
#pragma unroll
            for (int q = 0; q < 2; ++q) { cur_b[q] = nxt_b[q]; cur_c[q] = nxt_c[q]; }
#pragma unroll
            for (int q = 0; q < NS / 2; ++q) cur_dA[q] = nxt_dA[q];
        }
#else
#pragma unroll kWsUnroll
        for (int t = 0; t < steps; ++t) {
            const float2 dq = dd[t * DC + c];
            const float* row = bc + t * 2 * N + s * NS;
            const float2 dl2 = make_float2(dq.x, dq.x);
            const float2 dx2 = make_float2(dq.y, dq.y);
            float2 yacc[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};  // two short chains
#pragma unroll
            for (int q = 0; q < NS / 2; q += 2) {
                const float4 b4 = *reinterpret_cast<const float4*>(row + 2 * q);
                float4 c4;
                if (FULL) c4 = *reinterpret_cast<const float4*>(row + N + 2 * q);
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const float2 arg = __fmul2_rn(dl2, a2[q + r]);
                    const float2 dA = make_float2(ex2_sfu(arg.x), ex2_sfu(arg.y));
                    const float2 bb = r ? make_float2(b4.z, b4.w) : make_float2(b4.x, b4.y);
                    h[q + r] = __ffma2_rn(dA, h[q + r], __fmul2_rn(dx2, bb));
                    if (FULL) {
                        const float2 cc = r ? make_float2(c4.z, c4.w) : make_float2(c4.x, c4.y);
                        yacc[r] = __ffma2_rn(cc, h[q + r], yacc[r]);
                    }
                }
            }
            if (FULL) {
                const float2 y2 = __fadd2_rn(yacc[0], yacc[1]);
                ys[t * DC + c] = y2.x + y2.y;
            } else {
                dsum += dq.x;
            }
        }
#endif
#endif
        mbar_arrive(&done[i]);
    }
    if (!ok || !dval) return;
    float* dst = nullptr;
    if (FULL) {
        if (p.last_state && k == p.nchunk - 1) dst = p.last_state + ((int64_t)b * p.dim + d) * N + s * NS;
    } else {
        dst = p.carry + (((int64_t)b * p.nchunk + k) * p.dim + d) * N + s * NS;
        if (s == 0) p.dsum[((int64_t)b * p.nchunk + k) * p.dim + d] = dsum;
    }
    if (dst) {
#pragma unroll
        for (int q = 0; q < NS / 2; q += 2)
            *reinterpret_cast<float4*>(dst + 2 * q) = make_float4(h[q].x, h[q].y, h[q + 1].x, h[q + 1].y);
    }
}

}  // namespace ssm
