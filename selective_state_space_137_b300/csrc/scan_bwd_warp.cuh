// scan_bwd_warp.cuh -- the reverse sweep of the backward in the one-warp
// layout of the forward's tiled scan (dstate 16, bf16 or fp32 I/O, 16-byte
// rows).  The gradients are those of scan_bwd.cuh (same formulas, same
// launches around it: chunk aggregates, carries, the final reduce).  The
// state before every tile comes from checkpoints: the training forward's, or
// those the one-warp scan's MODE_STATES pass writes right before this sweep.
//
// A warp owns 16 channels of one sequence over one chunk of time, walked in
// tiles of 16 steps (the checkpoint spacing).  Lane (p, s) = (lane & 7,
// lane >> 3) owns the channel pair (2p, 2p + 1) and four states of both
// channels, the pair in the two halves of an f32x2 register.  A CTA holds W
// such warps side by side along the channels (W chosen by the host); the
// warps share nothing and never wait for one another: each writes the sums of
// its dB and dC terms over its 16 channels (a [T][2N] tile in shared memory,
// copied out after the tile's steps) to its own rows of the partial sums in
// global memory, which the final reduce adds in a fixed order (the result
// does not depend on timing).
//
// Per tile (reverse order):
//   pre-pass  per token, once (lane p, steps s, s + 4, s + 8, s + 12): Delta,
//             Delta x, dyc = dout silu(z), the factors of dz and of ddelta;
//             B and C widened to fp32 (B_n, B_n) pairs;
//   recompute the tile's states forward from its checkpoint, kept in
//             registers (H steps at a time);
//   reverse   per step and state:  g = dyc C + G,  G <- g dA,  q = G h_{t-1},
//             dA += Delta q, and three sums over the lane's states -- g B, A q
//             and C h (the per-token gradients) -- finished over the four
//             state quarters by shuffles; the dB = g Delta x and dC = dyc h
//             terms summed over the warp's 16 channels by shuffles and
//             stored (one 128-byte row per step);
//   post-pass per token: dx, ddelta, dz from the state sums, cast, TMA store.
//
// Shuffle reductions without selects.  Slot q of a lane holds state
// 4s + 2 (b2 ^ (q >> 1)) + (q & 1), b2 = bit 2 of the lane: lanes l and l ^ 4
// hold the two halves of their four states in opposite slots, so the first
// round of the channel sum keeps slots 0, 1 and sends slots 2, 3 on every
// lane.  Lanes with s >= 2 hold the channel pair as (2p + 1, 2p): the first
// round of the state sum (partner l ^ 16) keeps the low half and sends the
// high half on every lane.  (The per-token pairs are kept in shared memory in
// both channel orders for this.)
//
// The recurrence and its adjoint are those of the recurrent mode (stage 2 of
// "Mamba的三大创新"); see scan_bwd.cuh for the derivation.
#pragma once
#include "common.cuh"
#include "scan_bwd.cuh"
#include "tile_io.cuh"
#include "tma.cuh"

namespace ssm {

template <typename IO>
struct BwdWarpCfg {
    static constexpr int N = 16, DC = 16, NP = 8, T = kBwdT;
    static constexpr int ESZ = (int)sizeof(IO);
    // TMA ring depth: three stages of bf16 tiles, two of fp32 (7 and 6 warps a CTA fit)
    static constexpr int NST = ESZ == 2 ? 3 : 2;
    static constexpr int WMAX = ESZ == 2 ? 7 : 6;
    static constexpr int TOK = T * DC * ESZ;                  // one [T][16] token tile
    static constexpr int ROW = T * N * ESZ;                   // one [T][N] B or C tile
    static constexpr int OFF_X = 0, OFF_DL = TOK, OFF_DO = 2 * TOK, OFF_Z = 3 * TOK;
    static constexpr int OFF_B = 4 * TOK, OFF_C = 4 * TOK + ROW;
    static constexpr int STAGE = round_up(4 * TOK + 2 * ROW, 128);
    static constexpr int OFF_DD = NST * STAGE;                // float4 [2][T][NP] (Delta, Delta x), both orders
    static constexpr int OFF_DY = OFF_DD + 2 * T * NP * 16;   // float2 [2][T][NP] dyc, both orders
    static constexpr int OFF_ZS = OFF_DY + 2 * T * NP * 8;    // float4 [T][NP] (dz factor, softplus')
    static constexpr int OFF_XS = OFF_ZS + T * NP * 16;       // float2 [T][NP] x
    static constexpr int OFF_BP = OFF_XS + T * NP * 8;        // float4 [T][N / 2] (B_n, B_n, B_n+1, B_n+1)
    static constexpr int OFF_CP = OFF_BP + T * N * 8;         // the same for C
    static constexpr int OFF_SV = OFF_CP + T * N * 8;         // float2 [T][32] state sums
    static constexpr int OFF_RD = OFF_SV + T * 32 * 8;        // float [T][2N] dB | dC sums of the tile
    static constexpr int OFF_OB = OFF_RD + T * 2 * N * 4;     // IO [3][T][DC] dx, ddelta, dz
    static constexpr int OFF_BAR = round_up(OFF_OB + 3 * TOK, 16);
    static constexpr int WARP = round_up(OFF_BAR + NST * 8, 128);   // one warp's shared memory
    static constexpr int smem(int w) { return w * WARP; }
    static_assert(TOK % 128 == 0 && ROW % 128 == 0 && OFF_OB % 128 == 0, "TMA buffers 128-byte aligned");
};

// sigmoid of a pair (the SFU form of scan_bwd.cuh)
__device__ __forceinline__ float2 sigmoid2(float2 u) { return make_float2(sigmoid_fast(u.x), sigmoid_fast(u.y)); }

template <typename IO, int H, bool SP, bool ZG>
__global__ void __launch_bounds__(256, 1)
    scan_bwd_warp_kernel(const __grid_constant__ BwdMaps maps, BwdParams p) {
    using Cfg = BwdWarpCfg<IO>;
    constexpr int N = 16, T = Cfg::T, DC = Cfg::DC, NP = Cfg::NP, NST = Cfg::NST;
    constexpr unsigned FULL = 0xffffffffu;
    static_assert(H == 8 || H == 16, "state history of 8 or 16 steps");
    extern __shared__ __align__(1024) unsigned char smem[];
    const int W = (int)(blockDim.x >> 5);
    const int warp = (int)(threadIdx.x >> 5), lane = (int)(threadIdx.x & 31);
    unsigned char* ws = smem + warp * Cfg::WARP;
    uint64_t* full = reinterpret_cast<uint64_t*>(ws + Cfg::OFF_BAR);
    const int b = blockIdx.y, k = blockIdx.z;
    const int64_t unit = (int64_t)blockIdx.x * W + warp;   // this warp's 16-channel block
    const int d0 = (int)(unit * DC);
    if (d0 >= p.dim) return;   // a warp of the last CTA past the channels
    if (lane == 0) {
        for (int i = 0; i < NST; ++i) mbar_init(&full[i], 1);
        fence_barrier_init();
    }
    __syncwarp();

    const int64_t t0 = (int64_t)k * p.chunk_len;
    int64_t t1 = t0 + p.chunk_len;
    if (t1 > p.seqlen) t1 = p.seqlen;
    const int ntile = (int)((t1 - t0 + T - 1) / T);
    const int nload = ntile;
    const bool dz_on = ZG && p.dz != nullptr;
    const int64_t tile0 = t0 / T;

    const int pp = lane & 7, s = lane >> 3, hi = lane >> 4, m = s & 1;
    const int b0 = pp & 1, b1 = (pp >> 1) & 1, b2 = (pp >> 2) & 1;
    const int o_lane = 16 * b0 + 4 * s + 2 * b2 + b1;   // the dB | dC output this lane ends with
    // the two halves of a pair: channels cx (low) and cy (high)
    const int64_t cx = (int64_t)d0 + 2 * pp + hi, cy = (int64_t)d0 + 2 * pp + 1 - hi;
    const bool vx = cx < p.dim, vy = cy < p.dim;
    // natural order (c0, c0 + 1) of the pre- and post-passes
    const int64_t c0 = (int64_t)d0 + 2 * pp;
    const bool v0 = c0 < p.dim, v1 = c0 + 1 < p.dim;
    const float2 bias2 = make_float2((p.delta_bias && v0) ? __ldg(p.delta_bias + c0) : 0.f,
                                     (p.delta_bias && v1) ? __ldg(p.delta_bias + c0 + 1) : 0.f);
    const float2 D2 = make_float2((p.D && v0) ? __ldg(p.D + c0) : 0.f, (p.D && v1) ? __ldg(p.D + c0 + 1) : 0.f);
    auto nst = [&](int q) { return 4 * s + 2 * (b2 ^ (q >> 1)) + (q & 1); };   // state of slot q

    float4* DD = reinterpret_cast<float4*>(ws + Cfg::OFF_DD);
    float2* DY = reinterpret_cast<float2*>(ws + Cfg::OFF_DY);
    float4* ZS = reinterpret_cast<float4*>(ws + Cfg::OFF_ZS);
    float2* XS = reinterpret_cast<float2*>(ws + Cfg::OFF_XS);
    float4* BP = reinterpret_cast<float4*>(ws + Cfg::OFF_BP);
    float4* CP = reinterpret_cast<float4*>(ws + Cfg::OFF_CP);
    float2* SV = reinterpret_cast<float2*>(ws + Cfg::OFF_SV);
    IO* OB = reinterpret_cast<IO*>(ws + Cfg::OFF_OB);

    // ---- per-channel state: A log2 e, the incoming adjoint G
    float2 a2[4], G[4], dAacc[4];
    {
        const int64_t bk = (int64_t)b * p.nchunk + k;
        const float* gx = nullptr;
        const float* gy = nullptr;
        if (p.nchunk > 1) {
            gx = p.ebuf + (bk * p.dim + cx) * N;
            gy = p.ebuf + (bk * p.dim + cy) * N;
        } else if (p.dlast) {
            gx = p.dlast + ((int64_t)b * p.dim + cx) * N;
            gy = p.dlast + ((int64_t)b * p.dim + cy) * N;
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int n = nst(q);
            a2[q] = make_float2(vx ? __ldg(p.A + cx * N + n) * kLog2e : 0.f,
                                vy ? __ldg(p.A + cy * N + n) * kLog2e : 0.f);
            G[q] = make_float2((vx && gx) ? gx[n] : 0.f, (vy && gy) ? gy[n] : 0.f);
            dAacc[q] = make_float2(0.f, 0.f);
        }
    }
    auto ck_row = [&](int j, int64_t c) {
        return p.ckpt + (((int64_t)b * p.ntiles + tile0 + j) * p.dim + c) * N;
    };

    // ---- TMA ring: load v is tile ntile - 1 - v (x, delta, dout, z, B, C)
    auto issue = [&](int v) {   // lane 0
        unsigned char* st = ws + (v % NST) * Cfg::STAGE;
        const int r = (int)(t0 + (int64_t)(ntile - 1 - v) * T);
        uint64_t* bar = &full[v % NST];
        mbar_arrive_expect_tx(bar, (uint32_t)((ZG ? 4 : 3) * Cfg::TOK + 2 * Cfg::ROW));
        tma_load_3d(st + Cfg::OFF_X, &maps.x, bar, d0, r, b);
        tma_load_3d(st + Cfg::OFF_DL, &maps.delta, bar, d0, r, b);
        tma_load_3d(st + Cfg::OFF_B, &maps.B, bar, 0, r, b);
        tma_load_3d(st + Cfg::OFF_DO, &maps.dout, bar, d0, r, b);
        if (ZG) tma_load_3d(st + Cfg::OFF_Z, &maps.z, bar, d0, r, b);
        tma_load_3d(st + Cfg::OFF_C, &maps.C, bar, 0, r, b);
    };
    int issued = nload < NST ? nload : NST;
    int waited = 0;
    if (lane == 0) {
        prefetch_tmap(&maps.x);
        prefetch_tmap(&maps.delta);
        prefetch_tmap(&maps.dout);
        prefetch_tmap(&maps.B);
        prefetch_tmap(&maps.C);
        for (int v = 0; v < issued; ++v) issue(v);
    }
    __syncwarp();
    auto wait_stage = [&](int v) -> bool {
        const bool landed =
            __all_sync(FULL, mbar_wait_bounded(&full[v % NST], (uint32_t)((v / NST) & 1)));
        if (landed) waited = v + 1;
        return landed;
    };
    auto refill = [&]() {   // after the warp's last read of the stage just consumed
        if (issued < nload) {
            if (lane == 0) issue(issued);
            ++issued;
        }
    };
    // ---- B or C tile [T][N] io -> (v, v) pairs; lane l writes float4 l, l + 32, ...
    auto widen = [&](const IO* src, float4* dst) {
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int f = lane + 32 * r;   // = t * (N / 2) + n / 2
            const float2 v = load2(src + 2 * f);
            dst[f] = make_float4(v.x, v.x, v.y, v.y);
        }
    };
    auto put_dd = [&](int t, float2 dt2, float2 dx2) {
        DD[t * NP + pp] = make_float4(dt2.x, dt2.y, dx2.x, dx2.y);
        DD[(T + t) * NP + pp] = make_float4(dt2.y, dt2.x, dx2.y, dx2.x);
    };
    auto delta_of = [&](float2 u2) {
        return SP ? make_float2(softplus_tiled<IO>(u2.x), softplus_tiled<IO>(u2.y)) : u2;
    };
    // steps past the end of a partial tile get Delta = Delta x = dyc = 0: their
    // recompute keeps the state (dA = 1) and their reverse step keeps G and adds
    // nothing to dA, dB, dC, so every tile runs all T steps with no guards
    auto pre_bwd = [&](const unsigned char* st, int steps) {
        const IO* xs = reinterpret_cast<const IO*>(st + Cfg::OFF_X);
        const IO* ds = reinterpret_cast<const IO*>(st + Cfg::OFF_DL);
        const IO* dos = reinterpret_cast<const IO*>(st + Cfg::OFF_DO);
        const IO* zs = reinterpret_cast<const IO*>(st + Cfg::OFF_Z);
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int t = s + 4 * r, o = t * DC + 2 * pp;
            const float2 x2 = load2(xs + o);
            const float2 r2 = load2(ds + o);
            const float2 u2 = make_float2(r2.x + bias2.x, r2.y + bias2.y);
            const float2 do2 = load2(dos + o);
            const bool live = t < steps;
            const float2 dt2 = live ? delta_of(u2) : make_float2(0.f, 0.f);
            put_dd(t, dt2, make_float2(dt2.x * x2.x, dt2.y * x2.y));
            float2 dyc2 = live ? do2 : make_float2(0.f, 0.f), zf2 = make_float2(0.f, 0.f);
            if (ZG) {
                const float2 z2 = load2(zs + o);
                const float2 sg = sigmoid2(z2);
                if (live) dyc2 = make_float2(do2.x * z2.x * sg.x, do2.y * z2.y * sg.y);
                zf2 = make_float2(do2.x * sg.x * (1.f + z2.x * (1.f - sg.x)),
                                  do2.y * sg.y * (1.f + z2.y * (1.f - sg.y)));
            }
            DY[t * NP + pp] = dyc2;
            DY[(T + t) * NP + pp] = make_float2(dyc2.y, dyc2.x);
            const float2 sgu = SP ? sigmoid2(u2) : make_float2(1.f, 1.f);
            ZS[t * NP + pp] = make_float4(zf2.x, zf2.y, sgu.x, sgu.y);
            XS[t * NP + pp] = x2;
        }
        widen(reinterpret_cast<const IO*>(st + Cfg::OFF_B), BP);
        widen(reinterpret_cast<const IO*>(st + Cfg::OFF_C), CP);
    };

    // ---- one step of the recompute: h = 2^(Delta A log2 e) h + (Delta x) B
    auto fwd_step = [&](int t, float2 (&hh)[4]) {
        const float4 dd = DD[(hi * T + t) * NP + pp];
        const float4 bl = BP[t * (N / 2) + 2 * s + b2], bh = BP[t * (N / 2) + 2 * s + 1 - b2];
        const float2 dt2 = make_float2(dd.x, dd.y), dx2 = make_float2(dd.z, dd.w);
        const float2 Bq[4] = {make_float2(bl.x, bl.y), make_float2(bl.z, bl.w), make_float2(bh.x, bh.y),
                              make_float2(bh.z, bh.w)};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float2 e = __fmul2_rn(dt2, a2[q]);
            hh[q] = __ffma2_rn(make_float2(ex2_sfu(e.x), ex2_sfu(e.y)), hh[q], __fmul2_rn(dx2, Bq[q]));
        }
    };

    // ---- one step of the reverse sweep at step t of the tile: hc = h_t, hp = h_{t-1}.
    // The shared-memory inputs of a step are read by bwd_load ahead of the
    // previous step's stores (the compiler cannot prove that they do not
    // overlap, so a load written after a store waits for it).
    // the tile's dB | dC sums, row t at 32 t.  The address is hidden from the
    // compiler: it then keeps a step's shared loads after the previous step's
    // stores, which holds the register count below the spill point (with the
    // buffers provably disjoint it hoists loads many steps ahead and spills)
    float* redw = reinterpret_cast<float*>(ws + Cfg::OFF_RD);
    asm("" : "+l"(redw));
    struct BwdIn {
        float4 dd, bl, bh, cl, ch;
        float2 dy;
    };
    auto bwd_load = [&](int t) {
        BwdIn in;
        in.dd = DD[(hi * T + t) * NP + pp];
        in.dy = DY[(hi * T + t) * NP + pp];
        in.bl = BP[t * (N / 2) + 2 * s + b2];
        in.bh = BP[t * (N / 2) + 2 * s + 1 - b2];
        in.cl = CP[t * (N / 2) + 2 * s + b2];
        in.ch = CP[t * (N / 2) + 2 * s + 1 - b2];
        return in;
    };
    auto bwd_step = [&](int t, const BwdIn& in, const float2 (&hc)[4], const float2 (&hp)[4]) {
        const float4 dd = in.dd, bl = in.bl, bh = in.bh, cl = in.cl, ch = in.ch;
        const float2 dt2 = make_float2(dd.x, dd.y), dx2 = make_float2(dd.z, dd.w), dy2 = in.dy;
        const float2 Bq[4] = {make_float2(bl.x, bl.y), make_float2(bl.z, bl.w), make_float2(bh.x, bh.y),
                              make_float2(bh.z, bh.w)};
        const float2 Cq[4] = {make_float2(cl.x, cl.y), make_float2(cl.z, cl.w), make_float2(ch.x, ch.y),
                              make_float2(ch.z, ch.w)};
        float2 s1, s2, yp = make_float2(0.f, 0.f);
        float vb[4], vc[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float2 e = __fmul2_rn(dt2, a2[q]);
            const float2 dA = make_float2(ex2_sfu(e.x), ex2_sfu(e.y));
            const float2 g = __ffma2_rn(dy2, Cq[q], G[q]);
            const float2 gd = __fmul2_rn(g, dA);
            G[q] = gd;
            const float2 qv = __fmul2_rn(gd, hp[q]);
            s1 = q ? __ffma2_rn(g, Bq[q], s1) : __fmul2_rn(g, Bq[q]);
            s2 = q ? __ffma2_rn(a2[q], qv, s2) : __fmul2_rn(a2[q], qv);
            dAacc[q] = __ffma2_rn(dt2, qv, dAacc[q]);
            const float2 pb = __fmul2_rn(g, dx2), pc = __fmul2_rn(dy2, hc[q]);
            vb[q] = pb.x + pb.y;   // dB term of state slot q, summed over the pair
            vc[q] = pc.x + pc.y;   // dC term
            if (ZG) yp = q ? __ffma2_rn(Cq[q], hc[q], yp) : __fmul2_rn(Cq[q], hc[q]);
        }
        // dB, dC over the 8 pairs of the warp: lane bits 2, 1, 0 (the adds of a
        // round paired in f32x2: one instruction for two sums)
        const float2 ra = __fadd2_rn(make_float2(vb[0], vb[1]),
                                     make_float2(__shfl_xor_sync(FULL, vb[2], 4), __shfl_xor_sync(FULL, vb[3], 4)));
        const float2 rc_ = __fadd2_rn(make_float2(vc[0], vc[1]),
                                      make_float2(__shfl_xor_sync(FULL, vc[2], 4), __shfl_xor_sync(FULL, vc[3], 4)));
        const float kb = b1 ? ra.y : ra.x, eb = b1 ? ra.x : ra.y;
        const float kc = b1 ? rc_.y : rc_.x, ec = b1 ? rc_.x : rc_.y;
        const float2 rbc = __fadd2_rn(make_float2(kb, kc),
                                      make_float2(__shfl_xor_sync(FULL, eb, 2), __shfl_xor_sync(FULL, ec, 2)));
        const float keep = b0 ? rbc.y : rbc.x, send = b0 ? rbc.x : rbc.y;
        redw[t * 32 + o_lane] = keep + __shfl_xor_sync(FULL, send, 1);
        // g B, A q, C h over the four state quarters: lane bits 4, 3
        const float2 S12 = __fadd2_rn(make_float2(s1.x, s2.x),
                                      make_float2(__shfl_xor_sync(FULL, s1.y, 16), __shfl_xor_sync(FULL, s2.y, 16)));
        const float S1 = S12.x, S2 = S12.y;
        const float YP = ZG ? yp.x + __shfl_xor_sync(FULL, yp.y, 16) : 0.f;
        const float ka = m ? YP : S1, ea = m ? S1 : YP;
        const float kz = m ? 0.f : S2, ez = m ? S2 : 0.f;
        SV[t * 32 + lane] = __fadd2_rn(make_float2(ka, kz),
                                       make_float2(__shfl_xor_sync(FULL, ea, 8), __shfl_xor_sync(FULL, ez, 8)));
    };

    // ---- per-token gradients of a tile from the state sums; one TMA store per tensor
    float2 dD2 = make_float2(0.f, 0.f), dbias2 = make_float2(0.f, 0.f);
    auto post = [&](int64_t ts, int steps) {
        if (lane == 0) bulk_wait_read<0>();   // the previous tile's stores have read OB
        __syncwarp();
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int t = s + 4 * r;
            if (t < steps) {
                const float2 sa0 = SV[t * 32 + pp], ya0 = SV[t * 32 + pp + 8];
                const float2 sa1 = SV[t * 32 + pp + 16], ya1 = SV[t * 32 + pp + 24];
                const float4 dd = DD[t * NP + pp];
                const float2 dyc2 = DY[t * NP + pp];
                const float4 zs = ZS[t * NP + pp];
                const float2 x2 = XS[t * NP + pp];
                const float2 dxo = make_float2(fmaf(dd.x, sa0.x, dyc2.x * D2.x), fmaf(dd.y, sa1.x, dyc2.y * D2.y));
                const float2 du = make_float2(fmaf(x2.x, sa0.x, kLn2 * sa0.y) * zs.z,
                                              fmaf(x2.y, sa1.x, kLn2 * sa1.y) * zs.w);
                store2(OB + t * DC + 2 * pp, dxo.x, dxo.y);
                store2(OB + T * DC + t * DC + 2 * pp, du.x, du.y);
                if (dz_on)
                    store2(OB + 2 * T * DC + t * DC + 2 * pp, zs.x * fmaf(D2.x, x2.x, ya0.x),
                           zs.y * fmaf(D2.y, x2.y, ya1.x));
                dbias2.x += du.x;
                dbias2.y += du.y;
                dD2.x = fmaf(dyc2.x, x2.x, dD2.x);
                dD2.y = fmaf(dyc2.y, x2.y, dD2.y);
            }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            tma_store_3d(&maps.dx, OB, d0, (int)ts, b);
            tma_store_3d(&maps.ddelta, OB + T * DC, d0, (int)ts, b);
            if (dz_on) tma_store_3d(&maps.dz, OB + 2 * T * DC, d0, (int)ts, b);
            bulk_commit();
        }
    };

    bool ok = true;
    // ---- reverse sweep
    for (int jj = 0; ok && jj < ntile; ++jj) {
        const int v = jj, j = ntile - 1 - jj;
        const int64_t ts = t0 + (int64_t)j * T;
        const int steps = (int)((t1 - ts) < T ? (t1 - ts) : T);
        float2 hs[4];   // the state before the tile
#pragma unroll
        for (int hq = 0; hq < 2; ++hq) {
            const int n = nst(2 * hq);
            const float2 ax = vx ? *reinterpret_cast<const float2*>(ck_row(j, cx) + n) : make_float2(0.f, 0.f);
            const float2 ay = vy ? *reinterpret_cast<const float2*>(ck_row(j, cy) + n) : make_float2(0.f, 0.f);
            hs[2 * hq] = make_float2(ax.x, ay.x);
            hs[2 * hq + 1] = make_float2(ax.y, ay.y);
        }
        if (!wait_stage(v)) {
            ok = false;
            break;
        }
        pre_bwd(ws + (v % NST) * Cfg::STAGE, steps);
        __syncwarp();
        refill();
#pragma unroll
        for (int blk = T / H - 1; blk >= 0; --blk) {   // all T steps (see pre_bwd)
            const int base = blk * H;
            float2 hc[4], hp0[4], hist[H][4];
#pragma unroll
            for (int q = 0; q < 4; ++q) hc[q] = hs[q];
#pragma unroll
            for (int t = 0; t < base; ++t) fwd_step(t, hc);   // the steps before the block
#pragma unroll
            for (int q = 0; q < 4; ++q) hp0[q] = hc[q];
#pragma unroll
            for (int i = 0; i < H; ++i) {
                fwd_step(base + i, hc);
#pragma unroll
                for (int q = 0; q < 4; ++q) hist[i][q] = hc[q];
            }
            BwdIn cur = bwd_load(base + H - 1);
#pragma unroll
            for (int i = H - 1; i >= 0; --i) {
                const BwdIn nxt = i > 0 ? bwd_load(base + i - 1) : cur;
                if (i > 0) bwd_step(base + i, cur, hist[i], hist[i - 1]);
                else bwd_step(base, cur, hist[0], hp0);
                cur = nxt;
            }
        }
        __syncwarp();
        {   // the tile's sums to this warp's rows of the partial sums
            float* dst = p.pBC + ((unit * p.batch + b) * p.seqlen + ts) * 32 + lane;
#pragma unroll
            for (int t = 0; t < T; ++t)
                if (t < steps) __stcg(dst + t * 32, redw[t * 32 + lane]);
        }
        post(ts, steps);
        __syncwarp();   // the pre-pass of the next tile rewrites what the post-pass read
    }

    if (lane == 0) {
        bulk_wait<0>();
        if (!ok) {   // let the loads still in flight land before the warp exits
            for (int v = waited; v < issued; ++v)
                mbar_wait_bounded(&full[v % NST], (uint32_t)((v / NST) & 1), 100000000ull);
        }
    }
    if (!ok) return;

    // ---- chunk sums: dA (per state), dD and ddelta_bias (per channel), dinit
    const int64_t bk = (int64_t)b * p.nchunk + k;
#pragma unroll
    for (int hq = 0; hq < 2; ++hq) {
        const int n = nst(2 * hq);
        const float2 a = dAacc[2 * hq], c = dAacc[2 * hq + 1];
        if (vx) *reinterpret_cast<float2*>(p.pA + (bk * p.dim + cx) * N + n) = make_float2(a.x, c.x);
        if (vy) *reinterpret_cast<float2*>(p.pA + (bk * p.dim + cy) * N + n) = make_float2(a.y, c.y);
        if (k == 0 && p.dinit) {
            const float2 g0 = G[2 * hq], g1 = G[2 * hq + 1];
            if (vx) {
                p.dinit[((int64_t)b * p.dim + cx) * N + n] = g0.x;
                p.dinit[((int64_t)b * p.dim + cx) * N + n + 1] = g1.x;
            }
            if (vy) {
                p.dinit[((int64_t)b * p.dim + cy) * N + n] = g0.y;
                p.dinit[((int64_t)b * p.dim + cy) * N + n + 1] = g1.y;
            }
        }
    }
#pragma unroll
    for (int o = 8; o <= 16; o <<= 1) {
        dD2.x += __shfl_xor_sync(FULL, dD2.x, o);
        dD2.y += __shfl_xor_sync(FULL, dD2.y, o);
        dbias2.x += __shfl_xor_sync(FULL, dbias2.x, o);
        dbias2.y += __shfl_xor_sync(FULL, dbias2.y, o);
    }
    if (s == 0) {
        if (v0) {
            p.pD[bk * p.dim + c0] = dD2.x;
            p.pbias[bk * p.dim + c0] = dbias2.x;
        }
        if (v1) {
            p.pD[bk * p.dim + c0 + 1] = dD2.y;
            p.pbias[bk * p.dim + c0 + 1] = dbias2.y;
        }
    }
}

}  // namespace ssm
