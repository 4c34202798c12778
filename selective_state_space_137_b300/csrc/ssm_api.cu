// ssm_api.cu -- the C ABI of libssm_b300.so: argument checks, the choice of
// launch shape, and the launches.  Declarations and the contract of every
// entry point are in include/ssm.h.
#include "ssm.h"

#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include <algorithm>
#include <cstring>
#include <initializer_list>
#include <mutex>

#include <cudaTypedefs.h>
#include <nvtx3/nvToolsExt.h>

#include "common.cuh"
#include "conv.cuh"
#include "decode.cuh"
#include "gemm.cuh"
#include "lti.cuh"
#include "scan_bwd.cuh"
#include "scan_bwd_warp.cuh"
#include "scan_generic.cuh"
#include "tile_io.cuh"
#include "scan_warp.cuh"
#include "scan_ws.cuh"
#include "selftest.cuh"

namespace {

// An NVTX range around each entry point that enqueues GPU work, named after
// it: a profiler that records NVTX shows which library call issued which
// kernels.  With no tool attached a push or pop is one call through a
// pointer that is checked and skipped.
struct TraceRange {
    explicit TraceRange(const char* name) { nvtxRangePushA(name); }
    ~TraceRange() { nvtxRangePop(); }
};
#define SSM_TRACE(name) TraceRange ssm_trace_range_(name)

using ssm::DecodeParams;
using ssm::ScanParams;

constexpr int kVersion = 100;  // 0.1.0

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
// NULL counts as aligned (optional tensors); otherwise the address must be a
// multiple of `bytes`.
bool opt_aligned(const void* p, size_t bytes) {
    return p == nullptr || (reinterpret_cast<uintptr_t>(p) % bytes) == 0;
}
size_t io_size(const ssm_scan_desc* d) { return d->io_dtype == SSM_DTYPE_F32 ? 4 : 2; }

bool dstate_supported(int64_t n) {
    return n == 1 || n == 2 || n == 4 || n == 8 || n == 16 || n == 32 || n == 64;
}

ssm_status check_desc(const ssm_scan_desc* desc) {
    if (!desc) return SSM_ERR_INVALID_ARG;
    if (desc->batch < 0 || desc->seqlen < 0 || desc->dim < 0 || desc->dstate <= 0)
        return SSM_ERR_INVALID_ARG;
    if (desc->io_dtype != SSM_DTYPE_F32 && desc->io_dtype != SSM_DTYPE_BF16)
        return SSM_ERR_UNSUPPORTED;
    if (!dstate_supported(desc->dstate)) return SSM_ERR_UNSUPPORTED;
    // Index arithmetic is 64-bit; keep the per-tensor element counts well inside it.
    const double toks = (double)desc->batch * (double)desc->seqlen * (double)desc->dim;
    if (toks > 9.0e15) return SSM_ERR_UNSUPPORTED;
    return SSM_OK;
}

// Chunking of the time axis for the generic path: split only when there are
// too few (batch, channel) threads to occupy the GPU, and keep chunks long
// enough that the carry pass stays negligible.
int generic_nchunk(const ssm_scan_desc* d) {
    const int64_t chans = d->batch * d->dim;
    if (chans <= 0 || d->seqlen < 1024 || chans >= 32768) return 1;
    int64_t k = (65536 + chans - 1) / chans;
    const int64_t kmax = d->seqlen / 512;
    if (k > kmax) k = kmax;
    if (k > 1024) k = 1024;
    return k < 1 ? 1 : (int)k;
}

size_t workspace_for(const ssm_scan_desc* d, int nchunk) {
    if (nchunk <= 1) return 0;
    const size_t per = (size_t)d->batch * (size_t)nchunk * (size_t)d->dim;
    size_t bytes = per * (size_t)d->dstate * sizeof(float);   // carry
    bytes = (bytes + 255) & ~(size_t)255;
    bytes += per * sizeof(float);                            // dsum
    return bytes;
}

template <typename IO, int N, bool CONV = false, bool ZOH = false>
cudaError_t launch_generic(const ScanParams& p, cudaStream_t s) {
    const dim3 block(128);
    const unsigned gx = (unsigned)((p.dim + 127) / 128);
    if (p.nchunk > 1) {
        dim3 grid(gx, (unsigned)p.batch, (unsigned)(p.nchunk - 1));
        ssm::scan_generic_kernel<IO, N, ssm::MODE_AGG, CONV, ZOH><<<grid, block, 0, s>>>(p);
        const int64_t total = p.batch * p.dim * N;
        ssm::carry_kernel<<<(unsigned)((total + 255) / 256), 256, 0, s>>>(
            p.A, p.initial_state, p.carry, p.dsum, p.batch, p.dim, N, p.nchunk);
    }
    dim3 grid(gx, (unsigned)p.batch, (unsigned)p.nchunk);
    ssm::scan_generic_kernel<IO, N, ssm::MODE_FULL, CONV, ZOH><<<grid, block, 0, s>>>(p);
    return cudaGetLastError();
}

template <typename IO, bool CONV = false, bool ZOH = false>
cudaError_t dispatch_generic(int64_t n, const ScanParams& p, cudaStream_t s) {
    switch (n) {
        case 1: return launch_generic<IO, 1, CONV, ZOH>(p, s);
        case 2: return launch_generic<IO, 2, CONV, ZOH>(p, s);
        case 4: return launch_generic<IO, 4, CONV, ZOH>(p, s);
        case 8: return launch_generic<IO, 8, CONV, ZOH>(p, s);
        case 16: return launch_generic<IO, 16, CONV, ZOH>(p, s);
        case 32: return launch_generic<IO, 32, CONV, ZOH>(p, s);
        case 64: return launch_generic<IO, 64, CONV, ZOH>(p, s);
    }
    return cudaErrorInvalidValue;
}

template <typename IO, int N, bool CONV = false, bool ZOH = false>
cudaError_t launch_decode(const DecodeParams& p, cudaStream_t s) {
    const int64_t lanes = p.dim * ssm::DecodeShape<N>::LPC;   // per sequence
    const dim3 grid((unsigned)((lanes + 255) / 256), (unsigned)p.batch);
    if (CONV && !ZOH && p.vec && p.conv_width == 4)   // the usual width, fixed at compile time
        ssm::state_update_kernel<IO, N, CONV, ZOH, true, CONV && !ZOH ? 4 : 0><<<grid, 256, 0, s>>>(p);
    else if (p.vec)
        ssm::state_update_kernel<IO, N, CONV, ZOH, true><<<grid, 256, 0, s>>>(p);
    else
        ssm::state_update_kernel<IO, N, CONV, ZOH, false><<<grid, 256, 0, s>>>(p);
    return cudaGetLastError();
}

// Vector loads of the A, B and C slices need 16-byte (A) and 4-element (B, C)
// alignment of the bases; element-aligned callers get element loads.
bool decode_vec_ok(const ssm_scan_desc* d, const void* A, const void* B, const void* C) {
    const size_t v = 4 * io_size(d);
    return (reinterpret_cast<uintptr_t>(A) % 16) == 0 && (reinterpret_cast<uintptr_t>(B) % v) == 0 &&
           (reinterpret_cast<uintptr_t>(C) % v) == 0;
}

template <typename IO, bool CONV = false, bool ZOH = false>
cudaError_t dispatch_decode(int64_t n, const DecodeParams& p, cudaStream_t s) {
    switch (n) {
        case 1: return launch_decode<IO, 1, CONV, ZOH>(p, s);
        case 2: return launch_decode<IO, 2, CONV, ZOH>(p, s);
        case 4: return launch_decode<IO, 4, CONV, ZOH>(p, s);
        case 8: return launch_decode<IO, 8, CONV, ZOH>(p, s);
        case 16: return launch_decode<IO, 16, CONV, ZOH>(p, s);
        case 32: return launch_decode<IO, 32, CONV, ZOH>(p, s);
        case 64: return launch_decode<IO, 64, CONV, ZOH>(p, s);
    }
    return cudaErrorInvalidValue;
}

// ---------------------------------------------------------------------------
// Tiled paths: TMA-staged 16-step tiles of 16 channels, taken for bf16/fp32
// I/O with dstate 8, 16, 32 or 64, rows that are 16-byte multiples and
// 16-byte aligned tensors.
//   path 3 (scan_warp.cuh): one-warp CTAs, the first-order scan (and the
//          aggregate pass the backward's recompute uses);
//   path 2 (scan_ws.cuh): warp-specialised CTAs, for the exact zero-order
//          hold and the causal conv fused in front of the scan.

constexpr int kPlanSMs = 148;        // the plan is fixed for a 148-SM B300
constexpr int kChunkRound = 32;      // chunk lengths are multiples of this (and of both tiles)

// Path 2 (warp-specialised: helper warps for loads and per-token work, a scan
// warp for the recurrence).
#ifndef SSM_WS_T
#define SSM_WS_T 16          // time steps per tile
#endif
#ifndef SSM_WS_STAGES
#define SSM_WS_STAGES 4      // TMA ring depth
#endif
#ifndef SSM_WS_SLOTS
#define SSM_WS_SLOTS 2       // helper <-> scan hand-over slots
#endif
template <typename IO, int CK = 0, int N = 16>
using WsConfig = ssm::WsCfg<IO, SSM_WS_T, SSM_WS_STAGES, SSM_WS_SLOTS, CK, N>;
// Conv widths fused into the warp-specialised kernel (compile-time width);
// wider convs take the generic kernel.
constexpr int kWsMaxConvWidth = 4;

// Path 3 (one warp per CTA).  Two ring depths at dstate <= 16: 8 stages when
// the time axis is not cut (7 CTAs of 30 KB per SM), 6 for chunked long
// sequences, whose 25 KB CTAs let 8 chunks per SM run at once (measured on
// the long-sequence workload: 8 stages 4.75 ms, 6 stages 4.39 ms, 4 stages
// with 12 chunks 4.51 ms).
template <typename IO, int N>
using WarpConfig = ssm::WarpCfg<IO, N>;
template <typename IO, int N>
using WarpConfigChunked = ssm::WarpCfg<IO, N, (N <= 16 ? 6 : N == 32 ? 4 : 3)>;

bool tiled_dstate(int64_t n) { return n == 8 || n == 16 || n == 32 || n == 64; }

// Which tiled kernel a plan is for.
enum TiledKind { kKindWarp = 3, kKindWs = 2 };

// dc: channels per CTA; threads; smem: shared bytes per CTA; slots: resident
// CTAs per SM the register budget allows.  `chunked` picks the configuration a
// chunked launch uses.
struct TiledShape { int dc, threads, smem, slots; };

template <typename IO>
TiledShape tiled_shape_io(int64_t n, TiledKind kind, bool chunked) {
    switch (n) {
#define SSM_SHAPE_CASE(NN)                                                                         \
        case NN:                                                                                   \
            if (kind == kKindWarp && chunked)                                                      \
                return TiledShape{16, 32, WarpConfigChunked<IO, NN>::SMEM,                         \
                                  WarpConfigChunked<IO, NN>::MINB};                                \
            if (kind == kKindWarp)                                                                 \
                return TiledShape{16, 32, WarpConfig<IO, NN>::SMEM, WarpConfig<IO, NN>::MINB};     \
            return TiledShape{WsConfig<IO, 0, NN>::DC, WsConfig<IO, 0, NN>::THREADS,               \
                              WsConfig<IO, 0, NN>::SMEM, WsConfig<IO, 0, NN>::MINB};
        SSM_SHAPE_CASE(8) SSM_SHAPE_CASE(16) SSM_SHAPE_CASE(32) SSM_SHAPE_CASE(64)
#undef SSM_SHAPE_CASE
    }
    return {0, 0, 0, 0};
}

TiledShape tiled_shape(const ssm_scan_desc* d, TiledKind kind, bool chunked = false) {
    return d->io_dtype == SSM_DTYPE_F32 ? tiled_shape_io<float>(d->dstate, kind, chunked)
                                        : tiled_shape_io<__nv_bfloat16>(d->dstate, kind, chunked);
}

// Resident CTAs per SM of a tiled configuration (shared memory, threads, registers).
int resident_per_sm(const TiledShape& sh) {
    int per_sm = (228 * 1024) / (sh.smem + 1024);
    if (per_sm > 2048 / sh.threads) per_sm = 2048 / sh.threads;
    if (per_sm > sh.slots) per_sm = sh.slots;
    if (per_sm > 32) per_sm = 32;
    return per_sm;
}

// Shape-only eligibility for the tiled paths (pointer alignment is checked at call time).
bool tiled_shape_ok(const ssm_scan_desc* d) {
    if (!tiled_dstate(d->dstate)) return false;
    const int64_t e = d->io_dtype == SSM_DTYPE_F32 ? 4 : 2;
    if ((d->dim * e) % 16 != 0 || (d->dstate * e) % 16 != 0) return false;
    // TMA coordinates are 32-bit and the batch is a grid dimension
    if (d->seqlen >= (int64_t)1 << 31 || d->dim >= (int64_t)1 << 31 || d->batch > 65535) return false;
    return true;
}

// Chunks of the time axis for a tiled path: cut only when the (batch,
// channel-block) CTAs cannot fill the GPU; chunk lengths are multiples of
// kChunkRound, so every chunk but the last is whole tiles.
void tiled_chunks(const ssm_scan_desc* d, TiledKind kind, int* nchunk, int64_t* chunk_len) {
    const TiledShape sh = tiled_shape(d, kind);
    const int64_t groups = d->batch * ((d->dim + sh.dc - 1) / sh.dc);
    const int64_t target = (int64_t)kPlanSMs * resident_per_sm(sh);
    int64_t k = 1;
    if (groups > 0 && groups * 2 < target) {
        // as many chunks as the chunked configuration keeps resident, rounded
        // down: every CTA of the pass in one wave
        k = (int64_t)kPlanSMs * resident_per_sm(tiled_shape(d, kind, true)) / groups;
        const int64_t kmax = d->seqlen / (4 * kChunkRound);
        if (k > kmax) k = kmax;
        if (k > 4096) k = 4096;
        if (k < 1) k = 1;
    }
    int64_t len = (d->seqlen + k - 1) / k;
    len = (len + kChunkRound - 1) / kChunkRound * kChunkRound;
    if (len < kChunkRound) len = kChunkRound;
    *chunk_len = len;
    *nchunk = d->seqlen > 0 ? (int)((d->seqlen + len - 1) / len) : 1;
}

// Identifier of the calling thread's current CUDA context (0 when there is
// none).  Resources cached per device (copy streams, events, the address of
// the no-allocation scratch array) are keyed on it, so they are made again
// when the context changes (e.g. after cudaDeviceReset and a new primary
// context) instead of being used with the old context's handles.
unsigned long long current_context_id() {
    static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
    static PFN_cuCtxGetId_v12000 get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 4000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(f);
        f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(f);
    });
    CUcontext ctx = nullptr;
    if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
    unsigned long long id = 0;
    return get_id(ctx, &id) == CUDA_SUCCESS ? id : 0;
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

// Tensor map of a (batch, rows, cols) row-major tensor, box [box_rows][box_cols].
bool encode_3d(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int esz, int64_t cols,
               int64_t rows, int64_t batch, int box_cols, int box_rows) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)rows, (cuuint64_t)batch};
    const cuuint64_t strides[2] = {(cuuint64_t)(cols * esz), (cuuint64_t)(cols * rows * esz)};
    const cuuint32_t box[3] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, dt, 3, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The same with a box of box_cols x box_rows x box_batch.
bool encode_3d_box(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int esz, int64_t cols,
                   int64_t rows, int64_t batch, int box_cols, int box_rows, int box_batch) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)rows, (cuuint64_t)batch};
    const cuuint64_t strides[2] = {(cuuint64_t)(cols * esz), (cuuint64_t)(cols * rows * esz)};
    const cuuint32_t box[3] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows, (cuuint32_t)box_batch};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, dt, 3, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// agg_only: the chunk aggregates and carries alone (the chunk start states
// that the backward's recompute needs); out and z are not read.
template <typename IO, int CK, bool ZOH, int N>
cudaError_t launch_ws_n(const ssm_scan_desc* d, ScanParams p, cudaStream_t s, bool agg_only) {
    using Cfg = WsConfig<IO, CK, N>;
    const CUtensorMapDataType dt = sizeof(IO) == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                                   : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const int e = (int)sizeof(IO);
    ssm::TiledMaps maps;
    memset(&maps, 0, sizeof(maps));
    // with the conv, the x box also holds the K-1 raw inputs before the tile
    const int x_rows = Cfg::T + Cfg::HALO;
    bool ok = encode_3d(&maps.x, p.x, dt, e, d->dim, d->seqlen, d->batch, Cfg::DC, x_rows) &&
              encode_3d(&maps.delta, p.delta, dt, e, d->dim, d->seqlen, d->batch, Cfg::DC, Cfg::T) &&
              encode_3d(&maps.B, p.B, dt, e, Cfg::N, d->seqlen, d->batch, Cfg::N, Cfg::T) &&
              encode_3d(&maps.C, p.C, dt, e, Cfg::N, d->seqlen, d->batch, Cfg::N, Cfg::T);
    if (ok && !agg_only)
        ok = encode_3d(&maps.out, p.out, dt, e, d->dim, d->seqlen, d->batch, Cfg::DC, Cfg::T);
    if (ok && p.z && !agg_only)
        ok = encode_3d(&maps.z, p.z, dt, e, d->dim, d->seqlen, d->batch, Cfg::DC, Cfg::T);
    if (!ok) return cudaErrorInvalidValue;
    auto kfull = ssm::scan_ws_kernel<IO, Cfg, ssm::MODE_FULL, ZOH>;
    auto kagg = ssm::scan_ws_kernel<IO, Cfg, ssm::MODE_AGG, ZOH>;
    cudaError_t err = cudaFuncSetAttribute(kfull, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM);
    if (err == cudaSuccess)
        err = cudaFuncSetAttribute(kagg, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM);
    if (err != cudaSuccess) return err;
    const unsigned gx = (unsigned)((d->dim + Cfg::DC - 1) / Cfg::DC);
    if (p.nchunk > 1) {
        kagg<<<dim3(gx, (unsigned)d->batch, (unsigned)(p.nchunk - 1)), Cfg::THREADS, Cfg::SMEM, s>>>(maps, p);
        const int64_t total = p.batch * p.dim * Cfg::N;
        ssm::carry_kernel<<<(unsigned)((total + 255) / 256), 256, 0, s>>>(
            p.A, p.initial_state, p.carry, p.dsum, p.batch, p.dim, Cfg::N, p.nchunk);
    }
    if (agg_only) return cudaGetLastError();
    kfull<<<dim3(gx, (unsigned)d->batch, (unsigned)p.nchunk), Cfg::THREADS, Cfg::SMEM, s>>>(maps, p);
    return cudaGetLastError();
}

// The warp-specialised scan for dstate 8, 16, 32 or 64.
template <typename IO, int CK = 0, bool ZOH = false>
cudaError_t launch_ws(const ssm_scan_desc* d, ScanParams p, cudaStream_t s, bool agg_only = false) {
    switch (d->dstate) {
        case 8: return launch_ws_n<IO, CK, ZOH, 8>(d, p, s, agg_only);
        case 16: return launch_ws_n<IO, CK, ZOH, 16>(d, p, s, agg_only);
        case 32: return launch_ws_n<IO, CK, ZOH, 32>(d, p, s, agg_only);
        case 64: return launch_ws_n<IO, CK, ZOH, 64>(d, p, s, agg_only);
    }
    return cudaErrorInvalidValue;
}

template <typename IO>
cudaError_t launch_ws_conv(const ssm_scan_desc* d, const ScanParams& p, cudaStream_t s) {
    static_assert(kWsMaxConvWidth == 4, "one case per fused width");
    switch (p.conv_width) {
        case 1: return launch_ws<IO, 1>(d, p, s);
        case 2: return launch_ws<IO, 2>(d, p, s);
        case 3: return launch_ws<IO, 3>(d, p, s);
        case 4: return launch_ws<IO, 4>(d, p, s);
    }
    return cudaErrorInvalidValue;
}

// Path 3: the one-warp-CTA scan for dstate 8, 16, 32 or 64 (first-order
// input term).  agg_only: the chunk aggregates and carries alone (the chunk
// start states the backward's recompute needs); out, z and C are not read.
template <typename IO, int N, typename Cfg>
cudaError_t launch_warp_cfg(const ssm_scan_desc* d, ScanParams p, cudaStream_t s, bool agg_only) {
    const CUtensorMapDataType dt = sizeof(IO) == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                                   : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const int e = (int)sizeof(IO);
    ssm::TiledMaps maps;
    memset(&maps, 0, sizeof(maps));
    bool ok = encode_3d(&maps.x, p.x, dt, e, d->dim, d->seqlen, d->batch, Cfg::DC, Cfg::T) &&
              encode_3d(&maps.delta, p.delta, dt, e, d->dim, d->seqlen, d->batch, Cfg::DC, Cfg::T) &&
              encode_3d(&maps.B, p.B, dt, e, N, d->seqlen, d->batch, N, Cfg::T);
    if (ok && !agg_only)
        ok = encode_3d(&maps.C, p.C, dt, e, N, d->seqlen, d->batch, N, Cfg::T) &&
             encode_3d(&maps.out, p.out, dt, e, d->dim, d->seqlen, d->batch, Cfg::DC, Cfg::T);
    if (ok && p.z && !agg_only)
        ok = encode_3d(&maps.z, p.z, dt, e, d->dim, d->seqlen, d->batch, Cfg::DC, Cfg::T);
    if (!ok) return cudaErrorInvalidValue;
    // softplus and the gate are compile-time flags of the kernel
    const bool sp = p.softplus != 0, zg = p.z != nullptr;
    // the training forward (checkpoints) is a kernel of its own: the plain
    // forward is compiled without the checkpoint code
    const bool ck = p.ckpt != nullptr;
    using ssm::scan_warp_kernel;
    using ssm::MODE_FULL;
    auto kfull = ck ? (sp ? (zg ? scan_warp_kernel<IO, Cfg, MODE_FULL, true, true, 0, true>
                                : scan_warp_kernel<IO, Cfg, MODE_FULL, true, false, 0, true>)
                          : (zg ? scan_warp_kernel<IO, Cfg, MODE_FULL, false, true, 0, true>
                                : scan_warp_kernel<IO, Cfg, MODE_FULL, false, false, 0, true>))
                    : (sp ? (zg ? scan_warp_kernel<IO, Cfg, MODE_FULL, true, true>
                                : scan_warp_kernel<IO, Cfg, MODE_FULL, true, false>)
                          : (zg ? scan_warp_kernel<IO, Cfg, MODE_FULL, false, true>
                                : scan_warp_kernel<IO, Cfg, MODE_FULL, false, false>));
    auto kagg = sp ? ssm::scan_warp_kernel<IO, Cfg, ssm::MODE_AGG, true, false>
                   : ssm::scan_warp_kernel<IO, Cfg, ssm::MODE_AGG, false, false>;
    cudaError_t err = cudaFuncSetAttribute(kfull, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM);
    if (err == cudaSuccess)
        err = cudaFuncSetAttribute(kagg, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM);
    if (err != cudaSuccess) return err;
    const unsigned gx = (unsigned)((d->dim + Cfg::DC - 1) / Cfg::DC);
    if (p.nchunk > 1) {
        kagg<<<dim3(gx, (unsigned)d->batch, (unsigned)(p.nchunk - 1)), 32, Cfg::SMEM, s>>>(maps, p);
        const int64_t total = p.batch * p.dim * N;
        ssm::carry_kernel<<<(unsigned)((total + 255) / 256), 256, 0, s>>>(
            p.A, p.initial_state, p.carry, p.dsum, p.batch, p.dim, N, p.nchunk);
    }
    if (agg_only) return cudaGetLastError();
    kfull<<<dim3(gx, (unsigned)d->batch, (unsigned)p.nchunk), 32, Cfg::SMEM, s>>>(maps, p);
    return cudaGetLastError();
}

template <typename IO, int N>
cudaError_t launch_warp_n(const ssm_scan_desc* d, const ScanParams& p, cudaStream_t s, bool agg_only) {
    return p.nchunk > 1 ? launch_warp_cfg<IO, N, WarpConfigChunked<IO, N>>(d, p, s, agg_only)
                        : launch_warp_cfg<IO, N, WarpConfig<IO, N>>(d, p, s, agg_only);
}

// The one-warp scan in MODE_STATES (dstate 16): the state before every tile of
// every chunk into p.ckpt, each chunk from p.carry (nchunk > 1, filled by an
// aggregate pass and the carry) or the initial state.
template <typename IO, typename Cfg>
cudaError_t launch_warp_states_cfg(const ssm_scan_desc* d, const ScanParams& p, cudaStream_t s) {
    const CUtensorMapDataType dt = sizeof(IO) == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                                   : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const int e = (int)sizeof(IO);
    ssm::TiledMaps maps;
    memset(&maps, 0, sizeof(maps));
    const bool ok = encode_3d(&maps.x, p.x, dt, e, d->dim, d->seqlen, d->batch, Cfg::DC, Cfg::T) &&
                    encode_3d(&maps.delta, p.delta, dt, e, d->dim, d->seqlen, d->batch, Cfg::DC, Cfg::T) &&
                    encode_3d(&maps.B, p.B, dt, e, 16, d->seqlen, d->batch, 16, Cfg::T);
    if (!ok || !p.ckpt) return cudaErrorInvalidValue;
    auto kern = p.softplus ? ssm::scan_warp_kernel<IO, Cfg, ssm::MODE_STATES, true, false, 0, true>
                           : ssm::scan_warp_kernel<IO, Cfg, ssm::MODE_STATES, false, false, 0, true>;
    const cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM);
    if (err != cudaSuccess) return err;
    const unsigned gx = (unsigned)((d->dim + Cfg::DC - 1) / Cfg::DC);
    kern<<<dim3(gx, (unsigned)d->batch, (unsigned)p.nchunk), 32, Cfg::SMEM, s>>>(maps, p);
    return cudaGetLastError();
}
template <typename IO>
cudaError_t launch_warp_states(const ssm_scan_desc* d, const ScanParams& p, cudaStream_t s) {
    return p.nchunk > 1 ? launch_warp_states_cfg<IO, WarpConfigChunked<IO, 16>>(d, p, s)
                        : launch_warp_states_cfg<IO, WarpConfig<IO, 16>>(d, p, s);
}

// The one-warp scan with dt_proj fused in front (bf16 I/O, dstate 16, softplus):
// the chunked configuration's 6-stage ring plus the two fp32 raw-step tiles.
template <int R>
cudaError_t launch_warp_proj(const ssm_scan_desc* d, ScanParams p, cudaStream_t s) {
    using IO = __nv_bfloat16;
    using Cfg = WarpConfigChunked<IO, 16>;
    constexpr int SMEM = Cfg::SMEM + 2 * Cfg::T * Cfg::DC * 4;
    const CUtensorMapDataType dt = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    ssm::TiledMaps maps;
    memset(&maps, 0, sizeof(maps));
    bool ok = encode_3d(&maps.x, p.x, dt, 2, d->dim, d->seqlen, d->batch, Cfg::DC, Cfg::T) &&
              encode_3d(&maps.B, p.B, dt, 2, 16, d->seqlen, d->batch, 16, Cfg::T) &&
              encode_3d(&maps.C, p.C, dt, 2, 16, d->seqlen, d->batch, 16, Cfg::T) &&
              encode_3d(&maps.out, p.out, dt, 2, d->dim, d->seqlen, d->batch, Cfg::DC, Cfg::T);
    if (ok && p.z) ok = encode_3d(&maps.z, p.z, dt, 2, d->dim, d->seqlen, d->batch, Cfg::DC, Cfg::T);
    if (!ok) return cudaErrorInvalidValue;
    auto kfull = p.z ? ssm::scan_warp_kernel<IO, Cfg, ssm::MODE_FULL, true, true, R>
                     : ssm::scan_warp_kernel<IO, Cfg, ssm::MODE_FULL, true, false, R>;
    auto kagg = ssm::scan_warp_kernel<IO, Cfg, ssm::MODE_AGG, true, false, R>;
    cudaError_t err = cudaFuncSetAttribute(kfull, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
    if (err == cudaSuccess) err = cudaFuncSetAttribute(kagg, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
    if (err != cudaSuccess) return err;
    const unsigned gx = (unsigned)((d->dim + Cfg::DC - 1) / Cfg::DC);
    if (p.nchunk > 1) {
        kagg<<<dim3(gx, (unsigned)d->batch, (unsigned)(p.nchunk - 1)), 32, SMEM, s>>>(maps, p);
        const int64_t total = p.batch * p.dim * 16;
        ssm::carry_kernel<<<(unsigned)((total + 255) / 256), 256, 0, s>>>(
            p.A, p.initial_state, p.carry, p.dsum, p.batch, p.dim, 16, p.nchunk);
    }
    kfull<<<dim3(gx, (unsigned)d->batch, (unsigned)p.nchunk), 32, SMEM, s>>>(maps, p);
    return cudaGetLastError();
}

template <typename IO>
cudaError_t launch_warp(const ssm_scan_desc* d, const ScanParams& p, cudaStream_t s,
                        bool agg_only = false) {
    switch (d->dstate) {
        case 8: return launch_warp_n<IO, 8>(d, p, s, agg_only);
        case 16: return launch_warp_n<IO, 16>(d, p, s, agg_only);
        case 32: return launch_warp_n<IO, 32>(d, p, s, agg_only);
        case 64: return launch_warp_n<IO, 64>(d, p, s, agg_only);
    }
    return cudaErrorInvalidValue;
}

}  // namespace

extern "C" {

int ssm_version(void) { return kVersion; }

const char* ssm_status_string(ssm_status status) {
    switch (status) {
        case SSM_OK: return "SSM_OK";
        case SSM_ERR_INVALID_ARG: return "SSM_ERR_INVALID_ARG: invalid argument";
        case SSM_ERR_UNSUPPORTED: return "SSM_ERR_UNSUPPORTED: unsupported configuration";
        case SSM_ERR_CUDA: return "SSM_ERR_CUDA: CUDA launch failed";
        case SSM_ERR_TIMEOUT: return "SSM_ERR_TIMEOUT: a device-side wait timed out";
    }
    return "unknown ssm_status";
}

ssm_status ssm_scan_plan(const ssm_scan_desc* desc, ssm_scan_plan_info* info) {
    const ssm_status st = check_desc(desc);
    if (st != SSM_OK) return st;
    if (!info) return SSM_ERR_INVALID_ARG;
    int nchunk;
    int64_t chunk_len;
    const bool tiled = tiled_shape_ok(desc);
    if (tiled) {
        tiled_chunks(desc, kKindWarp, &nchunk, &chunk_len);
    } else {
        nchunk = generic_nchunk(desc);
    }
    info->path = tiled ? kKindWarp : 0;
    info->nchunk = nchunk;
    info->launches = (desc->batch == 0 || desc->dim == 0 || desc->seqlen == 0) ? 0
                     : (nchunk > 1 ? 3 : 1);
    info->reserved = 0;
    info->workspace = (int64_t)workspace_for(desc, nchunk);
    return SSM_OK;
}

size_t ssm_scan_workspace_size(const ssm_scan_desc* desc) {
    if (check_desc(desc) != SSM_OK) return 0;
    // Enough for any path: the tiled ones are taken only with 16-byte
    // aligned tensors, which is known at call time, and the exact-ZOH scan
    // and the fused conv take the warp-specialised kernel's plan.
    size_t need = workspace_for(desc, generic_nchunk(desc));
    if (tiled_shape_ok(desc)) {
        for (TiledKind kind : {kKindWarp, kKindWs}) {
            int nchunk;
            int64_t chunk_len;
            tiled_chunks(desc, kind, &nchunk, &chunk_len);
            const size_t t = workspace_for(desc, nchunk);
            if (t > need) need = t;
        }
    }
    return need;
}

}  // extern "C"

namespace {

// The scan behind ssm_scan_fwd (zoh = false) and ssm_scan_fwd_ex.
ssm_status scan_fwd_impl(const ssm_scan_desc* desc, bool zoh, const void* x, const void* delta,
                         const float* A, const void* B, const void* C, const float* D,
                         const void* z, const float* delta_bias, void* out, float* last_state,
                         const float* initial_state, void* workspace, size_t workspace_bytes,
                         void* stream, float* ckpt = nullptr) {
    const ssm_status st = check_desc(desc);
    if (st != SSM_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int64_t N = desc->dstate;
    const size_t state_bytes = (size_t)desc->batch * (size_t)desc->dim * (size_t)N * sizeof(float);

    const size_t esz = io_size(desc);
    if (!opt_aligned(x, esz) || !opt_aligned(delta, esz) || !opt_aligned(B, esz) ||
        !opt_aligned(C, esz) || !opt_aligned(z, esz) || !opt_aligned(out, esz) || !opt_aligned(A, 4) ||
        !opt_aligned(D, 4) || !opt_aligned(delta_bias, 4) || !opt_aligned(last_state, 4) ||
        !opt_aligned(initial_state, 4))
        return SSM_ERR_INVALID_ARG;

    if (desc->batch == 0 || desc->dim == 0) return SSM_OK;
    if (desc->seqlen == 0) {
        // No tokens: the final state is the initial state.
        if (last_state && last_state != initial_state) {
            cudaError_t e = initial_state
                ? cudaMemcpyAsync(last_state, initial_state, state_bytes, cudaMemcpyDeviceToDevice, s)
                : cudaMemsetAsync(last_state, 0, state_bytes, s);
            if (e != cudaSuccess) return SSM_ERR_CUDA;
        }
        return SSM_OK;
    }
    if (!x || !delta || !A || !B || !C || !out) return SSM_ERR_INVALID_ARG;

    bool tiled = tiled_shape_ok(desc) && aligned16(x) && aligned16(delta) &&
                 aligned16(B) && aligned16(C) && aligned16(out) && opt_aligned(z, 16) &&
                 opt_aligned(last_state, 16);
    // checkpoints every 16 tokens: the one-warp kernel (16-step tiles) or the
    // general one; the exact-ZOH scan takes the warp-specialised kernel
    if (ckpt && (zoh || WarpConfig<float, 16>::T != ssm::kCkptSteps)) tiled = false;
    const TiledKind kind = zoh ? kKindWs : kKindWarp;
    int nchunk;
    int64_t chunk_len;
    if (tiled) {
        tiled_chunks(desc, kind, &nchunk, &chunk_len);
    } else {
        nchunk = generic_nchunk(desc);
        chunk_len = (desc->seqlen + nchunk - 1) / nchunk;
        if (ckpt && nchunk > 1)   // chunk starts on a checkpoint
            chunk_len = (chunk_len + ssm::kCkptSteps - 1) / ssm::kCkptSteps * ssm::kCkptSteps;
        if (ckpt) nchunk = (int)((desc->seqlen + chunk_len - 1) / chunk_len);
    }
    const size_t need = workspace_for(desc, nchunk);
    if (need > 0 && (workspace == nullptr || workspace_bytes < need || !aligned16(workspace)))
        return SSM_ERR_INVALID_ARG;

    ScanParams p;
    p.ckpt = ckpt;
    p.ckpt_tiles = (desc->seqlen + ssm::kCkptSteps - 1) / ssm::kCkptSteps;
    p.x = x; p.delta = delta; p.A = A; p.B = B; p.C = C; p.D = D; p.z = z;
    p.delta_bias = delta_bias; p.out = out; p.last_state = last_state;
    p.initial_state = initial_state;
    p.batch = desc->batch; p.seqlen = desc->seqlen; p.dim = desc->dim;
    p.nchunk = nchunk;
    p.chunk_len = chunk_len;
    p.softplus = desc->delta_softplus ? 1 : 0;
    p.carry = nullptr; p.dsum = nullptr;
    if (nchunk > 1) {
        char* w = static_cast<char*>(workspace);
        const size_t per = (size_t)desc->batch * (size_t)nchunk * (size_t)desc->dim;
        p.carry = reinterpret_cast<float*>(w);
        p.dsum = reinterpret_cast<float*>(w + ((per * (size_t)N * sizeof(float) + 255) & ~(size_t)255));
    }
    // The chunk grid dimension is limited to 65535 and the batch to 65535.
    if (desc->batch > 65535) return SSM_ERR_UNSUPPORTED;

    cudaError_t e;
    const bool f32 = desc->io_dtype == SSM_DTYPE_F32;
    if (zoh) {
        // exact zero-order hold: the warp-specialised kernel for dstate 8 to 64,
        // the generic kernel (with the same chunk plan's workspace) otherwise
        if (tiled)
            e = f32 ? launch_ws<float, 0, true>(desc, p, s) : launch_ws<__nv_bfloat16, 0, true>(desc, p, s);
        else
            e = f32 ? dispatch_generic<float, false, true>(N, p, s)
                    : dispatch_generic<__nv_bfloat16, false, true>(N, p, s);
    } else if (tiled) {
        e = f32 ? launch_warp<float>(desc, p, s) : launch_warp<__nv_bfloat16>(desc, p, s);
    } else {
        e = f32 ? dispatch_generic<float>(N, p, s) : dispatch_generic<__nv_bfloat16>(N, p, s);
    }
    return e == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}

ssm_status check_opts(const ssm_scan_opts* o) {
    if (!o) return SSM_ERR_INVALID_ARG;
    if (o->discretization != SSM_DISC_EULER && o->discretization != SSM_DISC_ZOH)
        return SSM_ERR_INVALID_ARG;
    for (int i = 0; i < 3; ++i)
        if (o->reserved[i] != 0) return SSM_ERR_INVALID_ARG;
    return SSM_OK;
}

}  // namespace

extern "C" {

ssm_status ssm_scan_fwd(const ssm_scan_desc* desc, const void* x, const void* delta,
                        const float* A, const void* B, const void* C, const float* D,
                        const void* z, const float* delta_bias, void* out, float* last_state,
                        const float* initial_state, void* workspace, size_t workspace_bytes,
                        void* stream) {
    SSM_TRACE("ssm_scan_fwd");
    return scan_fwd_impl(desc, false, x, delta, A, B, C, D, z, delta_bias, out, last_state,
                         initial_state, workspace, workspace_bytes, stream);
}

size_t ssm_scan_checkpoint_size(const ssm_scan_desc* desc) {
    if (check_desc(desc) != SSM_OK) return 0;
    return (size_t)desc->batch * (size_t)((desc->seqlen + ssm::kCkptSteps - 1) / ssm::kCkptSteps) *
           (size_t)desc->dim * (size_t)desc->dstate * sizeof(float);
}

ssm_status ssm_scan_fwd_train(const ssm_scan_desc* desc, const void* x, const void* delta,
                              const float* A, const void* B, const void* C, const float* D,
                              const void* z, const float* delta_bias, void* out, float* last_state,
                              const float* initial_state, float* checkpoints, void* workspace,
                              size_t workspace_bytes, void* stream) {
    SSM_TRACE("ssm_scan_fwd_train");
    if (!checkpoints || !aligned16(checkpoints)) return SSM_ERR_INVALID_ARG;
    return scan_fwd_impl(desc, false, x, delta, A, B, C, D, z, delta_bias, out, last_state,
                         initial_state, workspace, workspace_bytes, stream, checkpoints);
}

ssm_status ssm_scan_fwd_ex(const ssm_scan_desc* desc, const ssm_scan_opts* opts, const void* x,
                           const void* delta, const float* A, const void* B, const void* C,
                           const float* D, const void* z, const float* delta_bias, void* out,
                           float* last_state, const float* initial_state, void* workspace,
                           size_t workspace_bytes, void* stream) {
    SSM_TRACE("ssm_scan_fwd_ex");
    const ssm_status so = check_opts(opts);
    if (so != SSM_OK) return so;
    return scan_fwd_impl(desc, opts->discretization == SSM_DISC_ZOH, x, delta, A, B, C, D, z,
                         delta_bias, out, last_state, initial_state, workspace, workspace_bytes,
                         stream);
}

ssm_status ssm_proj_scan_fwd(const ssm_scan_desc* desc, const ssm_proj_desc* proj, const void* x,
                             const void* dt_low, const void* W_dt, const float* A, const void* B,
                             const void* C, const float* D, const void* z,
                             const float* delta_bias, void* out, float* last_state,
                             const float* initial_state, void* workspace, size_t workspace_bytes,
                             void* stream) {
    SSM_TRACE("ssm_proj_scan_fwd");
    const ssm_status st = check_desc(desc);
    if (st != SSM_OK) return st;
    if (!proj || proj->dt_rank <= 0 || proj->reserved != 0) return SSM_ERR_INVALID_ARG;
    if (desc->io_dtype != SSM_DTYPE_BF16 || desc->dstate != 16 || !desc->delta_softplus ||
        (proj->dt_rank != 64 && proj->dt_rank != 128) || !tiled_shape_ok(desc))
        return SSM_ERR_UNSUPPORTED;
    for (const void* q : std::initializer_list<const void*>{x, dt_low, W_dt, B, C, z, out, last_state})
        if (!opt_aligned(q, 16)) return SSM_ERR_INVALID_ARG;
    if (!opt_aligned(A, 4) || !opt_aligned(D, 4) || !opt_aligned(delta_bias, 4) ||
        !opt_aligned(initial_state, 4))
        return SSM_ERR_INVALID_ARG;
    if (desc->batch == 0 || desc->dim == 0) return SSM_OK;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (desc->seqlen == 0) {
        const size_t state_bytes = (size_t)desc->batch * (size_t)desc->dim * 16 * sizeof(float);
        if (last_state && last_state != initial_state) {
            cudaError_t e = initial_state
                ? cudaMemcpyAsync(last_state, initial_state, state_bytes, cudaMemcpyDeviceToDevice, s)
                : cudaMemsetAsync(last_state, 0, state_bytes, s);
            if (e != cudaSuccess) return SSM_ERR_CUDA;
        }
        return SSM_OK;
    }
    if (!x || !dt_low || !W_dt || !A || !B || !C || !out) return SSM_ERR_INVALID_ARG;
    int nchunk;
    int64_t chunk_len;
    tiled_chunks(desc, kKindWarp, &nchunk, &chunk_len);
    const size_t need = workspace_for(desc, nchunk);
    if (need > 0 && (workspace == nullptr || workspace_bytes < need || !aligned16(workspace)))
        return SSM_ERR_INVALID_ARG;
    ScanParams p;
    p.x = x; p.delta = nullptr; p.A = A; p.B = B; p.C = C; p.D = D; p.z = z;
    p.delta_bias = delta_bias; p.out = out; p.last_state = last_state;
    p.initial_state = initial_state;
    p.batch = desc->batch; p.seqlen = desc->seqlen; p.dim = desc->dim;
    p.nchunk = nchunk;
    p.chunk_len = chunk_len;
    p.softplus = 1;
    p.carry = nullptr; p.dsum = nullptr;
    if (nchunk > 1) {
        char* w = static_cast<char*>(workspace);
        const size_t per = (size_t)desc->batch * (size_t)nchunk * (size_t)desc->dim;
        p.carry = reinterpret_cast<float*>(w);
        p.dsum = reinterpret_cast<float*>(w + ((per * 16 * sizeof(float) + 255) & ~(size_t)255));
    }
    p.dt_low = dt_low;
    p.W_dt = W_dt;
    const cudaError_t e = proj->dt_rank == 128 ? launch_warp_proj<128>(desc, p, s)
                                               : launch_warp_proj<64>(desc, p, s);
    return e == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}

ssm_status ssm_selftest_wait_timeout(int64_t limit_ns, void* stream) {
    if (limit_ns < 1000 || limit_ns > 5000000000LL) return SSM_ERR_INVALID_ARG;
    ssm::wait_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>((uint64_t)limit_ns);
    return cudaGetLastError() == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}

ssm_status ssm_get_device_status(void) {
    unsigned word = 0;
    if (cudaMemcpyFromSymbol(&word, ssm::g_ssm_device_error, sizeof(word)) != cudaSuccess)
        return SSM_ERR_CUDA;
    if (word == 0) return SSM_OK;
    const unsigned zero = 0;
    if (cudaMemcpyToSymbol(ssm::g_ssm_device_error, &zero, sizeof(zero)) != cudaSuccess)
        return SSM_ERR_CUDA;
    return SSM_ERR_TIMEOUT;
}

ssm_status ssm_get_async_status(void* workspace, void* stream) {
    (void)workspace;   // the error word is the device's, not the call's
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned word = 0;
    // read after the stream's earlier work, wait for this stream only
    if (cudaMemcpyFromSymbolAsync(&word, ssm::g_ssm_device_error, sizeof(word), 0,
                                  cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return SSM_ERR_CUDA;
    if (word == 0) return SSM_OK;
    const unsigned zero = 0;
    if (cudaMemcpyToSymbolAsync(ssm::g_ssm_device_error, &zero, sizeof(zero), 0,
                                cudaMemcpyHostToDevice, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return SSM_ERR_CUDA;
    return SSM_ERR_TIMEOUT;
}

}  // extern "C"

namespace {

ssm_status state_update_impl(const ssm_scan_desc* desc, bool zoh, float* state, const void* x,
                             const void* delta, const float* A, const void* B, const void* C,
                             const float* D, const void* z, const float* delta_bias, void* out,
                             void* stream) {
    const ssm_status st = check_desc(desc);
    if (st != SSM_OK) return st;
    const size_t esz = io_size(desc);
    // The state is accessed 16 bytes at a time when each lane owns 4+ states.
    if (!opt_aligned(state, desc->dstate >= 4 ? 16 : 4) || !opt_aligned(x, esz) ||
        !opt_aligned(delta, esz) || !opt_aligned(B, esz) || !opt_aligned(C, esz) ||
        !opt_aligned(z, esz) || !opt_aligned(out, esz) || !opt_aligned(A, 4) || !opt_aligned(D, 4) ||
        !opt_aligned(delta_bias, 4))
        return SSM_ERR_INVALID_ARG;
    if (desc->batch == 0 || desc->dim == 0) return SSM_OK;
    if (!state || !x || !delta || !A || !B || !C || !out) return SSM_ERR_INVALID_ARG;
    // grid: y = sequence (<= 65535), x = channel lanes (32-bit lane index)
    if (desc->batch > 65535 || desc->dim * 64 >= ((int64_t)1 << 31)) return SSM_ERR_UNSUPPORTED;

    DecodeParams p;
    p.state = state; p.x = x; p.delta = delta; p.A = A; p.B = B; p.C = C; p.D = D; p.z = z;
    p.delta_bias = delta_bias; p.out = out;
    p.batch = desc->batch; p.dim = desc->dim;
    p.softplus = desc->delta_softplus ? 1 : 0;
    p.vec = decode_vec_ok(desc, A, B, C);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const bool f32 = desc->io_dtype == SSM_DTYPE_F32;
    cudaError_t e;
    if (zoh)
        e = f32 ? dispatch_decode<float, false, true>(desc->dstate, p, s)
                : dispatch_decode<__nv_bfloat16, false, true>(desc->dstate, p, s);
    else
        e = f32 ? dispatch_decode<float>(desc->dstate, p, s)
                : dispatch_decode<__nv_bfloat16>(desc->dstate, p, s);
    return e == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}

}  // namespace

extern "C" {

ssm_status ssm_state_update(const ssm_scan_desc* desc, float* state, const void* x,
                            const void* delta, const float* A, const void* B, const void* C,
                            const float* D, const void* z, const float* delta_bias, void* out,
                            void* stream) {
    SSM_TRACE("ssm_state_update");
    return state_update_impl(desc, false, state, x, delta, A, B, C, D, z, delta_bias, out, stream);
}

ssm_status ssm_state_update_ex(const ssm_scan_desc* desc, const ssm_scan_opts* opts, float* state,
                               const void* x, const void* delta, const float* A, const void* B,
                               const void* C, const float* D, const void* z,
                               const float* delta_bias, void* out, void* stream) {
    SSM_TRACE("ssm_state_update_ex");
    const ssm_status so = check_opts(opts);
    if (so != SSM_OK) return so;
    return state_update_impl(desc, opts->discretization == SSM_DISC_ZOH, state, x, delta, A, B, C,
                             D, z, delta_bias, out, stream);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// The causal depthwise conv in front of the scan: standalone, fused into the
// scan, and fused into the decode step.
namespace {

ssm_status check_conv(const ssm_conv_desc* c) {
    if (!c) return SSM_ERR_INVALID_ARG;
    if (c->width < 1 || c->width > ssm::kMaxConvWidth) return SSM_ERR_UNSUPPORTED;
    if (c->activation != 0 && c->activation != 1) return SSM_ERR_INVALID_ARG;
    return SSM_OK;
}

// True when the byte ranges [a, a + n) and [b, b + n) intersect.
bool overlaps(const void* a, const void* b, size_t n) {
    if (!a || !b || n == 0) return false;
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + n && y < x + n;
}

#ifndef SSM_CONV_VEC16
#define SSM_CONV_VEC16 4     // bf16 channels per thread of the standalone conv (8-byte rows)
#endif
#ifndef SSM_CONV_MINCHUNK
#define SSM_CONV_MINCHUNK 64 // shortest time chunk per thread
#endif

// Time steps per thread of the standalone conv: enough threads to cover the
// GPU a few times over, and chunks long enough that the K-1 rows re-read at
// each chunk start stay a small fraction.
int64_t conv_chunk(int64_t seqlen, int64_t threads_per_step) {
    const int64_t target = (int64_t)kPlanSMs * 2048 * 2;
    int64_t nch = threads_per_step > 0 ? (target + threads_per_step - 1) / threads_per_step : 1;
    const int64_t most = seqlen / SSM_CONV_MINCHUNK > 1 ? seqlen / SSM_CONV_MINCHUNK : 1;
    if (nch > most) nch = most;
    if (nch > 65535) nch = 65535;
    if (nch < 1) nch = 1;
    return (seqlen + nch - 1) / nch;
}

template <typename IO, int VEC>
cudaError_t launch_conv(const ssm::ConvParams& p, cudaStream_t s) {
    const int64_t vecs = p.dim / VEC;
    const dim3 grid((unsigned)((vecs + 127) / 128), (unsigned)((p.seqlen + p.chunk - 1) / p.chunk),
                    (unsigned)p.batch);
    switch (p.width) {
        case 1: ssm::conv1d_kernel<IO, VEC, 1><<<grid, 128, 0, s>>>(p); break;
        case 2: ssm::conv1d_kernel<IO, VEC, 2><<<grid, 128, 0, s>>>(p); break;
        case 3: ssm::conv1d_kernel<IO, VEC, 3><<<grid, 128, 0, s>>>(p); break;
        case 4: ssm::conv1d_kernel<IO, VEC, 4><<<grid, 128, 0, s>>>(p); break;
        case 5: ssm::conv1d_kernel<IO, VEC, 5><<<grid, 128, 0, s>>>(p); break;
        case 6: ssm::conv1d_kernel<IO, VEC, 6><<<grid, 128, 0, s>>>(p); break;
        case 7: ssm::conv1d_kernel<IO, VEC, 7><<<grid, 128, 0, s>>>(p); break;
        case 8: ssm::conv1d_kernel<IO, VEC, 8><<<grid, 128, 0, s>>>(p); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

// The TMA-streamed form (16-byte rows and 16-byte aligned x, out).
template <typename IO, int K>
cudaError_t launch_conv_tma_k(const ssm::ConvMaps& maps, const ssm::ConvParams& p, cudaStream_t s) {
    using Cfg = ssm::ConvTmaCfg<IO, K>;
    auto k = ssm::conv1d_tma_kernel<IO, K>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM);
    if (e != cudaSuccess) return e;
    const dim3 grid((unsigned)((p.dim + ssm::kConvCC - 1) / ssm::kConvCC),
                    (unsigned)((p.seqlen + p.chunk - 1) / p.chunk), (unsigned)p.batch);
    k<<<grid, ssm::kConvCC, Cfg::SMEM, s>>>(maps, p);
    return cudaGetLastError();
}

template <typename IO>
cudaError_t launch_conv_tma(ssm::ConvParams p, cudaStream_t s) {
    const CUtensorMapDataType dt = sizeof(IO) == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                                   : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const int e = (int)sizeof(IO);
    // time chunks: multiples of the tile, about four waves of CTAs
    const int64_t blocks = ((p.dim + ssm::kConvCC - 1) / ssm::kConvCC) * p.batch;
    int64_t nch = blocks > 0 ? ((int64_t)kPlanSMs * 4 * 4 + blocks - 1) / blocks : 1;
    const int64_t most = p.seqlen / 128 > 1 ? p.seqlen / 128 : 1;
    if (nch > most) nch = most;
    if (nch > 65535) nch = 65535;
    if (nch < 1) nch = 1;
    int64_t chunk = (p.seqlen + nch - 1) / nch;
    chunk = (chunk + ssm::kConvTT - 1) / ssm::kConvTT * ssm::kConvTT;
    p.chunk = chunk;
    ssm::ConvMaps maps;
    memset(&maps, 0, sizeof(maps));
    const int H = p.width - 1;
    if (!encode_3d(&maps.x, p.x, dt, e, p.dim, p.seqlen, p.batch, ssm::kConvCC, ssm::kConvTT + H) ||
        !encode_3d(&maps.out, p.out, dt, e, p.dim, p.seqlen, p.batch, ssm::kConvCC, ssm::kConvTT))
        return cudaErrorInvalidValue;
    switch (p.width) {
        case 1: return launch_conv_tma_k<IO, 1>(maps, p, s);
        case 2: return launch_conv_tma_k<IO, 2>(maps, p, s);
        case 3: return launch_conv_tma_k<IO, 3>(maps, p, s);
        case 4: return launch_conv_tma_k<IO, 4>(maps, p, s);
        case 5: return launch_conv_tma_k<IO, 5>(maps, p, s);
        case 6: return launch_conv_tma_k<IO, 6>(maps, p, s);
        case 7: return launch_conv_tma_k<IO, 7>(maps, p, s);
        case 8: return launch_conv_tma_k<IO, 8>(maps, p, s);
    }
    return cudaErrorInvalidValue;
}

// Copy (or zero) the conv state when there are no tokens to push through it.
cudaError_t conv_state_passthrough(float* out, const float* in, size_t bytes, cudaStream_t s) {
    if (!out || out == in || bytes == 0) return cudaSuccess;
    return in ? cudaMemcpyAsync(out, in, bytes, cudaMemcpyDeviceToDevice, s)
              : cudaMemsetAsync(out, 0, bytes, s);
}

}  // namespace

extern "C" {

ssm_status ssm_conv1d_fwd(const ssm_scan_desc* desc, const ssm_conv_desc* conv, const void* x,
                          const float* w, const float* bias, const float* conv_state_in,
                          void* out, float* conv_state_out, void* stream) {
    SSM_TRACE("ssm_conv1d_fwd");
    if (!desc) return SSM_ERR_INVALID_ARG;
    if (desc->batch < 0 || desc->seqlen < 0 || desc->dim < 0) return SSM_ERR_INVALID_ARG;
    if (desc->io_dtype != SSM_DTYPE_F32 && desc->io_dtype != SSM_DTYPE_BF16)
        return SSM_ERR_UNSUPPORTED;
    ssm_status st = check_conv(conv);
    if (st != SSM_OK) return st;
    const size_t esz = io_size(desc);
    if (!opt_aligned(x, esz) || !opt_aligned(out, esz) || !opt_aligned(w, 4) ||
        !opt_aligned(bias, 4) || !opt_aligned(conv_state_in, 4) || !opt_aligned(conv_state_out, 4))
        return SSM_ERR_INVALID_ARG;
    const int H = conv->width - 1;
    const size_t state_bytes = (size_t)desc->batch * (size_t)desc->dim * (size_t)H * sizeof(float);
    if (overlaps(conv_state_in, conv_state_out, state_bytes)) return SSM_ERR_INVALID_ARG;
    if (desc->batch == 0 || desc->dim == 0) return SSM_OK;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (desc->seqlen == 0)
        return conv_state_passthrough(conv_state_out, conv_state_in, state_bytes, s) == cudaSuccess
                   ? SSM_OK : SSM_ERR_CUDA;
    if (!x || !w || !out) return SSM_ERR_INVALID_ARG;
    const size_t io_bytes = (size_t)desc->batch * (size_t)desc->seqlen * (size_t)desc->dim * esz;
    if (overlaps(x, out, io_bytes)) return SSM_ERR_INVALID_ARG;
    if (desc->batch > 65535) return SSM_ERR_UNSUPPORTED;

    // the TMA-streamed kernel when rows are 16-byte multiples and x, out aligned
    if ((desc->dim * (int64_t)esz) % 16 == 0 && aligned16(x) && aligned16(out) &&
        desc->seqlen < ((int64_t)1 << 31) - 64 && desc->dim < ((int64_t)1 << 31)) {
        ssm::ConvParams pt;
        pt.x = x; pt.w = w; pt.bias = bias; pt.state_in = conv_state_in; pt.out = out;
        pt.state_out = conv_state_out;
        pt.batch = desc->batch; pt.seqlen = desc->seqlen; pt.dim = desc->dim;
        pt.width = conv->width; pt.act = conv->activation; pt.chunk = 0;
        const cudaError_t et = desc->io_dtype == SSM_DTYPE_F32 ? launch_conv_tma<float>(pt, s)
                                                              : launch_conv_tma<__nv_bfloat16>(pt, s);
        return et == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
    }
    const int vec = desc->io_dtype == SSM_DTYPE_F32 ? 4 : SSM_CONV_VEC16;
    const bool wide = desc->dim % vec == 0 && aligned16(x) && aligned16(out);   // vector rows
    ssm::ConvParams p;
    p.x = x; p.w = w; p.bias = bias; p.state_in = conv_state_in; p.out = out;
    p.state_out = conv_state_out;
    p.batch = desc->batch; p.seqlen = desc->seqlen; p.dim = desc->dim;
    p.width = conv->width; p.act = conv->activation;
    p.chunk = conv_chunk(desc->seqlen, wide ? desc->dim / vec : desc->dim);
    if (((desc->dim / (wide ? vec : 1)) + 127) / 128 > 0x7fffffff) return SSM_ERR_UNSUPPORTED;
    cudaError_t e;
    if (desc->io_dtype == SSM_DTYPE_F32)
        e = wide ? launch_conv<float, 4>(p, s) : launch_conv<float, 1>(p, s);
    else
        e = wide ? launch_conv<__nv_bfloat16, SSM_CONV_VEC16>(p, s) : launch_conv<__nv_bfloat16, 1>(p, s);
    return e == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}

ssm_status ssm_conv_scan_fwd(const ssm_scan_desc* desc, const ssm_conv_desc* conv,
                             const void* x, const float* conv_w, const float* conv_bias,
                             const float* conv_state_in, float* conv_state_out,
                             const void* delta, const float* A, const void* B, const void* C,
                             const float* D, const void* z, const float* delta_bias, void* out,
                             float* last_state, const float* initial_state, void* workspace,
                             size_t workspace_bytes, void* stream) {
    SSM_TRACE("ssm_conv_scan_fwd");
    ssm_status st = check_desc(desc);
    if (st != SSM_OK) return st;
    st = check_conv(conv);
    if (st != SSM_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int64_t N = desc->dstate;
    const size_t state_bytes = (size_t)desc->batch * (size_t)desc->dim * (size_t)N * sizeof(float);
    const int H = conv->width - 1;
    const size_t cstate_bytes = (size_t)desc->batch * (size_t)desc->dim * (size_t)H * sizeof(float);

    const size_t esz = io_size(desc);
    if (!opt_aligned(x, esz) || !opt_aligned(delta, esz) || !opt_aligned(B, esz) ||
        !opt_aligned(C, esz) || !opt_aligned(z, esz) || !opt_aligned(out, esz) || !opt_aligned(A, 4) ||
        !opt_aligned(D, 4) || !opt_aligned(delta_bias, 4) || !opt_aligned(last_state, 4) ||
        !opt_aligned(initial_state, 4) || !opt_aligned(conv_w, 4) || !opt_aligned(conv_bias, 4) ||
        !opt_aligned(conv_state_in, 4) || !opt_aligned(conv_state_out, 4))
        return SSM_ERR_INVALID_ARG;
    if (overlaps(conv_state_in, conv_state_out, cstate_bytes)) return SSM_ERR_INVALID_ARG;

    if (desc->batch == 0 || desc->dim == 0) return SSM_OK;
    if (desc->seqlen == 0) {
        cudaError_t e = conv_state_passthrough(conv_state_out, conv_state_in, cstate_bytes, s);
        if (e == cudaSuccess && last_state && last_state != initial_state)
            e = initial_state
                ? cudaMemcpyAsync(last_state, initial_state, state_bytes, cudaMemcpyDeviceToDevice, s)
                : cudaMemsetAsync(last_state, 0, state_bytes, s);
        return e == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
    }
    if (!x || !delta || !A || !B || !C || !out || !conv_w) return SSM_ERR_INVALID_ARG;

    const bool tiled = tiled_shape_ok(desc) && aligned16(x) && aligned16(delta) &&
                       aligned16(B) && aligned16(C) && aligned16(out) && opt_aligned(z, 16) &&
                       opt_aligned(last_state, 16);
    // The conv is fused into the warp-specialised kernel (dstate 16, width up
    // to kWsMaxConvWidth) and into the generic one, which takes the rest.
    const bool ws = tiled && conv->width <= kWsMaxConvWidth;
    int nchunk;
    int64_t chunk_len;
    if (ws) {
        tiled_chunks(desc, kKindWs, &nchunk, &chunk_len);
    } else {
        nchunk = generic_nchunk(desc);
        chunk_len = (desc->seqlen + nchunk - 1) / nchunk;
    }
    const size_t need = workspace_for(desc, nchunk);
    if (need > 0 && (workspace == nullptr || workspace_bytes < need || !aligned16(workspace)))
        return SSM_ERR_INVALID_ARG;
    if (desc->batch > 65535) return SSM_ERR_UNSUPPORTED;

    ScanParams p;
    p.x = x; p.delta = delta; p.A = A; p.B = B; p.C = C; p.D = D; p.z = z;
    p.delta_bias = delta_bias; p.out = out; p.last_state = last_state;
    p.initial_state = initial_state;
    p.batch = desc->batch; p.seqlen = desc->seqlen; p.dim = desc->dim;
    p.nchunk = nchunk;
    p.chunk_len = chunk_len;
    p.softplus = desc->delta_softplus ? 1 : 0;
    p.carry = nullptr; p.dsum = nullptr;
    if (nchunk > 1) {
        char* w = static_cast<char*>(workspace);
        const size_t per = (size_t)desc->batch * (size_t)nchunk * (size_t)desc->dim;
        p.carry = reinterpret_cast<float*>(w);
        p.dsum = reinterpret_cast<float*>(w + ((per * (size_t)N * sizeof(float) + 255) & ~(size_t)255));
    }
    p.conv_w = conv_w; p.conv_bias = conv_bias;
    p.conv_state_in = H > 0 ? conv_state_in : nullptr;
    p.conv_state_out = H > 0 ? conv_state_out : nullptr;
    p.conv_width = conv->width; p.conv_act = conv->activation;

    cudaError_t e;
    if (ws)
        e = desc->io_dtype == SSM_DTYPE_F32 ? launch_ws_conv<float>(desc, p, s)
                                            : launch_ws_conv<__nv_bfloat16>(desc, p, s);
    else
        e = desc->io_dtype == SSM_DTYPE_F32 ? dispatch_generic<float, true>(N, p, s)
                                            : dispatch_generic<__nv_bfloat16, true>(N, p, s);
    return e == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}

ssm_status ssm_conv_state_update(const ssm_scan_desc* desc, const ssm_conv_desc* conv,
                                 float* conv_state, const float* conv_w, const float* conv_bias,
                                 float* state, const void* x, const void* delta, const float* A,
                                 const void* B, const void* C, const float* D, const void* z,
                                 const float* delta_bias, void* out, void* stream) {
    SSM_TRACE("ssm_conv_state_update");
    ssm_status st = check_desc(desc);
    if (st != SSM_OK) return st;
    st = check_conv(conv);
    if (st != SSM_OK) return st;
    const size_t esz = io_size(desc);
    if (!opt_aligned(state, desc->dstate >= 4 ? 16 : 4) || !opt_aligned(x, esz) ||
        !opt_aligned(delta, esz) || !opt_aligned(B, esz) || !opt_aligned(C, esz) ||
        !opt_aligned(z, esz) || !opt_aligned(out, esz) || !opt_aligned(A, 4) || !opt_aligned(D, 4) ||
        !opt_aligned(delta_bias, 4) || !opt_aligned(conv_state, 4) || !opt_aligned(conv_w, 4) ||
        !opt_aligned(conv_bias, 4))
        return SSM_ERR_INVALID_ARG;
    if (desc->batch == 0 || desc->dim == 0) return SSM_OK;
    if (!state || !x || !delta || !A || !B || !C || !out || !conv_w) return SSM_ERR_INVALID_ARG;
    if (conv->width > 1 && !conv_state) return SSM_ERR_INVALID_ARG;
    if (desc->batch > 65535 || desc->dim * 64 >= ((int64_t)1 << 31)) return SSM_ERR_UNSUPPORTED;

    DecodeParams p;
    p.state = state; p.x = x; p.delta = delta; p.A = A; p.B = B; p.C = C; p.D = D; p.z = z;
    p.delta_bias = delta_bias; p.out = out;
    p.batch = desc->batch; p.dim = desc->dim;
    p.softplus = desc->delta_softplus ? 1 : 0;
    p.conv_state = conv_state; p.conv_w = conv_w; p.conv_bias = conv_bias;
    p.conv_width = conv->width; p.conv_act = conv->activation;
    p.vec = decode_vec_ok(desc, A, B, C);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = desc->io_dtype == SSM_DTYPE_F32
                        ? dispatch_decode<float, true>(desc->dstate, p, s)
                        : dispatch_decode<__nv_bfloat16, true>(desc->dstate, p, s);
    return e == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// The selection projections (tcgen05 GEMMs).
namespace {

// 2-D bf16 tensor map of a row-major (rows, cols) matrix, box [box_rows][64],
// 128-byte swizzle (the tcgen05 K-major operand layout).
bool encode_2d_sw128(CUtensorMap* m, const void* base, int64_t cols, int64_t rows, int64_t ld,
                     int box_rows) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)(ld * 2)};
    const cuuint32_t box[2] = {(cuuint32_t)ssm::kGemmBK, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

#ifndef SSM_XPROJ_STAGES
#define SSM_XPROJ_STAGES 3   // TMA ring depth of x_proj (K = dim: a long loop)
#endif
#ifndef SSM_DTPROJ_BN
#define SSM_DTPROJ_BN 128    // dt_proj tile width
#endif
#ifndef SSM_DTPROJ_STAGES
#define SSM_DTPROJ_STAGES 2  // dt_proj ring depth (K = dt_rank: a few slabs)
#endif

template <int BN, int STAGES>
cudaError_t launch_gemm(const void* A, const void* Bw, int64_t M, int N, int K, const ssm::GemmParams& p,
                        cudaStream_t s) {
    using Cfg = ssm::GemmCfg<BN, STAGES>;
    ssm::GemmMaps maps;
    memset(&maps, 0, sizeof(maps));
    if (!encode_2d_sw128(&maps.a, A, K, M, K, ssm::kGemmBM) ||
        !encode_2d_sw128(&maps.b, Bw, K, N, K, BN))
        return cudaErrorInvalidValue;
    auto k = ssm::gemm_bf16_tn_kernel<BN, STAGES>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM);
    if (e != cudaSuccess) return e;
    const dim3 grid((unsigned)((M + ssm::kGemmBM - 1) / ssm::kGemmBM), (unsigned)((N + BN - 1) / BN));
    k<<<grid, ssm::kGemmThreads, Cfg::SMEM, s>>>(maps, p);
    return cudaGetLastError();
}

// The persistent form (dt_proj): as many CTAs as fit on the GPU at once
// (shared memory and the 512 TMEM columns of an SM), each walking tiles.
template <int BN, int STAGES>
cudaError_t launch_gemm_persistent(const void* A, const void* Bw, int64_t M, int N, int K,
                                   const ssm::GemmParams& p, cudaStream_t s) {
    using Cfg = ssm::GemmPCfg<BN, STAGES>;
    ssm::GemmMaps maps;
    memset(&maps, 0, sizeof(maps));
    if (!encode_2d_sw128(&maps.a, A, K, M, K, ssm::kGemmBM) ||
        !encode_2d_sw128(&maps.b, Bw, K, N, K, BN))
        return cudaErrorInvalidValue;
    auto k = ssm::gemm_bf16_tn_persistent_kernel<BN, STAGES>;
    const int nk = (K + ssm::kGemmBK - 1) / ssm::kGemmBK;
    const int smem = Cfg::smem(nk);   // the N tile's B slabs stay resident
    if (smem > 227 * 1024) return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    int per_sm = (228 * 1024) / (smem + 1024);
    if (per_sm > 512 / Cfg::TMEM_COLS) per_sm = 512 / Cfg::TMEM_COLS;
    if (per_sm > 2048 / ssm::kGemmPThreads) per_sm = 2048 / ssm::kGemmPThreads;
    if (per_sm < 1) per_sm = 1;
    const int64_t mtiles = (M + ssm::kGemmBM - 1) / ssm::kGemmBM, ntn = (N + BN - 1) / BN;
    if (mtiles * ntn > 0x7fffffff) return cudaErrorInvalidValue;
    // g CTAs per N tile, each walking every g-th M tile; the grid is ntn * g
    int64_t g = (int64_t)kPlanSMs * per_sm / ntn;
    if (g < 1) g = 1;
    if (g > mtiles) g = mtiles;
    k<<<(unsigned)(ntn * g), ssm::kGemmPThreads, smem, s>>>(maps, p);
    return cudaGetLastError();
}

// x_proj: the whole (R + 2N)-wide output in one tile column (BN = its size
// rounded up to 32).
cudaError_t launch_xproj(int bn, const void* A, const void* Bw, int64_t M, int N, int K,
                         const ssm::GemmParams& p, cudaStream_t s) {
    switch (bn) {
        case 32: return launch_gemm<32, SSM_XPROJ_STAGES>(A, Bw, M, N, K, p, s);
        case 64: return launch_gemm<64, SSM_XPROJ_STAGES>(A, Bw, M, N, K, p, s);
        case 96: return launch_gemm<96, SSM_XPROJ_STAGES>(A, Bw, M, N, K, p, s);
        case 128: return launch_gemm<128, SSM_XPROJ_STAGES>(A, Bw, M, N, K, p, s);
        case 160: return launch_gemm<160, SSM_XPROJ_STAGES>(A, Bw, M, N, K, p, s);
        case 192: return launch_gemm<192, SSM_XPROJ_STAGES>(A, Bw, M, N, K, p, s);
        case 224: return launch_gemm<224, SSM_XPROJ_STAGES>(A, Bw, M, N, K, p, s);
        case 256: return launch_gemm<256, SSM_XPROJ_STAGES>(A, Bw, M, N, K, p, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace

extern "C" ssm_status ssm_selection_proj_fwd(const ssm_scan_desc* desc, const ssm_proj_desc* proj,
                                             const void* x, const void* W_x, const void* W_dt,
                                             const float* delta_bias, void* dt_low, void* B,
                                             void* C, void* delta_raw, void* stream) {
    SSM_TRACE("ssm_selection_proj_fwd");
    if (!desc || !proj) return SSM_ERR_INVALID_ARG;
    if (desc->batch < 0 || desc->seqlen < 0 || desc->dim < 0 || desc->dstate <= 0 ||
        proj->dt_rank <= 0 || proj->reserved != 0)
        return SSM_ERR_INVALID_ARG;
    if (desc->io_dtype != SSM_DTYPE_BF16) return SSM_ERR_UNSUPPORTED;
    const int64_t R = proj->dt_rank, N = desc->dstate, Dm = desc->dim;
    const int64_t M = desc->batch * desc->seqlen;
    const int64_t NO = R + 2 * N;
    if (Dm % 8 != 0 || R % 8 != 0 || NO > 256 || Dm > ((int64_t)1 << 30) || M >= ((int64_t)1 << 31))
        return SSM_ERR_UNSUPPORTED;
    for (const void* q : std::initializer_list<const void*>{x, W_x, W_dt, dt_low, B, C, delta_raw})
        if (!opt_aligned(q, 16)) return SSM_ERR_INVALID_ARG;
    if (!opt_aligned(delta_bias, 4)) return SSM_ERR_INVALID_ARG;
    if (M == 0 || Dm == 0) return SSM_OK;
    if (!x || !W_x || !dt_low || !B || !C || (delta_raw && !W_dt)) return SSM_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    ssm::GemmParams p1;
    memset(&p1, 0, sizeof(p1));
    p1.M = M; p1.N = (int)NO; p1.K = (int)Dm;
    p1.seg[0] = {dt_low, R, 0, (int)R};
    p1.seg[1] = {B, N, (int)R, (int)N};
    p1.seg[2] = {C, N, (int)(R + N), (int)N};
    p1.nseg = 3;
    const int bn = (int)((NO + 31) / 32 * 32);
    cudaError_t e = launch_xproj(bn, x, W_x, M, (int)NO, (int)Dm, p1, s);
    if (e != cudaSuccess) return SSM_ERR_CUDA;
    if (delta_raw) {
        ssm::GemmParams p2;
        memset(&p2, 0, sizeof(p2));
        p2.M = M; p2.N = (int)Dm; p2.K = (int)R;
        p2.seg[0] = {delta_raw, Dm, 0, (int)Dm};
        p2.nseg = 1;
        p2.col_bias = delta_bias;
        p2.act = desc->delta_softplus ? 1 : 0;
        if (launch_gemm_persistent<SSM_DTPROJ_BN, SSM_DTPROJ_STAGES>(dt_low, W_dt, M, (int)Dm, (int)R,
                                                                     p2, s) != cudaSuccess)
            return SSM_ERR_CUDA;
    }
    return SSM_OK;
}

// ---------------------------------------------------------------------------
// The time-invariant model's convolution mode.
extern "C" {

ssm_status ssm_lti_kernel(const ssm_scan_desc* desc, const ssm_scan_opts* opts,
                          const float* delta, const float* A, const float* B, const float* C,
                          float* K, void* stream) {
    SSM_TRACE("ssm_lti_kernel");
    if (!desc || desc->dim < 0 || desc->seqlen < 0 || desc->dstate <= 0) return SSM_ERR_INVALID_ARG;
    if (!dstate_supported(desc->dstate)) return SSM_ERR_UNSUPPORTED;
    if (opts && check_opts(opts) != SSM_OK) return SSM_ERR_INVALID_ARG;
    if (!opt_aligned(delta, 4) || !opt_aligned(A, 4) || !opt_aligned(B, 4) || !opt_aligned(C, 4) ||
        !opt_aligned(K, 4))
        return SSM_ERR_INVALID_ARG;
    if (desc->dim == 0 || desc->seqlen == 0) return SSM_OK;
    if (!delta || !A || !B || !C || !K) return SSM_ERR_INVALID_ARG;
    const int64_t blocks = desc->dim * ((desc->seqlen + 255) / 256);
    if (blocks > 0x7fffffff) return SSM_ERR_UNSUPPORTED;
    ssm::LtiKernelParams p;
    p.delta = delta; p.A = A; p.B = B; p.C = C; p.K = K;
    p.dim = desc->dim; p.seqlen = desc->seqlen; p.N = (int)desc->dstate;
    p.zoh = (opts && opts->discretization == SSM_DISC_ZOH) ? 1 : 0;
    ssm::lti_kernel_kernel<<<(unsigned)blocks, 256, 0, static_cast<cudaStream_t>(stream)>>>(p);
    return cudaGetLastError() == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}

ssm_status ssm_lti_conv_fwd(const ssm_scan_desc* desc, const float* K, const void* x,
                            const float* D, const void* z, void* out, void* stream) {
    SSM_TRACE("ssm_lti_conv_fwd");
    if (!desc || desc->batch < 0 || desc->dim < 0 || desc->seqlen < 0) return SSM_ERR_INVALID_ARG;
    if (desc->io_dtype != SSM_DTYPE_F32 && desc->io_dtype != SSM_DTYPE_BF16)
        return SSM_ERR_UNSUPPORTED;
    const size_t esz = io_size(desc);
    if (!opt_aligned(K, 4) || !opt_aligned(x, esz) || !opt_aligned(D, 4) || !opt_aligned(z, esz) ||
        !opt_aligned(out, esz))
        return SSM_ERR_INVALID_ARG;
    if (desc->batch == 0 || desc->dim == 0 || desc->seqlen == 0) return SSM_OK;
    if (!K || !x || !out) return SSM_ERR_INVALID_ARG;
    const int64_t ty = (desc->seqlen + ssm::kLtiTo - 1) / ssm::kLtiTo;
    const int64_t tx = (desc->dim + ssm::kLtiCh - 1) / ssm::kLtiCh;
    if (ty > 65535 || desc->batch > 65535 || tx > 0x7fffffff) return SSM_ERR_UNSUPPORTED;
    ssm::LtiConvParams p;
    p.K = K; p.x = x; p.D = D; p.z = z; p.out = out;
    p.batch = desc->batch; p.seqlen = desc->seqlen; p.dim = desc->dim;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // bf16 I/O with 16-byte rows and bases: the tensor-core form
    if (desc->io_dtype == SSM_DTYPE_BF16 && desc->dim % 8 == 0 && desc->seqlen < ((int64_t)1 << 30) &&
        opt_aligned(x, 16) && opt_aligned(z, 16) && opt_aligned(out, 16) && desc->dim < ((int64_t)1 << 31)) {
        const CUtensorMapDataType dt = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
        ssm::LtiMmaMaps maps;
        memset(&maps, 0, sizeof(maps));
        const int C = ssm::kLtiMmaCh, T = ssm::kLtiMmaChunk, NB = ssm::kLtiMmaB;
        bool ok = encode_3d_box(&maps.x, x, dt, 2, desc->dim, desc->seqlen, desc->batch, C, T, NB) &&
                  encode_3d_box(&maps.out, out, dt, 2, desc->dim, desc->seqlen, desc->batch, C, T, NB);
        if (ok && z) ok = encode_3d_box(&maps.z, z, dt, 2, desc->dim, desc->seqlen, desc->batch, C, T, NB);
        if (!ok) return SSM_ERR_CUDA;
        auto kern = z ? ssm::lti_conv_mma_kernel<true> : ssm::lti_conv_mma_kernel<false>;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, ssm::LtiMmaCfg::SMEM) !=
            cudaSuccess)
            return SSM_ERR_CUDA;
        // persistent: as many CTAs as fit the GPU at once, shared by the batch blocks
        int dev = 0, sms = 0, per_sm = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 256, ssm::LtiMmaCfg::SMEM) !=
                cudaSuccess)
            return SSM_ERR_CUDA;
        const int64_t nby = (desc->batch + NB - 1) / NB;
        const int64_t items = (desc->dim / C) * ((desc->seqlen + T - 1) / T);
        const int64_t slots = std::max<int64_t>(1, (int64_t)sms * std::max(per_sm, 1) / nby);
        const dim3 g((unsigned)std::min(items, slots), (unsigned)nby);
        kern<<<g, 256, ssm::LtiMmaCfg::SMEM, s>>>(maps, p);
        return cudaGetLastError() == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
    }
    const dim3 grid((unsigned)tx, (unsigned)ty, (unsigned)desc->batch);
    if (desc->io_dtype == SSM_DTYPE_F32)
        ssm::lti_conv_kernel<float><<<grid, 256, 0, s>>>(p);
    else
        ssm::lti_conv_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(p);
    return cudaGetLastError() == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Backward (gradients of the scan).
namespace {

struct BwdPlan {
    int nchunk = 1;
    int warps = ssm::kBwdWarps;   // warps per CTA of the sweep
    int64_t chunk_len = 0, ntiles = 0, nblk = 0;
    // the one-warp-layout sweep (dstate 16, 16-byte rows): warps per CTA (0:
    // not used), channel blocks of the grid and dB | dC partial sums (one per
    // 16-channel warp); the sweeps above are its fallback when a call's
    // pointers are not 16-byte aligned
    int ww = 0;
    int64_t nblk_w = 0, npart_w = 0;
    size_t off_fstart = 0, off_fdsum = 0, off_ebuf = 0, off_bdsum = 0, off_ckpt = 0, off_pbc = 0,
           off_pa = 0, off_pd = 0, off_pbias = 0, bytes = 0;
};

size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }

// Warps per CTA of the sweep that are compiled: 5..8 for dstate 8 and 16,
// 6 or 8 for 32, 4 or 8 for 64 (the counts the picker below chooses for
// realistic shapes; the CTA's channel block stays a 16-byte TMA row), 8 for
// dstate below 8.
constexpr bool bwd_warps_ok(int n, int w) {
    return n < 8 ? w == ssm::kBwdWarps
                 : (n <= 16 ? (w >= 5 && w <= 8) : (n == 32 ? (w == 6 || w == 8) : (w == 4 || w == 8)));
}

int bwd_channels_per_cta(int64_t n, int w) {
    if (n != 1 && n != 2 && n != 4 && n != 8 && n != 16 && n != 32 && n != 64) return 0;
    const int lpc = n >= 4 ? (n / 4 > 32 ? 32 : (int)(n / 4)) : 1;
    return (32 / lpc) * w;
}

// Shared memory of the TMA-staged sweep (bytes), for the residency estimate.
template <int N, int W>
int bwd_smem_of(bool f32) {
    if constexpr (N < 8 || !bwd_warps_ok(N, W)) {
        return 0;
    } else {
        return f32 ? ssm::BwdTmaCfg<float, N, W>::SMEM : ssm::BwdTmaCfg<__nv_bfloat16, N, W>::SMEM;
    }
}
template <int N>
int bwd_smem_n(int w, bool f32) {
    switch (w) {
        case 4: return bwd_smem_of<N, 4>(f32);
        case 5: return bwd_smem_of<N, 5>(f32);
        case 6: return bwd_smem_of<N, 6>(f32);
        case 7: return bwd_smem_of<N, 7>(f32);
        case 8: return bwd_smem_of<N, 8>(f32);
    }
    return 0;
}
int bwd_sweep_smem(int64_t n, int w, bool f32) {
    switch (n) {
        case 8: return bwd_smem_n<8>(w, f32);
        case 16: return bwd_smem_n<16>(w, f32);
        case 32: return bwd_smem_n<32>(w, f32);
        case 64: return bwd_smem_n<64>(w, f32);
    }
    return 0;
}

// Warps per CTA for a grid of batch x channel blocks: the count that gives the
// busiest SM the fewest channels.  The CTAs of one wave land round-robin, so
// an SM holds ceil(ctas / 148) of them; a grid that needs a second wave (more
// CTAs than 148 x the CTAs that fit an SM at 128 registers) is charged for the
// wave.  Four-warp CTAs run about 15% slower per channel (measured), ties go
// to more warps.
int bwd_pick_warps(int64_t batch, int64_t dim, int64_t n, bool f32) {
    int best = ssm::kBwdWarps;
    double best_cost = 1e300;
    for (int w = 8; w >= 4; --w) {
        if (!bwd_warps_ok((int)n, w)) continue;
        const int64_t ch = bwd_channels_per_cta(n, w);
        const int64_t ctas = batch * ((dim + ch - 1) / ch);
        // CTAs per SM: registers (128 per thread) and shared memory (228 KB per
        // SM, 1 KB of it reserved per CTA)
        int64_t per_sm = 65536 / (w * 32 * 128);
        const int64_t sm_bytes = bwd_sweep_smem(n, w, f32);
        if (sm_bytes > 0 && 233472 / (sm_bytes + 1024) < per_sm) per_sm = 233472 / (sm_bytes + 1024);
        if (per_sm < 1) per_sm = 1;
        const int64_t slots = (int64_t)kPlanSMs * per_sm;
        const double slow = w == 4 ? 1.15 : 1.0;
        const double cost = ctas <= slots
                                ? (double)((ctas + kPlanSMs - 1) / kPlanSMs) * ch * slow
                                : (double)((ctas + slots - 1) / slots) * per_sm * ch * slow * 1.25;
        if (cost < best_cost) {
            best_cost = cost;
            best = w;
        }
    }
    return best;
}

// Shared memory of a CTA of the one-warp-layout sweep with w warps.
int bwd_warp_smem(int w, bool f32) {
    return f32 ? ssm::BwdWarpCfg<float>::smem(w) : ssm::BwdWarpCfg<__nv_bfloat16>::smem(w);
}

// The one-warp-layout sweep applies to dstate 16 with 16-byte rows.
bool bwd_warp_shape_ok(const ssm_scan_desc* d) {
    const int64_t e = (int64_t)io_size(d);
    return d->dstate == 16 && (d->dim * e) % 16 == 0 && d->seqlen < ((int64_t)1 << 31) &&
           d->dim < ((int64_t)1 << 31);
}

// Chunks and warps per CTA of the one-warp-layout sweep.  A warp-unit is one
// warp's 16 channels of one sequence over one chunk.  Chunks: one while there
// are at least 4 warp-units per SM, else enough to give each SM about 7.
// Warps per CTA: the fewest warp-steps on the busiest SM (CTAs land
// round-robin; a grid beyond the resident CTAs runs in waves); ties go to
// wider CTAs.
void bwd_warp_plan(const ssm_scan_desc* d, int64_t& k, int& ww, int64_t& nblk) {
    const bool f32 = d->io_dtype == SSM_DTYPE_F32;
    const int wmax = f32 ? ssm::BwdWarpCfg<float>::WMAX : ssm::BwdWarpCfg<__nv_bfloat16>::WMAX;
    const int64_t units = d->batch * ((d->dim + 15) / 16);
    const int64_t L = d->seqlen;
    k = 1;
    if (units < (int64_t)kPlanSMs * 4) {
        k = (int64_t)kPlanSMs * 7 / (units > 0 ? units : 1);
        const int64_t kmax = L / 512;
        if (k > kmax) k = kmax;
        if (k > 4096) k = 4096;
        if (k < 1) k = 1;
    }
    const double step_s = 26e-9;                        // one warp-step of a loaded SM (measured scale)
    const double steps = (double)((L + k - 1) / k);
    double best = 1e300;
    ww = wmax;
    nblk = (d->dim + 16 * wmax - 1) / (16 * wmax);
    for (int w = wmax; w >= 1; --w) {
        const int64_t blk = (d->dim + 16 * w - 1) / (16 * w);
        const int64_t ctas = d->batch * k * blk;
        int64_t per_sm = 233472 / (bwd_warp_smem(w, f32) + 1024);
        const int64_t by_regs = 65536 / (w * 32 * 224);
        if (by_regs < per_sm) per_sm = by_regs;
        if (per_sm < 1) per_sm = 1;
        const int64_t slots = (int64_t)kPlanSMs * per_sm;
        const int64_t busiest = ctas <= slots ? (ctas + kPlanSMs - 1) / kPlanSMs * w
                                              : (ctas + slots - 1) / slots * per_sm * w;
        const double t = (double)busiest * steps * step_s;
        if (t < best * 0.999) {
            best = t;
            ww = w;
            nblk = blk;
        }
    }
}

// Chunks of the time axis: one chunk unless the (sequence, channel-block)
// CTAs fill less than half of the GPU's 2 x 148 slots (each chunk beyond the
// first costs an aggregate pass forward and one backward).
BwdPlan bwd_plan(const ssm_scan_desc* d, bool with_ckpt = false) {
    BwdPlan pl;
    const int64_t N = d->dstate, L = d->seqlen;
    const int64_t ch = bwd_channels_per_cta(N, pl.warps);
    pl.nblk = ch > 0 ? (d->dim + ch - 1) / ch : 0;
    const int64_t groups = d->batch * pl.nblk;
    const int64_t slots = (int64_t)kPlanSMs * 2;
    int64_t k = 1;
    if (groups > 0 && groups * 2 >= slots) {   // one chunk: spread the CTAs evenly
        pl.warps = bwd_pick_warps(d->batch, d->dim, N, d->io_dtype == SSM_DTYPE_F32);
        const int64_t chw = bwd_channels_per_cta(N, pl.warps);
        pl.nblk = (d->dim + chw - 1) / chw;
    } else if (groups > 0) {
        k = slots / groups;   // rounded down: every CTA of the sweep in one wave
        const int64_t kmax = L / 512;
        if (k > kmax) k = kmax;
        if (k > 4096) k = 4096;
        if (k < 1) k = 1;
    }
    const int64_t T = ssm::kBwdT;
    int64_t len = (L + k - 1) / k;
    len = (len + T - 1) / T * T;
    if (len < T) len = T;
    pl.chunk_len = len;
    pl.nchunk = L > 0 ? (int)((L + len - 1) / len) : 1;
    pl.ntiles = (L + T - 1) / T;
    if (bwd_warp_shape_ok(d) && L > 0 && d->batch > 0 && d->dim > 0) {
        int64_t kw = 1;
        bwd_warp_plan(d, kw, pl.ww, pl.nblk_w);
        pl.npart_w = (d->dim + 15) / 16;
        int64_t lw = (L + kw - 1) / kw;
        lw = (lw + T - 1) / T * T;
        pl.chunk_len = lw;
        pl.nchunk = (int)((L + lw - 1) / lw);
    }
    const size_t B = (size_t)d->batch, D = (size_t)d->dim, K = (size_t)pl.nchunk;
    size_t o = 0;
    if (pl.nchunk > 1) {
        if (!with_ckpt) {   // chunk start states (the checkpoints hold them otherwise)
            pl.off_fstart = o; o = align256(o + B * K * D * N * 4);
            pl.off_fdsum = o;  o = align256(o + B * K * D * 4);
        }
        pl.off_ebuf = o;   o = align256(o + B * K * D * N * 4);
        pl.off_bdsum = o;  o = align256(o + B * K * D * 4);
    }
    pl.off_ckpt = o;
    if (!with_ckpt) o = align256(o + B * (size_t)pl.ntiles * D * N * 4);
    const size_t nblk_max = (size_t)(pl.nblk > pl.npart_w ? pl.nblk : pl.npart_w);
    pl.off_pbc = o;   o = align256(o + nblk_max * B * (size_t)L * 2 * N * 4);
    pl.off_pa = o;    o = align256(o + B * K * D * N * 4);
    pl.off_pd = o;    o = align256(o + B * K * D * 4);
    pl.off_pbias = o; o = align256(o + B * K * D * 4);
    pl.bytes = o;
    return pl;
}

// The TMA-staged reverse sweep (scan_bwd_tma_kernel) applies to dstate 8..64
// with 16-byte rows and 16-byte aligned token tensors (checked by the caller).
// The reverse sweep with W warps per CTA: TMA-staged when `tma`, else the
// register path.
template <typename IO, int N, int W>
cudaError_t launch_sweep(const BwdPlan& pl, const ssm::BwdParams& p, bool tma, cudaStream_t s) {
    if constexpr (!bwd_warps_ok(N, W)) {
        return cudaErrorInvalidValue;
    } else {
        using S = ssm::BwdShape<N, W>;
        const dim3 grid((unsigned)pl.nblk, (unsigned)p.batch, (unsigned)p.nchunk);
        if constexpr (N >= 8) {
            if (tma) {
                using Cfg = ssm::BwdTmaCfg<IO, N, W>;
                const CUtensorMapDataType dt = sizeof(IO) == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                                               : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
                const int e = (int)sizeof(IO);
                ssm::BwdMaps maps;
                memset(&maps, 0, sizeof(maps));
                const int64_t Dm = p.dim, L = p.seqlen, Bz = p.batch;
                bool ok = encode_3d(&maps.x, p.x, dt, e, Dm, L, Bz, Cfg::CH, Cfg::T) &&
                          encode_3d(&maps.delta, p.delta, dt, e, Dm, L, Bz, Cfg::CH, Cfg::T) &&
                          encode_3d(&maps.dout, p.dout, dt, e, Dm, L, Bz, Cfg::CH, Cfg::T) &&
                          encode_3d(&maps.B, p.B, dt, e, N, L, Bz, N, Cfg::T) &&
                          encode_3d(&maps.C, p.C, dt, e, N, L, Bz, N, Cfg::T) &&
                          encode_3d(&maps.dx, p.dx, dt, e, Dm, L, Bz, Cfg::CH, Cfg::T) &&
                          encode_3d(&maps.ddelta, p.ddelta, dt, e, Dm, L, Bz, Cfg::CH, Cfg::T);
                if (ok && p.z) ok = encode_3d(&maps.z, p.z, dt, e, Dm, L, Bz, Cfg::CH, Cfg::T);
                if (ok && p.dz) ok = encode_3d(&maps.dz, p.dz, dt, e, Dm, L, Bz, Cfg::CH, Cfg::T);
                if (!ok) return cudaErrorInvalidValue;
                auto kt = ssm::scan_bwd_tma_kernel<IO, N, W>;
                cudaError_t err =
                    cudaFuncSetAttribute(kt, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM);
                if (err != cudaSuccess) return err;
                kt<<<grid, W * 32, Cfg::SMEM, s>>>(maps, p);
                return cudaGetLastError();
            }
        }
        auto kb = ssm::scan_bwd_kernel<IO, N, W>;
        cudaError_t err = cudaFuncSetAttribute(kb, cudaFuncAttributeMaxDynamicSharedMemorySize, S::SMEM);
        if (err != cudaSuccess) return err;
        kb<<<grid, W * 32, S::SMEM, s>>>(p);
        return cudaGetLastError();
    }
}

// States recomputed per block of the one-warp-layout sweep (the tile's 16, or
// 8 at a time with the first half recomputed twice).
#ifndef SSM_BWD_HIST
#define SSM_BWD_HIST 16
#endif
constexpr int kBwdWarpHist = SSM_BWD_HIST;

// The one-warp-layout reverse sweep (dstate 16): pl.ww warps per CTA, TMA
// boxes of 16 channels x 16 steps.
template <typename IO>
cudaError_t launch_bwd_warp(const BwdPlan& pl, const ssm::BwdParams& p, cudaStream_t s) {
    using Cfg = ssm::BwdWarpCfg<IO>;
    const CUtensorMapDataType dt = sizeof(IO) == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                                   : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const int e = (int)sizeof(IO);
    ssm::BwdMaps maps;
    memset(&maps, 0, sizeof(maps));
    const int64_t Dm = p.dim, L = p.seqlen, Bz = p.batch;
    const int C = Cfg::DC, T = Cfg::T;
    bool ok = encode_3d(&maps.x, p.x, dt, e, Dm, L, Bz, C, T) &&
              encode_3d(&maps.delta, p.delta, dt, e, Dm, L, Bz, C, T) &&
              encode_3d(&maps.dout, p.dout, dt, e, Dm, L, Bz, C, T) &&
              encode_3d(&maps.B, p.B, dt, e, 16, L, Bz, 16, T) &&
              encode_3d(&maps.C, p.C, dt, e, 16, L, Bz, 16, T) &&
              encode_3d(&maps.dx, p.dx, dt, e, Dm, L, Bz, C, T) &&
              encode_3d(&maps.ddelta, p.ddelta, dt, e, Dm, L, Bz, C, T);
    if (ok && p.z) ok = encode_3d(&maps.z, p.z, dt, e, Dm, L, Bz, C, T);
    if (ok && p.dz) ok = encode_3d(&maps.dz, p.dz, dt, e, Dm, L, Bz, C, T);
    if (!ok || pl.ww < 1 || pl.ww > Cfg::WMAX) return cudaErrorInvalidValue;
    constexpr int H = kBwdWarpHist;
    const bool sp = p.softplus != 0, zg = p.z != nullptr;
    auto kern = sp ? (zg ? ssm::scan_bwd_warp_kernel<IO, H, true, true>
                         : ssm::scan_bwd_warp_kernel<IO, H, true, false>)
                   : (zg ? ssm::scan_bwd_warp_kernel<IO, H, false, true>
                         : ssm::scan_bwd_warp_kernel<IO, H, false, false>);
    const int smem = Cfg::smem(pl.ww);
    const cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (err != cudaSuccess) return err;
    kern<<<dim3((unsigned)pl.nblk_w, (unsigned)p.batch, (unsigned)p.nchunk), 32 * pl.ww, smem, s>>>(maps, p);
    return cudaGetLastError();
}

template <typename IO, int N>
cudaError_t launch_bwd(const ssm_scan_desc* desc, const BwdPlan& pl, ssm::BwdParams p,
                       const ScanParams& fp, float* dB, float* dC, float* dA, float* dD,
                       float* dbias, bool tma, cudaStream_t s) {
    if (p.nchunk > 1) {
        dim3 grid((unsigned)((p.dim + 127) / 128), (unsigned)p.batch, (unsigned)(p.nchunk - 1));
        const int64_t total = p.batch * p.dim * N;
        if (!p.ckpt_given) {
            // chunk start states, as the forward's chunked path computes them: the
            // one-warp kernel's aggregate pass where it applies (16-byte rows and
            // bases, which the TMA-staged sweep needs too; chunk lengths are
            // multiples of its 16-step tile), else the general kernel's
            bool done = false;
            if constexpr (N == 8 || N == 16 || N == 32 || N == 64) {
                if (tma && tiled_shape_ok(desc)) {
                    const cudaError_t e = launch_warp<IO>(desc, fp, s, true);
                    if (e != cudaSuccess) return e;
                    done = true;
                }
            }
            if (!done) {
                ssm::scan_generic_kernel<IO, N, ssm::MODE_AGG><<<grid, 128, 0, s>>>(fp);
                ssm::carry_kernel<<<(unsigned)((total + 255) / 256), 256, 0, s>>>(
                    p.A, p.initial_state, fp.carry, fp.dsum, p.batch, p.dim, N, p.nchunk);
            }
        }
        const int at = ssm::kAggThreads;
        const dim3 agrid((unsigned)((p.dim * ssm::BwdShape<N>::LPC + at - 1) / at), (unsigned)p.batch,
                         (unsigned)(p.nchunk - 1));
        ssm::scan_bwd_agg_kernel<IO, N><<<agrid, at, 0, s>>>(p);
        ssm::scan_bwd_carry_kernel<<<(unsigned)((total + 255) / 256), 256, 0, s>>>(
            p.A, p.dlast, p.ebuf, p.bdsum, p.batch, p.dim, N, p.nchunk);
    }
    cudaError_t err = cudaErrorInvalidValue;
    int64_t nblk = pl.nblk;
    bool swept = false;
    if constexpr (N == 16) {
        if (tma && pl.ww > 0) {
            // this sweep reads the state before every tile: without the training
            // forward's checkpoints, the one-warp scan writes them first
            err = cudaSuccess;
            if (!p.ckpt_given) {
                ScanParams sp = fp;
                sp.ckpt = p.ckpt;
                sp.ckpt_tiles = p.ntiles;
                err = launch_warp_states<IO>(desc, sp, s);
                p.ckpt_given = 1;
            }
            if (err == cudaSuccess) err = launch_bwd_warp<IO>(pl, p, s);
            nblk = pl.npart_w;
            swept = true;
        }
    }
    if (!swept) {
        switch (pl.warps) {
            case 4: err = launch_sweep<IO, N, 4>(pl, p, tma, s); break;
            case 5: err = launch_sweep<IO, N, 5>(pl, p, tma, s); break;
            case 6: err = launch_sweep<IO, N, 6>(pl, p, tma, s); break;
            case 7: err = launch_sweep<IO, N, 7>(pl, p, tma, s); break;
            case 8: err = launch_sweep<IO, N, 8>(pl, p, tma, s); break;
            default: err = cudaErrorInvalidValue;
        }
    }
    if (err != cudaSuccess) return err;
    const int64_t nout = p.batch * p.seqlen * 2 * N + p.dim * N + 2 * p.dim;
    ssm::scan_bwd_reduce_kernel<N><<<(unsigned)((nout + 255) / 256), 256, 0, s>>>(
        p, (int)nblk, dB, dC, dA, dD, dbias);
    return cudaGetLastError();
}

template <typename IO>
cudaError_t dispatch_bwd(const ssm_scan_desc* desc, int64_t n, const BwdPlan& pl, const ssm::BwdParams& p, const ScanParams& fp,
                         float* dB, float* dC, float* dA, float* dD, float* dbias, bool tma,
                         cudaStream_t s) {
    switch (n) {
        case 1: return launch_bwd<IO, 1>(desc, pl, p, fp, dB, dC, dA, dD, dbias, false, s);
        case 2: return launch_bwd<IO, 2>(desc, pl, p, fp, dB, dC, dA, dD, dbias, false, s);
        case 4: return launch_bwd<IO, 4>(desc, pl, p, fp, dB, dC, dA, dD, dbias, false, s);
        case 8: return launch_bwd<IO, 8>(desc, pl, p, fp, dB, dC, dA, dD, dbias, tma, s);
        case 16: return launch_bwd<IO, 16>(desc, pl, p, fp, dB, dC, dA, dD, dbias, tma, s);
        case 32: return launch_bwd<IO, 32>(desc, pl, p, fp, dB, dC, dA, dD, dbias, tma, s);
        case 64: return launch_bwd<IO, 64>(desc, pl, p, fp, dB, dC, dA, dD, dbias, tma, s);
    }
    return cudaErrorInvalidValue;
}

// Shape and alignment rules of the TMA-staged backward.
bool bwd_tma_ok(const ssm_scan_desc* d, std::initializer_list<const void*> tok) {
    if (d->dstate < 8) return false;
    const int64_t e = (int64_t)io_size(d);
    if ((d->dim * e) % 16 != 0 || (d->dstate * e) % 16 != 0) return false;
    if (d->seqlen >= ((int64_t)1 << 31) || d->dim >= ((int64_t)1 << 31)) return false;
    for (const void* q : tok)
        if (!opt_aligned(q, 16)) return false;
    return true;
}

}  // namespace

extern "C" {

size_t ssm_scan_bwd_workspace_size(const ssm_scan_desc* desc) {
    if (check_desc(desc) != SSM_OK) return 0;
    if (desc->batch == 0 || desc->dim == 0 || desc->seqlen == 0) return 0;
    return bwd_plan(desc).bytes;
}

size_t ssm_scan_bwd_ex_workspace_size(const ssm_scan_desc* desc, int with_checkpoints) {
    if (check_desc(desc) != SSM_OK) return 0;
    if (desc->batch == 0 || desc->dim == 0 || desc->seqlen == 0) return 0;
    return bwd_plan(desc, with_checkpoints != 0).bytes;
}

ssm_status ssm_scan_bwd_plan(const ssm_scan_desc* desc, int with_checkpoints,
                             ssm_scan_bwd_plan_info* info) {
    if (!info) return SSM_ERR_INVALID_ARG;
    const ssm_status st = check_desc(desc);
    if (st != SSM_OK) return st;
    memset(info, 0, sizeof(*info));
    if (desc->batch == 0 || desc->dim == 0 || desc->seqlen == 0) return SSM_OK;
    const BwdPlan pl = bwd_plan(desc, with_checkpoints != 0);
    info->nchunk = pl.nchunk;
    info->warps = pl.ww ? pl.ww : pl.warps;
    info->channels = pl.ww ? 16 * pl.ww : bwd_channels_per_cta(desc->dstate, pl.warps);
    info->ctas = (pl.ww ? pl.nblk_w : pl.nblk) * desc->batch * pl.nchunk;
    info->workspace = (int64_t)pl.bytes;
    return SSM_OK;
}

ssm_status ssm_scan_bwd(const ssm_scan_desc* desc, const void* x, const void* delta,
                        const float* A, const void* B, const void* C, const float* D,
                        const void* z, const float* delta_bias, const float* initial_state,
                        const void* dout, const float* dlast_state, void* dx, void* ddelta,
                        float* dA, float* dB, float* dC, float* dD, void* dz,
                        float* ddelta_bias, float* dinitial_state, void* workspace,
                        size_t workspace_bytes, void* stream) {
    SSM_TRACE("ssm_scan_bwd");
    return ssm_scan_bwd_ex(desc, x, delta, A, B, C, D, z, delta_bias, initial_state, dout,
                           dlast_state, nullptr, dx, ddelta, dA, dB, dC, dD, dz, ddelta_bias,
                           dinitial_state, workspace, workspace_bytes, stream);
}

ssm_status ssm_scan_bwd_ex(const ssm_scan_desc* desc, const void* x, const void* delta,
                           const float* A, const void* B, const void* C, const float* D,
                           const void* z, const float* delta_bias, const float* initial_state,
                           const void* dout, const float* dlast_state, const float* checkpoints,
                           void* dx, void* ddelta, float* dA, float* dB, float* dC, float* dD,
                           void* dz, float* ddelta_bias, float* dinitial_state, void* workspace,
                           size_t workspace_bytes, void* stream) {
    SSM_TRACE("ssm_scan_bwd_ex");
    const ssm_status st = check_desc(desc);
    if (st != SSM_OK) return st;
    const size_t esz = io_size(desc);
    if (!opt_aligned(x, esz) || !opt_aligned(delta, esz) || !opt_aligned(B, esz) ||
        !opt_aligned(C, esz) || !opt_aligned(z, esz) || !opt_aligned(dout, esz) ||
        !opt_aligned(dx, esz) || !opt_aligned(ddelta, esz) || !opt_aligned(dz, esz) ||
        !opt_aligned(A, 4) || !opt_aligned(D, 4) || !opt_aligned(delta_bias, 4) ||
        !opt_aligned(initial_state, 4) || !opt_aligned(dlast_state, 4) || !opt_aligned(dA, 4) ||
        !opt_aligned(dB, 4) || !opt_aligned(dC, 4) || !opt_aligned(dD, 4) ||
        !opt_aligned(ddelta_bias, 4) || !opt_aligned(dinitial_state, 4))
        return SSM_ERR_INVALID_ARG;
    if (dz && !z) return SSM_ERR_INVALID_ARG;
    if (checkpoints && !aligned16(checkpoints)) return SSM_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int64_t N = desc->dstate;
    const size_t Bz = (size_t)desc->batch, L = (size_t)desc->seqlen, Dm = (size_t)desc->dim;
    if (desc->batch == 0 || desc->dim == 0 || desc->seqlen == 0) {
        // No token reaches the loss through the scan: every sum is empty, and
        // the initial state's gradient is the final state's.
        cudaError_t e = cudaSuccess;
        auto zero = [&](void* ptr, size_t bytes) {
            if (ptr && bytes && e == cudaSuccess) e = cudaMemsetAsync(ptr, 0, bytes, s);
        };
        zero(dA, Dm * N * 4);
        zero(dD, Dm * 4);
        zero(ddelta_bias, Dm * 4);
        zero(dB, Bz * L * N * 4);
        zero(dC, Bz * L * N * 4);
        if (dinitial_state && e == cudaSuccess) {
            const size_t sb = Bz * Dm * N * 4;
            if (dlast_state)
                e = sb ? cudaMemcpyAsync(dinitial_state, dlast_state, sb, cudaMemcpyDeviceToDevice, s)
                       : cudaSuccess;
            else
                zero(dinitial_state, sb);
        }
        return e == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
    }
    if (!x || !delta || !A || !B || !C || !dout || !dx || !ddelta || !dA || !dB || !dC)
        return SSM_ERR_INVALID_ARG;
    if (desc->batch > 65535) return SSM_ERR_UNSUPPORTED;
    const bool with_ckpt = checkpoints != nullptr;
    const BwdPlan pl = bwd_plan(desc, with_ckpt);
    if (pl.nblk > 0x7fffffff || pl.nchunk > 65535) return SSM_ERR_UNSUPPORTED;
    if (workspace == nullptr || workspace_bytes < pl.bytes || !aligned16(workspace))
        return SSM_ERR_INVALID_ARG;
    char* w = static_cast<char*>(workspace);

    ScanParams fp;   // forward aggregate pass (chunk start states)
    fp.x = x; fp.delta = delta; fp.A = A; fp.B = B; fp.C = C; fp.D = nullptr; fp.z = nullptr;
    fp.delta_bias = delta_bias; fp.out = nullptr; fp.last_state = nullptr;
    fp.initial_state = initial_state;
    fp.batch = desc->batch; fp.seqlen = desc->seqlen; fp.dim = desc->dim;
    fp.nchunk = pl.nchunk; fp.chunk_len = pl.chunk_len;
    fp.softplus = desc->delta_softplus ? 1 : 0;
    fp.carry = (pl.nchunk > 1 && !with_ckpt) ? reinterpret_cast<float*>(w + pl.off_fstart) : nullptr;
    fp.dsum = (pl.nchunk > 1 && !with_ckpt) ? reinterpret_cast<float*>(w + pl.off_fdsum) : nullptr;

    ssm::BwdParams p;
    p.x = x; p.delta = delta; p.A = A; p.B = B; p.C = C; p.D = D; p.z = z;
    p.delta_bias = delta_bias; p.initial_state = initial_state; p.dout = dout;
    p.dlast = dlast_state; p.dx = dx; p.ddelta = ddelta; p.dz = dz; p.dinit = dinitial_state;
    p.fstart = fp.carry;
    p.ebuf = pl.nchunk > 1 ? reinterpret_cast<float*>(w + pl.off_ebuf) : nullptr;
    p.bdsum = pl.nchunk > 1 ? reinterpret_cast<float*>(w + pl.off_bdsum) : nullptr;
    p.ckpt = with_ckpt ? const_cast<float*>(checkpoints) : reinterpret_cast<float*>(w + pl.off_ckpt);
    p.ckpt_given = with_ckpt ? 1 : 0;
    p.pBC = reinterpret_cast<float*>(w + pl.off_pbc);
    p.pA = reinterpret_cast<float*>(w + pl.off_pa);
    p.pD = reinterpret_cast<float*>(w + pl.off_pd);
    p.pbias = reinterpret_cast<float*>(w + pl.off_pbias);
    p.batch = desc->batch; p.seqlen = desc->seqlen; p.dim = desc->dim;
    p.chunk_len = pl.chunk_len; p.ntiles = pl.ntiles; p.nchunk = pl.nchunk;
    p.softplus = desc->delta_softplus ? 1 : 0;
    const size_t v = (size_t)(ssm::BwdShape<16>::SPL) * esz;   // 4 elements for every dstate >= 4
    p.vec = (reinterpret_cast<uintptr_t>(B) % v) == 0 && (reinterpret_cast<uintptr_t>(C) % v) == 0;

    const bool tma = bwd_tma_ok(desc, {x, delta, B, C, z, dout, dx, ddelta, dz});
    const cudaError_t e = desc->io_dtype == SSM_DTYPE_F32
        ? dispatch_bwd<float>(desc, N, pl, p, fp, dB, dC, dA, dD, ddelta_bias, tma, s)
        : dispatch_bwd<__nv_bfloat16>(desc, N, pl, p, fp, dB, dC, dA, dD, ddelta_bias, tma, s);
    return e == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// The scan over host-resident tensors, pipelined over slices (whole sequences
// or runs of steps of one sequence).
namespace {

constexpr int kHostBufs = 2;   // slices in flight per stage
constexpr int kMaxDevices = 256;

struct HostLayout {
    int64_t bs = 0;                   // sequences per slice
    int64_t ts = 0;                   // steps per slice (< L only with bs == 1)
    size_t tok = 0, bc = 0, st = 0;   // bytes per slice: (bs, ts, D) io, (bs, ts, N) io, (bs, D, N) fp32
    size_t scan_ws = 0;               // ssm_scan_fwd workspace of one slice
    size_t per_buf = 0, total = 0;
    // offsets inside one buffer
    size_t o_x = 0, o_dl = 0, o_z = 0, o_b = 0, o_c = 0, o_out = 0, o_h0 = 0, o_h1 = 0, o_ws = 0;
};

// Slices: slice_batch > 0 takes that many whole sequences; slice_batch < 0
// takes -slice_batch steps of one sequence (the state carried from slice to
// slice on the device); 0 picks: whole sequences while one sequence's x is at
// most 16 MB (at least 2 slices when there are 2 sequences), else 16 MB runs
// of steps of one sequence (multiples of 64 steps).  Small slices keep the
// pipeline's ends short: the first slice's copy in and the last one's scan
// and copy out are not overlapped.
constexpr int64_t kHostSliceBytes = 16ll << 20;

void host_slice(const ssm_scan_desc* d, int64_t slice_batch, int64_t* bs, int64_t* ts) {
    *ts = d->seqlen;
    if (slice_batch > 0) {
        *bs = slice_batch < d->batch ? slice_batch : d->batch;
        return;
    }
    if (slice_batch < 0) {
        *bs = 1;
        *ts = -slice_batch < d->seqlen ? -slice_batch : d->seqlen;
        return;
    }
    const int64_t step = d->dim * (int64_t)io_size(d);
    const int64_t per_seq = d->seqlen * step;
    if (per_seq > kHostSliceBytes && step > 0) {
        *bs = 1;
        int64_t t = (kHostSliceBytes / step) / 64 * 64;
        if (t < 64) t = 64;
        *ts = t < d->seqlen ? t : d->seqlen;
        return;
    }
    int64_t b = per_seq > 0 ? kHostSliceBytes / per_seq : d->batch;
    if (b < 1) b = 1;
    if (d->batch >= 2 && b > d->batch / 2) b = d->batch / 2;
    *bs = b < 1 ? 1 : b;
}

HostLayout host_layout(const ssm_scan_desc* d, int64_t slice_batch) {
    HostLayout h;
    host_slice(d, slice_batch, &h.bs, &h.ts);
    const size_t e = io_size(d);
    h.tok = (size_t)h.bs * (size_t)h.ts * (size_t)d->dim * e;
    h.bc = (size_t)h.bs * (size_t)h.ts * (size_t)d->dstate * e;
    h.st = (size_t)h.bs * (size_t)d->dim * (size_t)d->dstate * sizeof(float);
    ssm_scan_desc sd = *d;
    sd.batch = h.bs;
    sd.seqlen = h.ts;
    h.scan_ws = ssm_scan_workspace_size(&sd);
    size_t o = 0;
    h.o_x = o;   o = align256(o + h.tok);
    h.o_dl = o;  o = align256(o + h.tok);
    h.o_z = o;   o = align256(o + h.tok);
    h.o_b = o;   o = align256(o + h.bc);
    h.o_c = o;   o = align256(o + h.bc);
    h.o_out = o; o = align256(o + h.tok);
    h.o_h0 = o;  o = align256(o + h.st);
    h.o_h1 = o;  o = align256(o + h.st);
    h.o_ws = o;  o = align256(o + h.scan_ws);
    h.per_buf = o;
    h.total = o * kHostBufs;
    return h;
}

// The copy streams and events of the host pipeline, made once per device and
// context and kept.  g_copy_mutex is held while a call enqueues its work, so
// two host threads never interleave their records and waits on the events.
struct CopyStreams {
    unsigned long long ctx = 0;
    cudaStream_t in = nullptr, out = nullptr;
    cudaEvent_t start = nullptr, ev_in[kHostBufs] = {}, ev_done[kHostBufs] = {}, ev_out[kHostBufs] = {};
};
std::mutex g_copy_mutex;
CopyStreams g_copy_streams[kMaxDevices];

// Needs g_copy_mutex held.
cudaError_t copy_streams(CopyStreams** cs) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    CopyStreams& c = g_copy_streams[dev];
    const unsigned long long ctx = current_context_id();
    if (!c.in || ctx == 0 || c.ctx != ctx) {
        CopyStreams n;
        e = cudaStreamCreateWithFlags(&n.in, cudaStreamNonBlocking);
        if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&n.out, cudaStreamNonBlocking);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&n.start, cudaEventDisableTiming);
        for (int i = 0; i < kHostBufs && e == cudaSuccess; ++i) {
            e = cudaEventCreateWithFlags(&n.ev_in[i], cudaEventDisableTiming);
            if (e == cudaSuccess) e = cudaEventCreateWithFlags(&n.ev_done[i], cudaEventDisableTiming);
            if (e == cudaSuccess) e = cudaEventCreateWithFlags(&n.ev_out[i], cudaEventDisableTiming);
        }
        if (e != cudaSuccess) return e;
        n.ctx = current_context_id();
        c = n;
    }
    *cs = &c;
    return cudaSuccess;
}

}  // namespace

extern "C" size_t ssm_scan_fwd_host_workspace_size(const ssm_scan_desc* desc, int64_t slice_batch) {
    if (check_desc(desc) != SSM_OK || desc->batch == 0 || desc->dim == 0 || desc->seqlen == 0) return 0;
    return host_layout(desc, slice_batch).total;
}

extern "C" ssm_status ssm_scan_fwd_host(const ssm_scan_desc* desc, int64_t slice_batch, const void* x,
                                        const void* delta, const float* A, const void* B,
                                        const void* C, const float* D, const void* z,
                                        const float* delta_bias, void* out, float* last_state,
                                        const float* initial_state, void* workspace,
                                        size_t workspace_bytes, void* stream) {
    SSM_TRACE("ssm_scan_fwd_host");
    const ssm_status st = check_desc(desc);
    if (st != SSM_OK) return st;
    if (desc->batch == 0 || desc->dim == 0) return SSM_OK;
    if (desc->seqlen == 0) {
        if (last_state) {
            const size_t sb = (size_t)desc->batch * (size_t)desc->dim * (size_t)desc->dstate * 4;
            if (initial_state) memcpy(last_state, initial_state, sb);
            else memset(last_state, 0, sb);
        }
        return SSM_OK;
    }
    if (!x || !delta || !A || !B || !C || !out) return SSM_ERR_INVALID_ARG;
    const HostLayout h = host_layout(desc, slice_batch);
    if (!workspace || workspace_bytes < h.total || (reinterpret_cast<uintptr_t>(workspace) & 255))
        return SSM_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(g_copy_mutex);
    CopyStreams* csp = nullptr;
    if (copy_streams(&csp) != cudaSuccess) return SSM_ERR_CUDA;
    const CopyStreams& cs = *csp;
    cudaStream_t comp = static_cast<cudaStream_t>(stream);
    char* ws = static_cast<char*>(workspace);
    const size_t e = io_size(desc);
    const int64_t ngroups = (desc->batch + h.bs - 1) / h.bs;
    const int64_t ntime = (desc->seqlen + h.ts - 1) / h.ts;
    const int64_t nsl = ngroups * ntime;

    // events: start; per buffer "inputs in", "scanned", "outputs out"
    cudaEvent_t ev_start = cs.start;
    const cudaEvent_t* ev_in = cs.ev_in;
    const cudaEvent_t* ev_done = cs.ev_done;
    const cudaEvent_t* ev_out = cs.ev_out;

    cudaError_t err = cudaEventRecord(ev_start, comp);
    if (err == cudaSuccess) err = cudaStreamWaitEvent(cs.in, ev_start, 0);
    if (err == cudaSuccess) err = cudaStreamWaitEvent(cs.out, ev_start, 0);
    ssm_status res = SSM_OK;
    for (int64_t i = 0; i < nsl && err == cudaSuccess && res == SSM_OK; ++i) {
        const int bi = (int)(i % kHostBufs);
        char* buf = ws + (size_t)bi * h.per_buf;
        const int64_t g = i / ntime, j = i % ntime;   // batch group, run of steps
        const int64_t b0 = g * h.bs, t0 = j * h.ts;
        const int64_t nb = desc->batch - b0 < h.bs ? desc->batch - b0 : h.bs;
        const int64_t nt = desc->seqlen - t0 < h.ts ? desc->seqlen - t0 : h.ts;
        // a slice is contiguous in host memory: whole sequences, or (ntime > 1)
        // a run of steps of one sequence
        const size_t tok = (size_t)nb * (size_t)nt * (size_t)desc->dim * e;
        const size_t tok_off = ((size_t)b0 * (size_t)desc->seqlen + (size_t)t0) * (size_t)desc->dim * e;
        const size_t bc = (size_t)nb * (size_t)nt * (size_t)desc->dstate * e;
        const size_t bc_off = ((size_t)b0 * (size_t)desc->seqlen + (size_t)t0) * (size_t)desc->dstate * e;
        const size_t sb = (size_t)nb * (size_t)desc->dim * (size_t)desc->dstate * 4;
        const size_t sb_off = (size_t)b0 * (size_t)desc->dim * (size_t)desc->dstate * 4;
        // copies in: the buffer's previous slice must have been scanned and copied out
        if (i >= kHostBufs) err = cudaStreamWaitEvent(cs.in, ev_out[bi], 0);
        auto h2d = [&](size_t off, const void* src, size_t n) {
            if (err == cudaSuccess && src && n)
                err = cudaMemcpyAsync(buf + off, static_cast<const char*>(src), n,
                                      cudaMemcpyHostToDevice, cs.in);
        };
        h2d(h.o_x, static_cast<const char*>(x) + tok_off, tok);
        h2d(h.o_dl, static_cast<const char*>(delta) + tok_off, tok);
        if (z) h2d(h.o_z, static_cast<const char*>(z) + tok_off, tok);
        h2d(h.o_b, static_cast<const char*>(B) + bc_off, bc);
        h2d(h.o_c, static_cast<const char*>(C) + bc_off, bc);
        if (initial_state && j == 0)
            h2d(h.o_h0, reinterpret_cast<const char*>(initial_state) + sb_off, sb);
        if (err == cudaSuccess) err = cudaEventRecord(ev_in[bi], cs.in);
        // the scan of the slice on the caller's stream; a later run of steps
        // starts from the state the previous one (the other buffer) ended in,
        // which the scans' order on the stream keeps valid
        if (err == cudaSuccess) err = cudaStreamWaitEvent(comp, ev_in[bi], 0);
        if (err != cudaSuccess) break;
        const float* h_start = nullptr;
        if (j > 0)
            h_start = reinterpret_cast<const float*>(ws + (size_t)((i - 1) % kHostBufs) * h.per_buf + h.o_h1);
        else if (initial_state)
            h_start = reinterpret_cast<const float*>(buf + h.o_h0);
        const bool keep_state = last_state || j + 1 < ntime;
        ssm_scan_desc sd = *desc;
        sd.batch = nb;
        sd.seqlen = nt;
        res = ssm_scan_fwd(&sd, buf + h.o_x, buf + h.o_dl, A, buf + h.o_b, buf + h.o_c, D,
                           z ? buf + h.o_z : nullptr, delta_bias, buf + h.o_out,
                           keep_state ? reinterpret_cast<float*>(buf + h.o_h1) : nullptr, h_start,
                           h.scan_ws ? buf + h.o_ws : nullptr, h.scan_ws, comp);
        if (res != SSM_OK) break;
        err = cudaEventRecord(ev_done[bi], comp);
        // copies out
        if (err == cudaSuccess) err = cudaStreamWaitEvent(cs.out, ev_done[bi], 0);
        if (err == cudaSuccess)
            err = cudaMemcpyAsync(static_cast<char*>(out) + tok_off, buf + h.o_out, tok,
                                  cudaMemcpyDeviceToHost, cs.out);
        if (err == cudaSuccess && last_state && j + 1 == ntime)
            err = cudaMemcpyAsync(reinterpret_cast<char*>(last_state) + sb_off, buf + h.o_h1, sb,
                                  cudaMemcpyDeviceToHost, cs.out);
        if (err == cudaSuccess) err = cudaEventRecord(ev_out[bi], cs.out);
    }
    // the caller's stream reaches the end of this call once everything has landed
    if (err == cudaSuccess && res == SSM_OK) {
        const int last = (int)((nsl - 1) % kHostBufs);
        err = cudaStreamWaitEvent(comp, ev_out[last], 0);
        if (err == cudaSuccess && nsl > 1)
            err = cudaStreamWaitEvent(comp, ev_out[(last + 1) % kHostBufs], 0);
    }
    if (res != SSM_OK) return res;
    return err == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}

// ---------------------------------------------------------------------------
// ssm_scan_fwd_noalloc: the scan for callers that cannot allocate device
// memory.  Its chunk-carry scratch is this file-scope device array instead of
// a caller workspace; see include/ssm.h for the contract.
namespace {

__device__ __align__(256) unsigned char g_noalloc_scratch[SSM_NOALLOC_SCRATCH_BYTES];

constexpr int kNoAllocMaxDevices = 256;
std::mutex g_noalloc_mutex;
struct NoAllocSlot {
    unsigned long long ctx = 0;
    void* addr = nullptr;
};
NoAllocSlot g_noalloc_addr[kNoAllocMaxDevices];

// Device address of g_noalloc_scratch on the current device.  In host code
// the array's name is only a host-side stand-in, so the address is looked up
// with cudaGetSymbolAddress (that device current) once per device and
// context, and cached; a new context (e.g. after cudaDeviceReset) looks it
// up again.
cudaError_t noalloc_scratch_address(void** addr) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kNoAllocMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    NoAllocSlot& slot = g_noalloc_addr[dev];
    const unsigned long long ctx = current_context_id();
    if (slot.addr == nullptr || ctx == 0 || slot.ctx != ctx) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);   // makes the context current if needed
        if (e != cudaSuccess) return e;
        slot.addr = p;
        slot.ctx = current_context_id();
    }
    *addr = slot.addr;
    return cudaSuccess;
}

}  // namespace

extern "C" ssm_status ssm_scan_fwd_noalloc(const ssm_scan_desc* desc, const void* x,
                                           const void* delta, const float* A, const void* B,
                                           const void* C, const float* D, const void* z,
                                           const float* delta_bias, void* out,
                                           float* last_state, const float* initial_state,
                                           void* stream) {
    SSM_TRACE("ssm_scan_fwd_noalloc");
    const ssm_status st = check_desc(desc);
    if (st != SSM_OK) return st;
    const size_t need = ssm_scan_workspace_size(desc);
    if (need > (size_t)SSM_NOALLOC_SCRATCH_BYTES) return SSM_ERR_UNSUPPORTED;
    void* scratch = nullptr;
    if (need > 0 && noalloc_scratch_address(&scratch) != cudaSuccess) return SSM_ERR_CUDA;
    return ssm_scan_fwd(desc, x, delta, A, B, C, D, z, delta_bias, out, last_state,
                        initial_state, scratch, need, stream);
}
