// tile_io.cuh -- helpers shared by the TMA-tiled kernels (the scan paths, the
// conv, the backward): the tensor maps of a scan, 16-byte vector packing of
// io elements, paired loads and stores of two adjacent io elements, and the
// SFU forms of softplus and silu used for bf16 I/O.
#pragma once
#include "common.cuh"
#include "scan_generic.cuh"
#include "tma.cuh"

namespace ssm {

struct TiledMaps {
    CUtensorMap x, delta, z, B, C, out;
};

__host__ __device__ constexpr int round_up(int v, int a) { return (v + a - 1) / a * a; }

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

}  // namespace ssm
