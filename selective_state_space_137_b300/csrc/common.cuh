// common.cuh -- small device helpers shared by the scan and decode kernels.
#pragma once
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace ssm {

constexpr float kLog2e = 1.4426950408889634f;   // log2(e)
constexpr float kLn2 = 0.6931471805599453f;     // ln(2)

// Load one io element as fp32.
__device__ __forceinline__ float load_f32(const float* p) { return __ldg(p); }
__device__ __forceinline__ float load_f32(const __nv_bfloat16* p) {
    return __bfloat162float(__ldg(p));
}
// Store fp32 as an io element (bf16: round to nearest even).
__device__ __forceinline__ void store_io(float* p, float v) { *p = v; }
__device__ __forceinline__ void store_io(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }

// 2^v on the special-function unit (flush-to-zero for results below 2^-126).
__device__ __forceinline__ float ex2_sfu(float v) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(v));
    return r;
}

// softplus(u) = log(1 + e^u).  Above u = 20 the correction log1p(e^-u) is
// below 2.1e-9 and u itself is returned.
__device__ __forceinline__ float softplus_accurate(float u) {
    return u > 20.f ? u : log1pf(expf(u));
}

// silu(v) = v * sigmoid(v).
__device__ __forceinline__ float silu_accurate(float v) { return v / (1.f + expf(-v)); }

// ---- packed fp32 pairs (f32x2 in one 64-bit register): one issue slot for two
// lanes of FP work.
typedef unsigned long long f32x2;

__device__ __forceinline__ f32x2 pk2(float lo, float hi) {
    f32x2 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void upk2(f32x2 v, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ f32x2 fma2(f32x2 a, f32x2 b, f32x2 c) {
    f32x2 r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
__device__ __forceinline__ f32x2 mul2(f32x2 a, f32x2 b) {
    f32x2 r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ f32x2 add2(f32x2 a, f32x2 b) {
    f32x2 r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

// bf16 tensor-core product of one m16n8k16 tile: d += a b (fp32 accumulate).
// Fragments (lane = 4 g + q): a0 = A[g][2q, 2q+1], a1 = A[g+8][2q, 2q+1],
// a2 = A[g][2q+8, 2q+9], a3 = A[g+8][2q+8, 2q+9]; b0 = B[2q, 2q+1][g],
// b1 = B[2q+8, 2q+9][g]; d = D[g][2q, 2q+1], D[g+8][2q, 2q+1] (low element first).
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                               uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

}  // namespace ssm
