// Device-side helpers shared by the WTConv kernels (sm_103a).
//
// Notation follows "Fast and Memory-Efficient Wavelet Convolutions via I/O-Aware
// Reformulation" (Aflalo et al.): X^(l) is the level-l low-pass carrier, Y^(l) the
// four Haar subbands of X^(l-1) (§4.1 Eq. 5), Z^(l) the filtered, scaled subbands.
//
// Inside the kernels the Haar subbands are kept UNNORMALIZED: U = 2 Y, i.e.
//   U_LL = a+b+c+d, U_LH = a+b-c-d, U_HL = a-b+c-d, U_HH = a-b-c+d,
// and the exact power-of-two factors (1/2 of the analysis, 2^-l of the synthesis,
// Eq. 7) are folded into the level kernels when they are staged (§4.1 notes that the
// transform needs only signed additions and power-of-two scaling).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace wt {

constexpr int kMaxLevels = 12;

// ---------------------------------------------------------------------------------
// Global-memory I/O in the layer's dtype (float or bfloat16), widened to float.
// ---------------------------------------------------------------------------------
template <typename T>
struct IO;

template <>
struct IO<float> {
    static __device__ __forceinline__ float ld(const float* p) { return __ldg(p); }
    static __device__ __forceinline__ float2 ld2(const float* p) {
        return __ldg(reinterpret_cast<const float2*>(p));
    }
    static __device__ __forceinline__ float4 ld4(const float* p) {
        return __ldg(reinterpret_cast<const float4*>(p));
    }
    static __device__ __forceinline__ void st(float* p, float v) { *p = v; }
    static __device__ __forceinline__ void st4(float* p, float4 v) {
        *reinterpret_cast<float4*>(p) = v;
    }
};

template <>
struct IO<__nv_bfloat16> {
    static __device__ __forceinline__ float bf(uint32_t bits16) {
        return __uint_as_float(bits16 << 16);
    }
    static __device__ __forceinline__ float ld(const __nv_bfloat16* p) {
        return __bfloat162float(*p);
    }
    static __device__ __forceinline__ float2 ld2(const __nv_bfloat16* p) {
        const uint32_t u = __ldg(reinterpret_cast<const unsigned int*>(p));
        return make_float2(bf(u & 0xffffu), bf(u >> 16));
    }
    static __device__ __forceinline__ float4 ld4(const __nv_bfloat16* p) {
        const uint2 u = __ldg(reinterpret_cast<const uint2*>(p));
        return make_float4(bf(u.x & 0xffffu), bf(u.x >> 16), bf(u.y & 0xffffu), bf(u.y >> 16));
    }
    static __device__ __forceinline__ void st(__nv_bfloat16* p, float v) {
        *p = __float2bfloat16_rn(v);
    }
    static __device__ __forceinline__ void st4(__nv_bfloat16* p, float4 v) {
        __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y);
        __nv_bfloat162 hi = __floats2bfloat162_rn(v.z, v.w);
        uint2 u;
        u.x = *reinterpret_cast<uint32_t*>(&lo);
        u.y = *reinterpret_cast<uint32_t*>(&hi);
        *reinterpret_cast<uint2*>(p) = u;
    }
};

template <>
struct IO<__half> {
    static __device__ __forceinline__ float ld(const __half* p) { return __half2float(*p); }
    static __device__ __forceinline__ float2 ld2(const __half* p) {
        const unsigned int u = __ldg(reinterpret_cast<const unsigned int*>(p));
        return __half22float2(*reinterpret_cast<const __half2*>(&u));
    }
    static __device__ __forceinline__ float4 ld4(const __half* p) {
        const uint2 u = __ldg(reinterpret_cast<const uint2*>(p));
        const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&u.x));
        const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&u.y));
        return make_float4(a.x, a.y, b.x, b.y);
    }
    static __device__ __forceinline__ void st(__half* p, float v) { *p = __float2half_rn(v); }
    static __device__ __forceinline__ void st4(__half* p, float4 v) {
        __half2 lo = __floats2half2_rn(v.x, v.y);
        __half2 hi = __floats2half2_rn(v.z, v.w);
        uint2 u;
        u.x = *reinterpret_cast<uint32_t*>(&lo);
        u.y = *reinterpret_cast<uint32_t*>(&hi);
        *reinterpret_cast<uint2*>(p) = u;
    }
};

// ---------------------------------------------------------------------------------
// Haar butterfly on one 2x2 block (a b / c d), unnormalized (Eq. 5 times 2).
// ---------------------------------------------------------------------------------
__device__ __forceinline__ float4 haar_u(float a, float b, float c, float d) {
    const float s0 = a + b, s1 = c + d, d0 = a - b, d1 = c - d;
    return make_float4(s0 + s1, s0 - s1, d0 + d1, d0 - d1);
}

__device__ __forceinline__ float4 f4_zero() { return make_float4(0.f, 0.f, 0.f, 0.f); }

// Synthesis of one coefficient tuple at within-block parity (ry, rx) (App. A Eq. 12/13;
// the 1/2 is folded into the weights): z.LL + s_y z.LH + s_x z.HL + s_y s_x z.HH.
template <int RY, int RX>
__device__ __forceinline__ float synth(const float4& z) {
    const float t0 = RY ? (z.x - z.y) : (z.x + z.y);
    const float t1 = RY ? (z.z - z.w) : (z.z + z.w);
    return RX ? (t0 - t1) : (t0 + t1);
}

// Same with the signs given at run time (0 = +, 1 = -).
__device__ __forceinline__ float synth_rt(const float4& z, int by, int bx) {
    const float t0 = by ? (z.x - z.y) : (z.x + z.y);
    const float t1 = by ? (z.z - z.w) : (z.z + z.w);
    return bx ? (t0 - t1) : (t0 + t1);
}

}  // namespace wt

namespace wt {

// ---------------------------------------------------------------------------------
// Packed fp32 pairs (sm_100+ f32x2 arithmetic): two independent lanes of work per
// instruction on an aligned register pair. Where the operands of a loop are not pairs
// already (a window read at odd pixel offsets), building them costs moves that scalar
// FMAs do not need; the base loops measured faster scalar for k >= 5.
// ---------------------------------------------------------------------------------
typedef unsigned long long f2x;

__device__ __forceinline__ f2x pk2(float lo, float hi) {
    f2x r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ float2 upk2(f2x v) {
    float2 r;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
    return r;
}
__device__ __forceinline__ f2x fma2(f2x a, f2x b, f2x c) {
    f2x d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ f2x add2(f2x a, f2x b) {
    f2x d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ f2x sub2(f2x a, f2x b) {
    f2x d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
// Scalar acc.lo += a * b on the low lane of a packed accumulator (the high lane is kept).
__device__ __forceinline__ void fma_lo(f2x& acc, float a, float b) {
    asm("{\n\t.reg .f32 lo, hi;\n\t"
        "mov.b64 {lo, hi}, %0;\n\t"
        "fma.rn.f32 lo, %1, %2, lo;\n\t"
        "mov.b64 %0, {lo, hi};\n\t}"
        : "+l"(acc)
        : "f"(a), "f"(b));
}

}  // namespace wt
