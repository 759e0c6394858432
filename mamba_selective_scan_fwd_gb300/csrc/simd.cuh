// Packed-pair f32 arithmetic (sm_100+ f32x2 instructions), the MUFU
// approximations used on the hot path, and bf16 <-> f32 bit conversions.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace ss {

// ---------------------------------------------------------------- f32x2
#ifdef SS_SCALAR_PAIRS
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
    return make_float2(fmaf(a.x, b.x, c.x), fmaf(a.y, b.y, c.y));
}
__device__ __forceinline__ float2 mul2(float2 a, float2 b) { return make_float2(a.x * b.x, a.y * b.y); }
__device__ __forceinline__ float2 add2(float2 a, float2 b) { return make_float2(a.x + b.x, a.y + b.y); }
#else
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
    float2 r;
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
        "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(r.x), "=f"(r.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return r;
}

__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
    float2 r;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(r.x), "=f"(r.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return r;
}

__device__ __forceinline__ float2 add2(float2 a, float2 b) {
    float2 r;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(r.x), "=f"(r.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return r;
}

#endif

__device__ __forceinline__ float2 splat2(float v) { return make_float2(v, v); }

// ---------------------------------------------------------------- MUFU
// 2^x with the hardware approximation (PTX ex2.approx.ftz.f32); results
// below the normal range flush to zero.
__device__ __forceinline__ float ex2a(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float lg2a(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float rcpa(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

constexpr float kLn2 = 0.6931471805599453f;
constexpr float kLog2eF = 1.4426950408889634f;

// softplus(x) = log(1 + e^x) = max(x, 0) + log1p(e) with e = e^-|x| in (0, 1].
// log1p(e) = 2 atanh(s) with s = e / (2 + e) in (0, 1/3], summed as the odd
// series 2 s (1 + s^2/3 + s^4/5 + ... + s^14/15); the first omitted term is
// below 1.1e-8 relative, so the result keeps f32 relative accuracy for every
// x (unlike log2 of 1 + e, whose hardware approximation has an absolute error
// bound near 1).
__device__ __forceinline__ float softplus_fast(float x) {
    const float e = ex2a(-fabsf(x) * kLog2eF);
    const float s = e * rcpa(2.f + e);
    const float s2 = s * s;
    float p = 1.f / 15.f;
    p = fmaf(p, s2, 1.f / 13.f);
    p = fmaf(p, s2, 1.f / 11.f);
    p = fmaf(p, s2, 1.f / 9.f);
    p = fmaf(p, s2, 1.f / 7.f);
    p = fmaf(p, s2, 1.f / 5.f);
    p = fmaf(p, s2, 1.f / 3.f);
    p = fmaf(p, s2, 1.f);
    return fmaxf(x, 0.f) + 2.f * s * p;
}

// sigmoid(x) = 1 / (1 + e^-x)
__device__ __forceinline__ float sigmoid_fast(float x) { return rcpa(1.f + ex2a(-x * kLog2eF)); }

// Two values at a time with packed f32x2 arithmetic (the MUFU steps stay
// scalar): the softplus of softplus_fast, together with sigmoid(x) from the
// same e = e^-|x| (sigmoid(x) = 1 / (1 + e) for x >= 0, e / (1 + e) below).
__device__ __forceinline__ void softplus_sigmoid2(float2 x, float2& sp, float2& sg) {
    const float2 e = make_float2(ex2a(-fabsf(x.x) * kLog2eF), ex2a(-fabsf(x.y) * kLog2eF));
    const float2 t = add2(e, splat2(2.f));
    const float2 s = mul2(e, make_float2(rcpa(t.x), rcpa(t.y)));
    const float2 s2 = mul2(s, s);
    float2 p = splat2(1.f / 15.f);
    p = fma2(p, s2, splat2(1.f / 13.f));
    p = fma2(p, s2, splat2(1.f / 11.f));
    p = fma2(p, s2, splat2(1.f / 9.f));
    p = fma2(p, s2, splat2(1.f / 7.f));
    p = fma2(p, s2, splat2(1.f / 5.f));
    p = fma2(p, s2, splat2(1.f / 3.f));
    p = fma2(p, s2, splat2(1.f));
    sp = fma2(add2(s, s), p, make_float2(fmaxf(x.x, 0.f), fmaxf(x.y, 0.f)));
    const float2 d = add2(e, splat2(1.f));
    const float2 r = make_float2(rcpa(d.x), rcpa(d.y));
    const float2 er = mul2(e, r);
    sg = make_float2(x.x >= 0.f ? r.x : er.x, x.y >= 0.f ? r.y : er.y);
}

__device__ __forceinline__ float2 softplus2(float2 x) {
    float2 sp, sg;
    softplus_sigmoid2(x, sp, sg);
    return sp;
}

__device__ __forceinline__ float2 sigmoid2(float2 x) {
    const float2 e = make_float2(ex2a(-x.x * kLog2eF), ex2a(-x.y * kLog2eF));
    const float2 d = add2(e, splat2(1.f));
    return make_float2(rcpa(d.x), rcpa(d.y));
}

// ---------------------------------------------------------------- bf16 bits
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// The low bf16 of w as f32 by a byte permute (kept off the FP32 pipe, where a
// shift may be issued as an integer multiply-add).
__device__ __forceinline__ float bf16lo_prmt(uint32_t w) {
    uint32_t r;
    asm("prmt.b32 %0, %1, %2, 0x1044;" : "=r"(r) : "r"(w), "r"(0u));
    return __uint_as_float(r);
}

// Four consecutive bf16 values at p (8-byte aligned shared memory) as f32.
__device__ __forceinline__ void ld_bf16x4(const void* p, float (&v)[4]) {
    const uint2 w = *reinterpret_cast<const uint2*>(p);
    v[0] = bf16lo_prmt(w.x);
    v[1] = bf16hi(w.x);
    v[2] = bf16lo_prmt(w.y);
    v[3] = bf16hi(w.y);
}

// Round-to-nearest-even f32 -> bf16 of two values, packed lo | hi << 16.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

}  // namespace ss
