// Shared device helpers and the launch plan of the sm_103a selective scan.
//
// Thread layout used by every scan kernel: a block of kThreads threads covers
// CH = kThreads / G channels of one batch row and one time chunk; the G
// adjacent lanes of a channel each own S = N / G of its states (S <= 8), so
// the N-state recurrence of a channel lives in registers across G lanes.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace ss {

constexpr int kThreads = 128;    // threads per scan block
constexpr int kTc = 8;           // backward sub-chunk length (steps kept in registers)
constexpr int kMinChunk = 64;    // shortest time chunk the planner creates
constexpr int64_t kTargetThreads = 32768;  // parallelism the planner aims for
constexpr float kLog2e = 1.4426950408889634f;
constexpr unsigned kFull = 0xffffffffu;

struct Plan {
    int S, G, CH;      // states per lane, lanes per channel, channels per block
    int64_t K;         // number of time chunks
    int64_t Lc;        // chunk length (multiple of kTc); the last chunk may be shorter
    int64_t tiles;     // channel tiles per batch row
    int64_t nsub;      // kTc sub-chunks per chunk
};

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// A pure function of the problem sizes: the same sizes always give the same
// chunking, hence bit-identical results.
inline Plan make_plan(int64_t Bsz, int64_t L, int64_t Dch, int64_t N) {
    Plan p;
    p.S = N < 8 ? (int)N : 8;
    p.G = (int)(N / p.S);
    p.CH = kThreads / p.G;
    p.tiles = ceil_div(Dch, p.CH);
    int64_t lanes = Bsz * Dch * p.G;
    int64_t K = 1;
    if (lanes > 0 && lanes < kTargetThreads) K = ceil_div(kTargetThreads, lanes);
    int64_t kmax = ceil_div(L, kMinChunk);
    if (K > kmax) K = kmax;
    if (K < 1) K = 1;
    int64_t Lc = ceil_div(ceil_div(L, K), kTc) * kTc;
    if (Lc < kTc) Lc = kTc;
    p.K = ceil_div(L, Lc);
    if (p.K < 1) p.K = 1;
    p.Lc = Lc;
    p.nsub = Lc / kTc;
    return p;
}

// ---------------------------------------------------------------- element I/O

template <typename T> __device__ __forceinline__ float ld(const T* p);
template <> __device__ __forceinline__ float ld<float>(const float* p) { return __ldg(p); }
template <> __device__ __forceinline__ float ld<__nv_bfloat16>(const __nv_bfloat16* p) {
    return __bfloat162float(__ldg(p));
}

template <typename T> __device__ __forceinline__ void st(T* p, float v);
template <> __device__ __forceinline__ void st<float>(float* p, float v) { *p = v; }
template <> __device__ __forceinline__ void st<__nv_bfloat16>(__nv_bfloat16* p, float v) {
    *p = __float2bfloat16_rn(v);
}

// Load S consecutive io elements (S * sizeof(T) bytes, naturally aligned) as floats.
template <int S> __device__ __forceinline__ void ld_row_f32(const float* p, float (&v)[S]) {
    if constexpr (S % 4 == 0) {
#pragma unroll
        for (int i = 0; i < S; i += 4) {
            float4 q = __ldg(reinterpret_cast<const float4*>(p + i));
            v[i] = q.x; v[i + 1] = q.y; v[i + 2] = q.z; v[i + 3] = q.w;
        }
    } else if constexpr (S == 2) {
        float2 q = __ldg(reinterpret_cast<const float2*>(p));
        v[0] = q.x; v[1] = q.y;
    } else {
        v[0] = __ldg(p);
    }
}

// bf16 -> f32 is exact: the bf16 bits become the top half of the f32.
template <int S> __device__ __forceinline__ void ld_row_bf16(const __nv_bfloat16* p, float (&v)[S]) {
    if constexpr (S == 8) {
        uint4 q = __ldg(reinterpret_cast<const uint4*>(p));
        const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int i = 0; i < 4; i++) {
            v[2 * i] = __uint_as_float(w[i] << 16);
            v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    } else if constexpr (S == 4) {
        uint2 q = __ldg(reinterpret_cast<const uint2*>(p));
        v[0] = __uint_as_float(q.x << 16); v[1] = __uint_as_float(q.x & 0xffff0000u);
        v[2] = __uint_as_float(q.y << 16); v[3] = __uint_as_float(q.y & 0xffff0000u);
    } else if constexpr (S == 2) {
        uint32_t q = __ldg(reinterpret_cast<const unsigned int*>(p));
        v[0] = __uint_as_float(q << 16); v[1] = __uint_as_float(q & 0xffff0000u);
    } else {
        v[0] = __bfloat162float(__ldg(p));
    }
}

template <typename T, int S> __device__ __forceinline__ void ld_row(const T* p, float (&v)[S]) {
    if constexpr (sizeof(T) == 4) {
        ld_row_f32<S>(reinterpret_cast<const float*>(p), v);
    } else {
        ld_row_bf16<S>(reinterpret_cast<const __nv_bfloat16*>(p), v);
    }
}

// ---------------------------------------------------------------- activations
// softplus(x) = log(1 + e^x); above 20 the correction log1p(e^-x) < 2.1e-9 is
// below f32 resolution of x and x itself is returned.
__device__ __forceinline__ float softplus_f(float x) { return x > 20.f ? x : log1pf(expf(x)); }
__device__ __forceinline__ float sigmoid_f(float x) { return 1.f / (1.f + expf(-x)); }

// Sum of v over the G adjacent lanes of a channel (xor butterfly; every lane
// ends with the same, order-fixed sum).
template <int G> __device__ __forceinline__ float group_sum(float v) {
#pragma unroll
    for (int m = 1; m < G; m <<= 1) v += __shfl_xor_sync(kFull, v, m);
    return v;
}

}  // namespace ss
