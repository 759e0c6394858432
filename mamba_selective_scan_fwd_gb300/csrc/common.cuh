// Shared device helpers of the sm_103a selective scan.
//
// Thread layout used by every scan kernel: a warp covers CH = 32 / G channels
// of one batch row and one time chunk; the G adjacent lanes of a channel each
// own S = N / G of its states (S <= 8), so the N-state recurrence of a channel
// lives in registers across G lanes.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace ss {

constexpr unsigned kFull = 0xffffffffu;

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// ---------------------------------------------------------------- element I/O

template <typename T> __device__ __forceinline__ void st(T* p, float v);
template <> __device__ __forceinline__ void st<float>(float* p, float v) { *p = v; }
template <> __device__ __forceinline__ void st<__nv_bfloat16>(__nv_bfloat16* p, float v) {
    *p = __float2bfloat16_rn(v);
}
template <> __device__ __forceinline__ void st<__half>(__half* p, float v) { *p = __float2half_rn(v); }

}  // namespace ss
