// One recurrence step for autoregressive decoding: the selective scan of
// baracuda-kernels `selective_scan.rs` ("Algorithm summary") for a single
// time step, continuing from a state held between calls (the per-layer SSM
// state mamba-rs keeps for inference), updated in place:
//
//   delta_eff = softplus?(delta + bias);  h[n] = exp(delta_eff * A[d,n]) * h[n] + delta_eff * B[n] * u
//   y = (sum_n h[n] * C[n] + D * u) * silu(z)
//
// The step reads and rewrites the whole [Bsz, Dch, N] state, so it is bound
// by HBM: a thread owns S (up to 16) consecutive states of one channel, moved
// as 16-byte vectors, G = N / S adjacent threads share a channel and combine
// their readouts with shuffles, and a warp covers a contiguous run of the
// state.  The state is touched once per step: its loads and stores are
// streaming (evict-first) accesses.
#include "common.cuh"
#include "kernels.h"
#include "simd.cuh"
#include "tiles.cuh"

namespace ss {

template <int N>
struct DCfg {
    static constexpr int S = N >= 16 ? 16 : N;  // states per thread
    static constexpr int G = N / S;           // threads per channel
};

template <typename T>
__device__ __forceinline__ float ld_io(const T* p, int64_t i) {
    if constexpr (sizeof(T) == 4) {
        return __ldg(reinterpret_cast<const float*>(p) + i);
    } else if constexpr (std::is_same<T, __half>::value) {
        return __half2float(__ushort_as_half(__ldg(reinterpret_cast<const unsigned short*>(p) + i)));
    } else {
        return __uint_as_float((uint32_t)__ldg(reinterpret_cast<const unsigned short*>(p) + i) << 16);
    }
}

template <typename T, int N>
__global__ void __launch_bounds__(256) k_decode(DecodeArgs a) {
    constexpr int S = DCfg<N>::S, G = DCfg<N>::G;
    const int64_t gid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t rows = a.Bsz * a.Dch;
    // every thread of a warp takes part in the shuffles; threads past the end
    // work on a clamped channel and store nothing
    const bool live = gid < rows * G;
    const int64_t row = live ? gid / G : rows - 1;  // b * Dch + d
    const int g = (int)(gid % G);
    const int64_t b = row / a.Dch, d = row % a.Dch;
    const int n0 = g * S;
    const T* u = static_cast<const T*>(a.u);
    const T* delta = static_cast<const T*>(a.delta);
    const T* Bm = static_cast<const T*>(a.B);
    const T* Cm = static_cast<const T*>(a.C);
    const T* z = static_cast<const T*>(a.z);

    const float uu = ld_io(u, row);
    float x = ld_io(delta, row);
    if (a.delta_bias) x += a.delta_bias[d];
    const float dl = a.softplus ? softplus_fast(x) : x;
    float h[S], Av[S], Bv[S], Cv[S];
    if constexpr (S % 4 == 0) {
#pragma unroll
        for (int q = 0; q < S; q += 4) {
            const float4 hv = __ldcs(reinterpret_cast<const float4*>(a.state + row * N + n0 + q));
            const float4 av = __ldg(reinterpret_cast<const float4*>(a.A + d * N + n0 + q));
            h[q] = hv.x; h[q + 1] = hv.y; h[q + 2] = hv.z; h[q + 3] = hv.w;
            Av[q] = av.x; Av[q + 1] = av.y; Av[q + 2] = av.z; Av[q + 3] = av.w;
        }
        // B and C values of the thread's states: S io elements each, naturally aligned
        constexpr int BW = S * (int)sizeof(T) / 4;
        uint32_t wb[BW], wc[BW];
        load_words<S * (int)sizeof(T), BW>(Bm + b * N + n0, wb);
        load_words<S * (int)sizeof(T), BW>(Cm + b * N + n0, wc);
#pragma unroll
        for (int s = 0; s < S; s++) {
            Bv[s] = elem<T>(wb, s);
            Cv[s] = elem<T>(wc, s);
        }
    } else {
#pragma unroll
        for (int s = 0; s < S; s++) {
            h[s] = a.state[row * N + n0 + s];
            Av[s] = __ldg(a.A + d * N + n0 + s);
            Bv[s] = ld_io(Bm, b * N + n0 + s);
            Cv[s] = ld_io(Cm, b * N + n0 + s);
        }
    }
    float yp = 0.f;
#pragma unroll
    for (int s = 0; s < S; s++) {
        const float A = a.a_is_log ? -expf(Av[s]) : Av[s];
        const float dA = ex2a(dl * A * kLog2eF);
        h[s] = fmaf(dA, h[s], dl * Bv[s] * uu);
        yp = fmaf(Cv[s], h[s], yp);
    }
    // readout summed over the G threads of the channel, in a fixed order
#pragma unroll
    for (int m = 1; m < G; m <<= 1) yp += __shfl_xor_sync(kFull, yp, m);
    if (!live) return;
    if constexpr (S % 4 == 0) {
#pragma unroll
        for (int q = 0; q < S; q += 4)
            __stcs(reinterpret_cast<float4*>(a.state + row * N + n0 + q), make_float4(h[q], h[q + 1], h[q + 2], h[q + 3]));
    } else {
#pragma unroll
        for (int s = 0; s < S; s++) a.state[row * N + n0 + s] = h[s];
    }
    if (g == 0) {
        float yv = yp + (a.D ? a.D[d] * uu : 0.f);
        if (z) {
            const float zz = ld_io(z, row);
            yv *= zz * sigmoid_fast(zz);
        }
        st(static_cast<T*>(a.y) + row, yv);
    }
}

template <typename T, int N>
cudaError_t launch_decode_t(const DecodeArgs& a, cudaStream_t st) {
    const int64_t threads = a.Bsz * a.Dch * DCfg<N>::G;
    prof_mark(st);
    k_decode<T, N><<<(unsigned)ceil_div(threads, 256), 256, 0, st>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t st) {
#define SS_DEC_N(T)                                          \
    switch (a.N) {                                           \
        case 1: return launch_decode_t<T, 1>(a, st);         \
        case 2: return launch_decode_t<T, 2>(a, st);         \
        case 4: return launch_decode_t<T, 4>(a, st);         \
        case 8: return launch_decode_t<T, 8>(a, st);         \
        case 16: return launch_decode_t<T, 16>(a, st);       \
        case 32: return launch_decode_t<T, 32>(a, st);       \
        default: return cudaErrorInvalidValue;               \
    }
    if (a.dtype == 0) { SS_DEC_N(float) }
    if (a.dtype == 1) { SS_DEC_N(__half) }
    SS_DEC_N(__nv_bfloat16)
#undef SS_DEC_N
}

}  // namespace ss
