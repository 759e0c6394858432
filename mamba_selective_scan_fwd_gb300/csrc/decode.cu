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
// streaming (evict-first) accesses.  For N = 16 and at least 256 channels a
// channel-major form (k_decode_cm below) keeps each channel's A in registers
// across batch rows and shares each row's B / C through uniform loads, which
// leaves the L1 data pipe to the state (about 82 % of the HBM copy bandwidth
// at Bsz = 512, D = 5120, against 69 % for the row-major form).
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

// NW 32-bit words (a multiple of 4) at p, an address common to the whole warp,
// through the uniform load path (PTX ldu).
template <int NW>
__device__ __forceinline__ void ldu_words(const void* p, uint32_t (&w)[NW]) {
#pragma unroll
    for (int v = 0; v < NW / 4; v++) {
        asm volatile("ldu.global.v4.u32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(w[4 * v]), "=r"(w[4 * v + 1]), "=r"(w[4 * v + 2]), "=r"(w[4 * v + 3])
                     : "l"(static_cast<const uint4*>(p) + v));
    }
}

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

// Channel-major form for N = 16 (all of a channel's states in one thread): a
// block of 256 threads takes 256 consecutive channels and `rows` consecutive
// batch rows, the rows per block chosen so that the grid is one wave of
// resident blocks.  A thread keeps its channel's A, D and bias in registers across
// the rows, the block's threads share each row's B and C (one uniform load for
// the warp), and the next row's state and per-(b, d) inputs are loaded while
// the current row computes.  Per row the shared-memory / L1 data pipe then
// carries little more than the state itself, which the row-major form above
// shares with A, B and C loads per thread.
template <typename T>
constexpr int dec_cm_blocks_per_sm() { return sizeof(T) == 4 ? 2 : 3; }

template <typename T>
__global__ void __launch_bounds__(256, dec_cm_blocks_per_sm<T>()) k_decode_cm(DecodeArgs a, int rows) {
    constexpr int N = 16;
    const int64_t d = (int64_t)blockIdx.x * 256 + threadIdx.x;
    // batch rows fit in 32 bits (the C ABI caps Bsz at 2^20)
    const int b0 = (int)blockIdx.y * rows;
    const int b1 = b0 + rows < (int)a.Bsz ? b0 + rows : (int)a.Bsz;
    const bool live = d < a.Dch;
    const int64_t dc = live ? d : a.Dch - 1;  // lanes past Dch compute on a clamped channel and store nothing
    const T* u = static_cast<const T*>(a.u);
    const T* delta = static_cast<const T*>(a.delta);
    const T* Bm = static_cast<const T*>(a.B);
    const T* Cm = static_cast<const T*>(a.C);
    const T* z = static_cast<const T*>(a.z);
    float A2[N];
#pragma unroll
    for (int q = 0; q < N; q += 4) {
        const float4 av = __ldg(reinterpret_cast<const float4*>(a.A + dc * N + q));
        const float v[4] = {av.x, av.y, av.z, av.w};
#pragma unroll
        for (int k = 0; k < 4; k++) A2[q + k] = (a.a_is_log ? -expf(v[k]) : v[k]) * kLog2eF;
    }
    const float bias = a.delta_bias ? a.delta_bias[dc] : 0.f;
    const float Dv = a.D ? a.D[dc] : 0.f;
    constexpr int BW = N * (int)sizeof(T) / 4;

    // row b's inputs: state (16 floats), u, delta, z
    float h[N], hn[N];
    float uu = 0.f, xd = 0.f, zz = 0.f, un = 0.f, xn = 0.f, zn = 0.f;
    auto load = [&](int b, float (&hs)[N], float& uo, float& xo, float& zo) {
        const int64_t row = b * a.Dch + dc;
#pragma unroll
        for (int q = 0; q < N; q += 4) {
            const float4 hv = __ldcs(reinterpret_cast<const float4*>(a.state + row * N + q));
            hs[q] = hv.x; hs[q + 1] = hv.y; hs[q + 2] = hv.z; hs[q + 3] = hv.w;
        }
        uo = ld_io(u, row);
        xo = ld_io(delta, row);
        zo = z ? ld_io(z, row) : 0.f;
    };
    if (b0 < b1) load(b0, h, uu, xd, zz);
    for (int b = b0; b < b1; b++) {
        // the next row's inputs (the last row's again after it, unused): no branch
        // splits the row's loads from its arithmetic
        load(b + 1 < b1 ? b + 1 : b, hn, un, xn, zn);
        // B and C of row b: the same words for every thread of the block
        uint32_t wb[BW], wc[BW];
        ldu_words<BW>(Bm + b * N, wb);
        ldu_words<BW>(Cm + b * N, wc);
        const float x = xd + bias;
        // softplus and the gate selected by the call's flags rather than branched on
        const float sp = softplus_fast(x);
        const float dl = a.softplus ? sp : x;
        const float dlu = dl * uu;
        float yp = 0.f;
#pragma unroll
        for (int n = 0; n < N; n++) {
            const float dA = ex2a(dl * A2[n]);
            h[n] = fmaf(dA, h[n], dlu * elem<T>(wb, n));
            yp = fmaf(elem<T>(wc, n), h[n], yp);
        }
        const float gz = zz * sigmoid_fast(zz);
        const float yv = (yp + Dv * uu) * (z ? gz : 1.f);
        if (live) {
            const int64_t row = b * a.Dch + d;
#pragma unroll
            for (int q = 0; q < N; q += 4)
                __stcs(reinterpret_cast<float4*>(a.state + row * N + q), make_float4(h[q], h[q + 1], h[q + 2], h[q + 3]));
            st(static_cast<T*>(a.y) + row, yv);
        }
#pragma unroll
        for (int n = 0; n < N; n++) h[n] = hn[n];
        uu = un; xd = xn; zz = zn;
    }
}

template <typename T, int N>
cudaError_t launch_decode_t(const DecodeArgs& a, cudaStream_t st) {
    prof_mark(st);
    if constexpr (N == 16) {
        if (a.Dch >= 256) {
            // one wave: as many row blocks per channel block as the resident blocks allow
            int dev = 0, sms = 0;
            if (cudaGetDevice(&dev) != cudaSuccess ||
                cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
                return cudaErrorInvalidValue;
            const int64_t gx = ceil_div(a.Dch, 256);
            int64_t gy = (int64_t)sms * dec_cm_blocks_per_sm<T>() / gx;
            gy = gy < 1 ? 1 : (gy > a.Bsz ? a.Bsz : gy);
            const int64_t rows = ceil_div(a.Bsz, gy);
            const dim3 grid((unsigned)gx, (unsigned)ceil_div(a.Bsz, rows));
            k_decode_cm<T><<<grid, 256, 0, st>>>(a, (int)rows);
            return cudaGetLastError();
        }
    }
    const int64_t threads = a.Bsz * a.Dch * DCfg<N>::G;
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
