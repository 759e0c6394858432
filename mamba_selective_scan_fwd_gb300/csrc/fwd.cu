// Forward selective scan (baracuda-kernels `selective_scan.rs`, module doc
// "Algorithm summary"):
//
//   delta_eff = softplus?(delta + bias);  a = exp(delta_eff * A[d,n]);
//   h = a * h + delta_eff * B[t,n] * u;   y = (sum_n h * C[t,n] + D * u) * silu(z)
//
// The time axis is cut into K chunks (K = 1 whenever batch x channels alone
// fill the GPU).  A chunk summary (P, H) -- the product of a over the chunk
// and the chunk's end state started from zero -- combines associatively:
// state_after = P * state_before + H.  k_fwd_summary writes the summaries of
// chunks 0..K-2; k_fwd_main folds those before its chunk into the carry-in
// state and walks its chunk writing y.
#include "common.cuh"
#include "kernels.h"

namespace ss {

template <typename T, int S, int G>
__global__ void __launch_bounds__(kThreads) k_fwd_summary(FwdArgs a, Plan p, int64_t k_lo, int64_t k_hi) {
    constexpr int CH = kThreads / G;
    const int tid = threadIdx.x;
    const int ch = tid / G, g = tid % G;
    int64_t blk = blockIdx.x;
    const int64_t tile = blk % p.tiles;
    blk /= p.tiles;
    const int64_t nk = k_hi - k_lo;
    const int64_t k = k_lo + blk % nk;
    const int64_t b = blk / nk;
    const int64_t d_raw = tile * CH + ch;
    const bool valid = d_raw < a.Dch;
    const int64_t d = valid ? d_raw : a.Dch - 1;
    const int n0 = g * S;
    const T* u = static_cast<const T*>(a.u);
    const T* delta = static_cast<const T*>(a.delta);
    const T* Bm = static_cast<const T*>(a.B);

    float A2[S];
#pragma unroll
    for (int s = 0; s < S; s++) A2[s] = a.A[d * a.N + n0 + s] * kLog2e;
    const float bias = a.delta_bias ? a.delta_bias[d] : 0.f;

    float h[S], P[S];
#pragma unroll
    for (int s = 0; s < S; s++) { h[s] = 0.f; P[s] = 1.f; }
    const int64_t t0 = k * p.Lc;
    const int64_t t1 = t0 + p.Lc < a.L ? t0 + p.Lc : a.L;
    for (int64_t t = t0; t < t1; t++) {
        const int64_t idx = (b * a.L + t) * a.Dch + d;
        float dl = ld(delta + idx) + bias;
        if (a.softplus) dl = softplus_f(dl);
        const float du = dl * ld(u + idx);
        float Bv[S];
        ld_row<T, S>(Bm + (b * a.L + t) * a.N + n0, Bv);
#pragma unroll
        for (int s = 0; s < S; s++) {
            const float da = exp2f(dl * A2[s]);
            h[s] = fmaf(da, h[s], du * Bv[s]);
            P[s] *= da;
        }
    }
    if (valid) {
        float2* out = reinterpret_cast<float2*>(a.ws_fsum) + ((b * a.Dch + d) * p.K + k) * a.N + n0;
#pragma unroll
        for (int s = 0; s < S; s++) out[s] = make_float2(P[s], h[s]);
    }
}

template <typename T, int S, int G>
__global__ void __launch_bounds__(kThreads) k_fwd_main(FwdArgs a, Plan p) {
    constexpr int CH = kThreads / G;
    const int tid = threadIdx.x;
    const int ch = tid / G, g = tid % G;
    int64_t blk = blockIdx.x;
    const int64_t tile = blk % p.tiles;
    blk /= p.tiles;
    const int64_t k = blk % p.K;
    const int64_t b = blk / p.K;
    const int64_t d_raw = tile * CH + ch;
    const bool valid = d_raw < a.Dch;
    const int64_t d = valid ? d_raw : a.Dch - 1;
    const int n0 = g * S;
    const T* u = static_cast<const T*>(a.u);
    const T* delta = static_cast<const T*>(a.delta);
    const T* Bm = static_cast<const T*>(a.B);
    const T* Cm = static_cast<const T*>(a.C);
    const T* z = static_cast<const T*>(a.z);
    T* y = static_cast<T*>(a.y);

    float A2[S];
#pragma unroll
    for (int s = 0; s < S; s++) A2[s] = a.A[d * a.N + n0 + s] * kLog2e;
    const float bias = a.delta_bias ? a.delta_bias[d] : 0.f;
    const float Dd = a.D ? a.D[d] : 0.f;

    float h[S];
#pragma unroll
    for (int s = 0; s < S; s++) h[s] = 0.f;
    if (k > 0) {
        const float2* sm = reinterpret_cast<const float2*>(a.ws_fsum) + (b * a.Dch + d) * p.K * a.N + n0;
        for (int64_t j = 0; j < k; j++) {
#pragma unroll
            for (int s = 0; s < S; s++) {
                const float2 ph = sm[j * a.N + s];
                h[s] = fmaf(ph.x, h[s], ph.y);
            }
        }
    }
    const int64_t t0 = k * p.Lc;
    const int64_t t1 = t0 + p.Lc < a.L ? t0 + p.Lc : a.L;
    for (int64_t t = t0; t < t1; t++) {
        const int64_t idx = (b * a.L + t) * a.Dch + d;
        float dl = ld(delta + idx) + bias;
        if (a.softplus) dl = softplus_f(dl);
        const float uu = ld(u + idx);
        const float du = dl * uu;
        float Bv[S], Cv[S];
        ld_row<T, S>(Bm + (b * a.L + t) * a.N + n0, Bv);
        ld_row<T, S>(Cm + (b * a.L + t) * a.N + n0, Cv);
        float acc = 0.f;
#pragma unroll
        for (int s = 0; s < S; s++) {
            const float da = exp2f(dl * A2[s]);
            h[s] = fmaf(da, h[s], du * Bv[s]);
            acc = fmaf(h[s], Cv[s], acc);
        }
        acc = group_sum<G>(acc);
        if (g == 0 && valid) {
            float yv = fmaf(Dd, uu, acc);
            if (z) {
                const float zz = ld(z + idx);
                yv *= zz * sigmoid_f(zz);
            }
            st(y + idx, yv);
        }
    }
    if (k == p.K - 1 && a.last_state && valid) {
#pragma unroll
        for (int s = 0; s < S; s++) a.last_state[(b * a.Dch + d) * a.N + n0 + s] = h[s];
    }
}

template <typename T, int S, int G>
cudaError_t launch_fwd_t(const FwdArgs& a, const Plan& p, cudaStream_t st) {
    if (p.K > 1) {
        const int64_t blocks = p.tiles * a.Bsz * (p.K - 1);
        k_fwd_summary<T, S, G><<<(unsigned)blocks, kThreads, 0, st>>>(a, p, 0, p.K - 1);
    }
    const int64_t blocks = p.tiles * a.Bsz * p.K;
    k_fwd_main<T, S, G><<<(unsigned)blocks, kThreads, 0, st>>>(a, p);
    return cudaGetLastError();
}

// The backward reuses the summary kernel over all K chunks.
template <typename T, int S, int G>
cudaError_t launch_fwd_summary_t(const FwdArgs& a, const Plan& p, cudaStream_t st) {
    const int64_t blocks = p.tiles * a.Bsz * p.K;
    k_fwd_summary<T, S, G><<<(unsigned)blocks, kThreads, 0, st>>>(a, p, 0, p.K);
    return cudaGetLastError();
}

#define SS_DISPATCH_N(T, FN, ...)                                  \
    switch (a.N) {                                                 \
        case 1: return FN<T, 1, 1>(__VA_ARGS__);                   \
        case 2: return FN<T, 2, 1>(__VA_ARGS__);                   \
        case 4: return FN<T, 4, 1>(__VA_ARGS__);                   \
        case 8: return FN<T, 8, 1>(__VA_ARGS__);                   \
        case 16: return FN<T, 8, 2>(__VA_ARGS__);                  \
        case 32: return FN<T, 8, 4>(__VA_ARGS__);                  \
        default: return cudaErrorInvalidValue;                     \
    }

cudaError_t launch_fwd(const FwdArgs& a, const Plan& p, cudaStream_t st) {
    if (a.dtype == 0) { SS_DISPATCH_N(float, launch_fwd_t, a, p, st) }
    SS_DISPATCH_N(__nv_bfloat16, launch_fwd_t, a, p, st)
}

cudaError_t launch_fwd_summary(const FwdArgs& a, const Plan& p, cudaStream_t st) {
    if (a.dtype == 0) { SS_DISPATCH_N(float, launch_fwd_summary_t, a, p, st) }
    SS_DISPATCH_N(__nv_bfloat16, launch_fwd_summary_t, a, p, st)
}

}  // namespace ss
