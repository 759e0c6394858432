// Backward selective scan: the chain rule of the forward definition
// (baracuda-kernels `selective_scan.rs`, "Algorithm summary") for the loss
// sum(dy * y), structured like mamba-rs `gpu/backward.rs` -- B2 gating
// backward, B3 SSM BPTT with local gradients followed by fixed-order
// reductions, B4 softplus backward on the raw delta -- but fused into one
// pass per chunk, recomputing the states instead of storing B*D*L*N of them,
// and without atomics.
//
// Per step t (states n, channel d):
//   g       = dy * silu(z)                       dz = dy * y0 * sig(z) * (1 + z (1 - sig(z)))
//   lam_n   = g * C_n + a_{t+1,n} lam_{t+1,n}    (the "carry" a_{t+1} lam_{t+1} flows backward)
//   du      = g D + Delta sum_n lam_n B_n
//   dDelta  = sum_n A_n lam_n a_n h_{t-1,n} + u sum_n lam_n B_n,  ddelta = dDelta * sig(x) (softplus)
//   dA_n   += Delta lam_n a_n h_{t-1,n};  dB_n += lam_n Delta u;  dC_n += g h_n
//
// Chunks: the forward summaries (P, H) give each chunk's carry-in state; the
// reverse summaries M_k = a_{s_k} lam_{s_k} (lam computed with a zero
// incoming carry) combine as rho_{k-1} = M_k + P_k rho_k and give each
// chunk's carry-in adjoint.  Inside a chunk, phase 1 walks forward storing
// the state at every kTc-step sub-chunk start; phase 2 visits the sub-chunks
// backwards, recomputes a and h of the sub-chunk in registers and runs the
// adjoint.  dB/dC are reduced over a block's channels through shared memory
// and over channel tiles by a second kernel; dA/dD/ddelta_bias per
// (batch, chunk) partials are reduced by a third.  All sums run in a fixed
// order, so the result is bit-reproducible.
#include "common.cuh"
#include "kernels.h"

namespace ss {

template <typename T, int S, int G>
__global__ void __launch_bounds__(kThreads) k_bwd_rev_summary(BwdArgs a, Plan p) {
    constexpr int CH = kThreads / G;
    const FwdArgs& f = a.f;
    const int tid = threadIdx.x;
    const int ch = tid / G, g = tid % G;
    int64_t blk = blockIdx.x;
    const int64_t tile = blk % p.tiles;
    blk /= p.tiles;
    const int64_t nk = p.K - 1;
    const int64_t k = 1 + blk % nk;
    const int64_t b = blk / nk;
    const int64_t d_raw = tile * CH + ch;
    const bool valid = d_raw < f.Dch;
    const int64_t d = valid ? d_raw : f.Dch - 1;
    const int n0 = g * S;
    const T* delta = static_cast<const T*>(f.delta);
    const T* Cm = static_cast<const T*>(f.C);
    const T* z = static_cast<const T*>(f.z);
    const T* dy = static_cast<const T*>(a.dy);

    float A2[S];
#pragma unroll
    for (int s = 0; s < S; s++) A2[s] = f.A[d * f.N + n0 + s] * kLog2e;
    const float bias = f.delta_bias ? f.delta_bias[d] : 0.f;
    float carry[S];
#pragma unroll
    for (int s = 0; s < S; s++) carry[s] = 0.f;
    const int64_t t0 = k * p.Lc;
    const int64_t t1 = t0 + p.Lc < f.L ? t0 + p.Lc : f.L;
    for (int64_t t = t1 - 1; t >= t0; t--) {
        const int64_t idx = (b * f.L + t) * f.Dch + d;
        float dl = ld(delta + idx) + bias;
        if (f.softplus) dl = softplus_f(dl);
        float gg = ld(dy + idx);
        if (z) {
            const float zz = ld(z + idx);
            gg *= zz * sigmoid_f(zz);
        }
        float Cv[S];
        ld_row<T, S>(Cm + (b * f.L + t) * f.N + n0, Cv);
#pragma unroll
        for (int s = 0; s < S; s++) {
            const float lam = fmaf(gg, Cv[s], carry[s]);
            carry[s] = exp2f(dl * A2[s]) * lam;
        }
    }
    if (valid) {
        float* out = a.ws_rsum + ((b * f.Dch + d) * p.K + k) * f.N + n0;
#pragma unroll
        for (int s = 0; s < S; s++) out[s] = carry[s];
    }
}

template <typename T, int S, int G>
__global__ void __launch_bounds__(kThreads) k_bwd_main(BwdArgs a, Plan p) {
    extern __shared__ float smem[];  // [2][CH][kTc][N]: per-channel dB / dC contributions of one sub-chunk
    constexpr int CH = kThreads / G;
    const FwdArgs& f = a.f;
    const int tid = threadIdx.x;
    const int ch = tid / G, g = tid % G;
    int64_t blk = blockIdx.x;
    const int64_t tile = blk % p.tiles;
    blk /= p.tiles;
    const int64_t k = blk % p.K;
    const int64_t b = blk / p.K;
    const int64_t d_raw = tile * CH + ch;
    const bool valid = d_raw < f.Dch;
    const float vmask = valid ? 1.f : 0.f;
    const int64_t d = valid ? d_raw : f.Dch - 1;
    const int n0 = g * S;
    const int64_t N = f.N, L = f.L, Dch = f.Dch;
    const T* u = static_cast<const T*>(f.u);
    const T* delta = static_cast<const T*>(f.delta);
    const T* Bm = static_cast<const T*>(f.B);
    const T* Cm = static_cast<const T*>(f.C);
    const T* z = static_cast<const T*>(f.z);
    const T* dy = static_cast<const T*>(a.dy);

    float Av[S], A2[S];
#pragma unroll
    for (int s = 0; s < S; s++) {
        Av[s] = f.A[d * N + n0 + s];
        A2[s] = Av[s] * kLog2e;
    }
    const float bias = f.delta_bias ? f.delta_bias[d] : 0.f;
    const float Dd = f.D ? f.D[d] : 0.f;
    const int64_t row = b * Dch + d;

    // carry-in state (forward summaries of the chunks before k)
    float h[S];
#pragma unroll
    for (int s = 0; s < S; s++) h[s] = 0.f;
    if (k > 0) {
        const float2* fs = reinterpret_cast<const float2*>(f.ws_fsum) + row * p.K * N + n0;
        for (int64_t j = 0; j < k; j++) {
#pragma unroll
            for (int s = 0; s < S; s++) {
                const float2 ph = fs[j * N + s];
                h[s] = fmaf(ph.x, h[s], ph.y);
            }
        }
    }
    // carry-in adjoint (reverse summaries of the chunks after k)
    float carry[S];
#pragma unroll
    for (int s = 0; s < S; s++) carry[s] = 0.f;
    if (k + 1 < p.K) {
        const float2* fs = reinterpret_cast<const float2*>(f.ws_fsum) + row * p.K * N + n0;
        const float* rs = a.ws_rsum + row * p.K * N + n0;
        for (int64_t j = p.K - 1; j > k; j--) {
#pragma unroll
            for (int s = 0; s < S; s++) carry[s] = fmaf(fs[j * N + s].x, carry[s], rs[j * N + s]);
        }
    }

    const int64_t t0 = k * p.Lc;
    const int64_t t1 = t0 + p.Lc < L ? t0 + p.Lc : L;
    const int64_t nsub = (t1 - t0 + kTc - 1) / kTc;
    float* ck = a.ws_ckpt + ((row * G + g) * p.K + k) * p.nsub * S;

    // phase 1: forward walk, keeping the state at each sub-chunk start
    for (int64_t j = 0; j < nsub; j++) {
        if (valid) {
#pragma unroll
            for (int s = 0; s < S; s++) ck[j * S + s] = h[s];
        }
#pragma unroll
        for (int i = 0; i < kTc; i++) {
            const int64_t t = t0 + j * kTc + i;
            if (t < t1) {
                const int64_t idx = (b * L + t) * Dch + d;
                float dl = ld(delta + idx) + bias;
                if (f.softplus) dl = softplus_f(dl);
                const float du = dl * ld(u + idx);
                float Bv[S];
                ld_row<T, S>(Bm + (b * L + t) * N + n0, Bv);
#pragma unroll
                for (int s = 0; s < S; s++) h[s] = fmaf(exp2f(dl * A2[s]), h[s], du * Bv[s]);
            }
        }
    }
    __syncthreads();  // checkpoints of channel Dch-1 are re-read by the clamped lanes of this block

    float dA_acc[S];
#pragma unroll
    for (int s = 0; s < S; s++) dA_acc[s] = 0.f;
    float dD_acc = 0.f, db_acc = 0.f;
    float* sB = smem + (size_t)ch * kTc * N;
    float* sC = smem + (size_t)(CH + ch) * kTc * N;

    // phase 2: sub-chunks in reverse order
    for (int64_t j = nsub - 1; j >= 0; j--) {
        const int64_t ts = t0 + j * kTc;
        float hs[S];
#pragma unroll
        for (int s = 0; s < S; s++) hs[s] = ck[j * S + s];
        float av[kTc][S], hv[kTc][S], dlv[kTc];
        {
            float hh[S];
#pragma unroll
            for (int s = 0; s < S; s++) hh[s] = hs[s];
#pragma unroll
            for (int i = 0; i < kTc; i++) {
                const int64_t t = ts + i;
                dlv[i] = 0.f;
                if (t < t1) {
                    const int64_t idx = (b * L + t) * Dch + d;
                    float dl = ld(delta + idx) + bias;
                    if (f.softplus) dl = softplus_f(dl);
                    dlv[i] = dl;
                    const float du = dl * ld(u + idx);
                    float Bv[S];
                    ld_row<T, S>(Bm + (b * L + t) * N + n0, Bv);
#pragma unroll
                    for (int s = 0; s < S; s++) {
                        av[i][s] = exp2f(dl * A2[s]);
                        hh[s] = fmaf(av[i][s], hh[s], du * Bv[s]);
                        hv[i][s] = hh[s];
                    }
                } else {
#pragma unroll
                    for (int s = 0; s < S; s++) { av[i][s] = 0.f; hv[i][s] = hh[s]; }
                }
            }
        }
#pragma unroll
        for (int i = kTc - 1; i >= 0; i--) {
            const int64_t t = ts + i;
            if (t < t1) {
                const int64_t idx = (b * L + t) * Dch + d;
                const float uu = ld(u + idx);
                const float dyv = ld(dy + idx);
                float gg = dyv, zz = 0.f, sz = 0.f;
                if (z) {
                    zz = ld(z + idx);
                    sz = sigmoid_f(zz);
                    gg = dyv * zz * sz;
                }
                float Bv[S], Cv[S];
                ld_row<T, S>(Bm + (b * L + t) * N + n0, Bv);
                ld_row<T, S>(Cm + (b * L + t) * N + n0, Cv);
                const float dlu = dlv[i] * uu * vmask;
                const float gm = gg * vmask;
                float du_p = 0.f, dd_p = 0.f, y0_p = 0.f;
#pragma unroll
                for (int s = 0; s < S; s++) {
                    const float lam = fmaf(gg, Cv[s], carry[s]);
                    du_p = fmaf(lam, Bv[s], du_p);
                    const float hp = i > 0 ? hv[i - 1][s] : hs[s];
                    const float cn = av[i][s] * lam;
                    const float q = cn * hp;
                    dd_p = fmaf(Av[s], q, dd_p);
                    dA_acc[s] = fmaf(dlv[i], q, dA_acc[s]);
                    y0_p = fmaf(Cv[s], hv[i][s], y0_p);
                    sB[i * N + n0 + s] = lam * dlu;
                    sC[i * N + n0 + s] = gm * hv[i][s];
                    carry[s] = cn;
                }
                du_p = group_sum<G>(du_p);
                dd_p = group_sum<G>(dd_p);
                y0_p = group_sum<G>(y0_p);
                if (g == 0 && valid) {
                    a.du[idx] = fmaf(gg, Dd, dlv[i] * du_p);
                    const float dDelta = fmaf(uu, du_p, dd_p);
                    float dx = dDelta;
                    if (f.softplus) dx *= sigmoid_f(ld(delta + idx) + bias);
                    a.ddelta[idx] = dx;
                    if (z) a.dz[idx] = dyv * fmaf(Dd, uu, y0_p) * sz * fmaf(zz, 1.f - sz, 1.f);
                    dD_acc = fmaf(gg, uu, dD_acc);
                    db_acc += dx;
                }
            } else {
#pragma unroll
                for (int s = 0; s < S; s++) {
                    sB[i * N + n0 + s] = 0.f;
                    sC[i * N + n0 + s] = 0.f;
                }
            }
        }
        __syncthreads();
        // sum the block's channels for every (tensor, step, state) of this sub-chunk
        const int per = kTc * (int)N;
        for (int o = tid; o < 2 * per; o += kThreads) {
            const int tensor = o / per, r = o % per;
            const int64_t t = ts + r / N;
            if (t < t1) {
                const float* src = smem + (size_t)tensor * CH * per + r;
                float acc = 0.f;
                for (int c = 0; c < CH; c++) acc += src[(size_t)c * per];
                a.ws_bc[(((size_t)tensor * p.tiles + tile) * f.Bsz + b) * L * N + t * N + r % N] = acc;
            }
        }
        __syncthreads();
    }
    if (valid) {
        float* o = a.ws_dA + ((b * p.K + k) * Dch + d) * N + n0;
#pragma unroll
        for (int s = 0; s < S; s++) o[s] = dA_acc[s];
        if (g == 0) {
            a.ws_dD[(b * p.K + k) * Dch + d] = dD_acc;
            a.ws_db[(b * p.K + k) * Dch + d] = db_acc;
        }
    }
}

// dB / dC: sum of the per-tile partials, tiles in ascending order.
__global__ void k_bwd_reduce_bc(BwdArgs a, Plan p) {
    const int64_t bln = a.f.Bsz * a.f.L * a.f.N;
    const int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= 2 * bln) return;
    const int tensor = e >= bln ? 1 : 0;
    const int64_t r = e - tensor * bln;
    const float* src = a.ws_bc + (size_t)tensor * p.tiles * bln + r;
    float acc = 0.f;
    for (int64_t tl = 0; tl < p.tiles; tl++) acc += src[tl * bln];
    (tensor ? a.dC : a.dB)[r] = acc;
}

// dA / dD / ddelta_bias: sum over (batch, chunk) partials in ascending order.
__global__ void k_bwd_reduce_params(BwdArgs a, Plan p) {
    const int64_t Dch = a.f.Dch, N = a.f.N;
    const int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t parts = a.f.Bsz * p.K;
    if (e < Dch * N) {
        float acc = 0.f;
        for (int64_t q = 0; q < parts; q++) acc += a.ws_dA[q * Dch * N + e];
        a.dA[e] = acc;
    }
    if (e < Dch) {
        if (a.dD) {
            float acc = 0.f;
            for (int64_t q = 0; q < parts; q++) acc += a.ws_dD[q * Dch + e];
            a.dD[e] = acc;
        }
        if (a.ddelta_bias) {
            float acc = 0.f;
            for (int64_t q = 0; q < parts; q++) acc += a.ws_db[q * Dch + e];
            a.ddelta_bias[e] = acc;
        }
    }
}

template <typename T, int S, int G>
cudaError_t launch_bwd_t(const BwdArgs& a, const Plan& p, cudaStream_t st) {
    constexpr int CH = kThreads / G;
    constexpr size_t kSmemMax = 2 * (size_t)CH * kTc * (S * G) * sizeof(float);
    const size_t smem = 2 * (size_t)CH * kTc * a.f.N * sizeof(float);
    // the attribute is per function and current device; setting it again is harmless
    cudaError_t attr = cudaFuncSetAttribute(k_bwd_main<T, S, G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                            (int)kSmemMax);
    if (attr != cudaSuccess) return attr;
    if (p.K > 1) {
        cudaError_t e = launch_fwd_summary(a.f, p, st);
        if (e != cudaSuccess) return e;
        const int64_t blocks = p.tiles * a.f.Bsz * (p.K - 1);
        k_bwd_rev_summary<T, S, G><<<(unsigned)blocks, kThreads, 0, st>>>(a, p);
    }
    const int64_t blocks = p.tiles * a.f.Bsz * p.K;
    k_bwd_main<T, S, G><<<(unsigned)blocks, kThreads, smem, st>>>(a, p);
    const int64_t n_bc = 2 * a.f.Bsz * a.f.L * a.f.N;
    k_bwd_reduce_bc<<<(unsigned)ceil_div(n_bc, 256), 256, 0, st>>>(a, p);
    const int64_t n_par = a.f.Dch * a.f.N;
    k_bwd_reduce_params<<<(unsigned)ceil_div(n_par, 256), 256, 0, st>>>(a, p);
    return cudaGetLastError();
}

#define SS_DISPATCH_N(T, FN, ...)                                  \
    switch (a.f.N) {                                               \
        case 1: return FN<T, 1, 1>(__VA_ARGS__);                   \
        case 2: return FN<T, 2, 1>(__VA_ARGS__);                   \
        case 4: return FN<T, 4, 1>(__VA_ARGS__);                   \
        case 8: return FN<T, 8, 1>(__VA_ARGS__);                   \
        case 16: return FN<T, 8, 2>(__VA_ARGS__);                  \
        case 32: return FN<T, 8, 4>(__VA_ARGS__);                  \
        default: return cudaErrorInvalidValue;                     \
    }

cudaError_t launch_bwd(const BwdArgs& a, const Plan& p, cudaStream_t st) {
    if (a.f.dtype == 0) { SS_DISPATCH_N(float, launch_bwd_t, a, p, st) }
    SS_DISPATCH_N(__nv_bfloat16, launch_bwd_t, a, p, st)
}

}  // namespace ss
