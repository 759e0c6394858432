// Reverse chunk summaries of the backward, for units the plan cuts in time.
//
// For chunk k of a unit (k >= 1) the summary is the pair (sum of delta_eff
// over the chunk, M_k), M_k being the adjoint carry the chunk passes back
// from a zero incoming carry:
//   carry <- 0;  for t from the chunk's last step down to its first:
//       lam_n = g_t C_{t,n} + carry_n,   carry_n <- a_{t,n} lam_n,
// with a_{t,n} = exp(delta_eff_t A_n) and g = dy silu(z) (dy without z).
// The backward's main pass combines them as rho_{k-1} = M_k + P_k rho_k with
// P_k = exp(A sum delta_eff).  This is the first factor of the chain rule of
// the forward definition (baracuda-kernels `selective_scan.rs`, "Algorithm
// summary"; the recurrence of mamba-rs `gpu/backward.rs`, B3), restricted to
// the adjoint of the state.
//
// The walk is light (one exponential and two packed f32x2 operations per
// state pair and step) next to its per-(t, d) terms, so this kernel stages
// 32-step tiles (the forward's boxes), one tile ahead, with one block barrier
// per tile: the tile's per-(t, d) terms (delta_eff, g) go to a shared-memory
// buffer of their own by tile parity, and C is read in its io type straight
// from the tile's buffer.  The sum of delta_eff is formed by the prologue
// threads over their own items, then added across them in a fixed order.
// Block and lane layout are the backward main kernel's (BCfg): the summary
// entries land where the main pass reads them.
#pragma once

#include "common.cuh"
#include "kernels.h"
#include "simd.cuh"
#include "tiles.cuh"

namespace ss {

constexpr int kRsTT = kFwdRows;  // steps per tile of the reverse summary

template <typename T, int N>
struct RCfg {
    using B = BCfg<T, N>;
    static constexpr int NW = B::NW, NPW = B::NPW, S = B::S, SP = B::SP, G = B::G, PAIRS = B::PAIRS, CH = B::CH,
                         THREADS = B::THREADS, ESZ = B::ESZ;
    static constexpr int GRP = 8;                        // channels per prologue item
    static constexpr int NGRP = CH / GRP;                // items per step
    static constexpr int ITEMS = kRsTT * NGRP / THREADS; // items per thread per tile
    static constexpr int RW = GRP * ESZ / 4;             // 32-bit words of an item's run
    static_assert(kRsTT * NGRP % THREADS == 0, "whole items per thread");
    static_assert(THREADS % NGRP == 0, "a thread's items share one channel group");
};

// S consecutive io values of a B / C row in shared memory as f32.
template <typename T, int S>
__device__ __forceinline__ void ld_row(const T* p, float (&v)[S]) {
    if constexpr (std::is_same<T, __nv_bfloat16>::value && S == 4) {
        ld_bf16x4(p, v);
    } else if constexpr (sizeof(T) == 4) {
        ld_f32<S>(reinterpret_cast<const float*>(p), v);
    } else {
#pragma unroll
        for (int s = 0; s < S; s++) {
            if constexpr (std::is_same<T, __half>::value) v[s] = __half2float(p[s]);
            else v[s] = __bfloat162float(p[s]);
        }
    }
}

template <typename T, int N>
__global__ void __launch_bounds__(32 * scan_warps(N), 6) k_bwd_rsum(BwdArgs a, FPlan p, int si, int64_t k_lo,
                                                               const __grid_constant__ TmaMaps maps) {
    using C = RCfg<T, N>;
    constexpr int NPW = C::NPW, S = C::S, SP = C::SP, G = C::G, PAIRS = C::PAIRS, CH = C::CH,
                  THREADS = C::THREADS, GRP = C::GRP, NGRP = C::NGRP, ITEMS = C::ITEMS, RW = C::RW;
    // raw runs of delta, dy, z and the C rows of a tile, double buffered (a TMA
    // box each, or loaded by the prologue)
    __shared__ __align__(128) T sRaw[2][3][kRsTT][CH];
    __shared__ __align__(128) T sC[2][kRsTT][N];
    // (delta_eff of both channels, g of both channels) per step and channel pair,
    // double buffered by tile
    __shared__ float4 sDG[2][kRsTT][PAIRS];
    __shared__ __align__(8) uint64_t sBar[2];
    __shared__ float sBias[CH];
    // per-thread sums of delta_eff over its items (GRP channels), added at the end
    __shared__ float sSD[THREADS][GRP + 1];

    const FwdArgs& f = a.f;
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const Seg sgm = seg_at(p, si);
    const int64_t ul = (int64_t)blockIdx.x % sgm.nu;
    const int64_t k = k_lo + (int64_t)blockIdx.x / sgm.nu;
    const int64_t unit = sgm.u_lo + ul;
    const int64_t tile = unit % p.tiles_b, b = unit / p.tiles_b;
    const int64_t qs = sgm.s0 + ul * sgm.K + k;  // summary index
    const int64_t L = f.L, Dch = f.Dch;
    const int64_t d0 = tile * CH;
    const T* delta = static_cast<const T*>(f.delta);
    const T* z = static_cast<const T*>(f.z);
    const T* dy = static_cast<const T*>(a.dy);
    const T* Cm = static_cast<const T*>(f.C);

    for (int c = tid; c < CH; c += THREADS) {
        const int64_t dc = d0 + c < Dch ? d0 + c : Dch - 1;
        sBias[c] = f.delta_bias ? f.delta_bias[dc] : 0.f;
    }
    const int pp = lane / G, g = lane % G;
    const int c0 = 2 * pp;
    const int n0 = w * NPW + g * S;
    const bool okc[2] = {d0 + c0 < Dch, d0 + c0 + 1 < Dch};
    const int64_t dd[2] = {okc[0] ? d0 + c0 : Dch - 1, okc[1] ? d0 + c0 + 1 : Dch - 1};
    // A2 = A log2(e) of the lane's state pairs; channels past Dch run with a zero
    // exponent and, with dy = 0 there, keep a zero carry
    float2 A2[2][SP], carry[2][SP];
#pragma unroll
    for (int e = 0; e < 2; e++) {
#pragma unroll
        for (int j = 0; j < SP; j++) {
            const int s0 = 2 * j, s1 = S >= 2 ? 2 * j + 1 : 0;
            A2[e][j] = make_float2(okc[e] ? scan_A(f, dd[e] * N + n0 + s0) * kLog2eF : 0.f,
                                   okc[e] && S >= 2 ? scan_A(f, dd[e] * N + n0 + s1) * kLog2eF : 0.f);
            carry[e][j] = make_float2(0.f, 0.f);
        }
    }
    float sdp[GRP];  // this thread's sums of delta_eff, channels cg .. cg + GRP of its items
#pragma unroll
    for (int c = 0; c < GRP; c++) sdp[c] = 0.f;

    bool tma = f.use_tma != 0;
    if (tma && !(smem_aligned128(&sRaw[0][0][0][0]) && smem_aligned128(&sC[0][0][0]))) {
        if (tid == 0) atomicOr(f.status, kDevMisaligned);
        tma = false;
    }
    // per-thread loads of whole aligned runs (else element loads, zero past Dch)
    const bool vfast = ((Dch * (int64_t)sizeof(T)) % 16 == 0) && (d0 + CH <= Dch);
    const int64_t t_begin = k * sgm.Lc;
    const int64_t t_end = t_begin + sgm.Lc < L ? t_begin + sgm.Lc : L;
    const int64_t ntile = (t_end - t_begin + kRsTT - 1) / kRsTT;

    // TMA copies of tile mm into buffer mm & 1: delta, dy, z as [32][CH], C as [32][N]
    const TmaMaps& mp = maps;
    auto issue = [&](int64_t mm) {
        if (!tma || tid != 0) return;
        const int buf = (int)(mm & 1);
        constexpr uint32_t run = kRsTT * CH * C::ESZ, row = kRsTT * N * C::ESZ;
        mbar_expect_tx(&sBar[buf], (z ? 3 : 2) * run + row);
        const int x = (int)d0, y = (int)(t_begin + mm * kRsTT), zc = (int)b;
        tma_load_3d(&sRaw[buf][0][0][0], &mp.m[kMapDelta], x, y, zc, &sBar[buf]);
        tma_load_3d(&sRaw[buf][1][0][0], &mp.m[kMapDy], x, y, zc, &sBar[buf]);
        if (z) tma_load_3d(&sRaw[buf][2][0][0], &mp.m[kMapZ], x, y, zc, &sBar[buf]);
        tma_load_3d(&sC[buf][0][0], &mp.m[kMapC], 0, y, zc, &sBar[buf]);
    };
    if (tma && tid == 0) {
        mbar_init(&sBar[0], 1);
        mbar_init(&sBar[1], 1);
        fence_proxy_async_smem();
    }
    issue(ntile - 1);
    __syncthreads();  // sBias and the barriers
    // the thread's items cover the same channel group in every tile: its biases
    // stay in registers
    const int cg = (tid % NGRP) * GRP;
    float biasv[GRP];
#pragma unroll
    for (int c = 0; c < GRP; c++) biasv[c] = sBias[cg + c];

    for (int64_t m = ntile - 1; m >= 0; m--) {
        const int64_t t0 = t_begin + m * kRsTT;
        const int buf = (int)(m & 1);
        // tile m is the use (ntile - 1 - m) / 2 of its buffer: that phase's parity
        const uint32_t phase = (uint32_t)(((ntile - 1 - m) >> 1) & 1);
        bool ok = true;
        if (tma) ok = mbar_wait(&sBar[buf], phase);
        // ---- prologue: (step, GRP-channel group) items; steps past t_end get
        // delta_eff = g = 0, which leave the carry unchanged.  All of the items'
        // loads come first, then their arithmetic (no branch on the row's
        // validity: selects zero the rows past t_end, whose shared-memory runs
        // hold finite data -- TMA zero fill past the tensor, the next chunk
        // before it), then the stores: with no store between them, the items'
        // dependency chains interleave.
        uint32_t rd[ITEMS][RW], rg[ITEMS][RW], rz[ITEMS][RW];
#pragma unroll
        for (int it = 0; it < ITEMS; it++) {
            const int r = (tid + it * THREADS) / NGRP;
            const int64_t t = t0 + r;
#pragma unroll
            for (int v = 0; v < RW; v++) rd[it][v] = rg[it][v] = rz[it][v] = 0u;
            if (tma) {
                lds_words<GRP * C::ESZ, RW>(&sRaw[buf][0][r][cg], rd[it]);
                lds_words<GRP * C::ESZ, RW>(&sRaw[buf][1][r][cg], rg[it]);
                if (z) lds_words<GRP * C::ESZ, RW>(&sRaw[buf][2][r][cg], rz[it]);
            } else if (t < t_end) {
                const int64_t off = (b * L + t) * Dch + d0 + cg;
                load_run<T, GRP, RW>(delta, off, d0 + cg, Dch, vfast, rd[it]);
                load_run<T, GRP, RW>(dy, off, d0 + cg, Dch, vfast, rg[it]);
                if (z) load_run<T, GRP, RW>(z, off, d0 + cg, Dch, vfast, rz[it]);
            }
        }
        float4 dv[ITEMS][GRP / 2];
#pragma unroll
        for (int it = 0; it < ITEMS; it++) {
            const bool rv = t0 + (tid + it * THREADS) / NGRP < t_end;
#pragma unroll
            for (int c = 0; c < GRP; c += 2) {
                const float2 x = make_float2(elem<T>(rd[it], c) + biasv[c], elem<T>(rd[it], c + 1) + biasv[c + 1]);
                // selected by the call's flags rather than branched on (without z the run
                // rz holds zeros)
                const float2 spf = softplus2(x);
                const float2 sp = f.softplus ? spf : x;
                const float2 dyv = make_float2(elem<T>(rg[it], c), elem<T>(rg[it], c + 1));
                const float2 zz = make_float2(elem<T>(rz[it], c), elem<T>(rz[it], c + 1));
                const float2 gz = mul2(mul2(dyv, sigmoid2(zz)), zz);
                float2 gg = z ? gz : dyv;
                const float2 dl = rv ? sp : make_float2(0.f, 0.f);
                gg = rv ? gg : make_float2(0.f, 0.f);
                sdp[c] += dl.x;
                sdp[c + 1] += dl.y;
                dv[it][c / 2] = make_float4(dl.x, dl.y, gg.x, gg.y);
            }
        }
#pragma unroll
        for (int it = 0; it < ITEMS; it++) {
            const int r = (tid + it * THREADS) / NGRP;
#pragma unroll
            for (int c = 0; c < GRP; c += 2) sDG[buf][r][(cg + c) / 2] = dv[it][c / 2];
        }
        if (!tma) {
            // the C rows of the tile, zero past t_end
            for (int id = tid; id < kRsTT * N; id += THREADS) {
                const int r = id / N, n = id % N;
                const int64_t t = t0 + r;
                sC[buf][r][n] = t < t_end ? Cm[(b * L + t) * N + n] : T(0.f);
            }
        }
        // A thread whose wait for the tile ran out makes the block give up (the
        // block agrees here): the status word records it, and the thread that
        // issued the copies waits once more for them before shared memory is
        // released.
        if (__syncthreads_or(!ok)) {
            if (tid == 0) {
                atomicOr(f.status, kDevWaitTimeout);
                mbar_wait(&sBar[buf], phase);
            }
            return;
        }
        // every thread is past the walk of tile m + 1: its buffer takes tile m - 1
        if (m > 0) issue(m - 1);
        // ---- the walk, last step first
#pragma unroll
        for (int i = kRsTT - 1; i >= 0; i--) {
            const float4 dg = sDG[buf][i][pp];
            float Cv[S];
            ld_row<T, S>(&sC[buf][i][n0], Cv);
#pragma unroll
            for (int e = 0; e < 2; e++) {
                const float2 dl = splat2(e ? dg.y : dg.x), gg = splat2(e ? dg.w : dg.z);
#pragma unroll
                for (int j = 0; j < SP; j++) {
                    const float2 Cp = make_float2(Cv[2 * j], S >= 2 ? Cv[2 * j + 1] : 0.f);
                    const float2 x = mul2(dl, A2[e][j]);
                    const float2 lam = fma2(gg, Cp, carry[e][j]);
                    carry[e][j] = mul2(make_float2(ex2a(x.x), ex2a(x.y)), lam);
                }
            }
        }
    }

    // ---- the summary: M_k of every (channel, state) (zero past Dch), and the
    // chunk's sum of delta_eff per channel: the items' partial sums added over
    // the threads of a channel group in thread order
#pragma unroll
    for (int e = 0; e < 2; e++) {
        float* M = a.ws_rsum + (qs * CH + c0 + e) * N + n0;
#pragma unroll
        for (int j = 0; j < SP; j++) {
            M[2 * j] = carry[e][j].x;
            if (S >= 2) M[2 * j + 1] = carry[e][j].y;
        }
    }
#pragma unroll
    for (int c = 0; c < GRP; c++) sSD[tid][c] = sdp[c];
    __syncthreads();
    for (int c = tid; c < CH; c += THREADS) {
        const int q = c / GRP, cc = c % GRP;
        float s = 0.f;
        for (int th = q; th < THREADS; th += NGRP) s += sSD[th][cc];
        a.ws_rsd[qs * CH + c] = s;
    }
}

}  // namespace ss
