// Forward chunk summaries, for units the plan cuts in time.
//
// For chunk k of a unit (k < K - 1) the summary is the pair (sum of delta_eff
// over the chunk, H_k), H_k being the state the chunk's steps leave from a
// zero start: h <- a_t h + delta_eff_t B_t u_t over the chunk (the recurrence
// of the forward definition, baracuda-kernels `selective_scan.rs`, "Algorithm
// summary").  The forward's main pass folds them into each chunk's carry-in
// as h <- exp(A sum delta_eff_j) h + H_j over the earlier chunks j.
//
// The scan has no readout, so per step it is one exponential pair and three
// packed f32x2 operations per state pair next to the per-(t, d) softplus of
// the prologue.  Like the reverse summaries, this kernel stages 32-step tiles
// (delta, u and B through TMA, one tile ahead) with one block barrier per
// tile: the tile's (delta_eff, delta_eff u) and its B rows (widened to f32 for
// 16-bit io) go to shared-memory buffers of their own by tile parity.  The sum of
// delta_eff is formed by the prologue threads over their own items, then
// added across them in a fixed order.  Block and lane layout are the forward
// main kernel's (FCfg), registers pairing a lane's two channels at one state,
// so the summary entries land where the main pass reads them.
#pragma once

#include "common.cuh"
#include "kernels.h"
#include "simd.cuh"
#include "tiles.cuh"

namespace ss {

constexpr int kFsTT = kFwdRows;  // steps per tile of the forward summaries

template <typename T, int N>
struct FSCfg {
    static constexpr int NW = scan_warps(N), NPW = N / NW, S = lane_states(N), G = NPW / S, PAIRS = 32 / G,
                         CH = 2 * PAIRS, THREADS = 32 * NW, ESZ = (int)sizeof(T);
    static constexpr int GRP = 8;                         // channels per prologue item
    static constexpr int NGRP = CH / GRP;                 // items per step
    static constexpr int ITEMS = kFsTT * NGRP / THREADS;  // items per thread per tile
    static constexpr int RW = GRP * ESZ / 4;              // 32-bit words of an item's run
    static constexpr int ROWS = kFsTT * N / THREADS >= 1 ? kFsTT * N / THREADS : 1;  // B values per thread
    static_assert(CH == channels_per_block(N), "channel tile of the plan");
    static_assert(kFsTT * NGRP % THREADS == 0, "whole items per thread");
    static_assert(THREADS % NGRP == 0, "a thread's items share one channel group");
    static_assert(kFsTT * N % THREADS == 0, "whole B values per thread");
};

template <typename T, int N>
__global__ void __launch_bounds__(32 * scan_warps(N), 6) k_fwd_fsum(FwdArgs a, FPlan p, int si, int64_t k_lo,
                                                                  const __grid_constant__ TmaMaps maps) {
    using C = FSCfg<T, N>;
    constexpr int NPW = C::NPW, S = C::S, G = C::G, PAIRS = C::PAIRS, CH = C::CH, THREADS = C::THREADS,
                  GRP = C::GRP, NGRP = C::NGRP, ITEMS = C::ITEMS, RW = C::RW;
    // f32 io: the scan reads B straight from the tile's buffer (no widened copy),
    // which keeps the block at 36 KB so that 6 fit on an SM
    constexpr bool DIRECT = sizeof(T) == 4;
    // raw runs of delta, u and the B rows of a tile, double buffered (a TMA box
    // each, or loaded by the prologue)
    __shared__ __align__(128) T sRaw[2][2][kFsTT][CH];
    __shared__ __align__(128) T sBr[2][kFsTT][N];
    // (delta_eff of both channels, delta_eff u of both channels) per step and
    // channel pair, and the B rows widened to f32 (16-bit io), double buffered by tile
    __shared__ float4 sDU[2][kFsTT][PAIRS];
    __shared__ __align__(16) float sB[2][DIRECT ? 1 : kFsTT][DIRECT ? 4 : N];
    __shared__ __align__(8) uint64_t sBar[2];
    __shared__ float sBias[CH];
    // per-thread sums of delta_eff over its items, added at the end: in the raw
    // runs' buffer, free by then (every thread is past its last prologue)
    static_assert(sizeof(T) * 2 * 2 * kFsTT * CH >= sizeof(float) * THREADS * (GRP + 1), "room for the sums");
    float(*sSD)[GRP + 1] = reinterpret_cast<float(*)[GRP + 1]>(&sRaw[0][0][0][0]);

    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const Seg sgm = seg_at(p, si);
    const int64_t ul = (int64_t)blockIdx.x % sgm.nu;
    const int64_t k = k_lo + (int64_t)blockIdx.x / sgm.nu;
    const int64_t unit = sgm.u_lo + ul;
    const int64_t tile = unit % p.tiles_b, b = unit / p.tiles_b;
    const int64_t q = sgm.s0 + ul * sgm.K + k;  // summary index
    const int64_t L = a.L, Dch = a.Dch;
    const int64_t d0 = tile * CH;
    const T* u = static_cast<const T*>(a.u);
    const T* delta = static_cast<const T*>(a.delta);
    const T* Bm = static_cast<const T*>(a.B);

    for (int c = tid; c < CH; c += THREADS) {
        const int64_t dc = d0 + c < Dch ? d0 + c : Dch - 1;
        sBias[c] = a.delta_bias ? a.delta_bias[dc] : 0.f;
    }
    const int pp = lane / G, g = lane % G;
    const int c0 = 2 * pp;
    const bool ok0 = d0 + c0 < Dch, ok1 = d0 + c0 + 1 < Dch;
    const int64_t dA0 = ok0 ? d0 + c0 : Dch - 1, dA1 = ok1 ? d0 + c0 + 1 : Dch - 1;
    const int n0 = w * NPW + g * S;
    // A2 = A log2(e) of the lane's states, paired across its two channels;
    // channels past Dch run with a zero exponent and, with u = 0 there, keep a
    // zero state
    float2 A2[S], h[S];
#pragma unroll
    for (int s = 0; s < S; s++) {
        A2[s] = make_float2(ok0 ? scan_A(a, dA0 * N + n0 + s) * kLog2eF : 0.f,
                            ok1 ? scan_A(a, dA1 * N + n0 + s) * kLog2eF : 0.f);
        h[s] = make_float2(0.f, 0.f);
    }
    float sdp[GRP];  // this thread's sums of delta_eff, channels cg .. cg + GRP of its items
#pragma unroll
    for (int c = 0; c < GRP; c++) sdp[c] = 0.f;

    bool tma = a.use_tma != 0;
    if (tma && !(smem_aligned128(&sRaw[0][0][0][0]) && smem_aligned128(&sBr[0][0][0]))) {
        if (tid == 0) atomicOr(a.status, kDevMisaligned);
        tma = false;
    }
    const bool vfast = ((Dch * (int64_t)sizeof(T)) % 16 == 0) && (d0 + CH <= Dch);
    const int64_t t_begin = k * sgm.Lc;
    const int64_t t_end = t_begin + sgm.Lc < L ? t_begin + sgm.Lc : L;
    const int64_t ntile = (t_end - t_begin + kFsTT - 1) / kFsTT;

    // TMA copies of tile jt into buffer jt & 1: delta, u as [32][CH], B as [32][N]
    const TmaMaps& mp = maps;
    auto issue = [&](int64_t jt) {
        if (!tma || tid != 0) return;
        const int buf = (int)(jt & 1);
        constexpr uint32_t run = kFsTT * CH * C::ESZ, row = kFsTT * N * C::ESZ;
        mbar_expect_tx(&sBar[buf], 2 * run + row);
        const int x = (int)d0, y = (int)(t_begin + jt * kFsTT), zc = (int)b;
        tma_load_3d(&sRaw[buf][0][0][0], &mp.m[kMapDelta], x, y, zc, &sBar[buf]);
        tma_load_3d(&sRaw[buf][1][0][0], &mp.m[kMapU], x, y, zc, &sBar[buf]);
        tma_load_3d(&sBr[buf][0][0], &mp.m[kMapB], 0, y, zc, &sBar[buf]);
    };
    if (tma && tid == 0) {
        mbar_init(&sBar[0], 1);
        mbar_init(&sBar[1], 1);
        fence_proxy_async_smem();
    }
    issue(0);
    __syncthreads();  // sBias and the barriers

    for (int64_t jt = 0; jt < ntile; jt++) {
        const int64_t t0 = t_begin + jt * kFsTT;
        const int buf = (int)(jt & 1);
        // tile jt is the use jt / 2 of its buffer: that phase's parity
        const uint32_t phase = (uint32_t)((jt >> 1) & 1);
        bool ok = true;
        if (tma) ok = mbar_wait(&sBar[buf], phase);
        // ---- prologue: (step, GRP-channel group) items; steps past t_end get
        // delta_eff = 0, which leaves the state unchanged
#pragma unroll
        for (int it = 0; it < ITEMS; it++) {
            const int id = tid + it * THREADS;
            const int r = id / NGRP, cg = (id % NGRP) * GRP;
            const int64_t t = t0 + r;
            const bool rv = t < t_end;
            uint32_t rd[RW], ru[RW];
            if (rv) {
                if (tma) {
                    lds_words<GRP * C::ESZ, RW>(&sRaw[buf][0][r][cg], rd);
                    lds_words<GRP * C::ESZ, RW>(&sRaw[buf][1][r][cg], ru);
                } else {
                    const int64_t off = (b * L + t) * Dch + d0 + cg;
                    load_run<T, GRP, RW>(delta, off, d0 + cg, Dch, vfast, rd);
                    load_run<T, GRP, RW>(u, off, d0 + cg, Dch, vfast, ru);
                }
            }
#pragma unroll
            for (int c = 0; c < GRP; c += 2) {
                float2 dl = make_float2(0.f, 0.f), dlu = dl;
                if (rv) {
                    const float2 x = make_float2(elem<T>(rd, c) + sBias[cg + c], elem<T>(rd, c + 1) + sBias[cg + c + 1]);
                    const float2 spf = softplus2(x);  // selected, not branched on
                    dl = a.softplus ? spf : x;
                    dlu = mul2(dl, make_float2(elem<T>(ru, c), elem<T>(ru, c + 1)));
                }
                sdp[c] += dl.x;
                sdp[c + 1] += dl.y;
                sDU[buf][r][(cg + c) / 2] = make_float4(dl.x, dl.y, dlu.x, dlu.y);
            }
        }
        // the tile's B rows as f32 (zero past t_end): widened from the TMA box, or
        // loaded; f32 rows that TMA brought in are read where they landed
        if (!DIRECT || !tma) {
#pragma unroll
            for (int v = 0; v < C::ROWS; v++) {
                const int id = tid + v * THREADS;
                const int r = id / N, n = id % N;
                const int64_t t = t0 + r;
                float bv = 0.f;
                if (t < t_end) {
                    if (tma) bv = (float)sBr[buf][r][n];
                    else bv = (float)Bm[(b * L + t) * N + n];
                }
                if constexpr (DIRECT) sBr[buf][r][n] = bv;
                else sB[buf][r][n] = bv;
            }
        }
        // A thread whose wait for the tile ran out makes the block give up (the
        // block agrees here): the status word records it, and the thread that
        // issued the copies waits once more for them before shared memory is
        // released.
        if (__syncthreads_or(!ok)) {
            if (tid == 0) {
                atomicOr(a.status, kDevWaitTimeout);
                mbar_wait(&sBar[buf], phase);
            }
            return;
        }
        // every thread is past the scan of tile jt - 1: its buffer takes tile jt + 1
        if (jt + 1 < ntile) issue(jt + 1);
        // ---- the scan: h <- a h + delta_eff u B, two channels per packed operation,
        // software-pipelined by two steps: the decays and input terms of step
        // i + 2 are formed before the recurrence of step i
        float2 daQ[2][S], xbQ[2][S];
        auto prep = [&](int i, int sl) {
            const float4 du = sDU[buf][i][pp];
            const float2 dl2 = make_float2(du.x, du.y), dlu2 = make_float2(du.z, du.w);
            float Bv[S];
            if constexpr (DIRECT) ld_f32<S>(reinterpret_cast<const float*>(&sBr[buf][i][n0]), Bv);
            else ld_f32<S>(&sB[buf][i][n0], Bv);
#pragma unroll
            for (int s = 0; s < S; s++) {
                const float2 x = mul2(dl2, A2[s]);
                daQ[sl][s] = make_float2(ex2a(x.x), ex2a(x.y));
                xbQ[sl][s] = mul2(dlu2, splat2(Bv[s]));
            }
        };
        prep(0, 0);
        prep(1, 1);
#pragma unroll
        for (int i = 0; i < kFsTT; i++) {
            const int sl = i & 1;
            float2 da[S], xb[S];
#pragma unroll
            for (int s = 0; s < S; s++) {
                da[s] = daQ[sl][s];
                xb[s] = xbQ[sl][s];
            }
            if (i + 2 < kFsTT) prep(i + 2, sl);
#pragma unroll
            for (int s = 0; s < S; s++) h[s] = fma2(da[s], h[s], xb[s]);
        }
    }

    // ---- the summary: H_k of every (channel, state) (zero past Dch), and the
    // chunk's sum of delta_eff per channel, the items' partial sums added over
    // the threads of a channel group in thread order
    float* H0 = a.ws_fsum + (q * CH + c0) * N + n0;
#pragma unroll
    for (int s = 0; s < S; s++) {
        H0[s] = h[s].x;
        H0[N + s] = h[s].y;
    }
#pragma unroll
    for (int c = 0; c < GRP; c++) sSD[tid][c] = sdp[c];
    __syncthreads();
    for (int c = tid; c < CH; c += THREADS) {
        const int qg = c / GRP, cc = c % GRP;
        float s = 0.f;
        for (int th = qg; th < THREADS; th += NGRP) s += sSD[th][cc];
        a.ws_fsd[q * CH + c] = s;
    }
}

}  // namespace ss
