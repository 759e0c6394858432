// Forward selective scan (baracuda-kernels `selective_scan.rs`, module doc
// "Algorithm summary"):
//
//   delta_eff = softplus?(delta + bias);  a = exp(delta_eff * A[d,n]);
//   h = a * h + delta_eff * B[t,n] * u;   y = (sum_n h * C[t,n] + D * u) * silu(z)
//
// One block owns CH channels of one batch row and one time chunk (the block
// layout of kernels.h): lane (p, g) of warp w holds S states of the channel
// pair p, the states n0 = w N/NW + g S .. n0 + S of both channels.  The
// layout spends the SM's shared-memory / L1 data pipe sparingly: every B / C
// value a lane reads from shared memory serves two channels, and one 16-byte
// load brings delta_eff and delta_eff * u of both; each lane stores its two
// channels' partial readouts with one 8-byte store.
// Work per 32-step tile:
//   prologue  threads take (step, 8-channel group) items: load the group's
//             runs of u, delta, z (whole 16-byte vectors, four items per
//             64-byte row of the tile), compute delta_eff, delta_eff * u,
//             silu(z) and D * u once per (t, d) into shared memory; other
//             items copy the B and C rows of the tile;
//   scan      each lane walks the 32 steps for its 2 x S states with packed
//             f32x2 arithmetic (one MUFU ex2 per state per step) and stores
//             its two channels' partial readouts per step;
//   epilogue  threads take (step, 8-channel group) items again: add the
//             lanes' and warps' partial readouts and D * u (the pre-gate
//             readout y0, stored as f32 for the backward's dz when the
//             states are saved and z is given), apply the gate and store
//             the group's run of y.
// Modes: Y (y, last_state), YSave (also the state at every kSub-step
// sub-chunk start and y0), Ckpt (the backward's checkpoint pass: the states
// and y0 only, no gate and no y), Summary (a chunk's end state and sum of
// delta_eff, no readout).
// The time axis of a unit (batch row, channel tile) is cut into K chunks when
// the plan says so (kernels.h); a chunk summary -- its end state H from a zero
// start and its sum of delta_eff, which gives the product of its decays
// P = exp(A sum delta_eff) -- then yields the carry-in state of the chunks
// after it: h <- P h + H.
#pragma once

#include "common.cuh"
#include "kernels.h"
#include "simd.cuh"
#include "tiles.cuh"

namespace ss {

constexpr int kRow = 32;  // time steps per tile
static_assert(kRow % kSub == 0, "a tile holds whole checkpoint sub-chunks");

template <typename T, int N>
struct FCfg {
    static constexpr int NW = fwd_warps(N);         // warps per block (they split the states)
    static constexpr int NPW = N / NW;              // states per warp
    static constexpr int G = NPW >= 2 ? 2 : 1;      // lanes per channel pair
    static constexpr int S = NPW / G;               // states per lane (of each of its two channels)
    static constexpr int PAIRS = 32 / G;            // channel pairs per block
    static constexpr int CH = 2 * PAIRS;            // channels per block
    static constexpr int THREADS = 32 * NW;
    static constexpr int ESZ = (int)sizeof(T);
    static constexpr int GRP = 8;                   // channels per prologue / epilogue item
    static constexpr int NGRP = CH / GRP;           // items per step
    static constexpr int ITEMS = kRow * NGRP / THREADS;  // items per thread per tile
    static constexpr int RW = GRP * ESZ / 4;        // 32-bit words of an item's run of one tensor
    static constexpr int NB = N * ESZ;              // bytes of a B / C row
    static constexpr int NWd = NB >= 4 ? NB / 4 : 1;  // 32-bit words per B / C row
    // B / C staging: a step's row holds N / S state groups of 2 S floats (S of
    // B, then S of C), padded by 4 floats so that rows staged by consecutive
    // threads start in different bank groups.  f32 io is copied straight into
    // it (double buffered); bf16 rows are copied raw and converted once.
    static constexpr int BCF = 2 * N + 4;
    static constexpr bool BC_DIRECT = ESZ == 4;
    static constexpr bool BC_RAW = !BC_DIRECT && N * ESZ >= 4;
    static constexpr int BC_BUFS = BC_DIRECT ? 2 : 1;
    // raw row length (elements): rows of 32 bytes or more padded by 16 bytes, so
    // that the 16-byte loads of consecutive rows fall in different bank groups
    static constexpr int RAWP = NB >= 32 ? N + 16 / ESZ : N;
    static constexpr int YP = CH + 4;               // padded shared row of partial readouts (floats)
    // plane of one lane of a pair's partial readouts: kRow rows of YP floats,
    // planes 16 mod 32 floats apart so that the 8-byte stores of both lanes of
    // the pairs of a half warp hit 32 banks
    static constexpr int YPL = kRow * YP + 16;
    static_assert(kRow * NGRP % THREADS == 0, "whole items per thread");
    static_assert(CH == channels_per_block(N), "channel tile of the plan");
};

// Slot of channel pair pp in a per-step staging row of 16-byte units: pair
// 4 q + j (j-th pair of 8-channel group q) goes to 2 q + (j & 1) + 2 NGRP (j >> 1).
// Eight prologue threads of a quarter warp (two steps x four groups, same j)
// then hit eight different bank groups for a row of an odd number of units.
template <int NGRP>
__device__ __forceinline__ int pair_slot(int pp) {
    const int q = pp >> 2, j = pp & 3;
    return 2 * q + (j & 1) + 2 * NGRP * (j >> 1);
}

template <typename T, int N, int MODE>
__global__ void __launch_bounds__(32 * fwd_warps(N), fwd_warps(N) == 2 ? 4 : 8) k_fwd2(FwdArgs a, FPlan p, int si, int64_t k_lo,
                                                               float* ckpt) {
    constexpr bool SUMMARY = MODE == kModeSummary;
    constexpr bool NOY = MODE == kModeSummary;                       // no readout (a chunk summary)
    constexpr bool GATE = MODE == kModeY || MODE == kModeYSave;      // gate and y (the checkpoint pass has neither)
    constexpr bool SAVE = MODE == kModeYSave || MODE == kModeCkpt;   // store the sub-chunk start states
    using C = FCfg<T, N>;
    constexpr int NW = C::NW, NPW = C::NPW, S = C::S, G = C::G, CH = C::CH, THREADS = C::THREADS, GRP = C::GRP,
                  NGRP = C::NGRP, ITEMS = C::ITEMS, RW = C::RW, NWd = C::NWd, YP = C::YP, BCF = C::BCF;
    // per-(t, d) staging, one float4 per channel pair at pair_slot: (delta_eff,
    // delta_eff * u) and (gate, D * u) of both channels; rows of PAIRS + 1 units
    __shared__ float4 sDU[kRow][C::PAIRS + 1];
    __shared__ float4 sGD[NOY ? 1 : kRow][NOY ? 1 : C::PAIRS + 1];
    // B / C values by state group (f32); with f32 io double buffered, the next
    // tile's rows being copied in while the scan reads the current one's
    __shared__ __align__(16) float sBC[C::BC_BUFS][kRow][BCF];
    // raw bf16 B / C rows of the next tile (converted into sBC by the prologue)
    __shared__ __align__(16) T sBCraw[2][C::BC_RAW ? kRow : 1][C::BC_RAW ? C::RAWP : 2];
    // raw runs of delta, u, z of the next tile, copied in asynchronously by the
    // thread that later converts them
    __shared__ __align__(16) T sRaw[GATE ? 3 : 2][kRow][CH];
    // per-warp partial readouts, one plane per lane of a pair (float g YPL + i YP
    // + c: lane g's sum over its states, step i, channel c)
    __shared__ __align__(16) float sY[NOY ? 1 : NW][NOY ? 1 : G * C::YPL];
    __shared__ float sBias[CH], sDv[CH];

    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    // block -> (unit, chunk) of segment si; unit -> (batch row, channel tile)
    const Seg sgm = seg_at(p, si);
    const int64_t ul = (int64_t)blockIdx.x % sgm.nu;
    const int64_t k = k_lo + (int64_t)blockIdx.x / sgm.nu;
    const int64_t unit = sgm.u_lo + ul;
    const int64_t ntiles = p.tiles_b;
    const int64_t tile = unit % ntiles, b = unit / ntiles;
    const int64_t s_first = sgm.s0 + ul * sgm.K;  // summary index of the unit's chunk 0
    const int64_t L = a.L, Dch = a.Dch;
    const int64_t d0 = tile * CH;
    const bool fast = ((Dch * (int64_t)sizeof(T)) % 16 == 0) && (d0 + CH <= Dch);
    const T* u = static_cast<const T*>(a.u);
    const T* delta = static_cast<const T*>(a.delta);
    const T* Bm = static_cast<const T*>(a.B);
    const T* Cm = static_cast<const T*>(a.C);
    const T* z = static_cast<const T*>(a.z);

    for (int c = tid; c < CH; c += THREADS) {
        const int64_t dc = d0 + c < Dch ? d0 + c : Dch - 1;
        sBias[c] = a.delta_bias ? a.delta_bias[dc] : 0.f;
        sDv[c] = a.D ? a.D[dc] : 0.f;
    }

    // scan-lane identity: channel pair pp (channels c0, c0 + 1 of the block),
    // states n0 .. n0 + S of warp w
    const int pp = lane / G, g = lane % G;
    const int c0 = 2 * pp;
    const bool ok0 = d0 + c0 < Dch, ok1 = d0 + c0 + 1 < Dch;
    const int64_t dA0 = ok0 ? d0 + c0 : Dch - 1, dA1 = ok1 ? d0 + c0 + 1 : Dch - 1;
    const int n0 = w * NPW + g * S;
    const int sg = n0 / S;  // the lane's state group
    const int pslot = pair_slot<NGRP>(pp);
    const int64_t row0 = b * Dch + dA0, row1 = b * Dch + dA1;
    // the state starts at h0 (zero without one); a chunk summary starts from zero
    const bool from_h0 = !SUMMARY && a.h0 != nullptr;
    float A2[2][S], h[2][S];
    float sd0 = 0.f, sd1 = 0.f;  // summary: the chunk's sums of delta_eff
#pragma unroll
    for (int s = 0; s < S; s++) {
        // channels past Dch run with a zero exponent: their state stays exactly zero
        A2[0][s] = ok0 ? scan_A(a, dA0 * N + n0 + s) * kLog2eF : 0.f;
        A2[1][s] = ok1 ? scan_A(a, dA1 * N + n0 + s) * kLog2eF : 0.f;
        h[0][s] = from_h0 && ok0 ? a.h0[row0 * N + n0 + s] : 0.f;
        h[1][s] = from_h0 && ok1 ? a.h0[row1 * N + n0 + s] : 0.f;
    }
    if (!SUMMARY && k > 0) {
        // carry-in: h <- P_j h + H_j over the unit's chunks j < k, with
        // P_j = exp2(A2 * sum of delta_eff over chunk j)
        for (int64_t j = 0; j < k; j++) {
            const int64_t q = s_first + j;
            const float* H0 = a.ws_fsum + (q * CH + c0) * N + n0;
            const float sdj0 = a.ws_fsd[q * CH + c0], sdj1 = a.ws_fsd[q * CH + c0 + 1];
#pragma unroll
            for (int s = 0; s < S; s++) {
                h[0][s] = fmaf(ex2a(A2[0][s] * sdj0), h[0][s], H0[s]);
                h[1][s] = fmaf(ex2a(A2[1][s] * sdj1), h[1][s], H0[N + s]);
            }
        }
        // channels past Dch (read a clamped channel's summaries) keep a zero state,
        // so that every saved slot of theirs holds zero
#pragma unroll
        for (int s = 0; s < S; s++) {
            h[0][s] = ok0 ? h[0][s] : 0.f;
            h[1][s] = ok1 ? h[1][s] : 0.f;
        }
    }

    const int64_t t_begin = k * sgm.Lc;
    const int64_t t_end = t_begin + sgm.Lc < L ? t_begin + sgm.Lc : L;
    // saved states (layout of ckpt_bytes): one block of CH x N floats per
    // (sub-chunk slot t / kSub, batch, channel tile), the lane's slots in lane order
    const int64_t ck_stride = a.Bsz * ntiles * CH * N;
    float* ck_blk = SAVE ? ckpt + (t_begin / kSub) * ck_stride + (b * ntiles + tile) * (CH * N) : nullptr;
    float* ck0 = SAVE ? ck_blk + ckpt_slot(w, 0, lane, S) : nullptr;
    float* ck1 = SAVE ? ck_blk + ckpt_slot(w, 1, lane, S) : nullptr;

    // Asynchronous copies of the tile starting at tt: the thread's item runs
    // (when the tile's rows are whole aligned vectors) and the B / C rows (f32
    // into sBC[buf]; bf16 raw into sBCraw); one commit group.
    auto issue = [&](int64_t tt, int buf) {
        if (fast) {
#pragma unroll
            for (int it = 0; it < ITEMS; it++) {
                const int id = tid + it * THREADS;
                const int r = id / NGRP, cg = (id % NGRP) * GRP;
                const int64_t t = tt + r;
                if (t < t_end) {
                    const int64_t off = (b * L + t) * Dch + d0 + cg;
                    cp_async_bytes<GRP * C::ESZ>(&sRaw[0][r][cg], delta + off);
                    cp_async_bytes<GRP * C::ESZ>(&sRaw[1][r][cg], u + off);
                    if (GATE && z) cp_async_bytes<GRP * C::ESZ>(&sRaw[GATE ? 2 : 1][r][cg], z + off);
                }
            }
        }
        for (int id = tid; id < (NOY ? 1 : 2) * kRow; id += THREADS) {
            const int half = id / kRow, r = id % kRow;
            const int64_t t = tt + r;
            const T* src = (half ? Cm : Bm) + (b * L + (t < t_end ? t : 0)) * N;
            if constexpr (C::BC_DIRECT) {
                cp_async_bc_row<T, N, S>(reinterpret_cast<unsigned char*>(&sBC[buf][r][0]), half, src, t < t_end);
            } else if constexpr (C::BC_RAW) {
                if (t < t_end) cp_async_bytes<N * C::ESZ>(&sBCraw[half][r][0], src);
            }
        }
        cp_async_commit();
    };
    issue(t_begin, 0);
    __syncthreads();  // sBias / sDv

    for (int64_t t0 = t_begin; t0 < t_end; t0 += kRow) {
        const int buf = (int)(((t0 - t_begin) / kRow) & 1);
        cp_async_wait<0>();  // this thread's copies of the tile
        // ---- prologue: (step, 8-channel group) items, then the B / C rows
#pragma unroll
        for (int it = 0; it < ITEMS; it++) {
            const int id = tid + it * THREADS;
            const int r = id / NGRP, q = id % NGRP;
            const int64_t t = t0 + r;
            const bool rv = t < t_end;
            const int cg = q * GRP;  // first channel of the group
            uint32_t rd[RW], ru[RW], rz[RW];
            if (rv) {
                if (fast) {
                    lds_words<GRP * C::ESZ, RW>(&sRaw[0][r][cg], rd);
                    lds_words<GRP * C::ESZ, RW>(&sRaw[1][r][cg], ru);
                    if (GATE && z) lds_words<GRP * C::ESZ, RW>(&sRaw[GATE ? 2 : 1][r][cg], rz);
                } else {
                    const int64_t off = (b * L + t) * Dch + d0 + cg;
                    load_run<T, GRP, RW>(delta, off, d0 + cg, Dch, false, rd);
                    load_run<T, GRP, RW>(u, off, d0 + cg, Dch, false, ru);
                    if (GATE && z) load_run<T, GRP, RW>(z, off, d0 + cg, Dch, false, rz);
                }
            }
#pragma unroll
            for (int c = 0; c < GRP; c += 2) {
                // two channels at a time with packed arithmetic
                float2 dl = make_float2(0.f, 0.f), dlu = dl, gt = make_float2(1.f, 1.f), dun = dl;
                if (rv) {
                    const float2 x = make_float2(elem<T>(rd, c) + sBias[cg + c], elem<T>(rd, c + 1) + sBias[cg + c + 1]);
                    dl = a.softplus ? softplus2(x) : x;
                    const float2 uu = make_float2(elem<T>(ru, c), elem<T>(ru, c + 1));
                    dlu = mul2(dl, uu);
                    if (!NOY) {
                        if (GATE && z) {
                            const float2 zz = make_float2(elem<T>(rz, c), elem<T>(rz, c + 1));
                            gt = mul2(zz, sigmoid2(zz));
                        }
                        dun = mul2(make_float2(sDv[cg + c], sDv[cg + c + 1]), uu);
                    }
                }
                const int slot = pair_slot<NGRP>((cg + c) / 2);
                sDU[r][slot] = make_float4(dl.x, dlu.x, dl.y, dlu.y);
                if (!NOY) sGD[r][slot] = make_float4(gt.x, dun.x, gt.y, dun.y);
            }
        }
        if constexpr (!C::BC_DIRECT) {
            // bf16 B / C rows of the tile's steps, row id = (tensor, step), converted
            // by the thread that copied them (or loaded here when too short to copy)
            for (int id = tid; id < (NOY ? 1 : 2) * kRow; id += THREADS) {
                const int half = id / kRow, r = id % kRow;
                const int64_t t = t0 + r;
                uint32_t wv[NWd];
                if (t < t_end) {
                    if constexpr (C::BC_RAW) lds_words<C::NB, NWd>(&sBCraw[half][r][0], wv);
                    else load_words<C::NB, NWd>((half ? Cm : Bm) + (b * L + t) * N, wv);
                }
                stage_bc_row_f32<T, N, S, NWd>(&sBC[0][r][0], half, wv, t < t_end);
            }
        }
        __syncthreads();  // staging complete; every thread is done reading sRaw
        if (t0 + kRow < t_end) issue(t0 + kRow, buf ^ 1);

        // ---- scan: 32 steps of the lane's 2 x S states.  Steps past t_end (last
        // tile only) carry delta_eff = 0 and B = 0: the state stays unchanged.
        const int64_t jt = (t0 - t_begin) / kSub;
#pragma unroll 8
        for (int i = 0; i < kRow; i++) {
            if (SAVE && (i % kSub) == 0) {
                const int64_t jo = (jt + i / kSub) * ck_stride;
                // every slot is written: channels past Dch hold a zero state
                if constexpr (S % 4 == 0) {
#pragma unroll
                    for (int s = 0; s < S; s += 4) {
                        *reinterpret_cast<float4*>(ck0 + jo + s) = make_float4(h[0][s], h[0][s + 1], h[0][s + 2], h[0][s + 3]);
                        *reinterpret_cast<float4*>(ck1 + jo + s) = make_float4(h[1][s], h[1][s + 1], h[1][s + 2], h[1][s + 3]);
                    }
                } else {
#pragma unroll
                    for (int s = 0; s < S; s++) {
                        ck0[jo + s] = h[0][s];
                        ck1[jo + s] = h[1][s];
                    }
                }
            }
            const float4 du = sDU[i][pslot];
            if (SUMMARY) {
                sd0 += du.x;  // delta_eff of steps past t_end is zero
                sd1 += du.z;
            }
            float Bv[S], Cv[S];
            ld_bc_f32<S>(&sBC[C::BC_DIRECT ? buf : 0][i][sg * 2 * S], Bv, Cv);
            float yp[2];
            if constexpr (S >= 2) {
                float2 ya[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
                for (int e = 0; e < 2; e++) {
                    const float2 dl2 = splat2(e ? du.z : du.x), dlu2 = splat2(e ? du.w : du.y);
#pragma unroll
                    for (int s = 0; s < S; s += 2) {
                        const float2 ex = mul2(dl2, make_float2(A2[e][s], A2[e][s + 1]));
                        const float2 da = make_float2(ex2a(ex.x), ex2a(ex.y));
                        const float2 x = mul2(dlu2, make_float2(Bv[s], Bv[s + 1]));
                        const float2 hh = fma2(da, make_float2(h[e][s], h[e][s + 1]), x);
                        h[e][s] = hh.x;
                        h[e][s + 1] = hh.y;
                        if (!NOY) ya[e] = fma2(make_float2(Cv[s], Cv[s + 1]), hh, ya[e]);
                    }
                }
                yp[0] = ya[0].x + ya[0].y;
                yp[1] = ya[1].x + ya[1].y;
            } else {
#pragma unroll
                for (int e = 0; e < 2; e++) {
                    const float da = ex2a((e ? du.z : du.x) * A2[e][0]);
                    h[e][0] = fmaf(da, h[e][0], (e ? du.w : du.y) * Bv[0]);
                    yp[e] = Cv[0] * h[e][0];
                }
            }
            if (!NOY) {
                // both channels' partials of the lane; the epilogue adds the pair's lanes
                *reinterpret_cast<float2*>(&sY[w][g * C::YPL + i * YP + c0]) = make_float2(yp[0], yp[1]);
            }
        }
        __syncthreads();

        // ---- epilogue: (step, 8-channel group) items
        if (!NOY) {
#pragma unroll
            for (int it = 0; it < ITEMS; it++) {
                const int id = tid + it * THREADS;
                const int r = id / NGRP, q = id % NGRP;
                const int64_t t = t0 + r;
                const int cg = q * GRP;
                if (t < t_end) {
                    float yv[GRP], y0v[GRP];
#pragma unroll
                    for (int c = 0; c < GRP; c += 4) {
                        // per warp, the sum of its G lanes' planes; then the warps in order
                        float4 acc;
#pragma unroll
                        for (int ww = 0; ww < NW; ww++) {
                            float4 o = *reinterpret_cast<const float4*>(&sY[ww][r * YP + cg + c]);
                            if constexpr (G == 2) {
                                const float4 q = *reinterpret_cast<const float4*>(&sY[ww][C::YPL + r * YP + cg + c]);
                                o.x += q.x; o.y += q.y; o.z += q.z; o.w += q.w;
                            }
                            if (ww == 0) {
                                acc = o;
                            } else {
                                acc.x += o.x; acc.y += o.y; acc.z += o.z; acc.w += o.w;
                            }
                        }
                        const float4 g01 = sGD[r][pair_slot<NGRP>((cg + c) / 2)];
                        const float4 g23 = sGD[r][pair_slot<NGRP>((cg + c) / 2 + 1)];
                        // the pre-gate readout y0 = sum_n h C + D u, then the gate
                        y0v[c] = acc.x + g01.y;
                        y0v[c + 1] = acc.y + g01.w;
                        y0v[c + 2] = acc.z + g23.y;
                        y0v[c + 3] = acc.w + g23.w;
                        yv[c] = y0v[c] * g01.x;
                        yv[c + 1] = y0v[c + 1] * g01.z;
                        yv[c + 2] = y0v[c + 2] * g23.x;
                        yv[c + 3] = y0v[c + 3] * g23.z;
                    }
                    const int64_t off = (b * L + t) * Dch + d0 + cg;
                    if (a.y0 && z) {
                        // kept for the backward's dz (f32; the same alignment as the io runs)
                        float* y0row = a.y0 + off;
                        if (fast) {
#pragma unroll
                            for (int c = 0; c < GRP; c += 4)
                                *reinterpret_cast<float4*>(y0row + c) = make_float4(y0v[c], y0v[c + 1], y0v[c + 2], y0v[c + 3]);
                        } else {
#pragma unroll
                            for (int c = 0; c < GRP; c++)
                                if (d0 + cg + c < Dch) y0row[c] = y0v[c];
                        }
                    }
                    if (!GATE) continue;
                    T* yrow = static_cast<T*>(a.y) + off;
                    if (fast) {
                        uint32_t wv[RW];
                        if constexpr (sizeof(T) == 4) {
#pragma unroll
                            for (int c = 0; c < GRP; c++) wv[c] = __float_as_uint(yv[c]);
                        } else {
#pragma unroll
                            for (int c = 0; c < GRP; c += 2) wv[c >> 1] = pack2<T>(yv[c], yv[c + 1]);
                        }
#pragma unroll
                        for (int v = 0; v < RW / 4; v++)
                            reinterpret_cast<uint4*>(yrow)[v] =
                                make_uint4(wv[4 * v], wv[4 * v + 1], wv[4 * v + 2], wv[4 * v + 3]);
                    } else {
#pragma unroll
                        for (int c = 0; c < GRP; c++)
                            if (d0 + cg + c < Dch) st(yrow + c, yv[c]);
                    }
                }
            }
        }
        // the next prologue restages sDU / sGD / sBC; sY is read above and written
        // again only after the next prologue's barrier
    }

    if (SUMMARY) {
        // every entry of the part is written (channels past Dch: zero state)
        const int64_t q = s_first + k;
        float* H0 = a.ws_fsum + (q * CH + c0) * N + n0;
#pragma unroll
        for (int s = 0; s < S; s++) {
            H0[s] = h[0][s];
            H0[N + s] = h[1][s];
        }
        if (w == 0 && g == 0) *reinterpret_cast<float2*>(a.ws_fsd + q * CH + c0) = make_float2(sd0, sd1);
    } else if (MODE != kModeCkpt && k == sgm.K - 1 && a.last_state) {
#pragma unroll
        for (int s = 0; s < S; s++) {
            if (ok0) a.last_state[row0 * N + n0 + s] = h[0][s];
            if (ok1) a.last_state[row1 * N + n0 + s] = h[1][s];
        }
    }
}

// One launch of mode MODE over chunks k_lo .. k_hi of segment si.
template <typename T, int N, int MODE>
void launch_fwd_mode(const FwdArgs& a, const FPlan& p, int si, cudaStream_t st, int64_t k_lo, int64_t k_hi,
                     float* ckpt) {
    prof_mark(st);
    k_fwd2<T, N, MODE><<<(unsigned)(p.seg[si].nu * (k_hi - k_lo)), FCfg<T, N>::THREADS, 0, st>>>(a, p, si, k_lo,
                                                                                                ckpt);
}

// The chunk summaries of every chunked segment, then each segment's main pass.
template <typename T, int N>
cudaError_t launch_fwd2_t(const FwdArgs& a, const FPlan& p, cudaStream_t st, int mode, float* ckpt) {
    for (int si = 0; si < p.nseg; si++)
        if (p.seg[si].K > 1) launch_fwd_mode<T, N, kModeSummary>(a, p, si, st, 0, p.seg[si].K - 1, nullptr);
    for (int si = 0; si < p.nseg; si++) {
        const int64_t K = p.seg[si].K;
        if (mode == kModeCkpt) {
            launch_fwd_mode<T, N, kModeCkpt>(a, p, si, st, 0, K, ckpt);
        } else if (ckpt) {
            launch_fwd_mode<T, N, kModeYSave>(a, p, si, st, 0, K, ckpt);
        } else {
            launch_fwd_mode<T, N, kModeY>(a, p, si, st, 0, K, nullptr);
        }
    }
    return cudaGetLastError();
}

// Forward launcher of one io type: switches on N.
template <typename T>
cudaError_t launch_fwd2_io(const FwdArgs& a, const FPlan& p, cudaStream_t st, int mode, float* ckpt) {
    switch (a.N) {
        case 1: return launch_fwd2_t<T, 1>(a, p, st, mode, ckpt);
        case 2: return launch_fwd2_t<T, 2>(a, p, st, mode, ckpt);
        case 4: return launch_fwd2_t<T, 4>(a, p, st, mode, ckpt);
        case 8: return launch_fwd2_t<T, 8>(a, p, st, mode, ckpt);
        case 16: return launch_fwd2_t<T, 16>(a, p, st, mode, ckpt);
        case 32: return launch_fwd2_t<T, 32>(a, p, st, mode, ckpt);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace ss
