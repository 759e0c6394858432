// Forward selective scan (baracuda-kernels `selective_scan.rs`, module doc
// "Algorithm summary"):
//
//   delta_eff = softplus?(delta + bias);  a = exp(delta_eff * A[d,n]);
//   h = a * h + delta_eff * B[t,n] * u;   y = (sum_n h * C[t,n] + D * u) * silu(z)
//
// One block owns CH channels of one batch row and one time chunk (the block
// layout of kernels.h): lane (p, g) of warp w holds S states of the channel
// pair p, the states n0 = w NPW + g S .. n0 + S of both channels.
//
// The scan is bound by the SM's FP32 pipe and its MUFU together: per state
// and step it needs one ex2 and four FP32 operations (the exponent, the
// input term, the recurrence, the readout), and both units run at 32 such
// (t, d, n) elements per clock on an SM.  So every FP32 operation of the
// scan is a packed f32x2 instruction whose two halves are the lane's two
// channels at one state: delta_eff, delta_eff * u and the readout of both
// channels come and go as natural register pairs, and the B / C value of
// the state is the same scalar in both halves (a broadcast operand, which
// costs no instruction).  A lane's partial readout of one step is then one
// 8-byte store of both channels.
// Work per 32-step tile:
//   prologue  threads take (step, 8-channel group) items: the group's runs
//             of delta, u, z (copied in with the previous tile), delta_eff
//             and delta_eff * u of each channel pair into shared memory; the
//             runs of u and z stay in the thread's registers for its
//             epilogue items (the same items); the B / C rows of the tile
//             become f32 rows;
//   scan      each lane walks the 32 steps for its 2 x S states, storing the
//             state entering every kSub-th step when the states are kept
//             for the backward;
//   epilogue  the (step, 8-channel group) items add the lanes' and warps'
//             partial readouts and D * u (the pre-gate readout y0, stored
//             as f32 for the backward's dz when the states are kept and z
//             is given), apply the gate z sigmoid(z) and store the group's
//             run of y.  (Forming D * u and the gate here rather than in the
//             prologue keeps them out of shared memory: the tile's shared-
//             memory data pipe is the forward's busiest unit.)
// Modes: Y (y, last_state), YSave (also the states entering every kSub-th
// step and y0), Ckpt (the backward's checkpoint pass: the states and y0, no
// gate and no y), Summary (a chunk's end state and sum of delta_eff, no
// readout).
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

constexpr int kRow = kFwdRows;  // time steps per forward tile
static_assert(kRow % kSub == 0, "a tile holds whole save intervals");

template <typename T, int N>
struct FCfg {
    static constexpr int NW = scan_warps(N);        // warps per block (they split the states)
    static constexpr int NPW = N / NW;              // states per warp
    static constexpr int S = lane_states(N);        // states per lane (of each of its two channels)
    static constexpr int G = NPW / S;               // lanes per channel pair
    static constexpr int PAIRS = 32 / G;            // channel pairs per block
    static constexpr int CH = 2 * PAIRS;            // channels per block
    static constexpr int THREADS = 32 * NW;
    static constexpr int ESZ = (int)sizeof(T);
    static constexpr int GRP = 8;                   // channels per prologue / epilogue item
    static constexpr int NGRP = CH / GRP;           // items per step
    static constexpr int ITEMS = kRow * NGRP / THREADS;  // items per thread per tile
    static constexpr int RW = GRP * ESZ / 4;        // 32-bit words of an item's run of one tensor
    static constexpr int NB = N * ESZ;              // bytes of a B / C row
    // f32 B / C staging, one dense [step][N] array per tensor (the layout a TMA
    // box lands in).  f32 io is copied straight into it (double buffered);
    // 16-bit rows are copied raw and converted once.  (Unlike the backward, the
    // forward keeps no packed bf16 rows: widening them in the scan sits on the
    // path to the decays, and measured slower -- 0.476 -> 0.553 ms for the
    // Mamba-2.8B layer's main pass -- although it halves the scan's B / C
    // shared-memory wavefronts.)
    static constexpr bool BC_DIRECT = ESZ == 4;
    static constexpr bool BC_RAW = !BC_DIRECT && NB >= 4;
    static constexpr int BC_BUFS = BC_DIRECT ? 2 : 1;
    // 16-bit rows are copied and converted in units of BCV values of one row,
    // consecutive threads taking consecutive units (free of bank conflicts)
    static constexpr int BCV = N >= 4 ? 4 : N;
    static constexpr int BCU = N / BCV;             // units per row
    // the raw u / z runs of a thread's items stay in registers from its prologue
    // to its epilogue when they are few (else the prologue stages the gate and
    // D * u in shared memory)
    static constexpr bool KEEP = ITEMS * RW <= 16;
    static constexpr int YP = CH + 4;               // padded row of partial readouts (floats)
    // plane of one lane of a pair's partial readouts: kRow rows of YP floats,
    // planes 16 mod 32 floats apart so that the 8-byte stores of the lanes of
    // two planes hit different banks
    static constexpr int YPL = kRow * YP + 16;
    static_assert(kRow * NGRP % THREADS == 0, "whole items per thread");
    static_assert(CH == channels_per_block(N), "channel tile of the plan");
    static_assert(S * G * NW == N, "the lanes cover the states");
};

template <typename T, int N, int MODE>
__global__ void __launch_bounds__(32 * scan_warps(N), scan_warps(N) == 2 ? 4 : 8)
    k_fwd(FwdArgs a, FPlan p, int si, int64_t k_lo, float* ckpt, const __grid_constant__ TmaMaps maps) {
    constexpr bool SUMMARY = MODE == kModeSummary;
    constexpr bool NOY = MODE == kModeSummary;                       // no readout (a chunk summary)
    constexpr bool GATE = MODE == kModeY || MODE == kModeYSave;      // gate and y (the checkpoint pass has neither)
    constexpr bool SAVE = MODE == kModeYSave || MODE == kModeCkpt;   // store the states entering every kSub-th step
    using C = FCfg<T, N>;
    constexpr int NW = C::NW, NPW = C::NPW, S = C::S, G = C::G, PAIRS = C::PAIRS, CH = C::CH,
                  THREADS = C::THREADS, GRP = C::GRP, NGRP = C::NGRP, ITEMS = C::ITEMS, RW = C::RW,
                  YP = C::YP;
    // per-(t, d) staging of the scan, one float4 per channel pair:
    // (delta_eff of both channels, delta_eff * u of both channels)
    __shared__ float4 sDU[kRow][PAIRS + 1];
    // (gate of both channels, D * u of both channels) for the epilogue, when the
    // raw runs do not stay in registers
    __shared__ float4 sGD[NOY || C::KEEP ? 1 : kRow][NOY || C::KEEP ? 1 : PAIRS + 1];
    // B / C rows as f32 [tensor][buffer][step][N]; with f32 io double buffered,
    // the next tile's rows being copied in while the scan reads the current one's
    __shared__ __align__(128) float sBC[2][C::BC_BUFS][kRow][N];
    // raw 16-bit B / C rows of the next tile [tensor][step][N] (converted into sBC
    // by the prologue)
    __shared__ __align__(128) T sBCraw[2][C::BC_RAW ? kRow : 1][C::BC_RAW ? N : 8];
    // raw runs of delta, u, z of the next tile (a TMA box each, or copied in
    // asynchronously by the thread that later converts them)
    __shared__ __align__(128) T sRaw[GATE ? 3 : 2][kRow][CH];
    // completion of the TMA copies into the two tile buffers
    __shared__ __align__(8) uint64_t sBar[2];
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
    // TMA boxes land on 128-byte aligned shared memory; a block whose buffers are
    // not (never expected) records it and stages with asynchronous copies instead
    bool tma = a.use_tma != 0;
    if (tma && !(smem_aligned128(&sRaw[0][0][0]) && smem_aligned128(&sBC[0][0][0][0]) &&
                 smem_aligned128(&sBCraw[0][0][0]))) {
        if (threadIdx.x == 0) atomicOr(a.status, kDevMisaligned);
        tma = false;
    }
    // the tile's runs are read from shared memory: TMA boxes (zero-filled past Dch),
    // or whole aligned vectors copied in asynchronously
    // whole aligned vectors of y / y0 per row: stores need the tile inside Dch
    const bool sfast = ((Dch * (int64_t)sizeof(T)) % 16 == 0) && (d0 + CH <= Dch);
    const bool fast = tma || sfast;
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
    if (tma && tid == 0) {
        mbar_init(&sBar[0], 1);
        mbar_init(&sBar[1], 1);
        fence_proxy_async_smem();
    }

    // scan-lane identity: channel pair pp (channels c0, c0 + 1 of the block),
    // states n0 .. n0 + S of warp w
    const int pp = lane / G, g = lane % G;
    const int c0 = 2 * pp;
    const bool ok0 = d0 + c0 < Dch, ok1 = d0 + c0 + 1 < Dch;
    const int64_t dA0 = ok0 ? d0 + c0 : Dch - 1, dA1 = ok1 ? d0 + c0 + 1 : Dch - 1;
    const int n0 = w * NPW + g * S;
    const int64_t row0 = b * Dch + dA0, row1 = b * Dch + dA1;
    // the state starts at h0 (zero without one); a chunk summary starts from zero.
    // Registers pair the lane's two channels at one state: (channel c0, c0 + 1).
    const bool from_h0 = !SUMMARY && a.h0 != nullptr;
    float2 A2[S], h[S];
    float2 sdp = make_float2(0.f, 0.f);  // summary: the chunk's sums of delta_eff
#pragma unroll
    for (int s = 0; s < S; s++) {
        // channels past Dch run with a zero exponent: their state stays exactly zero
        A2[s] = make_float2(ok0 ? scan_A(a, dA0 * N + n0 + s) * kLog2eF : 0.f,
                            ok1 ? scan_A(a, dA1 * N + n0 + s) * kLog2eF : 0.f);
        h[s] = make_float2(from_h0 && ok0 ? a.h0[row0 * N + n0 + s] : 0.f,
                           from_h0 && ok1 ? a.h0[row1 * N + n0 + s] : 0.f);
    }
    if (!SUMMARY && k > 0) {
        // carry-in: h <- P_j h + H_j over the unit's chunks j < k, with
        // P_j = exp2(A2 * sum of delta_eff over chunk j)
        for (int64_t j = 0; j < k; j++) {
            const int64_t q = s_first + j;
            const float* H0 = a.ws_fsum + (q * CH + c0) * N + n0;
            const float2 sdj = make_float2(a.ws_fsd[q * CH + c0], a.ws_fsd[q * CH + c0 + 1]);
#pragma unroll
            for (int s = 0; s < S; s++) {
                const float2 e = mul2(A2[s], sdj);
                h[s] = fma2(make_float2(ex2a(e.x), ex2a(e.y)), h[s], make_float2(H0[s], H0[N + s]));
            }
        }
        // channels past Dch (read a clamped channel's summaries) keep a zero state,
        // so that every saved slot of theirs holds zero
#pragma unroll
        for (int s = 0; s < S; s++) h[s] = make_float2(ok0 ? h[s].x : 0.f, ok1 ? h[s].y : 0.f);
    }

    const int64_t t_begin = k * sgm.Lc;
    const int64_t t_end = t_begin + sgm.Lc < L ? t_begin + sgm.Lc : L;
    // saved states (layout of ckpt_bytes): one block of CH x N floats per
    // (batch, channel tile, slot t / kSub), the lane's 2 S floats at its slots
    float* ck_lane = SAVE ? ckpt + ckpt_block(p, b, tile, t_begin / kSub, N) + ckpt_slot(w, lane, S, 0) : nullptr;

    // Copies of the tile starting at tt into buffer buf.  With TMA: one thread
    // issues a box per tensor (delta, u, z as [kRow][CH], B and C as
    // [kRow][N]: f32 into sBC[.][buf], 16-bit raw into sBCraw) on the buffer's
    // barrier.  Otherwise: each thread copies its item runs (when the tile's
    // rows are whole aligned vectors) and B / C rows asynchronously; one commit
    // group.
    const TmaMaps& mp = maps;
    auto issue = [&](int64_t tt, int buf) {
        if (tma) {
            if (tid == 0) {
                constexpr uint32_t run = kRow * CH * C::ESZ, row = kRow * N * C::ESZ;
                mbar_expect_tx(&sBar[buf], (GATE && z ? 3 : 2) * run + (NOY ? 1 : 2) * row);
                const int x = (int)d0, y = (int)tt, zc = (int)b;
                tma_load_3d(&sRaw[0][0][0], &mp.m[kMapDelta], x, y, zc, &sBar[buf]);
                tma_load_3d(&sRaw[1][0][0], &mp.m[kMapU], x, y, zc, &sBar[buf]);
                if (GATE && z) tma_load_3d(&sRaw[GATE ? 2 : 1][0][0], &mp.m[kMapZ], x, y, zc, &sBar[buf]);
                if constexpr (C::BC_DIRECT) {
                    tma_load_3d(&sBC[0][buf][0][0], &mp.m[kMapB], 0, y, zc, &sBar[buf]);
                    if (!NOY) tma_load_3d(&sBC[1][buf][0][0], &mp.m[kMapC], 0, y, zc, &sBar[buf]);
                } else {
                    tma_load_3d(&sBCraw[0][0][0], &mp.m[kMapB], 0, y, zc, &sBar[buf]);
                    if (!NOY) tma_load_3d(&sBCraw[1][0][0], &mp.m[kMapC], 0, y, zc, &sBar[buf]);
                }
            }
            return;
        }
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
        if constexpr (C::BC_DIRECT) {
            for (int id = tid; id < (NOY ? 1 : 2) * kRow; id += THREADS) {
                const int half = id / kRow, r = id % kRow;
                const int64_t t = tt + r;
                float* dst = &sBC[half][buf][r][0];
                if (t < t_end) {
                    cp_async_bytes<N * 4>(dst, (half ? Cm : Bm) + (b * L + t) * N);
                } else {
#pragma unroll
                    for (int n = 0; n < N; n++) dst[n] = 0.f;
                }
            }
        } else if constexpr (C::BC_RAW) {
            // in the prologue's conversion units
            for (int id = tid; id < (NOY ? 1 : 2) * kRow * C::BCU; id += THREADS) {
                const int row = id / C::BCU, n = (id % C::BCU) * C::BCV;
                const int half = row / kRow, r = row % kRow;
                const int64_t t = tt + r;
                if (t < t_end) cp_async_bytes<C::BCV * C::ESZ>(&sBCraw[half][r][n], (half ? Cm : Bm) + (b * L + t) * N + n);
            }
        }
        cp_async_commit();
    };
    issue(t_begin, 0);
    __syncthreads();  // sBias / sDv, the barriers
    // the thread's prologue / epilogue items cover the same channel group in every
    // tile (THREADS is a multiple of NGRP): its biases and D stay in registers
    static_assert(THREADS % NGRP == 0, "one channel group per thread");
    const int cg = (tid % NGRP) * GRP;
    float biasv[GRP], dvv[GRP];
#pragma unroll
    for (int c = 0; c < GRP; c++) {
        biasv[c] = sBias[cg + c];
        dvv[c] = sDv[cg + c];
    }
    // raw runs of u and z of the thread's prologue items, kept in registers for
    // its epilogue items (the same (step, group) items), which form D * u and
    // the gate from them
    constexpr bool KEEP = C::KEEP;
    uint32_t kU[NOY || !KEEP ? 1 : ITEMS][RW], kZ[GATE && KEEP ? ITEMS : 1][RW];

    for (int64_t t0 = t_begin; t0 < t_end; t0 += kRow) {
        const int64_t jt = (t0 - t_begin) / kRow;  // tile index within the chunk
        const int buf = (int)(jt & 1);
        // the tile's copies: this thread's own (asynchronous copies), or the
        // TMA boxes (the buffer's barrier completes its phase jt / 2 mod 2)
        bool ok = true;
        if (tma) ok = mbar_wait(&sBar[buf], (uint32_t)((jt >> 1) & 1));
        else cp_async_wait<0>();
        // ---- prologue: (step, 8-channel group) items, then the B / C rows.  All
        // of the thread's shared-memory reads come first, then the arithmetic of
        // every item, then the stores: with no store between them, the items'
        // dependency chains (two MUFU steps and a polynomial each) interleave.
        // The terms are formed for every row without branching; rows past t_end
        // store zero delta_eff and input terms.  Shared-memory runs are read for
        // every row: TMA zero-fills rows past the tensor, and other rows past
        // t_end hold earlier data, discarded by the selects.
        // 16-bit B / C rows of the tile's steps, in units of BCV values of one row
        // (tensor, step), converted by the thread that copied them (or loaded here
        // when too short to copy)
        constexpr int BCV = C::BCV, BCU = C::BCU, VW = BCV * C::ESZ >= 4 ? BCV * C::ESZ / 4 : 1;
        constexpr int BCUT = C::BC_DIRECT ? 1 : (NOY ? 1 : 2) * kRow * BCU / THREADS;  // units per thread
        uint32_t wv[BCUT][VW];
        if constexpr (!C::BC_DIRECT) {
            static_assert((NOY ? 1 : 2) * kRow * BCU % THREADS == 0, "whole conversion units per thread");
#pragma unroll
            for (int k = 0; k < BCUT; k++) {
                const int id = tid + k * THREADS;
                const int row = id / BCU, n = (id % BCU) * BCV;
                const int half = row / kRow, r = row % kRow;
                const int64_t t = t0 + r;
#pragma unroll
                for (int v = 0; v < VW; v++) wv[k][v] = 0u;
                if (t < t_end) {
                    if constexpr (C::BC_RAW) lds_words<BCV * C::ESZ, VW>(&sBCraw[half][r][n], wv[k]);
                    else load_words<BCV * C::ESZ, VW>((half ? Cm : Bm) + (b * L + t) * N + n, wv[k]);
                }
            }
        }
        // (items in batches of IB, which bounds the registers they hold)
        constexpr int IB = ITEMS < 2 ? ITEMS : 2;
        static_assert(ITEMS % IB == 0, "whole batches of items");
#pragma unroll
        for (int ib = 0; ib < ITEMS; ib += IB) {
            uint32_t rd[IB][RW], ru[IB][RW], rz[IB][RW];
#pragma unroll
            for (int k = 0; k < IB; k++) {
                const int it = ib + k;
                const int id = tid + it * THREADS;
                const int r = id / NGRP;
                const int64_t t = t0 + r;
#pragma unroll
                for (int v = 0; v < RW; v++) rd[k][v] = ru[k][v] = rz[k][v] = 0u;
                if (fast) {
                    lds_words<GRP * C::ESZ, RW>(&sRaw[0][r][cg], rd[k]);
                    lds_words<GRP * C::ESZ, RW>(&sRaw[1][r][cg], ru[k]);
                    if (GATE && z) lds_words<GRP * C::ESZ, RW>(&sRaw[GATE ? 2 : 1][r][cg], rz[k]);
                } else if (t < t_end) {
                    const int64_t off = (b * L + t) * Dch + d0 + cg;
                    load_run<T, GRP, RW>(delta, off, d0 + cg, Dch, false, rd[k]);
                    load_run<T, GRP, RW>(u, off, d0 + cg, Dch, false, ru[k]);
                    if (GATE && z) load_run<T, GRP, RW>(z, off, d0 + cg, Dch, false, rz[k]);
                }
            }
            float4 dv[IB][GRP / 2], gd[NOY || KEEP ? 1 : IB][GRP / 2];
#pragma unroll
            for (int k = 0; k < IB; k++) {
                const int it = ib + k;
                const bool rv = t0 + (tid + it * THREADS) / NGRP < t_end;
#pragma unroll
                for (int c = 0; c < GRP; c += 2) {
                    // two channels at a time with packed arithmetic
                    const float2 x = make_float2(elem<T>(rd[k], c) + biasv[c], elem<T>(rd[k], c + 1) + biasv[c + 1]);
                    // formed unconditionally and selected by the call's flag: a branch, even a
                    // uniform one, would split the items' interleaved chains
                    const float2 spf = softplus2(x);
                    const float2 sp = a.softplus ? spf : x;
                    const float2 uu = make_float2(elem<T>(ru[k], c), elem<T>(ru[k], c + 1));
                    const float2 spu = mul2(sp, uu);
                    const float2 dl = rv ? sp : make_float2(0.f, 0.f), dlu = rv ? spu : make_float2(0.f, 0.f);
                    dv[k][c / 2] = make_float4(dl.x, dl.y, dlu.x, dlu.y);
                    if constexpr (!NOY && !KEEP) {
                        float2 gt = make_float2(1.f, 1.f);
                        if (GATE && z) {
                            const float2 zz = make_float2(elem<T>(rz[k], c), elem<T>(rz[k], c + 1));
                            gt = mul2(zz, sigmoid2(zz));
                        }
                        const float2 dun = mul2(make_float2(dvv[c], dvv[c + 1]), uu);
                        gd[k][c / 2] = make_float4(gt.x, gt.y, dun.x, dun.y);  // read for rows before t_end only
                    }
                }
                if constexpr (!NOY && KEEP) {
#pragma unroll
                    for (int v = 0; v < RW; v++) kU[it][v] = ru[k][v];
                }
                if constexpr (GATE && KEEP) {
#pragma unroll
                    for (int v = 0; v < RW; v++) kZ[it][v] = rz[k][v];
                }
            }
#pragma unroll
            for (int k = 0; k < IB; k++) {
                const int r = (tid + (ib + k) * THREADS) / NGRP;
#pragma unroll
                for (int c = 0; c < GRP; c += 2) {
                    sDU[r][(cg + c) / 2] = dv[k][c / 2];
                    if constexpr (!NOY && !KEEP) sGD[r][(cg + c) / 2] = gd[k][c / 2];
                }
            }
        }
        if constexpr (!C::BC_DIRECT) {
#pragma unroll
            for (int k = 0; k < BCUT; k++) {
                const int id = tid + k * THREADS;
                const int row = id / BCU, n = (id % BCU) * BCV;
                const int half = row / kRow, r = row % kRow;
                float* dst = &sBC[half][0][r][n];
#pragma unroll
                for (int v = 0; v < BCV; v++) dst[v] = elem<T>(wv[k], v);  // zero past t_end
            }
        }
        // Staging complete; every thread is done reading sRaw / sBCraw.  A thread
        // whose wait for the tile ran out makes the whole block give up (the
        // block agrees here, so no thread is left at a later barrier): the status
        // word records it and the thread that issued the copies waits once more
        // for them before the block's shared memory is released.
        if (__syncthreads_or(!ok)) {
            if (tid == 0) {
                atomicOr(a.status, kDevWaitTimeout);
                mbar_wait(&sBar[buf], (uint32_t)((jt >> 1) & 1));
            }
            return;
        }
        if (t0 + kRow < t_end) issue(t0 + kRow, buf ^ 1);

        // ---- scan: 32 steps of the lane's 2 x S states.  Steps past t_end (last
        // tile only) carry delta_eff = 0 and B = 0: the state stays unchanged.
        // Software-pipelined by two steps: the decays and input terms of step
        // i + 2 (loads, exponents, MUFU) are formed before the recurrence of
        // step i, which is the only part that waits on the previous state.
        const float* brow = &sBC[0][C::BC_DIRECT ? buf : 0][0][0];
        const float* crow = &sBC[1][C::BC_DIRECT ? buf : 0][0][0];
        // decays, input terms and C values of the next two steps, by step parity
        float2 daQ[2][S], xbQ[2][S];
        float cQ[2][S] = {};
        auto prep = [&](int i, int sl) {
            const float4 du = sDU[i][pp];
            const float2 dl2 = make_float2(du.x, du.y), dlu2 = make_float2(du.z, du.w);
            if (SUMMARY) sdp = add2(sdp, dl2);  // delta_eff of steps past t_end is zero
            float Bv[S];
            ld_f32<S>(brow + i * N + n0, Bv);
            if (!NOY) ld_f32<S>(crow + i * N + n0, cQ[sl]);
#pragma unroll
            for (int s = 0; s < S; s++) {
                const float2 ex = mul2(dl2, A2[s]);
                daQ[sl][s] = make_float2(ex2a(ex.x), ex2a(ex.y));
                xbQ[sl][s] = mul2(dlu2, splat2(Bv[s]));
            }
        };
        prep(0, 0);
        prep(1, 1);
#pragma unroll
        for (int i = 0; i < kRow; i++) {
            if (SAVE && (i % kSub) == 0) {
                // the state entering step t0 + i (S states of c0 at the lane's slot of
                // channel 0, S of c1 at its slot of channel 1); every slot is written:
                // channels past Dch hold a zero state, and the slots of the last tile
                // past the sequence end (L rounded up to 32) the final state
                float* dst = ck_lane + ((t0 - t_begin + i) / kSub) * (CH * N);  // consecutive slots
                constexpr int E1 = 32 * S;  // ckpt_slot(w, lane, S, 1) - ckpt_slot(w, lane, S, 0)
                if constexpr (S == 4) {
                    *reinterpret_cast<float4*>(dst) = make_float4(h[0].x, h[1].x, h[2].x, h[3].x);
                    *reinterpret_cast<float4*>(dst + E1) = make_float4(h[0].y, h[1].y, h[2].y, h[3].y);
                } else {
#pragma unroll
                    for (int s = 0; s < S; s++) {
                        dst[s] = h[s].x;
                        dst[E1 + s] = h[s].y;
                    }
                }
            }
            const int sl = i & 1;
            float2 da[S], xb[S];
            float Cv[S];
#pragma unroll
            for (int s = 0; s < S; s++) {
                da[s] = daQ[sl][s];
                xb[s] = xbQ[sl][s];
                Cv[s] = cQ[sl][s];
            }
            if (i + 2 < kRow) prep(i + 2, sl);
#pragma unroll
            for (int s = 0; s < S; s++) h[s] = fma2(da[s], h[s], xb[s]);
            if (!NOY) {
                float2 ya = mul2(splat2(Cv[0]), h[0]);
#pragma unroll
                for (int s = 1; s < S; s++) ya = fma2(splat2(Cv[s]), h[s], ya);
                // both channels' partials of the lane; the epilogue adds the pair's lanes
                *reinterpret_cast<float2*>(&sY[w][g * C::YPL + i * YP + c0]) = ya;
            }
        }
        __syncthreads();

        // ---- epilogue: (step, 8-channel group) items; all items' sums and gates
        // first (rows past t_end too: their partial readouts are finite), then the
        // stores of the rows before t_end
        if (!NOY) {
#pragma unroll
            for (int ib = 0; ib < ITEMS; ib += IB) {
                float yv[IB][GRP], y0v[IB][GRP];
#pragma unroll
                for (int k = 0; k < IB; k++) {
                    const int it = ib + k;
                    const int r = (tid + it * THREADS) / NGRP;
#pragma unroll
                    for (int c = 0; c < GRP; c += 4) {
                        // per warp, the sum of its G lanes' planes; then the warps in order
                        float4 acc;
#pragma unroll
                        for (int ww = 0; ww < NW; ww++) {
                            float4 o = *reinterpret_cast<const float4*>(&sY[ww][r * YP + cg + c]);
#pragma unroll
                            for (int gg = 1; gg < G; gg++) {
                                const float4 v = *reinterpret_cast<const float4*>(&sY[ww][gg * C::YPL + r * YP + cg + c]);
                                o.x += v.x; o.y += v.y; o.z += v.z; o.w += v.w;
                            }
                            if (ww == 0) {
                                acc = o;
                            } else {
                                acc.x += o.x; acc.y += o.y; acc.z += o.z; acc.w += o.w;
                            }
                        }
                        // the pre-gate readout y0 = sum_n h C + D u, then the gate
                        const float sum4[4] = {acc.x, acc.y, acc.z, acc.w};
#pragma unroll
                        for (int e = 0; e < 4; e += 2) {
                            const int cc = c + e;
                            float2 y0, gt = make_float2(1.f, 1.f);
                            if constexpr (KEEP) {
                                const float2 uu = make_float2(elem<T>(kU[it], cc), elem<T>(kU[it], cc + 1));
                                y0 = fma2(make_float2(dvv[cc], dvv[cc + 1]), uu, make_float2(sum4[e], sum4[e + 1]));
                                if constexpr (GATE) {
                                    const float2 zz = make_float2(elem<T>(kZ[it], cc), elem<T>(kZ[it], cc + 1));
                                    const float2 gz = mul2(zz, sigmoid2(zz));  // selected, not branched on
                                    gt = z ? gz : make_float2(1.f, 1.f);
                                }
                            } else {
                                const float4 gd = sGD[r][(cg + cc) / 2];
                                y0 = add2(make_float2(sum4[e], sum4[e + 1]), make_float2(gd.z, gd.w));
                                gt = make_float2(gd.x, gd.y);
                            }
                            y0v[k][cc] = y0.x;
                            y0v[k][cc + 1] = y0.y;
                            yv[k][cc] = y0.x * gt.x;
                            yv[k][cc + 1] = y0.y * gt.y;
                        }
                    }
                }
#pragma unroll
                for (int k = 0; k < IB; k++) {
                    const int64_t t = t0 + (tid + (ib + k) * THREADS) / NGRP;
                    if (t >= t_end) continue;
                    const int64_t off = (b * L + t) * Dch + d0 + cg;
                    if (a.y0 && z) {
                        // kept for the backward's dz (f32; the same alignment as the io runs)
                        float* y0row = a.y0 + off;
                        if (sfast) {
#pragma unroll
                            for (int c = 0; c < GRP; c += 4)
                                *reinterpret_cast<float4*>(y0row + c) =
                                    make_float4(y0v[k][c], y0v[k][c + 1], y0v[k][c + 2], y0v[k][c + 3]);
                        } else {
#pragma unroll
                            for (int c = 0; c < GRP; c++)
                                if (d0 + cg + c < Dch) y0row[c] = y0v[k][c];
                        }
                    }
                    if (!GATE) continue;
                    T* yrow = static_cast<T*>(a.y) + off;
                    if (sfast) {
                        uint32_t wv[RW];
                        if constexpr (sizeof(T) == 4) {
#pragma unroll
                            for (int c = 0; c < GRP; c++) wv[c] = __float_as_uint(yv[k][c]);
                        } else {
#pragma unroll
                            for (int c = 0; c < GRP; c += 2) wv[c >> 1] = pack2<T>(yv[k][c], yv[k][c + 1]);
                        }
#pragma unroll
                        for (int v = 0; v < RW / 4; v++)
                            reinterpret_cast<uint4*>(yrow)[v] = make_uint4(wv[4 * v], wv[4 * v + 1], wv[4 * v + 2], wv[4 * v + 3]);
                    } else {
#pragma unroll
                        for (int c = 0; c < GRP; c++)
                            if (d0 + cg + c < Dch) st(yrow + c, yv[k][c]);
                    }
                }
            }
        }
        // the next prologue restages sDU / sGD / sBC only after every thread has
        // passed the scan barrier above, i.e. after the scan's reads; the epilogue's
        // reads of sGD / sY come before this thread's next prologue writes, and the
        // other threads write them again only after the next prologue's barrier
    }

    if (SUMMARY) {
        // every entry of the part is written (channels past Dch: zero state)
        const int64_t q = s_first + k;
        float* H0 = a.ws_fsum + (q * CH + c0) * N + n0;
#pragma unroll
        for (int s = 0; s < S; s++) {
            H0[s] = h[s].x;
            H0[N + s] = h[s].y;
        }
        if (w == 0 && g == 0) *reinterpret_cast<float2*>(a.ws_fsd + q * CH + c0) = sdp;
    } else if (MODE != kModeCkpt && k == sgm.K - 1 && a.last_state) {
#pragma unroll
        for (int s = 0; s < S; s++) {
            if (ok0) a.last_state[row0 * N + n0 + s] = h[s].x;
            if (ok1) a.last_state[row1 * N + n0 + s] = h[s].y;
        }
    }
}

// One launch of mode MODE over chunks k_lo .. k_hi of segment si.
template <typename T, int N, int MODE>
void launch_fwd_mode(const FwdArgs& a, const FPlan& p, int si, cudaStream_t st, int64_t k_lo, int64_t k_hi,
                     float* ckpt, const TmaMaps& maps) {
    prof_mark(st);
    k_fwd<T, N, MODE><<<(unsigned)(p.seg[si].nu * (k_hi - k_lo)), FCfg<T, N>::THREADS, 0, st>>>(a, p, si, k_lo, ckpt,
                                                                                               maps);
}

}  // namespace ss

#include "fsum.cuh"

namespace ss {

// The chunk summaries of every chunked segment, then each segment's main pass.
// A summary launch of more blocks than one round of the main kernel's
// residency (4 two-warp blocks per SM) runs the dedicated k_fwd_fsum, built
// for 6 resident blocks per SM so that it still takes one wave.  Otherwise the
// summary mode of k_fwd, which is about 3 % faster per step on long chunks
// (measured: the Mamba-130M bf16 forward's 768-block summaries 0.096 -> 0.076
// ms with k_fwd_fsum; the long sequence's 576 blocks 0.509 -> 0.522 ms).
template <typename T, int N>
cudaError_t launch_fwd_t(const FwdArgs& a, const FPlan& p, cudaStream_t st, int mode, float* ckpt,
                         const TmaMaps& maps) {
    for (int si = 0; si < p.nseg; si++) {
        const int64_t K = p.seg[si].K;
        if (K < 2) continue;
        const int64_t blocks = p.seg[si].nu * (K - 1);
        if constexpr (scan_warps(N) == 2) {
            if (blocks > round_blocks(N)) {
                prof_mark(st);
                k_fwd_fsum<T, N><<<(unsigned)blocks, FSCfg<T, N>::THREADS, 0, st>>>(a, p, si, 0, maps);
                continue;
            }
        }
        launch_fwd_mode<T, N, kModeSummary>(a, p, si, st, 0, K - 1, nullptr, maps);
    }
    for (int si = 0; si < p.nseg; si++) {
        const int64_t K = p.seg[si].K;
        if (mode == kModeCkpt) {
            launch_fwd_mode<T, N, kModeCkpt>(a, p, si, st, 0, K, ckpt, maps);
        } else if (ckpt) {
            launch_fwd_mode<T, N, kModeYSave>(a, p, si, st, 0, K, ckpt, maps);
        } else {
            launch_fwd_mode<T, N, kModeY>(a, p, si, st, 0, K, nullptr, maps);
        }
    }
    return cudaGetLastError();
}

// Forward launcher of one io type: switches on N.
template <typename T>
cudaError_t launch_fwd_io(const FwdArgs& a, const FPlan& p, cudaStream_t st, int mode, float* ckpt,
                          const TmaMaps& maps) {
    switch (a.N) {
        case 1: return launch_fwd_t<T, 1>(a, p, st, mode, ckpt, maps);
        case 2: return launch_fwd_t<T, 2>(a, p, st, mode, ckpt, maps);
        case 4: return launch_fwd_t<T, 4>(a, p, st, mode, ckpt, maps);
        case 8: return launch_fwd_t<T, 8>(a, p, st, mode, ckpt, maps);
        case 16: return launch_fwd_t<T, 16>(a, p, st, mode, ckpt, maps);
        case 32: return launch_fwd_t<T, 32>(a, p, st, mode, ckpt, maps);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace ss
