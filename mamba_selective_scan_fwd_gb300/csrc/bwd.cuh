// Backward selective scan: the chain rule of the forward definition
// (baracuda-kernels `selective_scan.rs`, "Algorithm summary") for the loss
// sum(dy * y), with the gradient structure of mamba-rs `gpu/backward.rs`
// (B2 gating backward, B3 SSM BPTT with local gradients then fixed-order
// reductions, B4 softplus backward on the raw delta), fused into one reverse
// pass per channel tile, recomputing states instead of storing them, and
// without atomics.
//
// Per step t, state n of channel d (lam = adjoint of h, "carry" = a_{t+1} lam_{t+1}):
//   g      = dy * silu(z)               dz     = dy * y0 * sig(z) * (1 + z (1 - sig(z)))
//   lam_n  = g * C_n + carry_n          carry_n <- a_{t,n} * lam_n
//   du     = g * D + Delta * sum_n lam_n B_n
//   dDelta = sum_n A_n q_n + u * sum_n lam_n B_n      with q_n = a_{t,n} lam_n h_{t-1,n}
//   ddelta = dDelta * sig(delta + bias) under softplus, else dDelta
//   dA_n  += Delta * q_n;   dB_n += lam_n * Delta * u;   dC_n += g * h_{t,n}
//
// Work split (the block layout of the forward: CH channels of one batch row
// and one time chunk; for N >= 16 two warps split the states of every
// channel; a lane holds S states of a channel pair):
//   * the forward (ss_fwd_save) or a checkpoint pass stores the state
//     entering every kSub-th step, and the pre-gate readout y0 that dz needs;
//   * this kernel visits kSub-step tiles from the end of the chunk backwards
//     (staged by TMA in pairs of tiles for two-warp blocks).  The tile
//     prologue computes the per-(t, d) terms once (softplus and its
//     derivative, the gate, g, dz, which it stores at once): the walk's
//     (delta_eff, delta_eff * u, g) into shared memory, and u, the softplus
//     derivative, delta_eff and g in the item thread's registers for its
//     epilogue (in shared memory where they do not fit).  Each lane then
//     recomputes the tile's states forward from the saved one, keeping the
//     kSub states in registers, and walks the adjoint backwards, evaluating
//     each step's decays again, one step ahead of the adjoint that needs them
//     (MUFU has room to spare; the registers do not);
//   * per step each lane stores its two channels' sums over its states, and
//     each warp sums dB / dC of its states over the block's channels through
//     shared memory in a fixed order; the tile epilogue adds the lanes' and
//     warps' per-(t, d) sums and writes du and ddelta; a second kernel adds
//     the per-tile dB / dC partials, a third the per-(unit, chunk)
//     dA / dD / ddelta_bias partials.  Every sum has a fixed order: the
//     result is bit-reproducible.
// The walk is bound by the SM's FP32 pipe (eleven FP32 operations per state
// and step, against one or two MUFU operations), so every FP32 operation
// there is a packed f32x2 instruction on two states (s, s + 1) of one
// channel: states, decays, adjoints and their products stay natural
// register pairs, and the per-channel terms (delta_eff, delta_eff * u, g)
// enter as broadcast scalars, which cost no instruction.
// Chunks (units the plan cuts in time, kernels.h): each chunk's carry-in
// state is its first saved state; reverse summaries (P_k, M_k) -- the chunk's
// decay product, from its sum of delta_eff as exp(A sum delta_eff), and
// M_k = a_{s_k} lam_{s_k} with lam from a zero incoming carry -- combine as
// rho_{k-1} = M_k + P_k rho_k into each chunk's carry-in adjoint.
#pragma once

#include <atomic>

#include "common.cuh"
#include "kernels.h"
#include "simd.cuh"
#include "tiles.cuh"

namespace ss {

constexpr int kTT = kSub;  // backward tile: steps staged per prologue, one recompute window

template <typename T, int N>
struct BCfg {
    static constexpr int NW = scan_warps(N);        // warps per block (they split the states)
    static constexpr int NPW = N / NW;              // states per warp
    static constexpr int S = lane_states(N);        // states per lane (of each of its two channels)
    static constexpr int SP = S >= 2 ? S / 2 : 1;   // state pairs per channel (a lone state for S = 1)
    static constexpr int G = NPW / S;               // lanes per channel pair
    static constexpr int PAIRS = 32 / G;            // channel pairs per block
    static constexpr int CH = 2 * PAIRS;            // channels per block
    static constexpr int THREADS = 32 * NW;
    static constexpr int ESZ = (int)sizeof(T);
    // channels per prologue / epilogue item: 4, or 2 where that leaves a thread
    // without an item (N = 32: 16 channels per block)
    static constexpr int GRP = kTT * CH / THREADS >= 4 ? 4 : 2;
    static constexpr int NGRP = CH / GRP;           // items per step
    static constexpr int ITEMS = kTT * NGRP / THREADS;  // items per thread per tile
    static constexpr int RWH = GRP * ESZ >= 4 ? GRP * ESZ / 4 : 1;  // 32-bit words of an item's run
    static constexpr int NB = N * ESZ;
    // B / C staging: a step's row is B (N values) then C.  The lanes load S of
    // each per step as broadcasts, and the shared-memory data pipe -- which
    // bounds this kernel -- returns one 32-bit word per lane per cycle however
    // few distinct addresses a warp reads: so bf16 rows stay packed (a lane's
    // four states are two words, widened by ALU bit operations) and are copied
    // in raw, double buffered; f32 rows are copied straight in (double
    // buffered); f16 rows are converted by the prologue
    // (each staged as one dense [step][N] array per tensor: the layout a TMA
    // box lands in)
    static constexpr bool BC_PK = std::is_same<T, __nv_bfloat16>::value && S == 4;
    static constexpr bool BC_DIRECT = ESZ == 4;
    static constexpr bool BC_RAW = !BC_DIRECT && !BC_PK && NB >= 4;
    static constexpr int BC_BUFS = BC_DIRECT ? 2 : 1;
    // f16 rows are copied and converted in units of BCV values of one row,
    // consecutive threads taking consecutive units (free of bank conflicts)
    static constexpr int BCV = N >= 4 ? 4 : N;
    static constexpr int BCU = N / BCV;             // units per row
    // u and the softplus derivative of a thread's prologue items stay in its
    // registers for its epilogue items (the same items) when they are few; else
    // the prologue stages them in shared memory
    static constexpr bool KEEP = ITEMS * (RWH + GRP) <= 8;
    // likewise delta_eff and g (which the walk reads from shared memory)
    static constexpr bool KEEP2 = KEEP && ITEMS * GRP <= 4;
    static constexpr int EP = CH + 4;               // padded per-channel rows (floats)
    // plane of per-step channel sums of one lane of a pair: kTT rows of EP floats,
    // planes 16 mod 32 floats apart so that the 8-byte stores of the lanes of
    // two planes hit different banks
    static constexpr int OPL = kTT * EP + 16;
    // dB / dC staging of one warp: block (step j, tensor tau) holds PAIRS rows
    // of NPW floats (the warp's states, summed over the pair's two channels),
    // padded to a stride of NPW floats mod 32: the reads of reduce_staged (lane
    // = (block, run of states), one pair's row at a time) then cover the 32
    // banks exactly once per wavefront of lanes (8 lanes of 16-byte reads)
    static constexpr int BLK = PAIRS * NPW + ((NPW - PAIRS * NPW) % 32 + 32) % 32;
    static_assert(BLK % 32 == NPW % 32, "staging stride");
    // blocks per SM the register budget must allow: one round of the plan on
    // every SM (8 warps: 4 two-warp or 8 one-warp blocks), which leaves the
    // walk up to 255 registers
    static constexpr int MINB = NW == 2 ? 4 : 8;
    // Tiles per staging copy ("a pair"): two for two-warp blocks.  A TMA copy
    // holds its issuing thread for some 60 - 100 cycles whatever its size, so
    // the copies of a tile's eight tensors cost the issuing warp about as much
    // as the tile's recompute; a copy of two tiles halves that per step, for
    // 8 KB more shared memory (a one-warp block keeps one tile per copy: 8 of
    // them share an SM).
    static constexpr int TPP = NW == 2 ? 2 : 1;
    static_assert(kTT * NGRP % THREADS == 0, "whole items per thread");
    static_assert(CH == channels_per_block(N), "channel tile of the plan");
    static_assert(S * G * NW == N, "the lanes cover the states");
};

// Sum the kTT staged steps of one warp (block (j, tau) holds step t + j of
// tensor tau) over its PAIRS staged rows (channel pairs) and store the sums
// as the warp's states n_w .. n_w + NPW of the dB / dC partial rows bc0[t + j],
// bc1[t + j] (rows of N floats; steps at or past t_end are not stored).  Work
// unit: V consecutive states of one (step, tensor); the rows are added as a
// fixed pairwise tree (p, p + 1), then pairs of pairs, ...
template <int PAIRS, int NPW, int N, int BLK>
__device__ __forceinline__ void reduce_staged(const float* sR, float* bc0, float* bc1, int n_w, int64_t t,
                                              int64_t t_end, int lane) {
    constexpr int V = NPW % 4 == 0 ? 4 : (NPW % 2 == 0 ? 2 : 1);
    constexpr int UPB = NPW / V;                 // units per (step, tensor) block
    constexpr int UNITS = kTT * 2 * UPB;
#pragma unroll
    for (int u0 = 0; u0 < UNITS; u0 += 32) {
        const int unit = u0 + lane;
        if (UNITS % 32 == 0 || unit < UNITS) {
            const int blk = unit / UPB, nv = (unit % UPB) * V;
            const int j = blk / 2, tau = blk % 2;
            const float* src = sR + blk * BLK + nv;
            float* dst = (tau ? bc1 : bc0) + (t + j) * N + n_w + nv;
            if constexpr (V == 4) {
                float4 v[PAIRS];
#pragma unroll
                for (int c = 0; c < PAIRS; c++) v[c] = *reinterpret_cast<const float4*>(src + c * NPW);
#pragma unroll
                for (int wd = 1; wd < PAIRS; wd <<= 1) {
#pragma unroll
                    for (int c = 0; c < PAIRS; c += 2 * wd) {
                        const float2 lo = add2(make_float2(v[c].x, v[c].y), make_float2(v[c + wd].x, v[c + wd].y));
                        const float2 hi = add2(make_float2(v[c].z, v[c].w), make_float2(v[c + wd].z, v[c + wd].w));
                        v[c] = make_float4(lo.x, lo.y, hi.x, hi.y);
                    }
                }
                if (t + j < t_end) *reinterpret_cast<float4*>(dst) = v[0];
            } else if constexpr (V == 2) {
                float2 v[PAIRS];
#pragma unroll
                for (int c = 0; c < PAIRS; c++) v[c] = *reinterpret_cast<const float2*>(src + c * NPW);
#pragma unroll
                for (int wd = 1; wd < PAIRS; wd <<= 1) {
#pragma unroll
                    for (int c = 0; c < PAIRS; c += 2 * wd) v[c] = add2(v[c], v[c + wd]);
                }
                if (t + j < t_end) *reinterpret_cast<float2*>(dst) = v[0];
            } else {
                float v[PAIRS];
#pragma unroll
                for (int c = 0; c < PAIRS; c++) v[c] = src[c * NPW];
#pragma unroll
                for (int wd = 1; wd < PAIRS; wd <<= 1) {
#pragma unroll
                    for (int c = 0; c < PAIRS; c += 2 * wd) v[c] += v[c + wd];
                }
                if (t + j < t_end) dst[0] = v[0];
            }
        }
    }
}

// CPL consecutive f32 outputs at p (channel c0 of the row): vector stores
// when aligned and complete, else element stores up to Dch.
template <int CPL>
__device__ __forceinline__ void store_run(float* p, const float (&v)[CPL], int64_t c0, int64_t Dch, bool fast) {
    if (fast) {
        if constexpr (CPL % 4 == 0) {
#pragma unroll
            for (int c = 0; c < CPL; c += 4)
                *reinterpret_cast<float4*>(p + c) = make_float4(v[c], v[c + 1], v[c + 2], v[c + 3]);
            return;
        } else if constexpr (CPL == 2) {
            *reinterpret_cast<float2*>(p) = make_float2(v[0], v[1]);
            return;
        }
    }
#pragma unroll
    for (int c = 0; c < CPL; c++)
        if (c0 + c < Dch) p[c] = v[c];
}

// MODE kRevMain: the backward proper.  MODE kRevSummary: only the adjoint
// walk of chunks 1..K-1 from a zero carry, writing (sum of delta_eff, M_k).  STATE: the
// call has an incoming gradient of last_state or wants dh0 (a separate
// instantiation, so that the plain backward carries none of it).
constexpr int kRevMain = 0, kRevSummary = 1;

template <typename T, int N, int MODE, bool STATE>
__global__ void __launch_bounds__(32 * scan_warps(N), BCfg<T, N>::MINB) k_bwd(BwdArgs a, FPlan p, int si,
                                                                              int64_t k_lo,
                                                                              const __grid_constant__ TmaMaps maps) {
    using C = BCfg<T, N>;
    constexpr bool MAIN = MODE == kRevMain;
    constexpr int NW = C::NW, NPW = C::NPW, S = C::S, SP = C::SP, G = C::G, PAIRS = C::PAIRS, CH = C::CH,
                  THREADS = C::THREADS, GRP = C::GRP, NGRP = C::NGRP, ITEMS = C::ITEMS, RWH = C::RWH,
                  EP = C::EP, BLK = C::BLK, TPP = C::TPP;
    constexpr int kSTT = TPP * kTT;  // steps per staging copy
    // per-(t, d) staging of the walk, one entry per channel pair
    __shared__ float4 sDU[kTT][PAIRS + 1];  // (Delta of both channels, Delta*u of both channels)
    // g of both channels (rows of PAIRS + 1 entries: the prologue's 8-byte stores
    // of two rows, a half-warp, fall on distinct banks)
    __shared__ float2 sG[kTT][PAIRS + 1];
    // (u of both channels, sig(delta + bias) of both channels), for the epilogue
    // when they do not stay in registers
    __shared__ float4 sUS[MAIN && !C::KEEP ? kTT : 1][MAIN && !C::KEEP ? PAIRS + 1 : 1];
    // Staging is by pairs of TPP tiles (kSTT steps): tile m is part m % TPP of
    // pair m / TPP, whose buffer is (m / TPP) & 1.
    // B / C rows as f32 (B then C): with f32 io the pairs' rows double buffered,
    // the next pair's being copied in while the current one is walked; with f16
    // the current tile's rows, converted by its prologue
    __shared__ __align__(128) float sBC[2][C::BC_BUFS][C::BC_PK ? 1 : (C::BC_DIRECT ? kSTT : kTT)][C::BC_PK ? 4 : N];
    // packed bf16 B / C rows (B, then C) of the pairs, double buffered: the walk
    // reads them directly
    __shared__ __align__(128) T sBCpk[2][C::BC_PK ? 2 : 1][C::BC_PK ? kSTT : 1][C::BC_PK ? N : 8];
    // raw 16-bit B / C rows of the next pair (converted into sBC by the prologues)
    __shared__ __align__(128) T sBCraw[2][C::BC_RAW ? kSTT : 1][C::BC_RAW ? N : 8];
    // completion of the TMA copies into the two pair buffers
    __shared__ __align__(8) uint64_t sBar[2];
    // raw runs of delta, u, dy, z of the next pair, copied in asynchronously by
    // the thread that later converts them
    __shared__ __align__(128) T sRaw[4][kSTT][CH];
    // the forward's pre-gate readout y0 of the next pair (for dz), likewise
    __shared__ __align__(128) float sY0[MAIN ? kSTT : 1][MAIN ? CH : 4];
    // dB / dC contributions of the tile's kTT steps, per warp: block (j, tau)
    // holds a row of NPW floats per pair
    __shared__ __align__(16) float sR[MAIN ? NW : 1][MAIN ? kTT * 2 * BLK : 4];
    // per-step sums over a lane's states: sum lam B, sum A q, one plane per
    // lane of a pair (float g OPL + r EP + c: lane g's sum for step r, channel c)
    __shared__ __align__(16) float sOu[MAIN ? NW : 1][MAIN ? G * C::OPL : 4];
    __shared__ __align__(16) float sOd[MAIN ? NW : 1][MAIN ? G * C::OPL : 4];
    // dD / ddelta_bias partials of each epilogue thread's items at the end (thread fastest)
    __shared__ float sAcc[MAIN ? 2 : 1][MAIN ? ITEMS * GRP : 1][THREADS];
    // the states entering the tiles of a pair (the recompute windows' starts:
    // TPP saved-state blocks of 2 S floats per lane), double buffered
    __shared__ __align__(128) float sH[MAIN ? 2 : 1][MAIN ? TPP * THREADS * 2 * S : 4];
    __shared__ float sBias[CH], sDv[CH];

    const FwdArgs& f = a.f;
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    // block -> (unit, chunk) of segment si; unit -> (batch row, channel tile)
    const Seg sgm = seg_at(p, si);
    const int64_t ul = (int64_t)blockIdx.x % sgm.nu;
    const int64_t k = k_lo + (int64_t)blockIdx.x / sgm.nu;
    const int64_t unit = sgm.u_lo + ul;
    const int64_t tile = unit % p.tiles_b, b = unit / p.tiles_b;
    const int64_t q_first = sgm.q0 + ul * sgm.K;  // part of the unit's chunk 0
    const int64_t s_first = sgm.s0 + ul * sgm.K;  // its summary index
    const int64_t L = f.L, Dch = f.Dch;
    const int64_t d0 = tile * CH;
    const T* u = static_cast<const T*>(f.u);
    const T* delta = static_cast<const T*>(f.delta);
    const T* Bm = static_cast<const T*>(f.B);
    const T* Cm = static_cast<const T*>(f.C);
    const T* z = static_cast<const T*>(f.z);
    const T* dy = static_cast<const T*>(a.dy);

    for (int c = tid; c < CH; c += THREADS) {
        const int64_t dc = d0 + c < Dch ? d0 + c : Dch - 1;
        sBias[c] = f.delta_bias ? f.delta_bias[dc] : 0.f;
        sDv[c] = f.D ? f.D[dc] : 0.f;
    }

    // scan-lane identity: channel pair pp (channels c0, c0 + 1 of the block),
    // states n0 .. n0 + S of both (warp w holds n_w .. n_w + NPW)
    const int pp = lane / G, g = lane % G;
    const int c0 = 2 * pp;
    const bool ok[2] = {d0 + c0 < Dch, d0 + c0 + 1 < Dch};
    const int64_t dd[2] = {ok[0] ? d0 + c0 : Dch - 1, ok[1] ? d0 + c0 + 1 : Dch - 1};
    const int n_w = w * NPW;
    const int n0 = n_w + g * S;
    const int64_t row[2] = {b * Dch + dd[0], b * Dch + dd[1]};
    // Registers pair two states (s, s + 1) of one channel: X[c][j] holds states
    // n0 + 2 j, n0 + 2 j + 1 of channel c0 + c (S = 1: the lone state in .x).
    // A2 = A * log2(e); the dDelta partial sums below use A2 and are scaled back
    // by ln 2 in the epilogue.  Channels past Dch run with a zero exponent, state
    // and adjoint: with u = dy = z = 0 loaded there, everything they form stays
    // exactly zero, so their dB / dC contributions need no masking.
    // The adjoint carry into the end of the sequence is the incoming gradient of
    // last_state (zero without one); a reverse summary starts from zero.
    const bool from_dlast = MAIN && STATE && a.dlast != nullptr;
    float2 A2[2][SP], carry[2][SP], dA[2][SP];
    float sd[2] = {0.f, 0.f};  // reverse summary: the chunk's sums of delta_eff
#pragma unroll
    for (int e = 0; e < 2; e++) {
#pragma unroll
        for (int j = 0; j < SP; j++) {
            const int s0 = 2 * j, s1 = S >= 2 ? 2 * j + 1 : 0;
            A2[e][j] = make_float2(ok[e] ? scan_A(f, dd[e] * N + n0 + s0) * kLog2eF : 0.f,
                                   ok[e] && S >= 2 ? scan_A(f, dd[e] * N + n0 + s1) * kLog2eF : 0.f);
            carry[e][j] = make_float2(from_dlast && ok[e] ? a.dlast[row[e] * N + n0 + s0] : 0.f,
                                      from_dlast && ok[e] && S >= 2 ? a.dlast[row[e] * N + n0 + s1] : 0.f);
            dA[e][j] = make_float2(0.f, 0.f);
        }
    }
    if (MAIN && k + 1 < sgm.K) {
        // carry into the end of chunk k (rho_{j-1} = M_j + P_j rho_j over the
        // reverse summaries of the unit's chunks K-1 .. k+1, P_j = exp2(A2 * sum
        // of delta_eff over chunk j), from rho_{K-1} the carry into the end of
        // the sequence), which k_bwd_carry left over the summary of chunk k + 1
#pragma unroll
        for (int e = 0; e < 2; e++) {
            const float* M = a.ws_rsum + ((s_first + k + 1) * CH + c0 + e) * N + n0;
#pragma unroll
            for (int j = 0; j < SP; j++)
                carry[e][j] = ok[e] ? make_float2(M[2 * j], S >= 2 ? M[2 * j + 1] : 0.f) : make_float2(0.f, 0.f);
        }
    }
    // dD / ddelta_bias partials of the thread's epilogue items (the same channels
    // in every tile), added over the tiles in order; summed per channel at the end
    float accD[ITEMS * GRP], accB[ITEMS * GRP];
#pragma unroll
    for (int c = 0; c < ITEMS * GRP; c++) accD[c] = accB[c] = 0.f;
    // the raw run of u and the softplus derivatives of the thread's items, from
    // its prologue to its epilogue (when they stay in registers)
    uint32_t kU[C::KEEP ? ITEMS : 1][RWH];
    float kS[C::KEEP ? ITEMS : 1][GRP], kDl[C::KEEP2 ? ITEMS : 1][GRP], kG[C::KEEP2 ? ITEMS : 1][GRP];

    // TMA boxes land on 128-byte aligned shared memory; a block whose buffers are
    // not (never expected) records it and stages with asynchronous copies instead
    bool tma = f.use_tma != 0;
    if (tma && !(smem_aligned128(&sRaw[0][0][0]) && smem_aligned128(&sBC[0][0][0][0]) &&
                 smem_aligned128(&sBCpk[0][0][0][0]) && smem_aligned128(&sBCraw[0][0][0]) &&
                 smem_aligned128(&sY0[0][0]) && smem_aligned128(&sH[0][0]))) {
        if (tid == 0) atomicOr(f.status, kDevMisaligned);
        tma = false;
    }
    // the tile's runs are read from shared memory: TMA boxes (zero-filled past Dch),
    // or whole aligned vectors copied in asynchronously
    const bool pfast = tma || (((Dch * (int64_t)sizeof(T)) % 16 == 0) && (d0 + CH <= Dch));
    const bool ofast = (Dch % 4 == 0) && (d0 + CH <= Dch);
    const int64_t t_begin = k * sgm.Lc;
    const int64_t t_end = t_begin + sgm.Lc < L ? t_begin + sgm.Lc : L;
    const int64_t ntile = (t_end - t_begin + kTT - 1) / kTT;
    // saved states (layout of ckpt_bytes): one block of CH x N floats per
    // (batch, channel tile, slot), consecutive slots contiguous; the lane's 2 S
    // floats at its slots
    const float* ck_unit = a.ws_ckpt + ckpt_block(p, b, tile, t_begin / kSub, N);  // the chunk's first slot
    float* bc0 = a.ws_bc + ((int64_t)tile * f.Bsz + b) * L * N;                  // dB partials of this tile
    float* bc1 = a.ws_bc + ((int64_t)(p.tiles_b + tile) * f.Bsz + b) * L * N;    // dC partials
    float* sRw = &sR[MAIN ? w : 0][0];
    constexpr int HB = THREADS * 2 * S;  // floats of one saved-state block

    // Copies of tile pair pp (its tiles TPP pp .. TPP pp + TPP - 1) into buffer pp & 1.
    // With TMA: one thread issues a box per tensor (delta, u, dy, z as
    // [kSTT][CH], y0 as f32 [kSTT][CH], B and C as [kSTT][N]: bf16 packed into
    // sBCpk, f32 into sBC, f16 raw into sBCraw) and one bulk copy of the pair's
    // TPP blocks of saved states (CH x N floats each, in lane order) into sH,
    // on the buffer's barrier.  Otherwise, one commit group of asynchronous
    // copies: the thread's item runs and y0 runs of the pair's tiles (when the
    // rows are whole aligned vectors), the B / C rows, and the lane's states
    // entering the tiles into its own slots of sH; each thread converts the
    // runs it copied and the states are read by the lane that copied them.
    const TmaMaps& mp = maps;
    auto issue = [&](int64_t pp) {
        const int64_t tt = t_begin + pp * kSTT;
        const int buf = (int)(pp & 1);
        if (tma) {
            if (tid == 0) {
                constexpr uint32_t run = kSTT * CH * C::ESZ, row = kSTT * N * C::ESZ, state = TPP * CH * N * 4;
                const uint32_t bytes = (MAIN ? 3 : 2) * run + (z ? run : 0) + (MAIN && z ? kSTT * CH * 4 : 0) +
                                       (MAIN ? 2 : 1) * row + (MAIN ? state : 0);
                mbar_expect_tx(&sBar[buf], bytes);
                const int x = (int)d0, y = (int)tt, zc = (int)b;
                tma_load_3d(&sRaw[0][0][0], &mp.m[kMapDelta], x, y, zc, &sBar[buf]);
                if (MAIN) tma_load_3d(&sRaw[1][0][0], &mp.m[kMapU], x, y, zc, &sBar[buf]);
                tma_load_3d(&sRaw[2][0][0], &mp.m[kMapDy], x, y, zc, &sBar[buf]);
                if (z) tma_load_3d(&sRaw[3][0][0], &mp.m[kMapZ], x, y, zc, &sBar[buf]);
                if (MAIN && z) tma_load_3d(&sY0[0][0], &mp.m[kMapY0], x, y, zc, &sBar[buf]);
#pragma unroll
                for (int half = MAIN ? 0 : 1; half < 2; half++) {
                    void* dst;
                    if constexpr (C::BC_PK) dst = &sBCpk[half][buf][0][0];
                    else if constexpr (C::BC_DIRECT) dst = &sBC[half][buf][0][0];
                    else dst = &sBCraw[half][0][0];
                    tma_load_3d(dst, &mp.m[half ? kMapC : kMapB], 0, y, zc, &sBar[buf]);
                }
                // the pair's slots always exist: slots run to L rounded up to 32 steps
                if (MAIN) bulk_load(&sH[buf][0], ck_unit + (tt - t_begin) / kSub * (CH * N), state, &sBar[buf]);
            }
            return;
        }
        if (pfast) {
#pragma unroll
            for (int it = 0; it < ITEMS; it++) {
                const int id = tid + it * THREADS;
                const int r0 = id / NGRP, cg = (id % NGRP) * GRP;
#pragma unroll
                for (int hh = 0; hh < TPP; hh++) {
                    const int r = hh * kTT + r0;
                    const int64_t t = tt + r;
                    if (t < t_end) {
                        const int64_t off = (b * L + t) * Dch + d0 + cg;
                        cp_async_bytes<GRP * C::ESZ>(&sRaw[0][r][cg], delta + off);
                        cp_async_bytes<GRP * C::ESZ>(&sRaw[1][r][cg], u + off);
                        cp_async_bytes<GRP * C::ESZ>(&sRaw[2][r][cg], dy + off);
                        if (z) cp_async_bytes<GRP * C::ESZ>(&sRaw[3][r][cg], z + off);
                        if (MAIN && z) cp_async_bytes<GRP * 4>(&sY0[r][cg], a.y0 + off);
                    }
                }
            }
        }
        for (int id = tid; id < (MAIN ? 2 : 1) * kSTT; id += THREADS) {
            const int half = MAIN ? id / kSTT : 1, r = id % kSTT;
            const int64_t t = tt + r;
            const T* src = (half ? Cm : Bm) + (b * L + (t < t_end ? t : 0)) * N;
            if constexpr (C::BC_PK) {
                T* dst = &sBCpk[half][buf][r][0];
                if (t < t_end) {
                    cp_async_bytes<N * C::ESZ>(dst, src);
                } else {
#pragma unroll
                    for (int n = 0; n < N; n += 2) *reinterpret_cast<uint32_t*>(dst + n) = 0u;
                }
            } else if constexpr (C::BC_DIRECT) {
                float* dst = &sBC[half][buf][r][0];
                if (t < t_end) {
                    cp_async_bytes<N * 4>(dst, src);
                } else {
#pragma unroll
                    for (int n = 0; n < N; n++) dst[n] = 0.f;
                }
            }
        }
        if constexpr (C::BC_RAW) {
            // in the prologue's conversion units
            for (int id = tid; id < (MAIN ? 2 : 1) * kSTT * C::BCU; id += THREADS) {
                const int row = id / C::BCU, n = (id % C::BCU) * C::BCV;
                const int half = MAIN ? row / kSTT : 1, r = row % kSTT;
                const int64_t t = tt + r;
                if (t < t_end) cp_async_bytes<C::BCV * C::ESZ>(&sBCraw[half][r][n], (half ? Cm : Bm) + (b * L + t) * N + n);
            }
        }
        if (MAIN) {
            // the block's layout: the lane's S states of each channel at its two slots
#pragma unroll
            for (int hh = 0; hh < TPP; hh++) {
                const float* src = ck_unit + ((tt - t_begin) / kSub + hh) * (CH * N) + ckpt_slot(w, lane, S, 0);
                float* dst = &sH[buf][hh * HB + ckpt_slot(w, lane, S, 0)];
                cp_async_bytes<S * 4>(dst, src);
                cp_async_bytes<S * 4>(dst + 32 * S, src + 32 * S);
            }
        }
        cp_async_commit();
    };
    if (tma && tid == 0) {
        mbar_init(&sBar[0], 1);
        mbar_init(&sBar[1], 1);
        fence_proxy_async_smem();
    }
    const int64_t npair = (ntile + TPP - 1) / TPP;
    issue(npair - 1);
    __syncthreads();  // sBias / sDv and the barriers before the first prologue
    // the thread's prologue / epilogue items cover the same channel group in every
    // tile (THREADS is a multiple of NGRP): its biases and D stay in registers
    static_assert(THREADS % NGRP == 0, "one channel group per thread");
    float biasv[GRP], dvv[GRP];
#pragma unroll
    for (int c = 0; c < GRP; c++) {
        biasv[c] = sBias[(tid % NGRP) * GRP + c];
        dvv[c] = sDv[(tid % NGRP) * GRP + c];
    }

    for (int64_t m = ntile - 1; m >= 0; m--) {
        const int64_t t0 = t_begin + m * kTT;
        const int64_t pr = m / TPP;            // the tile's pair
        const int buf = (int)(pr & 1);         // its staging buffer
        const int part = (int)(m % TPP);       // the tile's part of the pair
        const int hrow = part * kTT;           // its rows within the pair's staging
        // the pair's copies, awaited by the first of its tiles to be visited (the
        // last one): this thread's own (asynchronous copies), or the TMA boxes
        // (the pairs are visited from the last, so the buffer's barrier completes
        // its phase (npair - 1 - pr) / 2 mod 2)
        const uint32_t phase = (uint32_t)(((npair - 1 - pr) >> 1) & 1);
        bool ok = true;
        if (part == TPP - 1 || m == ntile - 1) {
            if (tma) ok = mbar_wait(&sBar[buf], phase);
            else cp_async_wait<0>();
        }
        // ---- prologue: (step, GRP-channel group) items of the tile; dz is final here
#pragma unroll
        for (int it = 0; it < ITEMS; it++) {
            const int id = tid + it * THREADS;
            const int r = id / NGRP, q = id % NGRP;
            const int cg = q * GRP;
            const int64_t t = t0 + r;
            const bool rv = t < t_end;
            uint32_t rd[RWH], ru[RWH], rz[RWH], rg[RWH];
            float vy0[GRP];
#pragma unroll
            for (int c = 0; c < GRP; c++) vy0[c] = 0.f;
#pragma unroll
            for (int v = 0; v < RWH; v++) rd[v] = ru[v] = rz[v] = rg[v] = 0u;
            // The terms are formed for every row without branching (the thread's
            // items then interleave); rows past t_end keep zero terms.  Shared-
            // memory runs are read for every row: TMA zero-fills rows past the
            // tensor, and other rows past t_end hold earlier data, discarded below.
            if (pfast) {
                lds_words<GRP * C::ESZ, RWH>(&sRaw[0][hrow + r][cg], rd);
                lds_words<GRP * C::ESZ, RWH>(&sRaw[1][hrow + r][cg], ru);
                lds_words<GRP * C::ESZ, RWH>(&sRaw[2][hrow + r][cg], rg);
                if (z) lds_words<GRP * C::ESZ, RWH>(&sRaw[3][hrow + r][cg], rz);
                if (MAIN && z) ld_f32<GRP>(&sY0[hrow + r][cg], vy0);
            } else if (rv) {
                const int64_t off = (b * L + t) * Dch + d0 + cg;
                load_run<T, GRP, RWH>(delta, off, d0 + cg, Dch, false, rd);
                load_run<T, GRP, RWH>(u, off, d0 + cg, Dch, false, ru);
                load_run<T, GRP, RWH>(dy, off, d0 + cg, Dch, false, rg);
                if (z) load_run<T, GRP, RWH>(z, off, d0 + cg, Dch, false, rz);
                if (MAIN && z) {
                    const float* y0r = a.y0 + off;
#pragma unroll
                    for (int c = 0; c < GRP; c++) vy0[c] = d0 + cg + c < Dch ? y0r[c] : 0.f;
                }
            }
            if (!rv) {
                // discarded rows: zero u, dy, z and y0 (then g, dz and the dD terms
                // are exactly zero, whatever the staging held)
#pragma unroll
                for (int v = 0; v < RWH; v++) ru[v] = rg[v] = rz[v] = 0u;
#pragma unroll
                for (int c = 0; c < GRP; c++) vy0[c] = 0.f;
            }
            float vdz[GRP];
            float4 dv[GRP / 2];  // the item's sDU and sG entries, stored after its arithmetic
            float2 gv[GRP / 2];
#pragma unroll
            for (int c = 0; c < GRP; c += 2) {
                // two channels at a time with packed arithmetic
                float2 dl2, sg2, dz2 = make_float2(0.f, 0.f);
                const float2 x = make_float2(elem<T>(rd, c) + biasv[c], elem<T>(rd, c + 1) + biasv[c + 1]);
                // the softplus and the gate terms are formed unconditionally and selected
                // by the call's flags: a branch, even a uniform one, would split the
                // items' interleaved chains (without z the run rz holds zeros)
                {
                    float2 spd, sgd;
                    softplus_sigmoid2(x, spd, sgd);
                    dl2 = f.softplus ? spd : x;
                    sg2 = f.softplus ? sgd : make_float2(1.f, 1.f);
                }
                dl2 = rv ? dl2 : make_float2(0.f, 0.f);
                const float2 uu2 = make_float2(elem<T>(ru, c), elem<T>(ru, c + 1));
                const float2 dlu2 = mul2(dl2, uu2);
                const float2 dyv = make_float2(elem<T>(rg, c), elem<T>(rg, c + 1));
                float2 gg2;
                {
                    const float2 zz = make_float2(elem<T>(rz, c), elem<T>(rz, c + 1));
                    const float2 sz = sigmoid2(zz);
                    const float2 dsz = mul2(dyv, sz);
                    const float2 gz = mul2(dsz, zz);
                    // dz = dy sig(z) (1 + z (1 - sig(z))) y0
                    const float2 dzf = mul2(dsz, fma2(zz, add2(splat2(1.f), make_float2(-sz.x, -sz.y)), splat2(1.f)));
                    const float2 dzv = mul2(dzf, make_float2(vy0[c], vy0[c + 1]));
                    gg2 = z ? gz : dyv;
                    dz2 = z ? dzv : make_float2(0.f, 0.f);
                }
                const int pr = (cg + c) / 2;
                dv[c / 2] = make_float4(dl2.x, dl2.y, dlu2.x, dlu2.y);
                gv[c / 2] = gg2;
                if (MAIN) {
                    if constexpr (C::KEEP2) {
                        kDl[it][c] = dl2.x;
                        kDl[it][c + 1] = dl2.y;
                        kG[it][c] = gg2.x;
                        kG[it][c + 1] = gg2.y;
                    }
                    if constexpr (C::KEEP) {
                        kS[it][c] = sg2.x;
                        kS[it][c + 1] = sg2.y;
                    } else {
                        sUS[r][pr] = make_float4(uu2.x, uu2.y, sg2.x, sg2.y);
                    }
                    accD[it * GRP + c] = fmaf(gg2.x, uu2.x, accD[it * GRP + c]);  // g = u = 0 past t_end
                    accD[it * GRP + c + 1] = fmaf(gg2.y, uu2.y, accD[it * GRP + c + 1]);
                }
                vdz[c] = dz2.x; vdz[c + 1] = dz2.y;
            }
#pragma unroll
            for (int j = 0; j < GRP / 2; j++) {
                sDU[r][cg / 2 + j] = dv[j];
                sG[r][cg / 2 + j] = gv[j];
            }
            if (MAIN) {
                if (z && rv) store_run<GRP>(a.dz + (b * L + t) * Dch + d0 + cg, vdz, d0 + cg, Dch, ofast);
            }
            if constexpr (MAIN && C::KEEP) {
#pragma unroll
                for (int v = 0; v < RWH; v++) kU[it][v] = ru[v];
            }
        }
        if constexpr (!C::BC_DIRECT && !C::BC_PK) {
            // 16-bit B / C rows of the tile's steps (the reverse summary needs only C),
            // in units of BCV values of one row, converted by the thread that copied
            // them (or loaded here when too short to copy)
            constexpr int BCV = C::BCV, BCU = C::BCU, VW = BCV * C::ESZ >= 4 ? BCV * C::ESZ / 4 : 1;
            for (int id = tid; id < (MAIN ? 2 : 1) * kTT * BCU; id += THREADS) {
                const int row = id / BCU, n = (id % BCU) * BCV;
                const int half = MAIN ? row / kTT : 1, r = row % kTT;
                const int64_t t = t0 + r;
                uint32_t wv[VW];
                if (t < t_end) {
                    if constexpr (C::BC_RAW) lds_words<BCV * C::ESZ, VW>(&sBCraw[half][hrow + r][n], wv);
                    else load_words<BCV * C::ESZ, VW>((half ? Cm : Bm) + (b * L + t) * N + n, wv);
                }
                float* dst = &sBC[half][0][r][n];
#pragma unroll
                for (int v = 0; v < BCV; v++) dst[v] = t < t_end ? elem<T>(wv, v) : 0.f;
            }
        }
        // Staging complete; every thread is done reading sRaw / sY0 / sBCraw.  A
        // thread whose wait for the tile ran out makes the whole block give up
        // (the block agrees here, so no thread is left at a later barrier): the
        // status word records it and the thread that issued the copies waits once
        // more for them before the block's shared memory is released.
        if (__syncthreads_or(!ok)) {
            if (tid == 0) {
                atomicOr(f.status, kDevWaitTimeout);
                mbar_wait(&sBar[buf], phase);
            }
            return;
        }
        // the pair's staging has been read by all its tiles' prologues once its
        // first tile (part 0, visited last) passes this barrier
        if (part == 0 && pr > 0) issue(pr - 1);
        // S values of row i's B (half 0) or C (half 1) from the lane's states
        auto ld_bc = [&](int i, int half, float (&v)[S]) {
            if constexpr (C::BC_PK) ld_bf16x4(&sBCpk[half][buf][hrow + i][n0], v);
            else if constexpr (C::BC_DIRECT) ld_f32<S>(&sBC[half][buf][hrow + i][n0], v);
            else ld_f32<S>(&sBC[half][0][i][n0], v);
        };

        if constexpr (!MAIN) {
            // ---- reverse summary: adjoint walk from a zero carry and the chunk's
            // decay product, no states needed
            for (int i = kTT - 1; i >= 0; i--) {
                if (t0 + i >= t_end) continue;
                const float4 du = sDU[i][pp];
                const float2 g2 = sG[i][pp];
                sd[0] += du.x;
                sd[1] += du.y;
                float Cv[S];
                ld_bc(i, 1, Cv);
#pragma unroll
                for (int e = 0; e < 2; e++) {
                    const float2 dl = splat2(e ? du.y : du.x), gg = splat2(e ? g2.y : g2.x);
#pragma unroll
                    for (int j = 0; j < SP; j++) {
                        const float2 Cp = make_float2(Cv[2 * j], S >= 2 ? Cv[2 * j + 1] : 0.f);
                        const float2 x = mul2(dl, A2[e][j]);
                        const float2 lam = fma2(gg, Cp, carry[e][j]);
                        carry[e][j] = mul2(make_float2(ex2a(x.x), ex2a(x.y)), lam);
                    }
                }
            }
            __syncthreads();  // the walk has read what the next prologue restages
        } else {
            // ---- the tile's window: recompute its kTT states forward from the state
            // entering it, then walk the adjoint backwards.  Steps past the chunk end
            // (last tile only) hold Delta = g = 0 and B = C = 0 in the staging: they
            // leave the state and the adjoint unchanged and add nothing; only their
            // per-step stores are skipped.
            // the state entering the tile (the lane's slots in sH), as state pairs
            const float* hsrc = &sH[buf][part * HB + ckpt_slot(w, lane, S, 0)];
            auto load_hs = [&](float2 (&hs)[2][SP]) {
#pragma unroll
                for (int e = 0; e < 2; e++) {
                    float v[S];
                    ld_f32<S>(hsrc + e * 32 * S, v);  // ckpt_slot(w, lane, S, e)
#pragma unroll
                    for (int j = 0; j < SP; j++) hs[e][j] = make_float2(v[2 * j], S >= 2 ? v[2 * j + 1] : 0.f);
                }
            };
            float2 hv[kTT][2][SP];  // the states after each step of the window
            float2 hs[2][SP];       // the state entering it (kept for the walk's last step)
            {
                load_hs(hs);
#pragma unroll
                for (int i = 0; i < kTT; i++) {
                    const float4 du = sDU[i][pp];
                    float Bv[S];
                    ld_bc(i, 0, Bv);
#pragma unroll
                    for (int e = 0; e < 2; e++) {
                        const float2 dl = splat2(e ? du.y : du.x), dlu = splat2(e ? du.w : du.z);
#pragma unroll
                        for (int j = 0; j < SP; j++) {
                            const float2 Bp = make_float2(Bv[2 * j], S >= 2 ? Bv[2 * j + 1] : 0.f);
                            const float2 x = mul2(dl, A2[e][j]);
                            const float2 da = make_float2(ex2a(x.x), ex2a(x.y));
                            const float2 bu = mul2(dlu, Bp);
                            hv[i][e][j] = fma2(da, i > 0 ? hv[i - 1][e][j] : hs[e][j], bu);
                        }
                    }
                }
            }
            // the walk, software-pipelined by one step: the inputs and decays of
            // step i - 1 are formed before the adjoint of step i
            float4 duN;
            float2 gN, daN[2][SP];
            float BN[S], CN[S];
            auto prepw = [&](int i) {
                duN = sDU[i][pp];
                gN = sG[i][pp];
                ld_bc(i, 0, BN);
                ld_bc(i, 1, CN);
#pragma unroll
                for (int e = 0; e < 2; e++) {
                    const float2 dl = splat2(e ? duN.y : duN.x);
#pragma unroll
                    for (int j = 0; j < SP; j++) {
                        const float2 x = mul2(dl, A2[e][j]);
                        daN[e][j] = make_float2(ex2a(x.x), ex2a(x.y));
                    }
                }
            };
            prepw(kTT - 1);
#pragma unroll
            for (int i = kTT - 1; i >= 0; i--) {
                const float4 du = duN;
                const float2 g2 = gN;
                float2 da[2][SP];
                float Bv[S], Cv[S];
#pragma unroll
                for (int e = 0; e < 2; e++)
#pragma unroll
                    for (int j = 0; j < SP; j++) da[e][j] = daN[e][j];
#pragma unroll
                for (int s = 0; s < S; s++) {
                    Bv[s] = BN[s];
                    Cv[s] = CN[s];
                }
                if (i > 0) prepw(i - 1);
                float2 hp[2][SP];  // the states entering step i
                if (i > 0) {
#pragma unroll
                    for (int e = 0; e < 2; e++)
#pragma unroll
                        for (int j = 0; j < SP; j++) hp[e][j] = hv[i - 1][e][j];
                } else {
#pragma unroll
                    for (int e = 0; e < 2; e++)
#pragma unroll
                        for (int j = 0; j < SP; j++) hp[e][j] = hs[e][j];
                }
                float2 cB[SP], cC[SP];
                float sumB[2], sumQ[2];
#pragma unroll
                for (int e = 0; e < 2; e++) {
                    const float2 dl = splat2(e ? du.y : du.x), dlu = splat2(e ? du.w : du.z),
                                 gg = splat2(e ? g2.y : g2.x);
                    float2 sBp = make_float2(0.f, 0.f), sQp = sBp;
#pragma unroll
                    for (int j = 0; j < SP; j++) {
                        const float2 Bp = make_float2(Bv[2 * j], S >= 2 ? Bv[2 * j + 1] : 0.f);
                        const float2 Cp = make_float2(Cv[2 * j], S >= 2 ? Cv[2 * j + 1] : 0.f);
                        const float2 lam = fma2(gg, Cp, carry[e][j]);
                        sBp = fma2(lam, Bp, sBp);
                        const float2 cn = mul2(da[e][j], lam);
                        const float2 q = mul2(cn, hp[e][j]);
                        sQp = fma2(A2[e][j], q, sQp);
                        dA[e][j] = fma2(dl, q, dA[e][j]);
                        // dB / dC contributions summed over the pair's two channels
                        cB[j] = e ? fma2(lam, dlu, cB[j]) : mul2(lam, dlu);
                        cC[j] = e ? fma2(gg, hv[i][e][j], cC[j]) : mul2(gg, hv[i][e][j]);
                        carry[e][j] = cn;
                    }
                    sumB[e] = S >= 2 ? sBp.x + sBp.y : sBp.x;
                    sumQ[e] = S >= 2 ? sQp.x + sQp.y : sQp.x;
                }
                // the lane's sums over its states, both channels; the epilogue adds
                // the G lanes of the pair and the warps
                {
                    const int o = g * C::OPL + i * EP + c0;
                    *reinterpret_cast<float2*>(&sOu[w][o]) = make_float2(sumB[0], sumB[1]);
                    *reinterpret_cast<float2*>(&sOd[w][o]) = make_float2(sumQ[0], sumQ[1]);
                }
                // stage dB / dC contributions (summed over the pairs below)
                {
                    float* r0 = sRw + (2 * i) * BLK + pp * NPW + g * S;
                    float* r1 = r0 + BLK;
                    if constexpr (S == 4) {
                        *reinterpret_cast<float4*>(r0) = make_float4(cB[0].x, cB[0].y, cB[1].x, cB[1].y);
                        *reinterpret_cast<float4*>(r1) = make_float4(cC[0].x, cC[0].y, cC[1].x, cC[1].y);
                    } else if constexpr (S == 2) {
                        *reinterpret_cast<float2*>(r0) = cB[0];
                        *reinterpret_cast<float2*>(r1) = cC[0];
                    } else {
                        r0[0] = cB[0].x;
                        r1[0] = cC[0].x;
                    }
                }
            }
            __syncwarp();  // staged contributions visible to every lane of the warp
            reduce_staged<PAIRS, NPW, N, BLK>(sRw, bc0, bc1, n_w, t0, t_end, lane);
            __syncwarp();  // the sums have read the staging before the next tile restages it
            __syncthreads();  // every warp's per-step sums are in sOu / sOd
            // ---- epilogue: du, ddelta of the (step, GRP-channel group) items.
            // Steps past t_end (last tile only) are not stored and add nothing.
#pragma unroll
            for (int it = 0; it < ITEMS; it++) {
                const int id = tid + it * THREADS;
                const int r = id / NGRP, q = id % NGRP;
                const int cg = q * GRP;
                const int64_t t = t0 + r;
                const bool tv = t < t_end;
                // per warp, the sum of its G lanes' planes; then the warps in order
                float su[GRP], sdv[GRP];
#pragma unroll
                for (int ww = 0; ww < NW; ww++) {
                    float ou[GRP], od[GRP];
                    ld_f32<GRP>(&sOu[ww][r * EP + cg], ou);
                    ld_f32<GRP>(&sOd[ww][r * EP + cg], od);
#pragma unroll
                    for (int gg = 1; gg < G; gg++) {
                        float pu[GRP], pd[GRP];
                        ld_f32<GRP>(&sOu[ww][gg * C::OPL + r * EP + cg], pu);
                        ld_f32<GRP>(&sOd[ww][gg * C::OPL + r * EP + cg], pd);
#pragma unroll
                        for (int c = 0; c < GRP; c++) {
                            ou[c] += pu[c];
                            od[c] += pd[c];
                        }
                    }
#pragma unroll
                    for (int c = 0; c < GRP; c++) {
                        su[c] = ww == 0 ? ou[c] : su[c] + ou[c];
                        sdv[c] = ww == 0 ? od[c] : sdv[c] + od[c];
                    }
                }
                float vdu[GRP], vdx[GRP];
#pragma unroll
                for (int c = 0; c < GRP; c += 2) {
                    // two channels at a time with packed arithmetic; the item's per-(t, d)
                    // terms as its prologue staged them
                    const int pr = (cg + c) / 2;
                    float2 dl2, gg2;
                    if constexpr (C::KEEP2) {
                        dl2 = make_float2(kDl[it][c], kDl[it][c + 1]);
                        gg2 = make_float2(kG[it][c], kG[it][c + 1]);
                    } else {
                        const float4 dlu = sDU[r][pr];
                        dl2 = make_float2(dlu.x, dlu.y);
                        gg2 = sG[r][pr];
                    }
                    float4 us;
                    if constexpr (C::KEEP) us = make_float4(elem<T>(kU[it], c), elem<T>(kU[it], c + 1), kS[it][c], kS[it][c + 1]);
                    else us = sUS[r][pr];
                    const float2 Dv = make_float2(dvv[c], dvv[c + 1]);
                    const float2 su2 = make_float2(su[c], su[c + 1]);
                    const float2 du2 = fma2(gg2, Dv, mul2(dl2, su2));
                    const float2 dx2 = mul2(fma2(make_float2(us.x, us.y), su2,
                                                 mul2(make_float2(sdv[c], sdv[c + 1]), splat2(kLn2))),
                                            make_float2(us.z, us.w));
                    vdu[c] = du2.x; vdu[c + 1] = du2.y;
                    vdx[c] = dx2.x; vdx[c + 1] = dx2.y;
                }
#pragma unroll
                for (int c = 0; c < GRP; c++) accB[it * GRP + c] += tv ? vdx[c] : 0.f;
                if (tv) {
                    const int64_t off = (b * L + t) * Dch + d0 + cg;
                    store_run<GRP>(a.du + off, vdu, d0 + cg, Dch, ofast);
                    store_run<GRP>(a.ddelta + off, vdx, d0 + cg, Dch, ofast);
                }
            }
            // No barrier here: the epilogue reads the per-step sums (the next ones
            // are written after the next prologue's barrier) and the staged terms
            // of its own items, which only this thread's next prologue rewrites
            // (the walk's reads of them ended before the barrier above).
        }
    }

    const int64_t q = q_first + k;  // this block's part
    if constexpr (!MAIN) {
        // every entry of the summary is written (channels past Dch: zero carry)
        const int64_t qs = s_first + k;
#pragma unroll
        for (int e = 0; e < 2; e++) {
            float* M = a.ws_rsum + (qs * CH + c0 + e) * N + n0;
#pragma unroll
            for (int j = 0; j < SP; j++) {
                M[2 * j] = carry[e][j].x;
                if (S >= 2) M[2 * j + 1] = carry[e][j].y;
            }
        }
        if (w == 0 && g == 0) *reinterpret_cast<float2*>(a.ws_rsd + qs * CH + c0) = make_float2(sd[0], sd[1]);
    } else {
#pragma unroll
        for (int e = 0; e < 2; e++) {
            if (ok[e]) {
                float* o = a.ws_dA + (q * CH + c0 + e) * N + n0;
#pragma unroll
                for (int j = 0; j < SP; j++) {
                    o[2 * j] = dA[e][j].x;
                    if (S >= 2) o[2 * j + 1] = dA[e][j].y;
                }
                // after the walk of the first chunk the carry is a_0 lam_0, the gradient of h0
                if (STATE && k == 0 && a.dh0) {
#pragma unroll
                    for (int j = 0; j < SP; j++) {
                        a.dh0[row[e] * N + n0 + 2 * j] = carry[e][j].x;
                        if (S >= 2) a.dh0[row[e] * N + n0 + 2 * j + 1] = carry[e][j].y;
                    }
                }
            }
        }
        // dD / ddelta_bias of each channel: the partials of the items that own it
        // (one per step of the tile) added in step order
#pragma unroll
        for (int c = 0; c < ITEMS * GRP; c++) {
            sAcc[0][c][tid] = accD[c];
            sAcc[1][c][tid] = accB[c];
        }
        __syncthreads();
        for (int cc = tid; cc < CH; cc += THREADS) {
            if (d0 + cc < Dch) {
                const int qg = cc / GRP, c = cc % GRP;
                float aD = 0.f, ab = 0.f;
#pragma unroll
                for (int r = 0; r < kTT; r++) {
                    const int id = r * NGRP + qg;
                    const int th = id % THREADS, itr = id / THREADS;
                    aD += sAcc[0][itr * GRP + c][th];
                    ab += sAcc[1][itr * GRP + c][th];
                }
                a.ws_dD[q * CH + cc] = aD;
                a.ws_db[q * CH + cc] = ab;
            }
        }
    }
}

}  // namespace ss

#include "rsum.cuh"

namespace ss {

// Ask for the largest shared-memory carveout for `kernel`, so that shared
// memory does not cap residency: once per device (a kernel attribute of the
// current device, not a stream operation, so that calls captured into a CUDA
// graph after a first eager call on that device make no such call).  `done`
// holds one bit per device ordinal; threads that race both set it.
template <typename K>
cudaError_t prefer_max_shared(K kernel, std::atomic<uint64_t>& done) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = dev >= 0 && dev < 64 ? uint64_t(1) << dev : 0;
    if (bit != 0 && (done.load(std::memory_order_acquire) & bit) != 0) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                             (int)cudaSharedmemCarveoutMaxShared);
    if (e == cudaSuccess && bit != 0) done.fetch_or(bit, std::memory_order_release);
    return e;
}

template <typename T, int N>
cudaError_t launch_bwd_t(const BwdArgs& a, const FPlan& p, cudaStream_t st, float* ckpt_out, const TmaMaps& fmaps,
                         const TmaMaps& bmaps) {
    cudaError_t e = cudaSuccess;
    if (ckpt_out) {
        // checkpoint pass (with forward summaries first when the sequence is chunked)
        e = launch_fwd(a.f, p, st, kModeCkpt, ckpt_out, fmaps);
        if (e != cudaSuccess) return e;
    }
    constexpr int threads = BCfg<T, N>::THREADS;
    // reverse summaries of every chunked segment (chunks 1 .. K-1): the
    // dedicated kernel for two-warp blocks (32-step tiles through the forward's
    // maps), the main kernel's summary mode for one-warp blocks (whose 32- or
    // 64-channel tiles would need too much shared memory there)
    static std::atomic<uint64_t> rsum_carveout_done{0};
    if constexpr (BCfg<T, N>::NW == 2) {
        bool any = false;
        for (int si = 0; si < p.nseg; si++) any = any || p.seg[si].K > 1;
        if (any) {
            e = prefer_max_shared(k_bwd_rsum<T, N>, rsum_carveout_done);
            if (e != cudaSuccess) return e;
        }
    }
    for (int si = 0; si < p.nseg; si++) {
        const int64_t K = p.seg[si].K;
        if (K > 1) {
            prof_mark(st);
            const unsigned grid = (unsigned)(p.seg[si].nu * (K - 1));
            if constexpr (BCfg<T, N>::NW == 2) k_bwd_rsum<T, N><<<grid, threads, 0, st>>>(a, p, si, 1, fmaps);
            else k_bwd<T, N, kRevSummary, false><<<grid, threads, 0, st>>>(a, p, si, 1, bmaps);
        }
    }
    // their carry passes: each chunk's incoming adjoint carry from the later chunks' summaries
    for (int si = 0; si < p.nseg; si++) {
        if (p.seg[si].K < 2) continue;
        e = launch_bwd_carry(a, p, si, st);
        if (e != cudaSuccess) return e;
    }
    const bool state = a.dlast != nullptr || a.dh0 != nullptr;
    auto main_kernel = state ? k_bwd<T, N, kRevMain, true> : k_bwd<T, N, kRevMain, false>;
    // one bit per device ordinal: the carveout preference is set on that device
    static std::atomic<uint64_t> carveout_done[2] = {{0}, {0}};
    e = prefer_max_shared(main_kernel, carveout_done[state]);
    if (e != cudaSuccess) return e;
    for (int si = 0; si < p.nseg; si++) {
        prof_mark(st);
        main_kernel<<<(unsigned)(p.seg[si].nu * p.seg[si].K), threads, 0, st>>>(a, p, si, 0, bmaps);
    }
    return cudaGetLastError();
}

// Backward launcher of one io type: switches on N.
template <typename T>
cudaError_t launch_bwd_io(const BwdArgs& a, const FPlan& p, cudaStream_t st, float* ckpt_out, const TmaMaps& fmaps,
                          const TmaMaps& bmaps) {
    switch (a.f.N) {
        case 1: return launch_bwd_t<T, 1>(a, p, st, ckpt_out, fmaps, bmaps);
        case 2: return launch_bwd_t<T, 2>(a, p, st, ckpt_out, fmaps, bmaps);
        case 4: return launch_bwd_t<T, 4>(a, p, st, ckpt_out, fmaps, bmaps);
        case 8: return launch_bwd_t<T, 8>(a, p, st, ckpt_out, fmaps, bmaps);
        case 16: return launch_bwd_t<T, 16>(a, p, st, ckpt_out, fmaps, bmaps);
        case 32: return launch_bwd_t<T, 32>(a, p, st, ckpt_out, fmaps, bmaps);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace ss
