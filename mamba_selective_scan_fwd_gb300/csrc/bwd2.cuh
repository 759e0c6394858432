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
// channel):
//   * the forward (ss_fwd_save) or a checkpoint pass stores the state at the
//     start of every kSub-step sub-chunk, and the pre-gate readout y0 that
//     dz needs;
//   * this kernel visits kTT-step tiles from the end of the chunk backwards.
//     The tile prologue computes the per-(t, d) terms once (softplus and its
//     derivative, the gate, g, the dz factor): the walk's (delta_eff,
//     delta_eff * u, g) go to shared memory, and the thread keeps its items'
//     terms in registers for its own epilogue; then each sub-chunk is
//     recomputed forward from its saved state, keeping its states and decays
//     in registers, and the adjoint walks it backwards;
//   * per step each lane stores its two channels' partial sums over its
//     states, and each warp sums dB / dC of its states over the block's
//     channels through shared memory in a fixed order; the tile epilogue
//     adds the lanes' and warps' per-(t, d) sums, takes y0 from the forward,
//     and writes du, ddelta, dz; a second kernel adds the per-tile dB / dC
//     partials, a third the per-(unit, chunk) dA / dD / ddelta_bias
//     partials.  Every sum has a fixed order: the result is bit-reproducible.
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

constexpr int kTT = 8;   // backward tile: steps staged per prologue
constexpr int kRB = 4;   // steps whose dB / dC contributions are reduced together (one sub-chunk)
static_assert(kRB == kSub, "one staged sub-chunk of dB / dC contributions at a time");
static_assert(kTT % kSub == 0, "a tile holds whole sub-chunks");

template <typename T, int N>
struct BCfg {
    static constexpr int NW = fwd_warps(N);         // warps per block (they split the states)
    static constexpr int NPW = N / NW;              // states per warp
    static constexpr int G = NPW >= 2 ? 2 : 1;      // lanes per channel pair
    static constexpr int S = NPW / G;               // states per lane (of each of its two channels)
    static constexpr int PAIRS = 32 / G;            // channel pairs per block
    static constexpr int CH = 2 * PAIRS;            // channels per block
    static constexpr int THREADS = 32 * NW;
    static constexpr int ESZ = (int)sizeof(T);
    static constexpr int GRP = 4;                   // channels per prologue / epilogue item
    static constexpr int NGRP = CH / GRP;           // items per step
    static constexpr int ITEMS = kTT * NGRP / THREADS;  // items per thread per tile
    static constexpr int RWH = GRP * ESZ / 4;       // 32-bit words of an item's run of one tensor
    static constexpr int NB = N * ESZ;
    static constexpr int NWd = NB >= 4 ? NB / 4 : 1;
    // B / C staging as in the forward: N / S state groups of 2 S floats per step
    static constexpr int BCF = 2 * N + 4;
    static constexpr bool BC_DIRECT = ESZ == 4;
    static constexpr bool BC_RAW = !BC_DIRECT && N * ESZ >= 4;
    static constexpr int BC_BUFS = BC_DIRECT ? 2 : 1;
    // raw row length (elements): rows of 32 bytes or more padded by 16 bytes, so
    // that the 16-byte loads of consecutive rows fall in different bank groups
    static constexpr int RAWP = NB >= 32 ? N + 16 / ESZ : N;
    static constexpr int EP = CH + 4;               // padded per-channel rows (floats)
    static constexpr int GP = PAIRS + 8;            // padded per-pair float2 rows
    // plane of per-step channel sums of one lane of a pair: kTT rows of EP floats,
    // planes 16 mod 32 floats apart so that the 8-byte stores of both lanes of
    // the pairs of a half warp hit 32 banks
    static constexpr int OPL = kTT * EP + 16;
    // dB / dC staging of one warp: block (step slot j, tensor tau) holds PAIRS
    // rows of NPW floats (the warp's states, summed over the pair's two
    // channels); blocks are padded by 8 floats so that the 16 lanes of a half
    // warp reading 8-byte pairs of four consecutive blocks hit 32 banks
    static constexpr int BLK = PAIRS * NPW + 8;
    // blocks per SM the register budget must allow: one round of the plan on
    // every SM (8 warps: 4 two-warp or 8 one-warp blocks), which leaves the
    // scan up to 255 registers (N = 16 takes 237 and about 20 % less time
    // than at 168)
    static constexpr int MINB = NW == 2 ? 4 : 8;
    static_assert(kTT * NGRP % THREADS == 0, "whole items per thread");
    static_assert(CH == channels_per_block(N), "channel tile of the plan");
};

// Slot of channel pair pp in a per-step staging row: the two pairs of a
// 4-channel item go to slots q and q + PAIRS / 2; a quarter warp of prologue
// threads (eight items of one step) then hits eight different bank groups.
template <int PAIRS>
__device__ __forceinline__ int bpair_slot(int pp) {
    return (pp >> 1) + (PAIRS / 2) * (pp & 1);
}

template <int S>
__device__ __forceinline__ void ld_state(const float* p, float (&v)[S]) {
    if constexpr (S % 4 == 0) {
#pragma unroll
        for (int q = 0; q < S; q += 4) {
            const float4 f = *reinterpret_cast<const float4*>(p + q);
            v[q] = f.x; v[q + 1] = f.y; v[q + 2] = f.z; v[q + 3] = f.w;
        }
    } else if constexpr (S == 2) {
        const float2 f = *reinterpret_cast<const float2*>(p);
        v[0] = f.x; v[1] = f.y;
    } else {
        v[0] = p[0];
    }
}

// Stage one step's dB / dC contributions (slot j of kRB) in shared memory:
// block (j, tau) holds one row of NPW floats per channel pair, the warp's
// states summed over the pair's two channels.  Channels past Dch need no
// masking: their u, dy and z load as zero, so lam * Delta * u and g * h are
// exactly zero there.
template <int S, int NPW, int BLK>
__device__ __forceinline__ void stage_contrib(float* sR, int j, const float (&cB)[S], const float (&cC)[S], int pp,
                                              int gs) {
    float* r0 = sR + (2 * j) * BLK + pp * NPW + gs;
    float* r1 = r0 + BLK;
    if constexpr (S % 4 == 0) {
#pragma unroll
        for (int s = 0; s < S; s += 4) {
            *reinterpret_cast<float4*>(r0 + s) = make_float4(cB[s], cB[s + 1], cB[s + 2], cB[s + 3]);
            *reinterpret_cast<float4*>(r1 + s) = make_float4(cC[s], cC[s + 1], cC[s + 2], cC[s + 3]);
        }
    } else if constexpr (S == 2) {
        *reinterpret_cast<float2*>(r0) = make_float2(cB[0], cB[1]);
        *reinterpret_cast<float2*>(r1) = make_float2(cC[0], cC[1]);
    } else {
        r0[0] = cB[0];
        r1[0] = cC[0];
    }
}

// Sum the kRB staged steps of one warp (slot j holds time step t + j) over
// the CH staged rows (channel pairs) and store the sums as the warp's states
// n_w .. n_w + NPW of the dB / dC partial rows bc0[t + j], bc1[t + j] (rows
// of N floats; steps at or past t_end are not stored).  Work unit: a pair of
// consecutive states of one (step, tensor); the rows are added as a fixed
// pairwise tree (c, c + 1), then pairs of pairs, ...
template <int CH, int NPW, int N, int BLK>
__device__ __forceinline__ void reduce_staged(const float* sR, float* bc0, float* bc1, int n_w, int64_t t,
                                              int64_t t_end, int lane) {
    if constexpr (NPW % 2 == 0) {
        constexpr int UPB = NPW / 2;               // units per (step, tensor) block
        constexpr int UNITS = kRB * 2 * UPB;
#pragma unroll
        for (int u0 = 0; u0 < UNITS; u0 += 32) {
            const int unit = u0 + lane;
            if (UNITS % 32 == 0 || unit < UNITS) {
                const int blk = unit / UPB, n2 = (unit % UPB) * 2;
                const int j = blk / 2, tau = blk % 2;
                const float* src = sR + blk * BLK + n2;
                float2 v[CH];
#pragma unroll
                for (int c = 0; c < CH; c++) v[c] = *reinterpret_cast<const float2*>(src + c * NPW);
#pragma unroll
                for (int wd = 1; wd < CH; wd <<= 1) {
#pragma unroll
                    for (int c = 0; c < CH; c += 2 * wd) v[c] = add2(v[c], v[c + wd]);
                }
                if (t + j < t_end)
                    *reinterpret_cast<float2*>((tau ? bc1 : bc0) + (t + j) * N + n_w + n2) = v[0];
            }
        }
    } else {
        for (int o = lane; o < kRB * 2 * NPW; o += 32) {
            const int blk = o / NPW, n = o % NPW;
            const int j = blk / 2, tau = blk % 2;
            const float* src = sR + blk * BLK + n;
            float v[CH];
#pragma unroll
            for (int c = 0; c < CH; c++) v[c] = src[c * NPW];
#pragma unroll
            for (int wd = 1; wd < CH; wd <<= 1) {
#pragma unroll
                for (int c = 0; c < CH; c += 2 * wd) v[c] += v[c + wd];
            }
            if (t + j < t_end) (tau ? bc1 : bc0)[(t + j) * N + n_w + n] = v[0];
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
__global__ void __launch_bounds__(32 * fwd_warps(N), BCfg<T, N>::MINB) k_bwd2(BwdArgs a, FPlan p, int si,
                                                                               int64_t k_lo) {
    using C = BCfg<T, N>;
    constexpr bool MAIN = MODE == kRevMain;
    constexpr int NW = C::NW, NPW = C::NPW, S = C::S, G = C::G, PAIRS = C::PAIRS, CH = C::CH,
                  THREADS = C::THREADS, GRP = C::GRP, NGRP = C::NGRP, ITEMS = C::ITEMS, RWH = C::RWH,
                  NWd = C::NWd, BCF = C::BCF, EP = C::EP, GP = C::GP, BLK = C::BLK;
    // per-(t, d) staging of the scan, one entry per channel pair at bpair_slot
    __shared__ float4 sDU[kTT][PAIRS + 1];  // (Delta, Delta*u) of both channels
    __shared__ float2 sG[kTT][GP];          // g of both channels
    // B / C values by state group (f32); with f32 io double buffered, the next
    // tile's rows being copied in while the current tile is walked
    __shared__ __align__(16) float sBC[C::BC_BUFS][kTT][BCF];
    // raw bf16 B / C rows of the next tile (converted into sBC by the prologue)
    __shared__ __align__(16) T sBCraw[2][C::BC_RAW ? kTT : 1][C::BC_RAW ? C::RAWP : 2];
    // raw runs of delta, u, dy, z of the next tile, copied in asynchronously by
    // the thread that later converts them
    __shared__ __align__(16) T sRaw[4][kTT][CH];
    // dB / dC contributions of kRB steps, per warp: block (j, tau) holds a row of NPW floats per pair
    __shared__ __align__(16) float sR[MAIN ? NW : 1][MAIN ? kRB * 2 * BLK : 4];
    // per-step sums over a lane's states: sum lam B, sum A q, one plane per
    // lane of a pair (float g OPL + r EP + c: lane g's sum for step r, channel c)
    __shared__ __align__(16) float sOu[MAIN ? NW : 1][MAIN ? G * C::OPL : 4];
    __shared__ __align__(16) float sOd[MAIN ? NW : 1][MAIN ? G * C::OPL : 4];
    // the forward's pre-gate readout y0 of the tile, copied by the epilogue
    // thread that reads it, double buffered by tile
    __shared__ __align__(16) float sY0[MAIN ? 2 : 1][MAIN ? kTT : 1][MAIN ? CH : 4];
    // dD / ddelta_bias partials of each epilogue thread's items at the end (thread fastest)
    __shared__ float sAcc[MAIN ? 2 : 1][MAIN ? ITEMS * GRP : 1][THREADS];
    // restart states of a tile's sub-chunks, S floats per lane and channel
    // parity (one plane per parity: a warp's loads are contiguous), double
    // buffered by tile
    __shared__ __align__(16) float sH[MAIN ? 2 : 1][MAIN ? kTT / kSub : 1][2][MAIN ? THREADS * S : 4];
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
    const int sg = n0 / S;
    const int pslot = bpair_slot<PAIRS>(pp);
    const int64_t row[2] = {b * Dch + dd[0], b * Dch + dd[1]};
    // A2 = A * log2(e); the dDelta partial sums below use A2 and are scaled back
    // by ln 2 in the epilogue.  Channels past Dch run with a zero exponent, state
    // and adjoint: with u = dy = z = 0 loaded there, everything they form stays
    // exactly zero, so their dB / dC contributions need no masking.
    // The adjoint carry into the end of the sequence is the incoming gradient of
    // last_state (zero without one); a reverse summary starts from zero.
    const bool from_dlast = MAIN && STATE && a.dlast != nullptr;
    float A2[2][S], carry[2][S], dA[2][S];
    float sd[2] = {0.f, 0.f};  // reverse summary: the chunk's sums of delta_eff
#pragma unroll
    for (int e = 0; e < 2; e++) {
#pragma unroll
        for (int s = 0; s < S; s++) {
            A2[e][s] = ok[e] ? scan_A(f, dd[e] * N + n0 + s) * kLog2eF : 0.f;
            carry[e][s] = from_dlast && ok[e] ? a.dlast[row[e] * N + n0 + s] : 0.f;
            dA[e][s] = 0.f;
        }
    }
    if (MAIN && k + 1 < sgm.K) {
        // carry into the end of chunk k: rho_{j-1} = M_j + P_j rho_j from the
        // reverse summaries of the unit's chunks K-1 .. k+1 (P_j = exp2(A2 *
        // sum of delta_eff over chunk j)), with rho_{K-1} the carry into the end
        // of the sequence
#pragma unroll
        for (int e = 0; e < 2; e++) {
            for (int64_t j = sgm.K - 1; j > k; j--) {
                const int64_t q = s_first + j;
                const float* M = a.ws_rsum + (q * CH + c0 + e) * N + n0;
                const float sdj = a.ws_rsd[q * CH + c0 + e];
#pragma unroll
                for (int s = 0; s < S; s++) carry[e][s] = fmaf(ex2a(A2[e][s] * sdj), carry[e][s], M[s]);
            }
#pragma unroll
            for (int s = 0; s < S; s++) carry[e][s] = ok[e] ? carry[e][s] : 0.f;
        }
    }
    // dD / ddelta_bias partials of the thread's epilogue items (the same channels
    // in every tile), added over the tiles in order; summed per channel at the end
    float accD[ITEMS * GRP], accB[ITEMS * GRP];
#pragma unroll
    for (int c = 0; c < ITEMS * GRP; c++) accD[c] = accB[c] = 0.f;

    const bool pfast = ((Dch * (int64_t)sizeof(T)) % 16 == 0) && (d0 + CH <= Dch);
    const bool ofast = (Dch % 4 == 0) && (d0 + CH <= Dch);
    const int64_t t_begin = k * sgm.Lc;
    const int64_t t_end = t_begin + sgm.Lc < L ? t_begin + sgm.Lc : L;
    const int64_t ntile = (t_end - t_begin + kTT - 1) / kTT;
    // saved states (layout of ckpt_bytes): one block of CH x N floats per
    // (sub-chunk slot, batch, channel tile), the lane's slots in lane order
    const int64_t ck_stride = f.Bsz * p.tiles_b * CH * N;
    const float* ck_blk = a.ws_ckpt + (t_begin / kSub) * ck_stride + (b * p.tiles_b + tile) * (CH * N);
    const float* ck0 = ck_blk + ckpt_slot(w, 0, lane, S);
    const float* ck1 = ck_blk + ckpt_slot(w, 1, lane, S);
    float* bc0 = a.ws_bc + ((int64_t)tile * f.Bsz + b) * L * N;                  // dB partials of this tile
    float* bc1 = a.ws_bc + ((int64_t)(p.tiles_b + tile) * f.Bsz + b) * L * N;    // dC partials
    float* sRw = &sR[MAIN ? w : 0][0];

    // Asynchronous copies of tile mm, one commit group: the thread's item runs
    // (when the tile's rows are whole aligned vectors), the B / C rows (f32 into
    // sBC[mm & 1]; bf16 raw into sBCraw), and the
    // restart states of the tile's sub-chunks into the lane's own slots of
    // sH[mm & 1] (S floats per channel).  Each thread converts the runs it
    // copied; the states are read by the lane that copied them.
    auto issue = [&](int64_t mm) {
        const int64_t tt = t_begin + mm * kTT;
        const int buf = (int)(mm & 1);
        if (pfast) {
#pragma unroll
            for (int it = 0; it < ITEMS; it++) {
                const int id = tid + it * THREADS;
                const int r = id / NGRP, cg = (id % NGRP) * GRP;
                const int64_t t = tt + r;
                if (t < t_end) {
                    const int64_t off = (b * L + t) * Dch + d0 + cg;
                    cp_async_bytes<GRP * C::ESZ>(&sRaw[0][r][cg], delta + off);
                    cp_async_bytes<GRP * C::ESZ>(&sRaw[1][r][cg], u + off);
                    cp_async_bytes<GRP * C::ESZ>(&sRaw[2][r][cg], dy + off);
                    if (z) cp_async_bytes<GRP * C::ESZ>(&sRaw[3][r][cg], z + off);
                    if (MAIN && z) cp_async_bytes<GRP * 4>(&sY0[buf][r][cg], a.y0 + off);
                }
            }
        }
        for (int id = tid; id < (MAIN ? 2 : 1) * kTT; id += THREADS) {
            const int half = MAIN ? id / kTT : 1, r = id % kTT;
            const int64_t t = tt + r;
            const T* src = (half ? Cm : Bm) + (b * L + (t < t_end ? t : 0)) * N;
            if constexpr (C::BC_DIRECT) {
                cp_async_bc_row<T, N, S>(reinterpret_cast<unsigned char*>(&sBC[buf][r][0]), half, src, t < t_end);
            } else if constexpr (C::BC_RAW) {
                if (t < t_end) cp_async_bytes<N * C::ESZ>(&sBCraw[half][r][0], src);
            }
        }
        if (MAIN) {
#pragma unroll
            for (int sub = 0; sub < kTT / kSub; sub++) {
                const int64_t ts = tt + sub * kSub;
                if (ts < t_end) {
                    const int64_t j = (ts - t_begin) / kSub;
                    cp_async_bytes<S * 4>(&sH[buf][sub][0][tid * S], ck0 + j * ck_stride);
                    cp_async_bytes<S * 4>(&sH[buf][sub][1][tid * S], ck1 + j * ck_stride);
                }
            }
        }
        cp_async_commit();
    };
    issue(ntile - 1);
    __syncthreads();  // sBias / sDv before the first prologue

    for (int64_t m = ntile - 1; m >= 0; m--) {
        const int64_t t0 = t_begin + m * kTT;
        const int buf = (int)(m & 1);
        cp_async_wait<0>();  // this thread's copies of the tile
        // per-(t, d) terms of the thread's own items that its epilogue needs
        // again (Delta, g, u, sig(delta + bias), the dz factor): kept in registers
        float kDl[ITEMS][GRP], kG[ITEMS][GRP], kU[ITEMS][GRP], kS[ITEMS][GRP], kZ[ITEMS][GRP];
        // ---- prologue: (step, 4-channel group) items of the tile
#pragma unroll
        for (int it = 0; it < ITEMS; it++) {
            const int id = tid + it * THREADS;
            const int r = id / NGRP, q = id % NGRP;
            const int cg = q * GRP;
            const int64_t t = t0 + r;
            const bool rv = t < t_end;
            uint32_t rd[RWH], ru[RWH], rz[RWH], rg[RWH];
            if (rv) {
                if (pfast) {
                    lds_words<GRP * C::ESZ, RWH>(&sRaw[0][r][cg], rd);
                    lds_words<GRP * C::ESZ, RWH>(&sRaw[1][r][cg], ru);
                    lds_words<GRP * C::ESZ, RWH>(&sRaw[2][r][cg], rg);
                    if (z) lds_words<GRP * C::ESZ, RWH>(&sRaw[3][r][cg], rz);
                } else {
                    const int64_t off = (b * L + t) * Dch + d0 + cg;
                    load_run<T, GRP, RWH>(delta, off, d0 + cg, Dch, false, rd);
                    load_run<T, GRP, RWH>(u, off, d0 + cg, Dch, false, ru);
                    load_run<T, GRP, RWH>(dy, off, d0 + cg, Dch, false, rg);
                    if (z) load_run<T, GRP, RWH>(z, off, d0 + cg, Dch, false, rz);
                }
            }
            float dl[GRP], dlu[GRP], gg[GRP], uu[GRP], sgx[GRP], dzf[GRP];
#pragma unroll
            for (int c = 0; c < GRP; c += 2) {
                // two channels at a time with packed arithmetic
                float2 dl2 = make_float2(0.f, 0.f), sg2 = dl2, uu2 = dl2, dlu2 = dl2, gg2 = dl2, dz2 = dl2;
                if (rv) {
                    const float2 x = make_float2(elem<T>(rd, c) + sBias[cg + c], elem<T>(rd, c + 1) + sBias[cg + c + 1]);
                    if (f.softplus) {
                        softplus_sigmoid2(x, dl2, sg2);
                    } else {
                        dl2 = x;
                        sg2 = make_float2(1.f, 1.f);
                    }
                    uu2 = make_float2(elem<T>(ru, c), elem<T>(ru, c + 1));
                    dlu2 = mul2(dl2, uu2);
                    const float2 dyv = make_float2(elem<T>(rg, c), elem<T>(rg, c + 1));
                    gg2 = dyv;
                    if (z) {
                        const float2 zz = make_float2(elem<T>(rz, c), elem<T>(rz, c + 1));
                        const float2 sz = sigmoid2(zz);
                        const float2 dsz = mul2(dyv, sz);
                        gg2 = mul2(dsz, zz);
                        // dz factor dy sig(z) (1 + z (1 - sig(z)))
                        dz2 = mul2(dsz, fma2(zz, add2(splat2(1.f), make_float2(-sz.x, -sz.y)), splat2(1.f)));
                    }
                }
                dl[c] = dl2.x; dl[c + 1] = dl2.y; sgx[c] = sg2.x; sgx[c + 1] = sg2.y;
                uu[c] = uu2.x; uu[c + 1] = uu2.y; dlu[c] = dlu2.x; dlu[c + 1] = dlu2.y;
                gg[c] = gg2.x; gg[c + 1] = gg2.y; dzf[c] = dz2.x; dzf[c + 1] = dz2.y;
            }
#pragma unroll
            for (int c = 0; c < GRP; c += 2) {
                const int slot = bpair_slot<PAIRS>((cg + c) / 2);
                sDU[r][slot] = make_float4(dl[c], dlu[c], dl[c + 1], dlu[c + 1]);
                sG[r][slot] = make_float2(gg[c], gg[c + 1]);
            }
#pragma unroll
            for (int c = 0; c < GRP; c++) {
                kDl[it][c] = dl[c];
                kG[it][c] = gg[c];
                kU[it][c] = uu[c];
                kS[it][c] = sgx[c];
                kZ[it][c] = dzf[c];
            }
        }
        if constexpr (!C::BC_DIRECT) {
            // bf16 B / C rows of the tile's steps (the reverse summary needs only C),
            // converted by the thread that copied them (or loaded here when too short to copy)
            for (int id = tid; id < (MAIN ? 2 : 1) * kTT; id += THREADS) {
                const int half = MAIN ? id / kTT : 1, r = id % kTT;
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
        if (m > 0) issue(m - 1);

        if constexpr (!MAIN) {
            // ---- reverse summary: adjoint walk from a zero carry and the chunk's
            // decay product, no states needed
            for (int i = kTT - 1; i >= 0; i--) {
                if (t0 + i >= t_end) continue;
                const float4 du = sDU[i][pslot];
                const float2 g2 = sG[i][pslot];
                sd[0] += du.x;
                sd[1] += du.z;
                float Bv[S], Cv[S];
                ld_bc_f32<S>(&sBC[C::BC_DIRECT ? buf : 0][i][sg * 2 * S], Bv, Cv);
#pragma unroll
                for (int e = 0; e < 2; e++) {
#pragma unroll
                    for (int s = 0; s < S; s++) {
                        const float lam = fmaf(e ? g2.y : g2.x, Cv[s], carry[e][s]);
                        const float da = ex2a((e ? du.z : du.x) * A2[e][s]);
                        carry[e][s] = da * lam;
                    }
                }
            }
        } else {
            // ---- the tile's sub-chunks of kSub steps, last one first.  Steps past
            // the chunk end (last tile only) hold Delta = g = 0 and B = C = 0 in the
            // staging: they leave the state and the adjoint unchanged and add
            // nothing; only their per-step stores are skipped.
#pragma unroll
            for (int sub = kTT / kSub - 1; sub >= 0; sub--) {
                const int64_t ts = t0 + sub * kSub;
                if (ts >= t_end) continue;
                // the lane's restart states of channel parity e: hsrc[e], copied with the tile's rows
                const float* hsrc[2] = {&sH[buf][sub][0][tid * S], &sH[buf][sub][1][tid * S]};
                // recompute the states and decays of the sub-chunk
                float hv[kSub][2][S], av[kSub][2][S];
                {
                    float hh[2][S];
                    // (the saved state of a channel past Dch is zero: the forward keeps it so)
#pragma unroll
                    for (int e = 0; e < 2; e++) ld_state<S>(hsrc[e], hh[e]);
#pragma unroll
                    for (int i = 0; i < kSub; i++) {
                        const int r = sub * kSub + i;
                        const float4 du = sDU[r][pslot];
                        float Bv[S];
                        ld_b_f32<S>(&sBC[C::BC_DIRECT ? buf : 0][r][sg * 2 * S], Bv);
#pragma unroll
                        for (int e = 0; e < 2; e++) {
                            if constexpr (S >= 2) {
                                const float2 dl2 = splat2(e ? du.z : du.x), dlu2 = splat2(e ? du.w : du.y);
#pragma unroll
                                for (int s = 0; s < S; s += 2) {
                                    const float2 ex = mul2(dl2, make_float2(A2[e][s], A2[e][s + 1]));
                                    const float2 da = make_float2(ex2a(ex.x), ex2a(ex.y));
                                    const float2 x = mul2(dlu2, make_float2(Bv[s], Bv[s + 1]));
                                    const float2 nh = fma2(da, make_float2(hh[e][s], hh[e][s + 1]), x);
                                    hh[e][s] = nh.x; hh[e][s + 1] = nh.y;
                                    hv[i][e][s] = nh.x; hv[i][e][s + 1] = nh.y;
                                    av[i][e][s] = da.x; av[i][e][s + 1] = da.y;
                                }
                            } else {
                                const float da = ex2a((e ? du.z : du.x) * A2[e][0]);
                                hh[e][0] = fmaf(da, hh[e][0], (e ? du.w : du.y) * Bv[0]);
                                hv[i][e][0] = hh[e][0];
                                av[i][e][0] = da;
                            }
                        }
                    }
                }
                // adjoint walk
#pragma unroll
                for (int i = kSub - 1; i >= 0; i--) {
                    const int r = sub * kSub + i;
                    const float4 du = sDU[r][pslot];
                    const float2 g2 = sG[r][pslot];
                    float Bv[S], Cv[S];
                    ld_bc_f32<S>(&sBC[C::BC_DIRECT ? buf : 0][r][sg * 2 * S], Bv, Cv);
                    float sumB[2], sumQ[2];
                    float cB[S], cC[S];
                    if constexpr (S >= 2) {
                        float2 cb2[S / 2], cc2[S / 2];
#pragma unroll
                        for (int e = 0; e < 2; e++) {
                            const float2 g2e = splat2(e ? g2.y : g2.x), dl2 = splat2(e ? du.z : du.x),
                                         dlu2 = splat2(e ? du.w : du.y);
                            float2 dup = make_float2(0.f, 0.f), ddp = dup;
#pragma unroll
                            for (int s = 0; s < S; s += 2) {
                                const float2 Cp = make_float2(Cv[s], Cv[s + 1]);
                                const float2 hcur = make_float2(hv[i][e][s], hv[i][e][s + 1]);
                                float2 hprev;
                                if (i > 0) {
                                    hprev = make_float2(hv[i - 1][e][s], hv[i - 1][e][s + 1]);
                                } else {
                                    hprev = *reinterpret_cast<const float2*>(hsrc[e] + s);
                                }
                                const float2 lam = fma2(g2e, Cp, make_float2(carry[e][s], carry[e][s + 1]));
                                dup = fma2(lam, make_float2(Bv[s], Bv[s + 1]), dup);
                                const float2 cn = mul2(make_float2(av[i][e][s], av[i][e][s + 1]), lam);
                                const float2 q = mul2(cn, hprev);
                                ddp = fma2(make_float2(A2[e][s], A2[e][s + 1]), q, ddp);
                                const float2 na = fma2(dl2, q, make_float2(dA[e][s], dA[e][s + 1]));
                                dA[e][s] = na.x; dA[e][s + 1] = na.y;
                                // dB / dC contributions summed over the pair's two channels
                                cb2[s / 2] = e ? fma2(lam, dlu2, cb2[s / 2]) : mul2(lam, dlu2);
                                cc2[s / 2] = e ? fma2(g2e, hcur, cc2[s / 2]) : mul2(g2e, hcur);
                                carry[e][s] = cn.x; carry[e][s + 1] = cn.y;
                            }
                            sumB[e] = dup.x + dup.y;
                            sumQ[e] = ddp.x + ddp.y;
                        }
#pragma unroll
                        for (int s = 0; s < S; s += 2) {
                            cB[s] = cb2[s / 2].x; cB[s + 1] = cb2[s / 2].y;
                            cC[s] = cc2[s / 2].x; cC[s + 1] = cc2[s / 2].y;
                        }
                    } else {
#pragma unroll
                        for (int e = 0; e < 2; e++) {
                            const float ge = e ? g2.y : g2.x, dle = e ? du.z : du.x, dlue = e ? du.w : du.y;
                            const float hprev =
                                i > 0 ? hv[i - 1][e][0] : hsrc[e][0];
                            const float lam = fmaf(ge, Cv[0], carry[e][0]);
                            sumB[e] = lam * Bv[0];
                            const float cn = av[i][e][0] * lam;
                            const float q = cn * hprev;
                            sumQ[e] = A2[e][0] * q;
                            dA[e][0] = fmaf(dle, q, dA[e][0]);
                            cB[0] = e ? fmaf(lam, dlue, cB[0]) : lam * dlue;
                            cC[0] = e ? fmaf(ge, hv[i][e][0], cC[0]) : ge * hv[i][e][0];
                            carry[e][0] = cn;
                        }
                    }
                    // the lane's sums over its states, both channels; the epilogue adds
                    // the G lanes of the pair and the warps
                    {
                        const int o = g * C::OPL + r * EP + c0;
                        *reinterpret_cast<float2*>(&sOu[w][o]) = make_float2(sumB[0], sumB[1]);
                        *reinterpret_cast<float2*>(&sOd[w][o]) = make_float2(sumQ[0], sumQ[1]);
                    }
                    // stage dB / dC contributions (summed over the pairs below)
                    stage_contrib<S, NPW, BLK>(sRw, i, cB, cC, pp, g * S);
                }
                __syncwarp();  // staged contributions visible to every lane of the warp
                reduce_staged<PAIRS, NPW, N, BLK>(sRw, bc0, bc1, n_w, ts, t_end, lane);
                __syncwarp();  // the sums have read the staging before the next sub-chunk restages it
            }
            __syncthreads();  // every warp's per-step sums are in sOu / sOd
            // ---- epilogue: du, ddelta, dz of the (step, 4-channel group) items.
            // Steps past t_end (last tile only) are not stored and add nothing;
            // their per-step sums may be unwritten (a sub-chunk wholly past the
            // end is skipped).
#pragma unroll
            for (int it = 0; it < ITEMS; it++) {
                const int id = tid + it * THREADS;
                const int r = id / NGRP, q = id % NGRP;
                const int cg = q * GRP;
                const int64_t t = t0 + r;
                const bool tv = t < t_end;
                // per warp, the sum of its G lanes' planes; then the warps in order
                float4 su, sd;
#pragma unroll
                for (int ww = 0; ww < NW; ww++) {
                    const int o = r * EP + cg;
                    float4 ou = *reinterpret_cast<const float4*>(&sOu[ww][o]);
                    float4 od = *reinterpret_cast<const float4*>(&sOd[ww][o]);
                    if constexpr (G == 2) {
                        const float4 pu = *reinterpret_cast<const float4*>(&sOu[ww][C::OPL + o]);
                        const float4 pd = *reinterpret_cast<const float4*>(&sOd[ww][C::OPL + o]);
                        ou.x += pu.x; ou.y += pu.y; ou.z += pu.z; ou.w += pu.w;
                        od.x += pd.x; od.y += pd.y; od.z += pd.z; od.w += pd.w;
                    }
                    if (ww == 0) {
                        su = ou; sd = od;
                    } else {
                        su.x += ou.x; su.y += ou.y; su.z += ou.z; su.w += ou.w;
                        sd.x += od.x; sd.y += od.y; sd.z += od.z; sd.w += od.w;
                    }
                }
                // y0 for dz (only with a gate): staged with the tile's rows, else loaded here
                float vy0[GRP];
#pragma unroll
                for (int c = 0; c < GRP; c++) vy0[c] = 0.f;
                if (z && tv) {
                    if (pfast) {
                        const float4 q = *reinterpret_cast<const float4*>(&sY0[buf][r][cg]);
                        vy0[0] = q.x; vy0[1] = q.y; vy0[2] = q.z; vy0[3] = q.w;
                    } else {
                        const float* y0r = a.y0 + (b * L + t) * Dch + d0 + cg;
#pragma unroll
                        for (int c = 0; c < GRP; c++) vy0[c] = d0 + cg + c < Dch ? y0r[c] : 0.f;
                    }
                }
                const float vsu[4] = {su.x, su.y, su.z, su.w}, vsd[4] = {sd.x, sd.y, sd.z, sd.w};
                const float(&vdl)[GRP] = kDl[it];
                const float(&vg)[GRP] = kG[it];
                const float(&vu)[GRP] = kU[it];
                const float(&vs)[GRP] = kS[it];
                const float(&vz)[GRP] = kZ[it];
                float vdu[GRP], vdx[GRP], vdz[GRP];
#pragma unroll
                for (int c = 0; c < GRP; c += 2) {
                    // two channels at a time with packed arithmetic
                    const float2 Dv = make_float2(sDv[cg + c], sDv[cg + c + 1]);
                    const float2 su2 = make_float2(vsu[c], vsu[c + 1]), u2 = make_float2(vu[c], vu[c + 1]);
                    const float2 du2 = fma2(make_float2(vg[c], vg[c + 1]), Dv, mul2(make_float2(vdl[c], vdl[c + 1]), su2));
                    const float2 dx2 = mul2(fma2(u2, su2, mul2(make_float2(vsd[c], vsd[c + 1]), splat2(kLn2))),
                                            make_float2(vs[c], vs[c + 1]));
                    const float2 dz2 = mul2(make_float2(vz[c], vz[c + 1]), make_float2(vy0[c], vy0[c + 1]));
                    vdu[c] = du2.x; vdu[c + 1] = du2.y;
                    vdx[c] = dx2.x; vdx[c + 1] = dx2.y;
                    vdz[c] = dz2.x; vdz[c + 1] = dz2.y;
                }
#pragma unroll
                for (int c = 0; c < GRP; c++) {
                    accD[it * GRP + c] = fmaf(vg[c], vu[c], accD[it * GRP + c]);  // g = u = 0 past t_end
                    accB[it * GRP + c] += tv ? vdx[c] : 0.f;
                }
                if (tv) {
                    const int64_t off = (b * L + t) * Dch + d0 + cg;
                    store_run<GRP>(a.du + off, vdu, d0 + cg, Dch, ofast);
                    store_run<GRP>(a.ddelta + off, vdx, d0 + cg, Dch, ofast);
                    if (z) store_run<GRP>(a.dz + off, vdz, d0 + cg, Dch, ofast);
                }
            }
        }
        // The reverse summary's walk reads what the next prologue restages.  The
        // main pass needs no barrier here: its epilogue reads only the per-step
        // sums (the next ones are written after the next prologue's barrier)
        // and the staging entries of its own items, which the same thread
        // rewrites next.
        if constexpr (!MAIN) __syncthreads();
    }

    const int64_t q = q_first + k;  // this block's part
    if constexpr (!MAIN) {
        // every entry of the summary is written (channels past Dch: zero carry)
        const int64_t qs = s_first + k;
#pragma unroll
        for (int e = 0; e < 2; e++) {
            float* M = a.ws_rsum + (qs * CH + c0 + e) * N + n0;
#pragma unroll
            for (int s = 0; s < S; s++) M[s] = carry[e][s];
        }
        if (w == 0 && g == 0) *reinterpret_cast<float2*>(a.ws_rsd + qs * CH + c0) = make_float2(sd[0], sd[1]);
    } else {
#pragma unroll
        for (int e = 0; e < 2; e++) {
            if (ok[e]) {
                float* o = a.ws_dA + (q * CH + c0 + e) * N + n0;
#pragma unroll
                for (int s = 0; s < S; s++) o[s] = dA[e][s];
                // after the walk of the first chunk the carry is a_0 lam_0, the gradient of h0
                if (STATE && k == 0 && a.dh0) {
#pragma unroll
                    for (int s = 0; s < S; s++) a.dh0[row[e] * N + n0 + s] = carry[e][s];
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
cudaError_t launch_bwd2_t(const BwdArgs& a, const FPlan& p, cudaStream_t st, float* ckpt_out) {
    cudaError_t e = cudaSuccess;
    if (ckpt_out) {
        // checkpoint pass (with forward summaries first when the sequence is chunked)
        e = launch_fwd2(a.f, p, st, kModeCkpt, ckpt_out);
        if (e != cudaSuccess) return e;
    }
    constexpr int threads = BCfg<T, N>::THREADS;
    // reverse summaries of every chunked segment (chunks 1 .. K-1)
    for (int si = 0; si < p.nseg; si++) {
        const int64_t K = p.seg[si].K;
        if (K > 1) {
            prof_mark(st);
            k_bwd2<T, N, kRevSummary, false><<<(unsigned)(p.seg[si].nu * (K - 1)), threads, 0, st>>>(a, p, si, 1);
        }
    }
    const bool state = a.dlast != nullptr || a.dh0 != nullptr;
    auto main_kernel = state ? k_bwd2<T, N, kRevMain, true> : k_bwd2<T, N, kRevMain, false>;
    // one bit per device ordinal: the carveout preference is set on that device
    static std::atomic<uint64_t> carveout_done[2] = {{0}, {0}};
    e = prefer_max_shared(main_kernel, carveout_done[state]);
    if (e != cudaSuccess) return e;
    for (int si = 0; si < p.nseg; si++) {
        prof_mark(st);
        main_kernel<<<(unsigned)(p.seg[si].nu * p.seg[si].K), threads, 0, st>>>(a, p, si, 0);
    }
    return cudaGetLastError();
}

// Backward launcher of one io type: switches on N.
template <typename T>
cudaError_t launch_bwd2_io(const BwdArgs& a, const FPlan& p, cudaStream_t st, float* ckpt_out) {
    switch (a.f.N) {
        case 1: return launch_bwd2_t<T, 1>(a, p, st, ckpt_out);
        case 2: return launch_bwd2_t<T, 2>(a, p, st, ckpt_out);
        case 4: return launch_bwd2_t<T, 4>(a, p, st, ckpt_out);
        case 8: return launch_bwd2_t<T, 8>(a, p, st, ckpt_out);
        case 16: return launch_bwd2_t<T, 16>(a, p, st, ckpt_out);
        case 32: return launch_bwd2_t<T, 32>(a, p, st, ckpt_out);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace ss
