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
//     start of every kSub-step sub-chunk;
//   * this kernel visits kTT-step tiles from the end of the chunk backwards.
//     The tile prologue computes the per-(t, d) terms once (softplus and its
//     derivative, the gate, g, the dz factor) into shared memory; then each
//     sub-chunk is recomputed forward from its saved state, keeping its
//     states and decays in registers, and the adjoint walks it backwards;
//   * per step the G lanes of a channel combine their partial sums with a
//     shuffle, and each warp sums dB / dC of its states over the block's
//     channels through shared memory in a fixed order; the tile epilogue
//     adds the warps' per-(t, d) sums and writes du, ddelta, dz; a second
//     kernel adds the per-tile dB / dC partials, a third the per-(batch,
//     chunk) dA / dD / ddelta_bias partials.  Every sum has a fixed order:
//     the result is bit-reproducible.
// Chunks (only when batch x channels cannot fill the GPU): each chunk's
// carry-in state is its first saved state; reverse summaries (P_k, M_k) --
// the chunk's decay product and M_k = a_{s_k} lam_{s_k} with lam from a zero
// incoming carry -- combine as rho_{k-1} = M_k + P_k rho_k into each chunk's
// carry-in adjoint.
#include "common.cuh"
#include "kernels.h"
#include "simd.cuh"

namespace ss {

constexpr int kTT = 8;   // backward tile: steps staged per prologue
constexpr int kRB = 4;   // steps whose dB / dC contributions are reduced together (one sub-chunk)
static_assert(kRB == kSub, "one staged sub-chunk of dB / dC contributions at a time");
static_assert(kTT % kSub == 0, "a tile holds whole sub-chunks");

template <typename T, int N>
struct BCfg {
    static constexpr int NW = fwd_warps(N);         // warps per block (they split the states)
    static constexpr int NPW = N / NW;              // states per warp
    static constexpr int G = NPW >= 2 ? 2 : 1;      // lanes per channel
    static constexpr int S = NPW / G;               // states per lane
    static constexpr int CH = 32 / G;               // channels per block
    static constexpr int THREADS = 32 * NW;
    static constexpr int PARTS = THREADS / kTT;     // prologue / epilogue threads per step
    static constexpr int CPL = CH / PARTS;          // channels per prologue / epilogue thread
    static constexpr int RWH = CPL * (int)sizeof(T) / 4 > 0 ? CPL * (int)sizeof(T) / 4 : 1;
    static constexpr int NB = N * (int)sizeof(T);
    static constexpr int NWd = NB >= 4 ? NB / 4 : 1;
    static constexpr int NP = N + 4;
    // dB / dC staging of one warp: block (step slot j, tensor tau) holds CH
    // rows of NPW floats (the warp's states); blocks are padded by 8 floats
    // so that the 16 lanes of a half warp reading 8-byte pairs of four
    // consecutive blocks hit 32 different banks
    static constexpr int BLK = CH * NPW + 8;
    static constexpr int MINB = N >= 32 ? 1 : 9;    // blocks per SM the register budget must allow
    static_assert(CPL >= 2, "prologue runs of at least two channels");
    static_assert(CH == kChannelsPerBlock || N == 1, "channel tile of the plan");
};

template <typename T>
__device__ __forceinline__ float belem(const uint32_t* w, int j) {
    if constexpr (sizeof(T) == 4) {
        return __uint_as_float(w[j]);
    } else {
        return (j & 1) ? bf16hi(w[j >> 1]) : bf16lo(w[j >> 1]);
    }
}

template <int NBYTES, int NWORDS>
__device__ __forceinline__ void bload_words(const void* p, uint32_t (&w)[NWORDS]) {
    if constexpr (NBYTES % 16 == 0) {
#pragma unroll
        for (int v = 0; v < NBYTES / 16; v++) {
            const uint4 q = __ldg(reinterpret_cast<const uint4*>(p) + v);
            w[4 * v] = q.x; w[4 * v + 1] = q.y; w[4 * v + 2] = q.z; w[4 * v + 3] = q.w;
        }
    } else if constexpr (NBYTES == 8) {
        const uint2 q = __ldg(reinterpret_cast<const uint2*>(p));
        w[0] = q.x; w[1] = q.y;
    } else if constexpr (NBYTES == 4) {
        w[0] = __ldg(reinterpret_cast<const unsigned int*>(p));
    } else {
        w[0] = __ldg(reinterpret_cast<const unsigned short*>(p));
    }
}

// CPL contiguous io elements at (row offset off, channel c0): vector loads when
// aligned and complete, else element loads zero-filled past Dch.
template <typename T, int CPL, int RWH>
__device__ __forceinline__ void bload_half(const T* base, int64_t off, int64_t c0, int64_t Dch, bool fast,
                                           uint32_t (&w)[RWH]) {
    if (fast) {
        bload_words<CPL * (int)sizeof(T), RWH>(base + off, w);
    } else {
#pragma unroll
        for (int i = 0; i < RWH; i++) w[i] = 0u;
#pragma unroll
        for (int c = 0; c < CPL; c++) {
            if (c0 + c < Dch) {
                if constexpr (sizeof(T) == 4) {
                    w[c] = __ldg(reinterpret_cast<const unsigned int*>(base + off) + c);
                } else {
                    const uint32_t v = __ldg(reinterpret_cast<const unsigned short*>(base + off) + c);
                    w[c >> 1] |= (c & 1) ? (v << 16) : v;
                }
            }
        }
    }
}

template <int S>
__device__ __forceinline__ void bld_shared(const float* p, float (&v)[S]) {
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

// softplus(x) (as in simd.cuh) together with sigmoid(x), sharing e = e^-|x|.
__device__ __forceinline__ void softplus_and_sigmoid(float x, float& sp, float& sg) {
    const float e = ex2a(-fabsf(x) * kLog2eF);
    const float s = e * rcpa(2.f + e);
    const float s2 = s * s;
    float p = 1.f / 15.f;
    p = fmaf(p, s2, 1.f / 13.f);
    p = fmaf(p, s2, 1.f / 11.f);
    p = fmaf(p, s2, 1.f / 9.f);
    p = fmaf(p, s2, 1.f / 7.f);
    p = fmaf(p, s2, 1.f / 5.f);
    p = fmaf(p, s2, 1.f / 3.f);
    p = fmaf(p, s2, 1.f);
    sp = fmaxf(x, 0.f) + 2.f * s * p;
    const float r = rcpa(1.f + e);
    sg = x >= 0.f ? r : e * r;
}

// Asynchronous copy of S floats (a lane's saved state) from global to shared
// memory; both addresses are aligned to the copy size.
template <int S>
__device__ __forceinline__ void cp_async_state(float* dst, const float* src) {
    const unsigned sa = (unsigned)__cvta_generic_to_shared(dst);
    if constexpr (S % 4 == 0) {
#pragma unroll
        for (int q = 0; q < S; q += 4)
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sa + 4 * q), "l"(src + q) : "memory");
    } else {
        asm volatile("cp.async.ca.shared.global [%0], [%1], %2;" ::"r"(sa), "l"(src), "n"(S * 4) : "memory");
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
}

template <int PENDING>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(PENDING) : "memory");
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
// block (j, tau) holds CH rows of NPW floats, the warp's states of each
// channel.  Lanes of channels past Dch need no masking: their u, dy and z
// load as zero, so lam * Delta * u and g * h are exactly zero there.
template <int S, int NPW, int BLK>
__device__ __forceinline__ void stage_contrib(float* sR, int j, const float (&cB)[S], const float (&cC)[S], int ch,
                                              int gs) {
    float* r0 = sR + (2 * j) * BLK + ch * NPW + gs;
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
// the CH channels and store the sums as the warp's states n_w .. n_w + NPW of
// the dB / dC partial rows bc0[t + j], bc1[t + j] (rows of N floats; steps
// at or past t_end are not stored).  Work unit: a pair of consecutive states
// of one (step, tensor); the channels are added as a fixed pairwise tree
// (c, c + 1), then pairs of pairs, ...
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
// walk of chunks 1..K-1 from a zero carry, writing (P_k, M_k).
constexpr int kRevMain = 0, kRevSummary = 1;

template <typename T, int N, int MODE>
__global__ void __launch_bounds__(32 * fwd_warps(N), BCfg<T, N>::MINB) k_bwd2(BwdArgs a, FPlan p, int64_t k_lo,
                                                                               int64_t k_hi) {
    using C = BCfg<T, N>;
    constexpr bool MAIN = MODE == kRevMain;
    constexpr int NW = C::NW, NPW = C::NPW, S = C::S, G = C::G, CH = C::CH, CPL = C::CPL, RWH = C::RWH,
                  NWd = C::NWd, NP = C::NP, BLK = C::BLK;
    // per-(t, d) staging: rows padded by one element, so that both the row-parallel
    // prologue / epilogue (thread = step) and the scan (lane = channel) access them
    // without bank conflicts and with constant offsets
    __shared__ float4 sS[kTT][CH + 1];                    // (Delta, Delta*u, g, sig(x))
    __shared__ float2 sE[MAIN ? kTT : 1][CH + 1];         // (u, dz factor)
    __shared__ __align__(16) float sB[MAIN ? kTT : 1][NP];
    __shared__ __align__(16) float sC[kTT][NP];
    // dB / dC contributions of kRB steps, per warp: block (j, tau) holds CH rows of NPW floats
    __shared__ __align__(16) float sR[MAIN ? NW : 1][MAIN ? kRB * 2 * BLK : 4];
    // per-step, per-warp sums over the warp's states: (sum lam B, sum A q) and y0
    __shared__ float2 sOa[MAIN ? NW : 1][MAIN ? kTT : 1][CH + 1];
    __shared__ float sOb[MAIN ? NW : 1][MAIN ? kTT : 1][CH + 1];
    __shared__ float sBias[CH], sDv[CH];
    // per-thread dD / ddelta_bias partials of the epilogue threads (thread fastest)
    __shared__ float sAcc[MAIN ? 2 : 1][MAIN ? CPL : 1][C::THREADS];
    // restart states of the next two sub-chunks, one S-float slot per lane (double buffered)
    __shared__ __align__(16) float sH[MAIN ? 2 : 1][C::THREADS * S];

    const FwdArgs& f = a.f;
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    int64_t blk = blockIdx.x;
    const int64_t tile = blk % p.tiles_b;
    blk /= p.tiles_b;
    const int64_t nk = k_hi - k_lo;
    const int64_t k = k_lo + blk % nk;
    const int64_t b = blk / nk;
    const int64_t L = f.L, Dch = f.Dch;
    const int64_t d0 = tile * CH;
    const T* u = static_cast<const T*>(f.u);
    const T* delta = static_cast<const T*>(f.delta);
    const T* Bm = static_cast<const T*>(f.B);
    const T* Cm = static_cast<const T*>(f.C);
    const T* z = static_cast<const T*>(f.z);
    const T* dy = static_cast<const T*>(a.dy);

    if (tid < CH) {
        const int64_t dc = d0 + tid < Dch ? d0 + tid : Dch - 1;
        sBias[tid] = f.delta_bias ? f.delta_bias[dc] : 0.f;
        sDv[tid] = f.D ? f.D[dc] : 0.f;
    }

    // scan-lane identity: channel ch, states n0 .. n0 + S (warp w holds n_w .. n_w + NPW)
    const int ch = lane / G, g = lane % G;
    const bool ch_ok = d0 + ch < Dch;
    const int64_t d = ch_ok ? d0 + ch : Dch - 1;
    const int n_w = w * NPW;
    const int n0 = n_w + g * S;
    const int64_t row = b * Dch + d;
    // A2 = A * log2(e); the dDelta partial sum below uses A2 and is scaled back by ln 2 in the epilogue.
    // Lanes of channels past Dch run with a zero exponent, state and adjoint: with
    // u = dy = z = 0 loaded there, every quantity they form stays exactly zero
    // (whatever A of the clamped channel is), so their dB / dC contributions
    // need no masking.
    float A2[S], carry[S], dA[S], Pr[MAIN ? 1 : S];
#pragma unroll
    for (int s = 0; s < S; s++) {
        A2[s] = ch_ok ? f.A[d * N + n0 + s] * kLog2eF : 0.f;
        carry[s] = 0.f;
        dA[s] = 0.f;
        if (!MAIN) Pr[s] = 1.f;
    }
    if (MAIN && k + 1 < p.K) {
        // carry into the end of chunk k: rho_{j-1} = M_j + P_j rho_j from the
        // reverse summaries (P_j, M_j) of chunks K-1 .. k+1, with rho_{K-1} = 0
        const float2* rs = reinterpret_cast<const float2*>(a.ws_rsum) + row * p.K * N + n0;
        for (int64_t j = p.K - 1; j > k; j--) {
#pragma unroll
            for (int s = 0; s < S; s++) {
                const float2 pm = rs[j * N + s];
                carry[s] = fmaf(pm.x, carry[s], pm.y);
            }
        }
#pragma unroll
        for (int s = 0; s < S; s++) carry[s] = ch_ok ? carry[s] : 0.f;
    }

    // prologue / epilogue thread identity: step pr of the tile, channels pc0 .. pc0 + CPL
    const int pr = tid % kTT, ph = tid / kTT;
    const int pc0 = ph * CPL;
    const bool pfast = ((Dch * (int64_t)sizeof(T)) % 16 == 0) && (d0 + CH <= Dch) &&
                       ((CPL * (int)sizeof(T)) % 4 == 0);
    const bool ofast = (Dch % 4 == 0) && (d0 + CH <= Dch);
    // per-channel dD / ddelta_bias partials of this epilogue thread over its rows,
    // kept in the thread's own shared slots between tiles
    if (MAIN) {
#pragma unroll
        for (int c = 0; c < CPL; c++) { sAcc[0][c][tid] = 0.f; sAcc[1][c][tid] = 0.f; }
    }

    const int64_t t_begin = k * p.Lc;
    const int64_t t_end = t_begin + p.Lc < L ? t_begin + p.Lc : L;
    const int64_t ntile = (t_end - t_begin + kTT - 1) / kTT;
    // saved states, step-major: [k * (Lc / kSub) + j][Bsz * Dch][N]
    const int64_t ck_stride = f.Bsz * Dch * N;
    const float* ck = a.ws_ckpt + (k * (p.Lc / kSub)) * ck_stride + row * N + n0;
    float* bc0 = a.ws_bc + ((int64_t)tile * f.Bsz + b) * L * N;                  // dB partials of this tile
    float* bc1 = a.ws_bc + ((int64_t)(p.tiles_b + tile) * f.Bsz + b) * L * N;    // dC partials
    float* sRw = &sR[MAIN ? w : 0][0];
    __syncthreads();  // sBias / sDv and the sAcc slots before the first prologue

    // restart state of sub-chunk j lives in sH[j & 1][tid * S ..]; each lane copies
    // and reads only its own slot, so the copies need no barrier.  The last
    // sub-chunk's is requested here, each earlier one a sub-chunk ahead.
    if (MAIN) {
        const int64_t jlast = (t_end - t_begin + kSub - 1) / kSub - 1;
        cp_async_state<S>(&sH[jlast & 1][tid * S], ck + jlast * ck_stride);
    }

    for (int64_t m = ntile - 1; m >= 0; m--) {
        const int64_t t0 = t_begin + m * kTT;
        // ---- prologue: per-(t, d) terms of the tile's steps, staged in shared memory
        {
            const int64_t t = t0 + pr;
            const bool rv = t < t_end;
            const bool stage_b = MAIN && ph == 0, stage_c = ph == (MAIN ? 1 : 0);
            uint32_t rd[RWH], ru[RWH], rz[RWH], rg[RWH], rbc[NWd];
            if (rv) {
                const int64_t off = (b * L + t) * Dch + d0 + pc0;
                bload_half<T, CPL, RWH>(delta, off, d0 + pc0, Dch, pfast, rd);
                bload_half<T, CPL, RWH>(u, off, d0 + pc0, Dch, pfast, ru);
                bload_half<T, CPL, RWH>(dy, off, d0 + pc0, Dch, pfast, rg);
                if (z) bload_half<T, CPL, RWH>(z, off, d0 + pc0, Dch, pfast, rz);
                if (stage_b || stage_c) bload_words<C::NB, NWd>((stage_b ? Bm : Cm) + (b * L + t) * N, rbc);
            }
#pragma unroll
            for (int c = 0; c < CPL; c++) {
                const int cc = pc0 + c;
                float dl = 0.f, sgx = 0.f, uu = 0.f, gg = 0.f, dzf = 0.f;
                if (rv) {
                    const float x = belem<T>(rd, c) + sBias[cc];
                    if (f.softplus) {
                        softplus_and_sigmoid(x, dl, sgx);
                    } else {
                        dl = x;
                        sgx = 1.f;
                    }
                    uu = belem<T>(ru, c);
                    const float dyv = belem<T>(rg, c);
                    gg = dyv;
                    if (z) {
                        const float zz = belem<T>(rz, c);
                        const float sz = sigmoid_fast(zz);
                        gg = dyv * zz * sz;
                        dzf = dyv * sz * fmaf(zz, 1.f - sz, 1.f);
                    }
                }
                sS[pr][cc] = make_float4(dl, dl * uu, gg, sgx);
                if (MAIN) sE[pr][cc] = make_float2(uu, dzf);
            }
            // B row (MAIN) / C row of the thread's step; rows padded to N + 4 floats
            if (stage_b || stage_c) {
                float* dst = stage_b ? &sB[pr][0] : &sC[pr][0];
                if constexpr (N % 4 == 0) {
#pragma unroll
                    for (int n = 0; n < N; n += 4)
                        *reinterpret_cast<float4*>(dst + n) =
                            rv ? make_float4(belem<T>(rbc, n), belem<T>(rbc, n + 1), belem<T>(rbc, n + 2),
                                             belem<T>(rbc, n + 3))
                               : make_float4(0.f, 0.f, 0.f, 0.f);
                } else {
#pragma unroll
                    for (int n = 0; n < N; n++) dst[n] = rv ? belem<T>(rbc, n) : 0.f;
                }
            }
        }
        __syncthreads();

        if constexpr (!MAIN) {
            // ---- reverse summary: adjoint walk from a zero carry and the chunk's
            // decay product, no states needed
            for (int i = kTT - 1; i >= 0; i--) {
                if (t0 + i >= t_end) continue;
                const float4 ss = sS[i][ch];
                float Cv[S];
                bld_shared<S>(&sC[i][n0], Cv);
#pragma unroll
                for (int s = 0; s < S; s++) {
                    const float lam = fmaf(ss.z, Cv[s], carry[s]);
                    const float da = ex2a(ss.x * A2[s]);
                    carry[s] = da * lam;
                    Pr[s] *= da;
                }
            }
        } else {
            // ---- the tile's sub-chunks of kSub steps, last one first.  Steps past
            // the chunk end (last tile only) hold Delta = g = 0 and B = C = 0 in the
            // staging: they leave the state and the adjoint unchanged and add
            // nothing; only their per-step stores are skipped.
#pragma unroll 1
            for (int sub = kTT / kSub - 1; sub >= 0; sub--) {
                const int64_t ts = t0 + sub * kSub;
                if (ts >= t_end) continue;
                // request the previous sub-chunk's restart state, then wait for this one's
                const int64_t jsub = (ts - t_begin) / kSub;
                const float* hsrc = &sH[jsub & 1][tid * S];
                if (jsub > 0) {
                    cp_async_state<S>(&sH[(jsub - 1) & 1][tid * S], ck + (jsub - 1) * ck_stride);
                    cp_async_wait<1>();
                } else {
                    cp_async_wait<0>();
                }
                float hs[S];
                ld_state<S>(hsrc, hs);
#pragma unroll
                for (int s = 0; s < S; s++) hs[s] = ch_ok ? hs[s] : 0.f;
                // recompute the states and decays of the sub-chunk
                float hv[kSub][S], av[kSub][S];
                {
                    float hh[S];
#pragma unroll
                    for (int s = 0; s < S; s++) hh[s] = hs[s];
#pragma unroll
                    for (int i = 0; i < kSub; i++) {
                        const int r = sub * kSub + i;
                        const float4 ss = sS[r][ch];
                        float Bv[S];
                        bld_shared<S>(&sB[r][n0], Bv);
                        if constexpr (S >= 2) {
#pragma unroll
                            for (int s = 0; s < S; s += 2) {
                                const float2 e = mul2(splat2(ss.x), make_float2(A2[s], A2[s + 1]));
                                const float2 da = make_float2(ex2a(e.x), ex2a(e.y));
                                const float2 x = mul2(splat2(ss.y), make_float2(Bv[s], Bv[s + 1]));
                                const float2 nh = fma2(da, make_float2(hh[s], hh[s + 1]), x);
                                hh[s] = nh.x; hh[s + 1] = nh.y;
                                hv[i][s] = nh.x; hv[i][s + 1] = nh.y;
                                av[i][s] = da.x; av[i][s + 1] = da.y;
                            }
                        } else {
                            const float da = ex2a(ss.x * A2[0]);
                            hh[0] = fmaf(da, hh[0], ss.y * Bv[0]);
                            hv[i][0] = hh[0];
                            av[i][0] = da;
                        }
                    }
                }
                // adjoint walk
#pragma unroll
                for (int i = kSub - 1; i >= 0; i--) {
                    const int r = sub * kSub + i;
                    const float4 ss = sS[r][ch];
                    float Bv[S], Cv[S];
                    bld_shared<S>(&sB[r][n0], Bv);
                    bld_shared<S>(&sC[r][n0], Cv);
                    float du_p, dd_p, y0_p;
                    float cB[S], cC[S];
                    if constexpr (S >= 2) {
                        float2 dup = make_float2(0.f, 0.f), ddp = dup, y0p = dup;
                        const float2 g2 = splat2(ss.z), dl2 = splat2(ss.x), dlu2 = splat2(ss.y);
#pragma unroll
                        for (int s = 0; s < S; s += 2) {
                            const float2 Cp = make_float2(Cv[s], Cv[s + 1]);
                            const float2 hcur = make_float2(hv[i][s], hv[i][s + 1]);
                            const float2 hprev = i > 0 ? make_float2(hv[i - 1][s], hv[i - 1][s + 1])
                                                       : make_float2(ch_ok ? hsrc[s] : 0.f, ch_ok ? hsrc[s + 1] : 0.f);
                            const float2 lam = fma2(g2, Cp, make_float2(carry[s], carry[s + 1]));
                            dup = fma2(lam, make_float2(Bv[s], Bv[s + 1]), dup);
                            const float2 cn = mul2(make_float2(av[i][s], av[i][s + 1]), lam);
                            const float2 q = mul2(cn, hprev);
                            ddp = fma2(make_float2(A2[s], A2[s + 1]), q, ddp);
                            const float2 na = fma2(dl2, q, make_float2(dA[s], dA[s + 1]));
                            dA[s] = na.x; dA[s + 1] = na.y;
                            y0p = fma2(Cp, hcur, y0p);
                            const float2 cb = mul2(lam, dlu2), cc = mul2(g2, hcur);
                            cB[s] = cb.x; cB[s + 1] = cb.y;
                            cC[s] = cc.x; cC[s + 1] = cc.y;
                            carry[s] = cn.x; carry[s + 1] = cn.y;
                        }
                        du_p = dup.x + dup.y;
                        dd_p = ddp.x + ddp.y;
                        y0_p = y0p.x + y0p.y;
                    } else {
                        const float hprev = i > 0 ? hv[i - 1][0] : (ch_ok ? hsrc[0] : 0.f);
                        const float lam = fmaf(ss.z, Cv[0], carry[0]);
                        du_p = lam * Bv[0];
                        const float cn = av[i][0] * lam;
                        const float q = cn * hprev;
                        dd_p = A2[0] * q;
                        dA[0] = fmaf(ss.x, q, dA[0]);
                        y0_p = Cv[0] * hv[i][0];
                        cB[0] = lam * ss.y;
                        cC[0] = ss.z * hv[i][0];
                        carry[0] = cn;
                    }
                    // sums over the warp's states of the channel: lane g = 0 keeps
                    // (sum lam B, sum A q), lane g = 1 keeps y0
                    if constexpr (G == 2) {
                        const float x1 = __shfl_xor_sync(kFull, g == 0 ? y0_p : du_p, 1);
                        const float x2 = __shfl_xor_sync(kFull, dd_p, 1);
                        if (g == 0) sOa[w][r][ch] = make_float2(du_p + x1, dd_p + x2);
                        else sOb[w][r][ch] = x1 + y0_p;
                    } else {
                        sOa[w][r][ch] = make_float2(du_p, dd_p);
                        sOb[w][r][ch] = y0_p;
                    }
                    // stage dB / dC contributions (summed over the channels below)
                    stage_contrib<S, NPW, BLK>(sRw, i, cB, cC, ch, g * S);
                }
                __syncwarp();  // staged contributions visible to every lane of the warp
                reduce_staged<CH, NPW, N, BLK>(sRw, bc0, bc1, n_w, ts, t_end, lane);
                __syncwarp();  // the sums have read the staging before the next sub-chunk restages it
            }
            __syncthreads();  // every warp's per-step sums are in sOa / sOb
            // ---- epilogue: du, ddelta, dz of step t0 + pr for channels pc0 .. pc0 + CPL
            {
                // steps past t_end (last tile only) are not stored and add nothing; their
                // per-step sums may be unwritten (a sub-chunk wholly past the end is skipped)
                const int64_t t = t0 + pr;
                const bool tv = t < t_end;
                float vdu[CPL], vdx[CPL], vdz[CPL], eD[CPL], eb[CPL];
#pragma unroll
                for (int c = 0; c < CPL; c++) {
                    eD[c] = sAcc[0][c][tid];
                    eb[c] = sAcc[1][c][tid];
                }
#pragma unroll
                for (int c = 0; c < CPL; c++) {
                    const int cc = pc0 + c;
                    float2 so = sOa[0][pr][cc];
                    float y0 = sOb[0][pr][cc];
#pragma unroll
                    for (int q = 1; q < NW; q++) {
                        const float2 o = sOa[q][pr][cc];
                        so.x += o.x;
                        so.y += o.y;
                        y0 += sOb[q][pr][cc];
                    }
                    const float4 ss = sS[pr][cc];
                    const float2 se = sE[pr][cc];
                    vdu[c] = fmaf(ss.z, sDv[cc], ss.x * so.x);
                    vdx[c] = fmaf(se.x, so.x, so.y * kLn2) * ss.w;
                    vdz[c] = se.y * fmaf(sDv[cc], se.x, y0);
                    eD[c] = fmaf(ss.z, se.x, eD[c]);  // g = u = 0 on padded steps
                    eb[c] += tv ? vdx[c] : 0.f;
                }
#pragma unroll
                for (int c = 0; c < CPL; c++) {
                    sAcc[0][c][tid] = eD[c];
                    sAcc[1][c][tid] = eb[c];
                }
                if (tv) {
                    const int64_t off = (b * L + t) * Dch + d0 + pc0;
                    store_run<CPL>(a.du + off, vdu, d0 + pc0, Dch, ofast);
                    store_run<CPL>(a.ddelta + off, vdx, d0 + pc0, Dch, ofast);
                    if (z) store_run<CPL>(a.dz + off, vdz, d0 + pc0, Dch, ofast);
                }
            }
        }
        __syncthreads();  // the next prologue restages sS / sE / sB / sC
    }

    if constexpr (!MAIN) {
        if (ch_ok) {
            float2* out = reinterpret_cast<float2*>(a.ws_rsum) + (row * p.K + k) * N + n0;
#pragma unroll
            for (int s = 0; s < S; s++) out[s] = make_float2(Pr[s], carry[s]);
        }
    } else {
        if (ch_ok) {
            float* o = a.ws_dA + ((b * p.K + k) * Dch + d) * N + n0;
#pragma unroll
            for (int s = 0; s < S; s++) o[s] = dA[s];
        }
        // dD / ddelta_bias: the kTT threads sharing a channel set (consecutive
        // lanes of one warp) hold partials over their rows; combine them (xor
        // butterfly over the row bits, fixed order)
        float eD[CPL], eb[CPL];
#pragma unroll
        for (int c = 0; c < CPL; c++) {
            eD[c] = sAcc[0][c][tid];
            eb[c] = sAcc[1][c][tid];
        }
#pragma unroll
        for (int c = 0; c < CPL; c++) {
#pragma unroll
            for (int mk = 1; mk < kTT; mk <<= 1) {
                const float oD = __shfl_xor_sync(kFull, eD[c], mk), ob = __shfl_xor_sync(kFull, eb[c], mk);
                const bool low = (pr & mk) == 0;
                eD[c] = low ? eD[c] + oD : oD + eD[c];
                eb[c] = low ? eb[c] + ob : ob + eb[c];
            }
        }
        if (pr == 0) {
#pragma unroll
            for (int c = 0; c < CPL; c++) {
                if (d0 + pc0 + c < Dch) {
                    a.ws_dD[(b * p.K + k) * Dch + d0 + pc0 + c] = eD[c];
                    a.ws_db[(b * p.K + k) * Dch + d0 + pc0 + c] = eb[c];
                }
            }
        }
    }
}

// dB / dC: sum of the per-tile partials, tiles in ascending order.  A thread
// owns 4 consecutive outputs (16-byte streaming loads, 8 tiles in flight)
// when N is a multiple of 4, one output otherwise.
__global__ void k_bwd2_reduce_bc(BwdArgs a, FPlan p) {
    const int64_t bln = a.f.Bsz * a.f.L * a.f.N;
    const int64_t tiles = p.tiles_b;
    if (a.f.N % 4 == 0) {
        const int64_t q = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;  // float4 index over both tensors
        const int64_t nq = bln / 4;
        if (q >= 2 * nq) return;
        const int tensor = q >= nq ? 1 : 0;
        const int64_t r = q - tensor * nq;
        const float4* src = reinterpret_cast<const float4*>(a.ws_bc + (size_t)tensor * tiles * bln) + r;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        int64_t tl = 0;
        for (; tl + 8 <= tiles; tl += 8) {
            float4 v[8];
#pragma unroll
            for (int u = 0; u < 8; u++) v[u] = __ldcs(src + (tl + u) * nq);
#pragma unroll
            for (int u = 0; u < 8; u++) {
                acc.x += v[u].x; acc.y += v[u].y; acc.z += v[u].z; acc.w += v[u].w;
            }
        }
        for (; tl < tiles; tl++) {
            const float4 v = __ldcs(src + tl * nq);
            acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
        }
        reinterpret_cast<float4*>(tensor ? a.dC : a.dB)[r] = acc;
    } else {
        const int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
        if (e >= 2 * bln) return;
        const int tensor = e >= bln ? 1 : 0;
        const int64_t r = e - tensor * bln;
        const float* src = a.ws_bc + (size_t)tensor * tiles * bln + r;
        float acc = 0.f;
        for (int64_t tl = 0; tl < tiles; tl++) acc += src[tl * bln];
        (tensor ? a.dC : a.dB)[r] = acc;
    }
}

// dA / dD / ddelta_bias: sum over (batch, chunk) partials in ascending order.
__global__ void k_bwd2_reduce_params(BwdArgs a, FPlan p) {
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

template <typename T, int N>
cudaError_t launch_bwd2_t(const BwdArgs& a, const FPlan& p, cudaStream_t st, float* ckpt_out) {
    cudaError_t e = cudaSuccess;
    if (ckpt_out) {
        // checkpoint pass (with forward summaries first when the sequence is chunked)
        e = launch_fwd2(a.f, p, st, kModeCkpt, ckpt_out);
        if (e != cudaSuccess) return e;
    }
    constexpr int threads = BCfg<T, N>::THREADS;
    if (p.K > 1) {
        const int64_t blocks = p.tiles_b * a.f.Bsz * (p.K - 1);
        prof_mark(st);
        k_bwd2<T, N, kRevSummary><<<(unsigned)blocks, threads, 0, st>>>(a, p, 1, p.K);
    }
    const int64_t blocks = p.tiles_b * a.f.Bsz * p.K;
    // prefer the largest shared-memory carveout so that shared memory does not cap residency
    e = cudaFuncSetAttribute(k_bwd2<T, N, kRevMain>, cudaFuncAttributePreferredSharedMemoryCarveout,
                             (int)cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    prof_mark(st);
    k_bwd2<T, N, kRevMain><<<(unsigned)blocks, threads, 0, st>>>(a, p, 0, p.K);
    const int64_t n_bc = 2 * a.f.Bsz * a.f.L * a.f.N / (N % 4 == 0 ? 4 : 1);  // threads
    prof_mark(st);
    k_bwd2_reduce_bc<<<(unsigned)ceil_div(n_bc, 256), 256, 0, st>>>(a, p);
    const int64_t n_par = a.f.Dch * a.f.N;
    prof_mark(st);
    k_bwd2_reduce_params<<<(unsigned)ceil_div(n_par, 256), 256, 0, st>>>(a, p);
    return cudaGetLastError();
}

cudaError_t launch_bwd2(const BwdArgs& a, const FPlan& p, cudaStream_t st, float* ckpt_out) {
#define SS_BWD2_N(T)                                              \
    switch (a.f.N) {                                              \
        case 1: return launch_bwd2_t<T, 1>(a, p, st, ckpt_out);   \
        case 2: return launch_bwd2_t<T, 2>(a, p, st, ckpt_out);   \
        case 4: return launch_bwd2_t<T, 4>(a, p, st, ckpt_out);   \
        case 8: return launch_bwd2_t<T, 8>(a, p, st, ckpt_out);   \
        case 16: return launch_bwd2_t<T, 16>(a, p, st, ckpt_out); \
        case 32: return launch_bwd2_t<T, 32>(a, p, st, ckpt_out); \
        default: return cudaErrorInvalidValue;                    \
    }
    if (a.f.dtype == 0) { SS_BWD2_N(float) }
    SS_BWD2_N(__nv_bfloat16)
#undef SS_BWD2_N
}

}  // namespace ss
